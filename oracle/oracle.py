"""Python access to the fp64 CPU oracle (``sk_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the CPU
baseline leg of ``bench.py`` use this module; the product library never
imports it.  It shares no code with the CUDA path.

``build()`` compiles ``sk_oracle.c`` with the system C compiler into
``oracle/_build/libsk_oracle.so`` (IEEE double arithmetic, no fast-math,
OpenMP over independent output rows).  Every other function is argument
marshalling around the C functions, whose comments cite the page sections
they follow.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(values the pages print, closed forms, invariants, a library softmax on tiny
inputs, brute force); for the KV write step and the e4m3fn encoder by
``tests/test_kv_write_pins.py`` (round trips through the pinned decoder, IEEE
midpoints, PyTorch's float8 cast, a hand-written page image, attention on
directly built pages); and for the shuffled-page conversion by
``tests/test_shuffle_pins.py`` (NumPy's reshape and transpose of the printed
formula, a bijection on unique values, untouched blocks); none is marked
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sk_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsk_oracle.so")
_lock = threading.Lock()
_lib = None

KV_BF16 = 0
KV_FP8 = 1


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [os.environ.get("CC", "gcc"), "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.sko_e4m3fn_encode.restype = ctypes.c_uint8
        lib.sko_e4m3fn_encode.argtypes = [ctypes.c_float]
        lib.sko_reshape_and_cache.restype = None
        lib.sko_reshape_and_cache.argtypes = [P, P, P, i32, i32, i32, P, i32, ctypes.c_float, ctypes.c_float,
                                              i64, i32]
        lib.sko_std_to_shuffled.restype = None
        lib.sko_std_to_shuffled.argtypes = [P, i32, P, i32, i64, i32, i32, i32, P, P]
        lib.sko_bf16_to_double.restype = f64
        lib.sko_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.sko_e4m3fn_to_double.restype = f64
        lib.sko_e4m3fn_to_double.argtypes = [ctypes.c_uint8]
        lib.sko_fixed_nseg.restype = i32
        lib.sko_fixed_nseg.argtypes = [i32, i32, i32, i32]
        lib.sko_plan.restype = i32
        lib.sko_plan.argtypes = [P, P, i32, i32, i32, i32, i32, P, i32, P, P]
        common = [P, P, i32, f64, f64, P, i32, i32, P, P, i32, i32, i32, i32, f64, i32]
        lib.sko_attention.restype = None
        lib.sko_attention.argtypes = common + [P, i64, P, P]
        lib.sko_attention_split.restype = None
        lib.sko_attention_split.argtypes = common + [P, P, i32, i32, P, P, P, P, P]
        lib.sko_merge.restype = None
        lib.sko_merge.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P]
        lib.sko_num_threads.restype = i32
        lib.sko_num_threads.argtypes = []
        lib.sko_set_num_threads.restype = None
        lib.sko_set_num_threads.argtypes = [i32]
        _lib = lib
        return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def num_threads() -> int:
    """Threads the oracle's parallel loops use."""
    return int(_load().sko_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the oracle's parallel loops (n <= 0: every processor).  For
    timing only: every result is the same at any thread count."""
    _load().sko_set_num_threads(int(n))


def bf16_to_double(bits: int) -> float:
    return _load().sko_bf16_to_double(int(bits) & 0xFFFF)


def e4m3fn_to_double(code: int) -> float:
    return _load().sko_e4m3fn_to_double(int(code) & 0xFF)


def e4m3fn_encode(x) -> np.ndarray:
    """e4m3fn codes of binary32 values (nearest, ties to even, saturating)."""
    x = np.asarray(x, dtype=np.float32)
    f = _load().sko_e4m3fn_encode
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def reshape_and_cache(key_bits, value_bits, slot_mapping, kv_pages: np.ndarray, kv_dtype: int,
                      k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Writes the tokens' K/V rows into ``kv_pages`` ([NB, H_kv, page, 2D]; uint16
    bf16 bits or uint8 e4m3 codes) in place and returns it."""
    key_bits = _c(key_bits, np.uint16)
    value_bits = _c(value_bits, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    nt, hkv, d = key_bits.shape
    assert value_bits.shape == key_bits.shape and slot_mapping.shape == (nt,)
    nb, hkv2, page, d2 = kv_pages.shape
    assert hkv2 == hkv and d2 == 2 * d and kv_pages.flags.c_contiguous
    assert kv_pages.dtype == (np.uint16 if kv_dtype == KV_BF16 else np.uint8)
    _load().sko_reshape_and_cache(_ptr(key_bits), _ptr(value_bits), _ptr(slot_mapping), nt, hkv, d,
                                  _ptr(kv_pages), int(kv_dtype), float(k_scale), float(v_scale), nb, page)
    return kv_pages


def std_to_shuffled(kv_pages: np.ndarray, block_ids=None, k_shuf=None, v_shuf=None):
    """Standard pages [NB, H, N, 2D] (uint16 bf16 bits or uint8 e4m3 codes) to
    shuffled K [NB, H, D/x, N, x] and V [NB, H, N/x, D, x], x = 16 / element size.
    Outputs are created zeroed unless given (then written in place)."""
    kv_pages = np.ascontiguousarray(kv_pages)
    nb, h, n, d2 = kv_pages.shape
    d = d2 // 2
    es = kv_pages.dtype.itemsize
    x = 16 // es
    if k_shuf is None:
        k_shuf = np.zeros((nb, h, d // x, n, x), kv_pages.dtype)
    if v_shuf is None:
        v_shuf = np.zeros((nb, h, n // x, d, x), kv_pages.dtype)
    assert k_shuf.flags.c_contiguous and v_shuf.flags.c_contiguous
    ids = None if block_ids is None else _c(block_ids, np.int32)
    _load().sko_std_to_shuffled(_ptr(kv_pages), es, _ptr(ids), 0 if ids is None else ids.shape[0], nb, h, d, n,
                                _ptr(k_shuf), _ptr(v_shuf))
    return k_shuf, v_shuf


def fixed_nseg(bs: int, num_kv_heads: int, num_sms: int, seg_max: int = 64) -> int:
    return int(_load().sko_fixed_nseg(bs, num_kv_heads, num_sms, seg_max))


def plan(seq_lens, cu_q, num_kv_heads: int, num_sms: int, seg_max: int, tile: int,
         plan_capacity: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray, int]:
    """Returns (plan int32[plan_capacity], tok_nseg int32[NT], nseg int32[bs], n_items)."""
    seq_lens = _c(seq_lens, np.int32)
    cu_q = _c(cu_q, np.int32)
    bs = seq_lens.shape[0]
    p = np.zeros(plan_capacity, dtype=np.int32)
    tok = np.zeros(int(cu_q[-1]) if bs else 0, dtype=np.int32)
    nseg = np.zeros(bs, dtype=np.int32)
    n = _load().sko_plan(_ptr(seq_lens), _ptr(cu_q), bs, num_kv_heads, num_sms, seg_max, tile,
                         _ptr(p), plan_capacity, _ptr(tok), _ptr(nseg))
    if n < 0:
        raise ValueError("plan capacity too small")
    return p, tok, nseg, int(n)


def _problem_args(q_bits, kv, kv_dtype, k_scale, v_scale, block_table, page, seq_lens, cu_q,
                  num_q_heads, num_kv_heads, head_dim, sm_scale, causal):
    q_bits = _c(q_bits, np.uint16)
    kv = np.ascontiguousarray(kv)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    cu_q = _c(cu_q, np.int32)
    keep = (q_bits, kv, block_table, seq_lens, cu_q)
    args = [_ptr(q_bits), _ptr(kv), int(kv_dtype), float(k_scale), float(v_scale),
            _ptr(block_table), int(block_table.shape[1]), int(page), _ptr(seq_lens), _ptr(cu_q),
            int(seq_lens.shape[0]), int(num_q_heads), int(num_kv_heads), int(head_dim),
            float(sm_scale), int(causal)]
    return args, keep


def attention(q_bits, kv, kv_dtype, k_scale, v_scale, block_table, page, seq_lens, cu_q,
              num_q_heads, num_kv_heads, head_dim, sm_scale, causal=1, rows=None):
    """Unsplit fp64 attention.  q_bits: uint16 bf16 bits [NT, H_q, D]; kv: uint16 bf16 bits or
    uint8 e4m3 codes [NB, H_kv, page, 2D].  Returns (out [n_rows, D], lse [n_rows]); rows are
    flat t * H_q + hq indices (default: all, in order)."""
    args, keep = _problem_args(q_bits, kv, kv_dtype, k_scale, v_scale, block_table, page, seq_lens,
                               cu_q, num_q_heads, num_kv_heads, head_dim, sm_scale, causal)
    nt = int(np.asarray(cu_q)[-1])
    rows_a = None if rows is None else _c(rows, np.int64)
    n = nt * num_q_heads if rows is None else rows_a.shape[0]
    out = np.zeros((n, head_dim), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    _load().sko_attention(*args, _ptr(rows_a), int(n), _ptr(out), _ptr(lse))
    return out, lse


def attention_split(q_bits, kv, kv_dtype, k_scale, v_scale, block_table, page, seq_lens, cu_q,
                    num_q_heads, num_kv_heads, head_dim, sm_scale, causal, nseg, seg_tiles, tile,
                    seg_max):
    """Segment-by-segment fp64 evaluation merged by log-sum-exp.  Returns
    (part_o, part_m, part_l, out [NT*H_q, D], lse)."""
    args, keep = _problem_args(q_bits, kv, kv_dtype, k_scale, v_scale, block_table, page, seq_lens,
                               cu_q, num_q_heads, num_kv_heads, head_dim, sm_scale, causal)
    nt = int(np.asarray(cu_q)[-1])
    nseg = _c(nseg, np.int32)
    seg_tiles = _c(seg_tiles, np.int32)
    part_o = np.zeros((nt, seg_max, num_q_heads, head_dim), dtype=np.float64)
    part_m = np.full((nt, seg_max, num_q_heads), -np.inf, dtype=np.float64)
    part_l = np.zeros((nt, seg_max, num_q_heads), dtype=np.float64)
    out = np.zeros((nt * num_q_heads, head_dim), dtype=np.float64)
    lse = np.zeros(nt * num_q_heads, dtype=np.float64)
    _load().sko_attention_split(*args, _ptr(nseg), _ptr(seg_tiles), int(tile), int(seg_max),
                                _ptr(part_o), _ptr(part_m), _ptr(part_l), _ptr(out), _ptr(lse))
    return part_o, part_m, part_l, out, lse


def merge(part_o, part_m, part_l, tok_nseg, fixed_nseg_count, num_tokens, num_q_heads, head_dim,
          seg_max):
    """LSE merge of float32 partials; returns (out [NT*H_q, D], lse)."""
    part_o = _c(part_o, np.float32)
    part_m = _c(part_m, np.float32)
    part_l = _c(part_l, np.float32)
    tok = None if tok_nseg is None else _c(tok_nseg, np.int32)
    out = np.zeros((num_tokens * num_q_heads, head_dim), dtype=np.float64)
    lse = np.zeros(num_tokens * num_q_heads, dtype=np.float64)
    _load().sko_merge(_ptr(part_o), _ptr(part_m), _ptr(part_l), _ptr(tok), int(fixed_nseg_count),
                      int(num_tokens), int(num_q_heads), int(head_dim), int(seg_max), _ptr(out),
                      _ptr(lse))
    return out, lse


def fixed_segments(seq_lens, nseg_f: int, tile: int):
    """Per-sequence (nseg, seg_tiles) of the fixed split: nseg_f segments of
    ceil(tiles_s / nseg_f) tiles each (trailing segments may be empty)."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    tiles = (seq_lens + tile - 1) // tile
    seg_tiles = np.maximum(1, (tiles + nseg_f - 1) // nseg_f)
    return np.full(seq_lens.shape, nseg_f, dtype=np.int32), seg_tiles.astype(np.int32)


def planned_segments(plan_arr: np.ndarray, nseg: np.ndarray):
    """Per-sequence (nseg, seg_tiles) of a plan: every segment is plan[0] tiles."""
    return np.asarray(nseg, dtype=np.int32), np.full(nseg.shape, int(plan_arr[0]), dtype=np.int32)
