"""Python binding of libsk: length-aware split-KV paged decode/verify attention
on GB300 (sm_103a).

Argument marshalling only: every step of the path (plan, attention, merge)
and the KV write and page conversion around it run in the CUDA kernels of
``libsk.so``; torch supplies device memory and streams.  The functions carry
the C names (``sk_build_plan``, ``sk_paged_decode_attn``,
``sk_merge_segments``, ``sk_plan_cache_reset``, ``sk_reshape_and_cache``,
``sk_std_to_shuffled``) and take torch tensors; ``paged_decode_attention``
chains the three attention calls the way a serving step does.  If
``libsk.so`` has not been built, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

__all__ = [
    "SkError", "lib", "sk_tile_tokens", "sk_fixed_nseg", "sk_build_plan", "sk_plan_cache_reset",
    "sk_plan_launch_count", "sk_paged_decode_attn", "sk_merge_segments", "sk_get_device_status",
    "paged_decode_attention", "plan_capacity", "sk_plan_capacity", "sk_paged_decode_attention_static",
    "sk_static_scratch_bytes", "sk_reshape_and_cache", "sk_std_to_shuffled", "sk_set_wait_limit",
    "SK_OK", "SK_CACHED", "SK_ERR_TIMEOUT", "SK_KV_BF16", "SK_KV_FP8_E4M3", "SK_DEV_BAD_BLOCK",
    "SK_DEV_BAD_SEQ", "SK_DEV_TIMEOUT",
]

SK_OK = 0
SK_CACHED = 1
SK_ERR_TIMEOUT = -5
SK_KV_BF16 = 0
SK_KV_FP8_E4M3 = 1
SK_DEV_BAD_BLOCK = 0x1
SK_DEV_BAD_SEQ = 0x2
SK_DEV_TIMEOUT = 0x4

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsk.so")
_lock = threading.Lock()
_lib = None


class SkError(RuntimeError):
    pass


def lib():
    """Load libsk.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise SkError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
        L.sk_tile_tokens.restype = i32
        L.sk_tile_tokens.argtypes = []
        L.sk_fixed_nseg.restype = i32
        L.sk_fixed_nseg.argtypes = [i32, i32, i32, i32]
        L.sk_plan_capacity.restype = i32
        L.sk_plan_capacity.argtypes = [i32, i32, i32]
        L.sk_set_wait_limit.restype = ctypes.c_longlong
        L.sk_set_wait_limit.argtypes = [ctypes.c_longlong]
        L.sk_last_device_status.restype = i32
        L.sk_last_device_status.argtypes = []
        L.sk_build_plan.restype = i32
        L.sk_build_plan.argtypes = [P, u64, P, u64, i32, i32, i32, i32, i32, P, i32, P, P]
        L.sk_plan_cache_reset.restype = None
        L.sk_plan_cache_reset.argtypes = []
        L.sk_plan_launch_count.restype = ctypes.c_longlong
        L.sk_plan_launch_count.argtypes = []
        L.sk_paged_decode_attn.restype = i32
        L.sk_paged_decode_attn.argtypes = [P, P, i32, f32, f32, P, i32, i32, i32, P, P, P, i32,
                                           i32, i32, i32, i32, i32, i32, f32, i32, i32, i32,
                                           P, P, P, P]
        L.sk_merge_segments.restype = i32
        L.sk_merge_segments.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, P, P]
        L.sk_reshape_and_cache.restype = i32
        L.sk_reshape_and_cache.argtypes = [P, P, P, i32, i32, i32, P, i32, f32, f32, i32, i32, P]
        L.sk_std_to_shuffled.restype = i32
        L.sk_std_to_shuffled.argtypes = [P, i32, P, i32, i32, i32, i32, i32, P, P, P]
        L.sk_get_device_status.restype = i32
        L.sk_get_device_status.argtypes = [P, i32]
        L.sk_paged_decode_attention_static.restype = i32
        L.sk_paged_decode_attention_static.argtypes = [P, P, i32, f32, f32, P, i32, i32, i32, P, P,
                                                       i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                                       i32, i32, P, P, P]
        L.sk_static_scratch_bytes.restype = ctypes.c_size_t
        L.sk_static_scratch_bytes.argtypes = []
        L.sk_last_error.restype = ctypes.c_char_p
        L.sk_last_error.argtypes = []
        _lib = L
        return L


def _check(rc: int, name: str) -> int:
    if rc < 0:
        msg = lib().sk_last_error()
        raise SkError(f"{name} returned {rc}: {msg.decode() if msg else ''}")
    return rc


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t, dtype, name, dims=None):
    """Type, layout and rank of one argument (where it lives is checked by _on_cuda)."""
    if t is None:
        raise ValueError(f"{name} is required")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions, has {t.dim()}")


def _shape(t, shape, name):
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _on_cuda(**tensors):
    for name, t in tensors.items():
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _check_batch(q, kv_pages, block_table, seq_lens, cu_seqlens_q):
    """The shapes an attention call reads through raw pointers: q [NT, H_q, D], kv_pages
    [NB, H_kv, page, 2D] with H_kv dividing H_q, seq_lens [bs], cu_seqlens_q [bs + 1] and at
    least bs block-table rows.  Returns (nt, hq, d, nb, hkv, page, bs)."""
    nt, hq, d = q.shape
    nb, hkv, page, d2 = kv_pages.shape
    if d2 != 2 * d:
        raise ValueError(f"kv_pages last dimension is {d2}, expected 2 * head_dim = {2 * d}")
    if hkv < 1 or hq % hkv != 0:
        raise ValueError(f"{hq} query heads are not a multiple of {hkv} KV heads")
    bs = seq_lens.numel()
    if cu_seqlens_q.numel() != bs + 1:
        raise ValueError(f"cu_seqlens_q has {cu_seqlens_q.numel()} entries, expected bs + 1 = {bs + 1}")
    if block_table.shape[0] < bs:
        raise ValueError(f"block_table has {block_table.shape[0]} rows for {bs} sequences")
    return nt, hq, d, nb, hkv, page, bs


def sk_tile_tokens() -> int:
    return lib().sk_tile_tokens()


def sk_fixed_nseg(bs: int, num_kv_heads: int, num_sms: int, seg_max: int = 64) -> int:
    return lib().sk_fixed_nseg(bs, num_kv_heads, num_sms, seg_max)


def sk_plan_capacity(bs: int, num_kv_heads: int, num_sms: int) -> int:
    """Smallest valid plan buffer length for a batch (computed by the library)."""
    return _check(lib().sk_plan_capacity(int(bs), int(num_kv_heads), int(num_sms)), "sk_plan_capacity")


plan_capacity = sk_plan_capacity


def sk_set_wait_limit(cycles: int) -> int:
    """Sets the attention kernel's abortable-wait limit in SM cycles (negative:
    the default, about two seconds) for later launches; returns the previous one.
    A test hook for the timeout path."""
    return int(lib().sk_set_wait_limit(int(cycles)))


def sk_plan_cache_reset() -> None:
    lib().sk_plan_cache_reset()


def sk_plan_launch_count() -> int:
    return lib().sk_plan_launch_count()


def sk_build_plan(seq_lens, cu_seqlens_q, num_kv_heads: int, plan, tok_nseg, num_sms: int,
                  seg_max: int = 64, stream=None) -> int:
    """Returns SK_OK (plan kernel enqueued) or SK_CACHED (cache hit)."""
    import torch
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _need(plan, torch.int32, "plan", 1)
    _need(tok_nseg, torch.int32, "tok_nseg", 1)
    bs = seq_lens.numel()
    if cu_seqlens_q.numel() != bs + 1:
        raise ValueError(f"cu_seqlens_q has {cu_seqlens_q.numel()} entries, expected bs + 1 = {bs + 1}")
    _on_cuda(seq_lens=seq_lens, cu_seqlens_q=cu_seqlens_q, plan=plan, tok_nseg=tok_nseg)
    rc = lib().sk_build_plan(_ptr(seq_lens), seq_lens._version, _ptr(cu_seqlens_q),
                             cu_seqlens_q._version, bs, tok_nseg.numel(), num_kv_heads, num_sms,
                             seg_max, _ptr(plan), plan.numel(), _ptr(tok_nseg), _stream(stream))
    return _check(rc, "sk_build_plan")


def _kv_dtype(kv_pages) -> int:
    import torch
    if kv_pages.dtype == torch.bfloat16:
        return SK_KV_BF16
    if kv_pages.dtype in (torch.uint8, torch.float8_e4m3fn):
        return SK_KV_FP8_E4M3
    raise ValueError(f"kv_pages dtype {kv_pages.dtype}: expected bfloat16, uint8 or float8_e4m3fn")


def sk_paged_decode_attn(q, kv_pages, block_table, seq_lens, cu_seqlens_q, plan, part_o, part_m,
                         part_l, *, max_q_len: int, sm_scale: float, num_sms: int,
                         k_scale: float = 1.0, v_scale: float = 1.0, causal: bool = True,
                         stream=None) -> int:
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_pages, None, "kv_pages", 4)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _need(part_o, torch.float32, "part_o", 4)
    _need(part_m, torch.float32, "part_m", 3)
    _need(part_l, torch.float32, "part_l", 3)
    if plan is not None:
        _need(plan, torch.int32, "plan", 1)
    nt, hq, d, nb, hkv, page, bs = _check_batch(q, kv_pages, block_table, seq_lens, cu_seqlens_q)
    seg_max = part_o.shape[1]
    _shape(part_o, (nt, seg_max, hq, d), "part_o")
    _shape(part_m, (nt, seg_max, hq), "part_m")
    _shape(part_l, (nt, seg_max, hq), "part_l")
    _on_cuda(q=q, kv_pages=kv_pages, block_table=block_table, seq_lens=seq_lens, cu_seqlens_q=cu_seqlens_q,
             plan=plan, part_o=part_o, part_m=part_m, part_l=part_l)
    rc = lib().sk_paged_decode_attn(
        _ptr(q), _ptr(kv_pages), _kv_dtype(kv_pages), float(k_scale), float(v_scale),
        _ptr(block_table), block_table.shape[1], nb, page, _ptr(seq_lens), _ptr(cu_seqlens_q),
        _ptr(plan), plan.numel() if plan is not None else 0, seq_lens.numel(), nt, int(max_q_len),
        hq, hkv, d, float(sm_scale), 1 if causal else 0, int(num_sms), seg_max,
        _ptr(part_o), _ptr(part_m), _ptr(part_l), _stream(stream))
    return _check(rc, "sk_paged_decode_attn")


def sk_merge_segments(part_o, part_m, part_l, tok_nseg, out, lse=None, fixed_nseg: int = 0,
                      stream=None) -> int:
    import torch
    _need(part_o, torch.float32, "part_o", 4)
    _need(part_m, torch.float32, "part_m", 3)
    _need(part_l, torch.float32, "part_l", 3)
    _need(out, torch.bfloat16, "out", 3)
    if tok_nseg is not None:
        _need(tok_nseg, torch.int32, "tok_nseg", 1)
    if lse is not None:
        _need(lse, torch.float32, "lse", 2)
    nt, seg_max, hq, d = part_o.shape
    _shape(part_m, (nt, seg_max, hq), "part_m")
    _shape(part_l, (nt, seg_max, hq), "part_l")
    _shape(out, (nt, hq, d), "out")
    _shape(lse, (nt, hq), "lse")
    if tok_nseg is not None and tok_nseg.numel() != nt:
        raise ValueError(f"tok_nseg has {tok_nseg.numel()} entries for {nt} tokens")
    _on_cuda(part_o=part_o, part_m=part_m, part_l=part_l, tok_nseg=tok_nseg, out=out, lse=lse)
    rc = lib().sk_merge_segments(_ptr(part_o), _ptr(part_m), _ptr(part_l), _ptr(tok_nseg),
                                 int(fixed_nseg), nt, hq, d, seg_max, _ptr(out), _ptr(lse),
                                 _stream(stream))
    return _check(rc, "sk_merge_segments")


def sk_reshape_and_cache(key, value, slot_mapping, kv_pages, *, k_scale: float = 1.0,
                         v_scale: float = 1.0, stream=None) -> int:
    """Writes this step's K/V rows ([num_tokens, num_kv_heads, head_dim] bf16) into
    ``kv_pages`` ([num_blocks, num_kv_heads, page, 2*head_dim], bf16 or e4m3) at
    ``slot_mapping`` (int64 [num_tokens], negative = no slot), in place."""
    import torch
    _need(key, torch.bfloat16, "key", 3)
    _need(value, torch.bfloat16, "value", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(kv_pages, None, "kv_pages", 4)
    nt, hkv, d = key.shape
    if tuple(value.shape) != (nt, hkv, d) or slot_mapping.numel() != nt:
        raise ValueError("key, value and slot_mapping must agree on [num_tokens, num_kv_heads, head_dim]")
    nb, hkv2, page, d2 = kv_pages.shape
    if hkv2 != hkv or d2 != 2 * d:
        raise ValueError("kv_pages must be [num_blocks, num_kv_heads, page, 2 * head_dim]")
    _on_cuda(key=key, value=value, slot_mapping=slot_mapping, kv_pages=kv_pages)
    rc = lib().sk_reshape_and_cache(_ptr(key), _ptr(value), _ptr(slot_mapping), nt, hkv, d,
                                    _ptr(kv_pages), _kv_dtype(kv_pages), float(k_scale), float(v_scale),
                                    nb, page, _stream(stream))
    return _check(rc, "sk_reshape_and_cache")


def sk_std_to_shuffled(kv_pages, k_shuf, v_shuf, block_ids=None, stream=None) -> int:
    """Standard pages [NB, H, 16, 256] to shuffled K [NB, H, 128/x, 16, x] and
    V [NB, H, 16/x, 128, x] (x = 16 / element size), for ``block_ids`` (int32)
    or every block."""
    import torch
    _need(kv_pages, None, "kv_pages", 4)
    _need(k_shuf, kv_pages.dtype, "k_shuf", 5)
    _need(v_shuf, kv_pages.dtype, "v_shuf", 5)
    if block_ids is not None:
        _need(block_ids, torch.int32, "block_ids", 1)
    nb, hkv, page, d2 = kv_pages.shape
    d = d2 // 2
    x = 16 // kv_pages.element_size()
    if tuple(k_shuf.shape) != (nb, hkv, d // x, page, x) or tuple(v_shuf.shape) != (nb, hkv, page // x, d, x):
        raise ValueError("k_shuf must be [NB, H, D/x, page, x] and v_shuf [NB, H, page/x, D, x]")
    _on_cuda(kv_pages=kv_pages, k_shuf=k_shuf, v_shuf=v_shuf, block_ids=block_ids)
    rc = lib().sk_std_to_shuffled(_ptr(kv_pages), _kv_dtype(kv_pages), _ptr(block_ids),
                                  0 if block_ids is None else block_ids.numel(), nb, hkv, d, page,
                                  _ptr(k_shuf), _ptr(v_shuf), _stream(stream))
    return _check(rc, "sk_std_to_shuffled")


def sk_static_scratch_bytes() -> int:
    return lib().sk_static_scratch_bytes()


def sk_paged_decode_attention_static(q, kv_pages, block_table, seq_lens, cu_seqlens_q, out, lse=None,
                                     *, max_q_len: int, sm_scale: float, num_sms: int,
                                     k_scale: float = 1.0, v_scale: float = 1.0, causal: bool = True,
                                     seg_max: int = 64, use_plan: Optional[bool] = None,
                                     stream=None) -> int:
    """The whole call without device allocation: plan, per-token counts and
    partials live in the library's fixed 32 MiB device array.  For callers that
    cannot allocate; calls that overlap on the GPU race on that array.
    use_plan defaults to bs > 1, as in paged_decode_attention (bs == 1 takes the
    fixed split)."""
    import torch
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_pages, None, "kv_pages", 4)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _need(out, torch.bfloat16, "out", 3)
    if lse is not None:
        _need(lse, torch.float32, "lse", 2)
    nt, hq, d, nb, hkv, page, bs = _check_batch(q, kv_pages, block_table, seq_lens, cu_seqlens_q)
    _shape(out, (nt, hq, d), "out")
    _shape(lse, (nt, hq), "lse")
    if use_plan is None:
        use_plan = bs > 1
    _on_cuda(q=q, kv_pages=kv_pages, block_table=block_table, seq_lens=seq_lens, cu_seqlens_q=cu_seqlens_q,
             out=out, lse=lse)
    rc = lib().sk_paged_decode_attention_static(
        _ptr(q), _ptr(kv_pages), _kv_dtype(kv_pages), float(k_scale), float(v_scale),
        _ptr(block_table), block_table.shape[1], nb, page, _ptr(seq_lens), _ptr(cu_seqlens_q),
        1 if use_plan else 0, seq_lens.numel(), nt, int(max_q_len), hq, hkv, d, float(sm_scale),
        1 if causal else 0, int(num_sms), int(seg_max), _ptr(out), _ptr(lse), _stream(stream))
    return _check(rc, "sk_paged_decode_attention_static")


def sk_get_device_status(stream=None, clear: bool = True) -> int:
    """Synchronises and returns the mask of SK_DEV_* bits (0 when clean), the
    timeout bit included: the C call reports a timeout as SK_ERR_TIMEOUT and
    keeps the mask for sk_last_device_status()."""
    L = lib()
    rc = L.sk_get_device_status(_stream(stream), 1 if clear else 0)
    if rc == SK_ERR_TIMEOUT:
        return int(L.sk_last_device_status())
    return _check(rc, "sk_get_device_status")


def paged_decode_attention(q, kv_pages, block_table, seq_lens, cu_seqlens_q, *, max_q_len: int,
                           sm_scale: float, num_sms: int, k_scale: float = 1.0,
                           v_scale: float = 1.0, causal: bool = True, seg_max: int = 64,
                           use_plan: Optional[bool] = None, workspace=None, out=None, lse=None,
                           stream=None) -> Tuple[object, object]:
    """One attention call: plan (bs > 1, or when use_plan is True), split-KV
    attention, LSE merge.  ``workspace`` is an optional dict of preallocated
    buffers (plan, tok_nseg, part_o, part_m, part_l) reused across calls.
    Returns (out bf16 [NT, H_q, D], lse fp32 [NT, H_q])."""
    import torch
    nt, hq, d = q.shape
    hkv = kv_pages.shape[1]
    bs = seq_lens.numel()
    dev = q.device
    ws = workspace if workspace is not None else {}
    if use_plan is None:
        use_plan = bs > 1
    if "part_o" not in ws:
        ws["part_o"] = torch.empty((nt, seg_max, hq, d), dtype=torch.float32, device=dev)
        ws["part_m"] = torch.empty((nt, seg_max, hq), dtype=torch.float32, device=dev)
        ws["part_l"] = torch.empty((nt, seg_max, hq), dtype=torch.float32, device=dev)
    if use_plan and "plan" not in ws:
        ws["plan"] = torch.empty(plan_capacity(bs, hkv, num_sms), dtype=torch.int32, device=dev)
        ws["tok_nseg"] = torch.empty(nt, dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty((nt, hq, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((nt, hq), dtype=torch.float32, device=dev)
    plan = ws["plan"] if use_plan else None
    if use_plan:
        sk_build_plan(seq_lens, cu_seqlens_q, hkv, plan, ws["tok_nseg"], num_sms, seg_max, stream)
    sk_paged_decode_attn(q, kv_pages, block_table, seq_lens, cu_seqlens_q, plan, ws["part_o"],
                         ws["part_m"], ws["part_l"], max_q_len=max_q_len, sm_scale=sm_scale,
                         num_sms=num_sms, k_scale=k_scale, v_scale=v_scale, causal=causal,
                         stream=stream)
    fixed = 0 if use_plan else sk_fixed_nseg(bs, hkv, num_sms, seg_max)
    sk_merge_segments(ws["part_o"], ws["part_m"], ws["part_l"], ws["tok_nseg"] if use_plan else None,
                      out, lse, fixed_nseg=fixed, stream=stream)
    return out, lse
