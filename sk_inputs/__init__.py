"""Seeded synthetic inputs for split-KV paged decode/verify attention.

This module only *generates* inputs: batch lengths, query lengths, block
tables, query tensors and KV pages.  It holds none of the attention method's
arithmetic (no planning, no softmax, no merge), so both the CPU oracle and the
CUDA path can take their inputs from it without sharing any method code.

Page layout ("standard pages", vLLM RFC 59111 "NixlConnector: convert standard
KV pages to ROCm AITER shuffled pages", Background): every block holds, per KV
head, ``page`` token rows of ``2*D`` elements with K in ``[0, D)`` and V in
``[D, 2D)``.  The global cache is ``[num_blocks, H_kv, page, 2*D]``.

Workloads follow the shapes of SGLang PR 39172 ("gfx950 assembly attention:
length-aware split-KV for dynamic workload", Benchmarking and Profiling): a
uniform 16 x 119k verify batch, an agentic length mix with one 248k request
and 0/1/5/17-token sequences, a ragged draft-extend batch with fp8 KV, plus a
tiny decode case and a high-batch decode case.  The agentic trace of the page
is not available, so seeded log-uniform lengths rescaled to the page's token
totals stand in for it.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

HEAD_DIM = 128
PAGE = 16
NUM_SMS_PLAN = 148      # SM count the plan budget is quoted on
SEG_MAX = 64

KV_BF16 = 0
KV_FP8 = 1

BF16_NAN_BITS = 0x7FC0
FP8_NAN_CODE = 0x7F


@dataclasses.dataclass
class Workload:
    """One batch of the split-KV path: lengths, layout sizes and seeds."""
    name: str
    seq_lens: np.ndarray          # int32 [bs], KV length including this step's query tokens
    q_lens: np.ndarray            # int32 [bs]
    num_q_heads: int
    num_kv_heads: int
    kv_dtype: int = KV_BF16
    k_scale: float = 1.0
    v_scale: float = 1.0
    head_dim: int = HEAD_DIM
    page: int = PAGE
    causal: int = 1
    num_sms: int = NUM_SMS_PLAN
    seg_max: int = SEG_MAX
    seed: int = 0
    spare_blocks: int = 64
    block_table: Optional[np.ndarray] = None   # int32 [bs, stride]; -1 = unused
    num_blocks: int = 0

    @property
    def bs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def cu_q(self) -> np.ndarray:
        cu = np.zeros(self.bs + 1, dtype=np.int32)
        cu[1:] = np.cumsum(self.q_lens, dtype=np.int64).astype(np.int32)
        return cu

    @property
    def num_tokens(self) -> int:
        return int(self.q_lens.sum())

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.bs else 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def elem_bytes(self) -> int:
        return 1 if self.kv_dtype == KV_FP8 else 2

    @property
    def kv_bytes(self) -> int:
        """Bytes of K and V that one call has to read: sum_s L_s * H_kv * 2 * D * elem."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * 2 * self.head_dim * self.elem_bytes

    @property
    def bt_stride(self) -> int:
        return int(self.block_table.shape[1])


def _pages_for(length: int, page: int) -> int:
    return (int(length) + page - 1) // page


def assign_block_table(w: Workload, rng: np.random.Generator) -> None:
    """Fill ``w.block_table`` from a seeded permutation of every physical block id.

    ``num_blocks`` = pages the batch needs + ``spare_blocks``; sequence s takes
    the next ceil(L_s/page) ids of the permutation; unused slots hold -1.
    """
    pages = [_pages_for(L, w.page) for L in w.seq_lens]
    stride = max(1, max(pages) if pages else 1)
    w.num_blocks = int(sum(pages)) + w.spare_blocks
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    bt = np.full((w.bs, stride), -1, dtype=np.int32)
    k = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[k:k + n]
        k += n
    w.block_table = bt


def rescale_to_total(extras: np.ndarray, target: int) -> np.ndarray:
    """Scale positive reals to integers summing exactly to ``target``.

    floor(e_k * target / sum(e)), then +1 to the largest fractional parts
    (ties to the lower index) until the total is met.
    """
    e = np.asarray(extras, dtype=np.float64)
    exact = e * (float(target) / e.sum())
    base = np.floor(exact).astype(np.int64)
    rem = int(target - base.sum())
    frac = exact - base
    order = sorted(range(len(e)), key=lambda i: (-frac[i], i))
    for i in order[:rem]:
        base[i] += 1
    return base


def _log_uniform(rng: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))


AGENTIC_FIXED = [248000, 0, 1, 5, 17]


def agentic_lengths(rng: np.random.Generator, bs: int, total: int) -> np.ndarray:
    """{248000, 0, 1, 5, 17} + (bs-5) log-uniform lengths in [512, 200000] rescaled to ``total``."""
    n_extra = bs - len(AGENTIC_FIXED)
    extras = _log_uniform(rng, n_extra, 512.0, 200000.0)
    scaled = rescale_to_total(extras, total - sum(AGENTIC_FIXED))
    return np.array(AGENTIC_FIXED + [int(x) for x in scaled], dtype=np.int32)


def make_workload(name: str, seq_lens, q_lens, num_q_heads: int, num_kv_heads: int, seed: int,
                  kv_dtype: int = KV_BF16, k_scale: float = 1.0, v_scale: float = 1.0,
                  causal: int = 1, num_sms: int = NUM_SMS_PLAN, seg_max: int = SEG_MAX,
                  spare_blocks: int = 64, rng: Optional[np.random.Generator] = None) -> Workload:
    rng = rng if rng is not None else np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.broadcast_to(np.asarray(q_lens, dtype=np.int32), seq_lens.shape).copy()
    w = Workload(name=name, seq_lens=seq_lens, q_lens=q_lens, num_q_heads=num_q_heads,
                 num_kv_heads=num_kv_heads, kv_dtype=kv_dtype, k_scale=k_scale, v_scale=v_scale,
                 causal=causal, num_sms=num_sms, seg_max=seg_max, seed=seed,
                 spare_blocks=spare_blocks)
    assign_block_table(w, rng)
    return w


def config(index: int) -> Workload:
    """The benchmark workloads, numbered 1..8 (seed = 1000 + index).

    1 tiny decode      bs 2, L {5, 300}, q 1, 8/1 heads, bf16
    2 uniform verify   bs 16 x 119000, q 4, 32/2 heads, bf16
    3 agentic verify   bs 16, {248000,0,1,5,17} + 11 log-uniform, total 1,850,000, q 4, 32/2, bf16
    4 draft-extend     bs 20, same fixed five + 15 log-uniform, total 2,320,000, q ~ U{1..4},
                       16/2 heads, fp8 e4m3 KV (k_scale 0.5, v_scale 0.25)
    5 high-batch       bs 128 x 8192, q 1, 32/8 heads, bf16
    6 bs1 long         bs 1 x 110000, q 4, 32/2 heads, bf16 (the fixed-split bypass)
    7 bs1 longest      bs 1 x 248000, q 4, 32/2 heads, bf16 (the fixed-split bypass)
    8 uniform fp8      bs 16 x 119000, q 4, 32/2 heads, fp8 e4m3 KV (k_scale 0.5, v_scale 0.25):
                       workload 2 on e4m3 pages, 64 query rows per work item (about 512 KV
                       bytes per token, as in the page's benchmark rows)
    """
    seed = 1000 + index
    rng = np.random.default_rng(seed)
    if index == 1:
        return make_workload("tiny_decode_bs2", [5, 300], 1, 8, 1, seed, rng=rng)
    if index == 2:
        return make_workload("uniform_verify_16x119k_q4", [119000] * 16, 4, 32, 2, seed, rng=rng)
    if index == 3:
        lens = agentic_lengths(rng, 16, 1_850_000)
        return make_workload("agentic_verify_bs16_1.85M_q4", lens, 4, 32, 2, seed, rng=rng)
    if index == 4:
        lens = agentic_lengths(rng, 20, 2_320_000)
        q = rng.integers(1, 5, size=20).astype(np.int32)
        return make_workload("ragged_draft_extend_bs20_2.32M_fp8", lens, q, 16, 2, seed,
                             kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25, rng=rng)
    if index == 5:
        return make_workload("high_batch_decode_128x8192", [8192] * 128, 1, 32, 8, seed, rng=rng)
    if index == 6:
        return make_workload("bs1_long_110k_q4", [110000], 4, 32, 2, seed, rng=rng)
    if index == 7:
        return make_workload("bs1_long_248k_q4", [248000], 4, 32, 2, seed, rng=rng)
    if index == 8:
        return make_workload("uniform_verify_16x119k_q4_fp8", [119000] * 16, 4, 32, 2, seed,
                             kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25, rng=rng)
    raise ValueError(f"no workload {index}")


# ---------------------------------------------------------------------------
# tensors (torch is imported lazily so the length/table logic stays numpy-only)
# ---------------------------------------------------------------------------

def _randn_bf16(shape, seed: int, device, chunk: int = 1 << 26):
    import torch
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    n = flat.numel()
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        flat[i:i + m] = torch.randn(m, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_q(w: Workload, device="cpu"):
    """bf16 [num_tokens, H_q, D] ~ N(0, 1), seed 10*seed + 1."""
    return _randn_bf16((w.num_tokens, w.num_q_heads, w.head_dim), 10 * w.seed + 1, device)


def make_kv(w: Workload, device="cpu", poison_tail: bool = True, chunk_blocks: int = 4096):
    """KV pages [num_blocks, H_kv, page, 2*D].

    bf16: K and V ~ N(0, 1).  fp8: real K, V ~ N(0, 1) stored as OCP e4m3fn codes of
    K / k_scale and V / v_scale (clamped to +-448, rounded by torch's float8 cast),
    returned as uint8.  With ``poison_tail`` every token row past L_s in a
    sequence's last page is overwritten with NaN bits: the method must never
    read those rows into a result.
    """
    import torch
    shape = (w.num_blocks, w.num_kv_heads, w.page, 2 * w.head_dim)
    seed = 10 * w.seed + 2
    if w.kv_dtype == KV_BF16:
        kv = _randn_bf16(shape, seed, device)
    else:
        kv = torch.empty(shape, dtype=torch.uint8, device=device)
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        D = w.head_dim
        inv = torch.empty(2 * D, dtype=torch.float32, device=device)
        inv[:D] = 1.0 / w.k_scale
        inv[D:] = 1.0 / w.v_scale
        for b0 in range(0, w.num_blocks, chunk_blocks):
            b1 = min(w.num_blocks, b0 + chunk_blocks)
            x = torch.randn((b1 - b0,) + shape[1:], generator=g, device=device, dtype=torch.float32)
            x = (x * inv).clamp_(-448.0, 448.0)
            kv[b0:b1] = x.to(torch.float8_e4m3fn).view(torch.uint8)
    if poison_tail:
        poison_unused_rows(w, kv)
    return kv


def poison_unused_rows(w: Workload, kv) -> None:
    """Write NaN bits into the token rows past L_s of every sequence's last page."""
    import torch
    nan_bits = BF16_NAN_BITS if w.kv_dtype == KV_BF16 else FP8_NAN_CODE
    view = kv.view(torch.int16) if w.kv_dtype == KV_BF16 else kv
    val = nan_bits  # 0x7FC0 and 0x7F both fit the signed view
    for s, L in enumerate(w.seq_lens):
        L = int(L)
        if L == 0 or L % w.page == 0:
            continue
        blk = int(w.block_table[s, (L - 1) // w.page])
        view[blk, :, L % w.page:, :] = val


def fill_unused_blocks(w: Workload, kv) -> None:
    """Write NaN bits into every block that no sequence references."""
    import torch
    used = np.zeros(w.num_blocks, dtype=bool)
    used[w.block_table[w.block_table >= 0]] = True
    free = np.nonzero(~used)[0]
    if free.size == 0:
        return
    idx = torch.as_tensor(free, device=kv.device, dtype=torch.long)
    if w.kv_dtype == KV_BF16:
        kv.view(torch.int16)[idx] = BF16_NAN_BITS
    else:
        kv[idx] = FP8_NAN_CODE


def small_cases() -> List[Workload]:
    """Shapes of the page's accuracy tests (GQA 16 and 8, agentic skew with
    0/1/5/17-token sequences, bs 1/2/24/64, ragged q 1..4), scaled down so the
    oracle finishes every element in seconds; lengths still span several
    64-token tiles and end in ragged pages."""
    cases = []
    rng = np.random.default_rng(7)
    cases.append(make_workload("g16_q4_bs3", [700, 1333, 64], 4, 32, 2, 11, rng=rng))
    cases.append(make_workload("g8_q1_bs2_tiny", [5, 300], 1, 8, 1, 12, rng=rng))
    cases.append(make_workload("skew_0_1_5_17", [0, 1, 5, 17, 2049, 611], 4, 32, 2, 13, rng=rng))
    cases.append(make_workload("bs1_long", [4000], 4, 32, 2, 14, rng=rng))
    cases.append(make_workload("bs24_mixed", list(rng.integers(0, 900, size=24)), 1, 16, 2, 15, rng=rng))
    qr = rng.integers(1, 5, size=7).astype(np.int32)
    cases.append(make_workload("ragged_q_fp8", [3, 40, 129, 1000, 2, 777, 64], qr, 16, 2, 16,
                               kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25, rng=rng))
    cases.append(make_workload("bs64_decode_g4", list(rng.integers(1, 400, size=64)), 1, 32, 8, 17, rng=rng))
    cases.append(make_workload("g8_noncausal_q3", [50, 901], 3, 16, 2, 18, causal=0, rng=rng))
    return cases
