"""Small hand-built problems for the oracle pins and the GPU parity tests.

A problem is described by its logical K, V (per sequence, position, KV head,
dimension) and Q; ``build_problem`` writes the logical K/V into standard pages
[num_blocks, H_kv, page, 2*D] through a seeded random block table.  Values are
stored as bf16 bits or OCP e4m3fn codes, and the *decoded* stored values are
kept as the logical arrays, so a check compares against exactly what a kernel
can read.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional

import numpy as np
import torch

KV_BF16 = 0
KV_FP8 = 1


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    t = torch.as_tensor(np.clip(np.asarray(x, dtype=np.float32), -448, 448)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def e4m3_codes_to_f64(c: np.ndarray) -> np.ndarray:
    t = torch.as_tensor(np.asarray(c, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)
    return t.numpy()


@dataclasses.dataclass
class Problem:
    seq_lens: np.ndarray
    q_lens: np.ndarray
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page: int
    kv_dtype: int
    k_scale: float
    v_scale: float
    sm_scale: float
    causal: int
    block_table: np.ndarray
    q_bits: np.ndarray            # uint16 [NT, H_q, D]
    kv: np.ndarray                # uint16 or uint8 [NB, H_kv, page, 2D]
    K: List[np.ndarray]           # decoded stored codes, [L_s, H_kv, D] per sequence (before k_scale)
    V: List[np.ndarray]
    Q: np.ndarray                 # decoded [NT, H_q, D]

    @property
    def bs(self):
        return len(self.seq_lens)

    @property
    def cu_q(self):
        cu = np.zeros(self.bs + 1, dtype=np.int32)
        cu[1:] = np.cumsum(self.q_lens)
        return cu

    @property
    def num_tokens(self):
        return int(np.sum(self.q_lens))

    def oracle_args(self):
        return (self.q_bits, self.kv, self.kv_dtype, self.k_scale, self.v_scale, self.block_table,
                self.page, self.seq_lens, self.cu_q, self.num_q_heads, self.num_kv_heads,
                self.head_dim, self.sm_scale, self.causal)


def build_problem(seq_lens, q_lens, num_q_heads, num_kv_heads, head_dim=128, page=16,
                  kv_dtype=KV_BF16, k_scale=1.0, v_scale=1.0, causal=1, seed=0, spare=3,
                  kfun: Optional[Callable] = None, vfun: Optional[Callable] = None,
                  qfun: Optional[Callable] = None, sm_scale=None, garbage=np.nan) -> Problem:
    """kfun/vfun(s, p_array, h, d_array) -> values [len(p), D]; qfun(t, hq, d) -> [D].
    Defaults draw N(0,1).  Rows past L_s in last pages and spare blocks hold ``garbage``."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.broadcast_to(np.asarray(q_lens, dtype=np.int32), seq_lens.shape).copy()
    bs = len(seq_lens)
    D = head_dim
    npages = [(int(L) + page - 1) // page for L in seq_lens]
    stride = max(1, max(npages) if npages else 1)
    nb = sum(npages) + spare
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((bs, stride), -1, dtype=np.int32)
    k = 0
    for s, n in enumerate(npages):
        bt[s, :n] = perm[k:k + n]
        k += n
    raw = np.full((nb, num_kv_heads, page, 2 * D), garbage, dtype=np.float64)
    dims = np.arange(D)
    for s in range(bs):
        L = int(seq_lens[s])
        if L == 0:
            continue
        pos = np.arange(L)
        for h in range(num_kv_heads):
            kv_k = kfun(s, pos, h, dims) if kfun else rng.standard_normal((L, D)) / (k_scale if kv_dtype else 1.0)
            kv_v = vfun(s, pos, h, dims) if vfun else rng.standard_normal((L, D)) / (v_scale if kv_dtype else 1.0)
            blk = bt[s, pos // page]
            raw[blk, h, pos % page, :D] = kv_k
            raw[blk, h, pos % page, D:] = kv_v
    if kv_dtype == KV_BF16:
        kv = to_bf16_bits(raw)
        dec = bf16_bits_to_f64(kv)
    else:
        kv = to_e4m3_codes(raw)
        dec = e4m3_codes_to_f64(kv)
    Ks, Vs = [], []
    for s in range(bs):
        L = int(seq_lens[s])
        pos = np.arange(L)
        blk = bt[s, pos // page] if L else np.zeros(0, dtype=np.int32)
        Ks.append(dec[blk, :, pos % page, :D] if L else np.zeros((0, num_kv_heads, D)))
        Vs.append(dec[blk, :, pos % page, D:] if L else np.zeros((0, num_kv_heads, D)))
    nt = int(q_lens.sum())
    if qfun is not None:
        qv = np.zeros((nt, num_q_heads, D))
        for t in range(nt):
            for hq in range(num_q_heads):
                qv[t, hq] = qfun(t, hq, dims)
    else:
        qv = rng.standard_normal((nt, num_q_heads, D))
    q_bits = to_bf16_bits(qv)
    return Problem(seq_lens, q_lens, num_q_heads, num_kv_heads, D, page, kv_dtype, k_scale, v_scale,
                   (1.0 / np.sqrt(D)) if sm_scale is None else sm_scale, causal, bt, q_bits, kv,
                   Ks, Vs, bf16_bits_to_f64(q_bits))


def visible(problem: Problem, s: int, j: int) -> int:
    """Keys [0, n) visible to query token j of sequence s."""
    L = int(problem.seq_lens[s])
    q = int(problem.q_lens[s])
    if not problem.causal:
        return L
    return max(0, min(L, L - q + j + 1))


def dense_reference(problem: Problem):
    """Per-row attention written with scipy's softmax over densely gathered K/V."""
    from scipy.special import softmax, logsumexp
    G = problem.num_q_heads // problem.num_kv_heads
    cu = problem.cu_q
    out = np.zeros((problem.num_tokens, problem.num_q_heads, problem.head_dim))
    lse = np.full((problem.num_tokens, problem.num_q_heads), -np.inf)
    ks = problem.k_scale if problem.kv_dtype == KV_FP8 else 1.0
    vs = problem.v_scale if problem.kv_dtype == KV_FP8 else 1.0
    for s in range(problem.bs):
        for j in range(int(problem.q_lens[s])):
            t = cu[s] + j
            n = visible(problem, s, j)
            if n == 0:
                continue
            for hq in range(problem.num_q_heads):
                h = hq // G
                sc = problem.sm_scale * ks * (problem.K[s][:n, h, :] @ problem.Q[t, hq])
                out[t, hq] = vs * (softmax(sc) @ problem.V[s][:n, h, :])
                lse[t, hq] = logsumexp(sc)
    return out, lse


def repermute(problem: Problem, seed: int, extra_spare: int = 5) -> Problem:
    """Same logical K/V, moved to other physical blocks by a new seeded permutation."""
    rng = np.random.default_rng(seed)
    nb_old = problem.kv.shape[0]
    nb = nb_old + extra_spare
    perm = rng.permutation(nb).astype(np.int32)
    fill = problem.kv.reshape(-1)[0] * 0 + (0x7FC0 if problem.kv.dtype == np.uint16 else 0x7F)
    kv = np.full((nb,) + problem.kv.shape[1:], fill, dtype=problem.kv.dtype)
    bt = np.full_like(problem.block_table, -1)
    k = 0
    for s in range(problem.bs):
        for i in range(problem.block_table.shape[1]):
            old = problem.block_table[s, i]
            if old < 0:
                continue
            bt[s, i] = perm[k]
            kv[perm[k]] = problem.kv[old]
            k += 1
    return dataclasses.replace(problem, block_table=bt, kv=kv)
