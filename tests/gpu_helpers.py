"""Shared pieces of the GPU parity tests: move a problem to the device, run
the library path through the C ABI, and evaluate the oracle on the same
inputs (whole problems for small cases, single sequences for full sizes)."""
from __future__ import annotations

import numpy as np
import torch

import paged_split_kv_gb300 as sk
import sk_inputs as si
from oracle import oracle

TOL_BF16 = 1e-2
TOL_FP8 = 2e-2
TOL_PLAN_VS_FIXED = 8e-3


def tol_for(kv_dtype):
    return TOL_FP8 if kv_dtype == si.KV_FP8 else TOL_BF16


def dev():
    return torch.device("cuda:0")


def problem_tensors(pr, device):
    """Device tensors for a tests.helpers.Problem (host bits)."""
    q = torch.from_numpy(pr.q_bits.view(np.int16).copy()).view(torch.bfloat16).to(device)
    if pr.kv_dtype == si.KV_FP8:
        kv = torch.from_numpy(pr.kv.copy()).to(device)
    else:
        kv = torch.from_numpy(pr.kv.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return q, kv


def host_bits(q, kv, kv_dtype):
    q_bits = q.view(torch.int16).cpu().numpy().view(np.uint16)
    if kv_dtype == si.KV_FP8:
        kv_h = kv.cpu().numpy()
    else:
        kv_h = kv.view(torch.int16).cpu().numpy().view(np.uint16)
    return q_bits, kv_h


class Run:
    """Output of one library call (plan or fixed split) plus the buffers it used."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def run_library(case, q, kv, use_plan=True, seg_max=None, num_sms=None, block_table=None):
    """case: anything with seq_lens, q_lens, num_q_heads, num_kv_heads, kv_dtype, k_scale,
    v_scale, sm_scale, causal, block_table (numpy)."""
    d = q.device
    seg_max = seg_max or getattr(case, "seg_max", 64)
    num_sms = num_sms or getattr(case, "num_sms", 148)
    bt = torch.as_tensor(case.block_table if block_table is None else block_table, device=d)
    lens = torch.as_tensor(np.asarray(case.seq_lens, dtype=np.int32), device=d)
    cu_np = np.concatenate([[0], np.cumsum(case.q_lens)]).astype(np.int32)
    cu = torch.as_tensor(cu_np, device=d)
    nt, hq, D = q.shape
    bs = len(case.seq_lens)
    hkv = case.num_kv_heads
    cap = sk.plan_capacity(bs, hkv, num_sms)
    plan = torch.full((cap,), -7, dtype=torch.int32, device=d) if use_plan else None
    tok = torch.full((max(nt, 1),), -7, dtype=torch.int32, device=d)[:nt] if use_plan else None
    part_o = torch.full((nt, seg_max, hq, D), float("nan"), dtype=torch.float32, device=d)
    part_m = torch.full((nt, seg_max, hq), float("nan"), dtype=torch.float32, device=d)
    part_l = torch.full((nt, seg_max, hq), float("nan"), dtype=torch.float32, device=d)
    out = torch.full((nt, hq, D), float("nan"), dtype=torch.bfloat16, device=d)
    lse = torch.full((nt, hq), float("nan"), dtype=torch.float32, device=d)
    max_q = int(np.max(case.q_lens)) if bs else 0
    sk.sk_plan_cache_reset()
    if use_plan:
        rc = sk.sk_build_plan(lens, cu, hkv, plan, tok, num_sms, seg_max)
        assert rc == sk.SK_OK
    sk.sk_paged_decode_attn(q, kv, bt, lens, cu, plan, part_o, part_m, part_l, max_q_len=max_q,
                            sm_scale=case.sm_scale, num_sms=num_sms, k_scale=case.k_scale,
                            v_scale=case.v_scale, causal=bool(case.causal))
    fixed = 0 if use_plan else sk.sk_fixed_nseg(bs, hkv, num_sms, seg_max)
    sk.sk_merge_segments(part_o, part_m, part_l, tok, out, lse, fixed_nseg=fixed)
    torch.cuda.synchronize()
    status = sk.sk_get_device_status(clear=True)
    return Run(out=out, lse=lse, plan=plan, tok_nseg=tok, part_o=part_o, part_m=part_m,
               part_l=part_l, status=status, fixed=fixed, cu=cu_np, seg_max=seg_max,
               num_sms=num_sms)


def oracle_problem(pr):
    out, lse = oracle.attention(*pr.oracle_args())
    return out.reshape(pr.num_tokens, pr.num_q_heads, pr.head_dim), lse.reshape(pr.num_tokens, pr.num_q_heads)


def oracle_rows(w, q, kv, s, picks):
    """Oracle output for the (query token j, query head hq) rows ``picks`` of
    sequence ``s`` of full-size workload ``w``: the sequence is copied out alone
    (its pages, a fresh block table) and the oracle evaluates only those rows.
    Returns [(t, hq, out[D], lse)] with t the global token index."""
    L = int(w.seq_lens[s])
    qs = int(w.q_lens[s])
    cu = w.cu_q
    npg = (L + w.page - 1) // w.page
    blocks = torch.as_tensor(w.block_table[s, :npg].astype(np.int64), device=kv.device)
    kv_sub = kv.index_select(0, blocks) if npg else kv[:0]
    q_sub = q[cu[s]:cu[s] + qs]
    q_bits, kv_bits = host_bits(q_sub, kv_sub, w.kv_dtype)
    if npg == 0:
        kv_bits = np.zeros((1,) + tuple(kv.shape[1:]), dtype=kv_bits.dtype)
    bt = np.arange(max(npg, 1), dtype=np.int32)[None, :]
    picks = sorted(set(picks))
    rows = np.array([j * w.num_q_heads + h for j, h in picks], dtype=np.int64)
    out, lse = oracle.attention(q_bits, kv_bits, w.kv_dtype, w.k_scale, w.v_scale, bt, w.page,
                                np.array([L], np.int32), np.array([0, qs], np.int32),
                                w.num_q_heads, w.num_kv_heads, w.head_dim, w.sm_scale, w.causal,
                                rows=rows)
    return [(int(cu[s]) + j, h, o, l) for (j, h), o, l in zip(picks, out, lse)]


def oracle_sampled(w, q, kv, seqs, rows_per_seq, rng):
    """Oracle output for a few random (token, head) rows of each sequence in
    ``seqs`` of full-size workload ``w``.  Returns [(t, hq, out[D], lse)]."""
    res = []
    for s in seqs:
        qs = int(w.q_lens[s])
        if qs == 0:
            continue
        picks = [(int(rng.integers(0, qs)), int(rng.integers(0, w.num_q_heads))) for _ in range(rows_per_seq)]
        res += oracle_rows(w, q, kv, s, picks)
    return res


def row_relative_error(got_row, ref_row):
    """max |got - ref| over a row divided by max |ref| of that row (0 for an all-zero
    reference that the kernel also returned as zeros)."""
    scale = float(np.max(np.abs(ref_row)))
    err = float(np.max(np.abs(np.asarray(got_row, np.float64) - ref_row)))
    if scale == 0.0:
        return 0.0 if err == 0.0 else float("inf")
    return err / scale


def oracle_all_rows(w, q, kv):
    """Oracle output and lse of every (token, query head) row of workload ``w``
    (small workloads: one oracle call per sequence).  Returns (out [NT, H_q, D],
    lse [NT, H_q])."""
    out = np.zeros((w.num_tokens, w.num_q_heads, w.head_dim))
    lse = np.full((w.num_tokens, w.num_q_heads), -np.inf)
    cu = w.cu_q
    for s in range(w.bs):
        L = int(w.seq_lens[s])
        qs = int(w.q_lens[s])
        if qs == 0:
            continue
        npg = (L + w.page - 1) // w.page
        blocks = torch.as_tensor(w.block_table[s, :npg].astype(np.int64), device=kv.device)
        kv_sub = kv.index_select(0, blocks) if npg else kv[:0]
        q_bits, kv_bits = host_bits(q[cu[s]:cu[s] + qs], kv_sub, w.kv_dtype)
        if npg == 0:
            kv_bits = np.zeros((1,) + tuple(kv.shape[1:]), dtype=kv_bits.dtype)
        bt = np.arange(max(npg, 1), dtype=np.int32)[None, :]
        o, l = oracle.attention(q_bits, kv_bits, w.kv_dtype, w.k_scale, w.v_scale, bt, w.page,
                                np.array([L], np.int32), np.array([0, qs], np.int32), w.num_q_heads,
                                w.num_kv_heads, w.head_dim, w.sm_scale, w.causal)
        out[cu[s]:cu[s] + qs] = o.reshape(qs, w.num_q_heads, w.head_dim)
        lse[cu[s]:cu[s] + qs] = l.reshape(qs, w.num_q_heads)
    return out, lse


def segments_of(case, use_plan, num_sms=148, seg_max=64, tile=64):
    """(nseg, seg_tiles) per sequence from the oracle's own plan or fixed split."""
    lens = np.asarray(case.seq_lens, np.int32)
    cu = np.concatenate([[0], np.cumsum(case.q_lens)]).astype(np.int32)
    if use_plan:
        cap = 1 + max(num_sms // case.num_kv_heads, len(lens))
        p, tok, nseg, n = oracle.plan(lens, cu, case.num_kv_heads, num_sms, seg_max, tile, cap)
        return oracle.planned_segments(p, nseg)
    nf = oracle.fixed_nseg(len(lens), case.num_kv_heads, num_sms, seg_max)
    return oracle.fixed_segments(lens, nf, tile)
