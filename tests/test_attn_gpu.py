"""Attention + merge through the C ABI vs the fp64 oracle.

Small problems are compared element by element (bf16 output, log-sum-exp and
every segment partial); the five full-size workloads are compared on sampled
rows the oracle evaluates one by one, plus invariants that hold at any size.
Tolerances (max-abs): 1e-2 for bf16 KV, 2e-2 for fp8 KV, 8e-3 between the
planned and the fixed split on the same inputs."""
import math

import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
import sk_inputs as si
from gpu_helpers import (TOL_BF16, TOL_PLAN_VS_FIXED, oracle_all_rows, oracle_problem, oracle_sampled,
                         problem_tensors,
                         run_library, segments_of, tol_for, host_bits)
from helpers import KV_BF16, KV_FP8, build_problem, repermute
from oracle import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _small_problems():
    return [
        build_problem([0, 1, 5, 17, 700, 1333, 64, 257], [4, 4, 1, 2, 4, 3, 4, 1], 32, 2, seed=21),
        build_problem([5, 300], 1, 8, 1, seed=22),
        build_problem([2049, 611, 0, 1], 4, 16, 2, kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25, seed=23),
        build_problem([3, 40, 129, 1000, 2, 777, 64], [1, 3, 4, 2, 1, 4, 2], 16, 2, kv_dtype=KV_FP8,
                      k_scale=0.5, v_scale=0.25, seed=24),
        build_problem(list(range(1, 40)), 1, 32, 8, seed=25),
        build_problem([50, 901], 3, 16, 2, causal=0, seed=26),
        build_problem([4000], 4, 32, 2, seed=27),                # bs 1: long single sequence
        build_problem([130, 70], 8, 128, 8, seed=28),            # 128 rows per work item (G16 x q8)
        build_problem([300, 20], 2, 40, 4, seed=29),             # G = 10, rows not a power of two
        build_problem([700, 130, 2000, 9], [4, 4, 3, 4], 32, 2, kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25,
                      seed=30),                                  # fp8 with 64 rows per work item
        build_problem([900, 33, 2000], [12, 5, 10], 16, 2, kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25,
                      seed=33),                                  # fp8, up to 96 rows: two row blocks, the second partial
        build_problem([600, 1500, 7], [12, 12, 3], 64, 4, seed=34),   # G 16 x q 12 = 192 rows: three row blocks
        build_problem([300, 2000, 1], [1, 4, 2], 8, 8, seed=35),      # G 1 (plain multi-head attention)
        build_problem([500, 1500, 64], [3, 2, 1], 16, 4, kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25,
                      seed=36),                                  # fp8, 4 KV heads, 12 rows: the 16-row tile
        build_problem([400, 90, 1000], [10, 9, 1], 64, 4, causal=0, seed=37),   # not causal, 160 rows
        # fp8 P is split into two e4m3 terms: scores ~ N(0, 9) spread p over many orders of
        # magnitude (small terms near the e4m3 subnormals, early rescales)
        build_problem([3000, 517, 40], [4, 3, 1], 16, 2, kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25,
                      sm_scale=3.0 / math.sqrt(128), seed=38),
        # ... and scores near 0: every p near the top of the split's range
        build_problem([2500, 260], [4, 2], 16, 2, kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25,
                      sm_scale=0.01 / math.sqrt(128), seed=39),
        # ... and a late needle: one key far into the sequence beats the running max by ~2^16
        build_problem([3000, 700], [4, 4], 16, 2, kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25,
                      qfun=lambda t, hq, d: np.full(len(d), 0.5),
                      kfun=lambda s, p, h, d: np.where((p == (2890 if s == 0 else 590))[:, None], 2.0,
                                                       np.random.default_rng(100 + 7 * s + h).standard_normal(
                                                           (len(p), len(d)))) / 0.5,
                      seed=40),
    ]


@pytest.mark.parametrize("use_plan", [True, False])
@pytest.mark.parametrize("k", range(18))
def test_small_problem_elementwise(k, use_plan):
    pr = _small_problems()[k]
    q, kv = problem_tensors(pr, DEV)
    r = run_library(pr, q, kv, use_plan=use_plan)
    assert r.status == 0
    ref, ref_lse = oracle_problem(pr)
    got = r.out.float().cpu().numpy()
    tol = tol_for(pr.kv_dtype)
    assert np.isfinite(got).all()
    err = np.max(np.abs(got - ref))
    assert err <= tol, err
    lse = r.lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(lse), ~fin)
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0) <= 1e-3


@pytest.mark.parametrize("k", [0, 2, 3, 6, 9, 10, 11, 13, 14, 15, 16, 17])
def test_small_problem_partials(k):
    """Every segment partial: o / l and m + log l are the segment's unique output
    and log-sum-exp; a row that sees no key of the segment has (-inf, 0, 0)."""
    pr = _small_problems()[k]
    q, kv = problem_tensors(pr, DEV)
    for use_plan in (True, False):
        r = run_library(pr, q, kv, use_plan=use_plan)
        nseg, seg_tiles = segments_of(pr, use_plan)
        po, pm, pl, _, _ = oracle.attention_split(*pr.oracle_args(), nseg, seg_tiles, 64, r.seg_max)
        go, gm, gl = (x.cpu().numpy() for x in (r.part_o, r.part_m, r.part_l))
        cu = pr.cu_q
        tol = tol_for(pr.kv_dtype)
        for s in range(pr.bs):
            for t in range(cu[s], cu[s + 1]):
                for g in range(int(nseg[s])):
                    for h in range(pr.num_q_heads):
                        if pl[t, g, h] == 0:
                            assert gl[t, g, h] == 0 and np.isneginf(gm[t, g, h]) and not go[t, g, h].any()
                            continue
                        assert gl[t, g, h] > 0
                        assert abs((gm[t, g, h] + math.log(gl[t, g, h])) - (pm[t, g, h] + math.log(pl[t, g, h]))) < 1e-3
                        err = np.max(np.abs(go[t, g, h] / gl[t, g, h] - po[t, g, h] / pl[t, g, h]))
                        assert err <= tol, (s, t, g, h, err)


def _merged_partials(r, pr, use_plan, num_sms):
    """The library's fp32 segment partials of every row merged in fp64 on the host
    (M = max m_g, out = sum o_g e^(m_g - M) / sum l_g e^(m_g - M)): the attention result
    before the final rounding to bf16."""
    nseg, _ = segments_of(pr, use_plan, num_sms=num_sms)
    po, pm, pl = (x.cpu().numpy().astype(np.float64) for x in (r.part_o, r.part_m, r.part_l))
    out = np.zeros((pr.num_tokens, pr.num_q_heads, po.shape[-1]))
    for s in range(pr.bs):
        n = int(nseg[s])
        for t in range(pr.cu_q[s], pr.cu_q[s + 1]):
            m, l, o = pm[t, :n], pl[t, :n], po[t, :n]          # [n, H], [n, H], [n, H, D]
            live = l > 0
            M = np.where(live, m, -np.inf).max(axis=0, initial=-np.inf)
            wgt = np.where(live, np.exp(np.where(live, m, 0.0) - np.where(np.isfinite(M), M, 0.0)), 0.0)
            lam = (l * wgt).sum(axis=0)
            num = (o * wgt[:, :, None]).sum(axis=0)
            out[t] = np.where(lam[:, None] > 0, num / np.where(lam > 0, lam, 1.0)[:, None], 0.0)
    return out


def test_planned_vs_fixed_split_agree():
    """The planned and the fixed split of the same inputs agree within 8e-3, compared on
    the merged fp32 partials (the split's own effect); the bf16 outputs agree within 8e-3
    or one bf16 spacing of the larger value, since two results a hair apart can round to
    neighbouring bf16 values."""
    for pr in _small_problems():
        q, kv = problem_tensors(pr, DEV)
        a = run_library(pr, q, kv, use_plan=True, num_sms=24)
        b = run_library(pr, q, kv, use_plan=False, num_sms=24)
        ma, mb = _merged_partials(a, pr, True, 24), _merged_partials(b, pr, False, 24)
        err = float(np.max(np.abs(ma - mb)))
        assert err <= TOL_PLAN_VS_FIXED, err
        oa, ob = a.out.float().cpu().numpy(), b.out.float().cpu().numpy()
        big = np.maximum(np.abs(oa), np.abs(ob))
        spacing = np.exp2(np.floor(np.log2(np.maximum(big, 2.0 ** -126))) - 7)
        assert np.all(np.abs(oa - ob) <= np.maximum(TOL_PLAN_VS_FIXED, spacing))


def test_block_table_permutation_is_bit_identical():
    pr = _small_problems()[0]
    pr2 = repermute(pr, seed=5)
    q, kv = problem_tensors(pr, DEV)
    q2, kv2 = problem_tensors(pr2, DEV)
    a = run_library(pr, q, kv)
    b = run_library(pr2, q2, kv2)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_v_one_gives_one_and_needle():
    # V = 1: every row that sees a key returns exactly 1 (bf16)
    pr = build_problem([0, 1, 5, 17, 2500], 4, 32, 2, vfun=lambda s, p, h, d: np.ones((len(p), len(d))), seed=31)
    q, kv = problem_tensors(pr, DEV)
    r = run_library(pr, q, kv)
    got = r.out.float().cpu().numpy()
    ref, _ = oracle_problem(pr)
    seen = np.abs(ref).max(axis=-1) > 0
    assert np.all(np.abs(got[seen] - 1.0) <= 2 ** -8)
    assert np.all(got[~seen] == 0)

    def kf(s, p, h, d):
        k = np.zeros((len(p), len(d)))
        k[p == 1777, :] = 40.0 / np.sqrt(128)
        return k
    pr = build_problem([3000], 1, 2, 1, kfun=kf, qfun=lambda t, hq, d: np.ones(len(d)), seed=32)
    q, kv = problem_tensors(pr, DEV)
    r = run_library(pr, q, kv)
    want = pr.V[0][1777, 0]
    assert np.max(np.abs(r.out.float().cpu().numpy()[0, 0] - want)) <= 1e-2


def _run_workload(w, dev, use_plan=True):
    q = si.make_q(w, dev)
    kv = si.make_kv(w, dev)
    return q, kv, run_library(w, q, kv, use_plan=use_plan)


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5, 6, 7, 8])
def test_full_workload_sampled_rows(idx):
    w = si.config(idx)
    dev = torch.device(DEV)
    q, kv, r = _run_workload(w, dev)
    assert r.status == 0
    out = r.out.float()
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(1000 + idx)
    seqs = sorted(set([int(np.argmax(w.seq_lens))] + [int(x) for x in rng.integers(0, w.bs, size=6)]))
    samples = oracle_sampled(w, q, kv, seqs, 3, rng)
    tol = tol_for(w.kv_dtype)
    got = out.cpu().numpy()
    lse = r.lse.cpu().numpy()
    worst = 0.0
    for t, h, o, l in samples:
        worst = max(worst, float(np.max(np.abs(got[t, h] - o))))
        if np.isfinite(l):
            assert abs(lse[t, h] - l) <= 1e-3
        else:
            assert np.isneginf(lse[t, h])
    assert worst <= tol, worst
    # the planned and the fixed split agree on the same inputs
    r2 = run_library(w, q, kv, use_plan=False)
    diff = (r2.out.float() - out).abs().max().item()
    assert diff <= TOL_PLAN_VS_FIXED, diff


@pytest.mark.parametrize("use_plan", [True, False])
def test_page_accuracy_shapes_elementwise(use_plan):
    """The shapes of the page's accuracy tests, scaled down (GQA 16 and 8, agentic
    skew with 0/1/5/17-token sequences, bs 1/2/24/64, ragged q 1..4 on e4m3 pages,
    not causal): every output element and lse against the oracle, planned and
    fixed split."""
    dev = torch.device(DEV)
    for w in si.small_cases():
        q, kv, r = _run_workload(w, dev, use_plan=use_plan)
        assert r.status == 0, w.name
        ref, ref_lse = oracle_all_rows(w, q, kv)
        got = r.out.float().cpu().numpy()
        err = float(np.max(np.abs(got - ref), initial=0.0))
        assert err <= tol_for(w.kv_dtype), (w.name, err)
        lse = r.lse.cpu().numpy()
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isneginf(lse), ~fin), w.name
        assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) <= 1e-3, w.name


def test_uniform_16x70k_sampled_rows():
    """The page's uniform accuracy shape at full size: 16 sequences of 70000 keys,
    q 4, GQA 16 (32/2 heads): sampled rows against the oracle, planned vs fixed."""
    w = si.make_workload("uniform_16x70k", [70000] * 16, 4, 32, 2, seed=70)
    dev = torch.device(DEV)
    q, kv, r = _run_workload(w, dev)
    assert r.status == 0
    rng = np.random.default_rng(70)
    samples = oracle_sampled(w, q, kv, sorted(set(int(x) for x in rng.integers(0, 16, size=4))), 4, rng)
    got = r.out.float().cpu().numpy()
    worst = max(float(np.max(np.abs(got[t, h] - o))) for t, h, o, _ in samples)
    assert worst <= TOL_BF16, worst
    r2 = run_library(w, q, kv, use_plan=False)
    diff = (r2.out.float() - r.out.float()).abs().max().item()
    assert diff <= TOL_PLAN_VS_FIXED, diff


def test_maximum_batch_of_short_sequences():
    """The largest batch the calls accept (32767 sequences) of short requests: lengths
    0..40 with a fifth empty, q 1..2, 8/1 heads.  More non-empty sequences than the
    plan's budget, so every sequence is one segment (about 26000 CTAs); sampled rows
    against the oracle, every empty sequence's rows 0 with lse -inf, and the fixed
    split (one segment) equal to the plan."""
    rng = np.random.default_rng(32767)
    bs = 32767
    lens = rng.integers(0, 41, size=bs)
    lens[rng.random(bs) < 0.2] = 0
    w = si.make_workload("max_batch", lens, rng.integers(1, 3, size=bs), 8, 1, seed=97)
    dev = torch.device(DEV)
    q, kv, r = _run_workload(w, dev)
    assert r.status == 0
    out = r.out.float().cpu().numpy()
    lse = r.lse.cpu().numpy()
    assert np.isfinite(out).all()
    empty_tok = np.repeat(w.seq_lens == 0, w.q_lens)
    assert np.all(out[empty_tok] == 0.0) and np.all(np.isneginf(lse[empty_tok]))
    seqs = sorted(set(int(x) for x in rng.integers(0, bs, size=40)) | {0, bs - 1})
    worst = 0.0
    for t, h, o, l in oracle_sampled(w, q, kv, seqs, 2, rng):
        worst = max(worst, float(np.max(np.abs(out[t, h] - o))))
        if np.isfinite(l):
            assert abs(lse[t, h] - l) <= 1e-3
        else:
            assert np.isneginf(lse[t, h])
    assert worst <= TOL_BF16, worst
    r2 = run_library(w, q, kv, use_plan=False)
    assert r2.status == 0
    assert torch.equal(r2.out, r.out)


@pytest.mark.parametrize("seq_len,bs,q,hq,hkv,kv_dtype", [
    (8000, 16, 8, 32, 2, KV_BF16),      # 128 rows per work item: two row blocks
    (20000, 8, 20, 32, 2, KV_BF16),     # 320 rows: five row blocks
    (9000, 12, 12, 16, 2, KV_FP8),      # 96 rows, fp8
])
def test_many_rows_per_work_item_sampled(seq_len, bs, q, hq, hkv, kv_dtype):
    """Work items with more than 64 query rows (long drafts with wide GQA groups)
    run as row blocks of 64 on the tensor-core kernel: sampled rows vs the oracle,
    and the planned split vs the fixed one."""
    ks, vs = (0.5, 0.25) if kv_dtype == KV_FP8 else (1.0, 1.0)
    w = si.make_workload(f"rows_{hq // hkv * q}", [seq_len] * bs, q, hq, hkv, seed=40 + q,
                         kv_dtype=kv_dtype, k_scale=ks, v_scale=vs)
    q_t, kv, r = _run_workload(w, torch.device(DEV))
    assert r.status == 0
    rng = np.random.default_rng(7 + q)
    samples = oracle_sampled(w, q_t, kv, sorted(set(int(x) for x in rng.integers(0, bs, size=4))), 6, rng)
    got = r.out.float().cpu().numpy()
    worst = max(float(np.max(np.abs(got[t, h] - o))) for t, h, o, _ in samples)
    assert worst <= tol_for(kv_dtype), worst
    r2 = run_library(w, q_t, kv, use_plan=False)
    diff = (r2.out.float() - r.out.float()).abs().max().item()
    assert diff <= TOL_PLAN_VS_FIXED, diff


def test_long_sequences_with_v_one():
    """Agentic lengths (one 248k request, 0/1/5/17-token sequences) with V = 1:
    every row that sees a key must return exactly 1, at full length."""
    w = si.config(3)
    dev = torch.device(DEV)
    q = si.make_q(w, dev)
    kv = si.make_kv(w, dev, poison_tail=False)
    kv[..., w.head_dim:] = 1.0
    si.poison_unused_rows(w, kv)
    r = run_library(w, q, kv)
    assert r.status == 0
    out = r.out.float().cpu().numpy()
    for s in range(w.bs):
        for j in range(int(w.q_lens[s])):
            t = w.cu_q[s] + j
            n = max(0, min(int(w.seq_lens[s]), int(w.seq_lens[s]) - int(w.q_lens[s]) + j + 1))
            want = 1.0 if n > 0 else 0.0
            assert np.all(np.abs(out[t] - want) <= 2 ** -8), (s, j)


def test_repeated_calls_are_bit_identical_under_perturbed_timing():
    """Every kernel orders its work through barriers, so results may not depend on
    timing: the same call, repeated while unrelated GPU work shifts the schedule,
    returns bit-identical outputs (a missed wait shows up here as a flaky row)."""
    d = torch.device(DEV)
    noise = torch.randn((2048, 2048), device=d)
    for pr in (_small_problems()[0], _small_problems()[3], _small_problems()[6], _small_problems()[8], _small_problems()[9]):
        q, kv = problem_tensors(pr, DEV)
        ref, _ = oracle_problem(pr)
        first = None
        for i in range(12):
            if i % 3 == 1:
                noise = noise @ noise.T * 1e-3       # occupy the SMs right before the call
            r = run_library(pr, q, kv, use_plan=(i % 2 == 0), num_sms=24 if i % 4 < 2 else 148)
            got = r.out.view(torch.int16).clone()
            if i < 2:
                first = first if first is not None else {}
                first[i % 2, i % 4 < 2] = got
            key = (i % 2, i % 4 < 2)
            if key in (first or {}):
                assert torch.equal(got, first[key]), (i, key)
            else:
                first[key] = got
            assert np.max(np.abs(r.out.float().cpu().numpy() - ref)) <= tol_for(pr.kv_dtype)
