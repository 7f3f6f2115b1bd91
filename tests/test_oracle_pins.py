"""Pins for the fp64 CPU oracle: values the pages print, closed forms,
invariants, library routines on tiny inputs and brute force.  Each test is
chosen so that a plausible slip in the oracle (a dropped scale, a wrong head
or page index, K and V swapped, an off-by-one in the causal limit, a wrong
segment boundary) fails at least one of them.  No GPU is needed."""
import json
import math
import os

import numpy as np
import pytest
import torch

from helpers import (KV_BF16, KV_FP8, build_problem, dense_reference, repermute, visible)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TILE = 64


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- number formats

def test_e4m3fn_spot_values_from_spec(oracle):
    for code_s, val in _golden("e4m3fn_spot_values.json")["values"]:
        got = oracle.e4m3fn_to_double(int(code_s, 16))
        if val == "nan":
            assert math.isnan(got), code_s
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code_s


def test_e4m3fn_all_codes_match_torch(oracle):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3fn_to_double(c)
        if math.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], hex(c)


def test_bf16_decode_matches_torch(oracle):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    ref = torch.as_tensor(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b, r in zip(bits, ref):
        got = oracle.bf16_to_double(int(b))
        assert (math.isnan(got) and math.isnan(r)) or got == r


# --------------------------------------------------------------------------- fixed split

def test_fixed_split_matches_page_statements(oracle):
    g = _golden("fixed_split_pr39172.json")
    for st in g["statements"]:
        lo, hi = st["bs"]
        for bs in range(lo, hi + 1):
            assert oracle.fixed_nseg(bs, st["kv_heads"], st["num_sms"], 64) == st["nseg"], (st, bs)
    seg = g["segment_length"]
    nseg_f, seg_tiles = oracle.fixed_segments([seg["seq_len"]], seg["nseg"], TILE)
    tokens = int(seg_tiles[0]) * TILE
    assert abs(tokens - seg["tokens_per_segment_approx"]) / seg["tokens_per_segment_approx"] < 0.01


def test_fixed_split_edges(oracle):
    # 148 SMs: bs 1 with 2 kv heads -> 74 -> pow2floor 64; more work items than SMs -> 1
    assert oracle.fixed_nseg(1, 2, 148, 64) == 64
    assert oracle.fixed_nseg(1, 1, 148, 16) == 16
    assert oracle.fixed_nseg(16, 2, 148, 64) == 4      # 148 // 32 = 4
    assert oracle.fixed_nseg(128, 8, 148, 64) == 1
    assert oracle.fixed_nseg(3, 1, 148, 64) == 32      # 49 -> 32


# --------------------------------------------------------------------------- plan

def _expand(v, n):
    if isinstance(v, str):
        cnt, val = v.split(" x ")
        return [int(val)] * int(cnt)
    return v


def test_plan_golden_cases(oracle):
    g = _golden("plan_cases.json")
    for case in g["cases"]:
        lens = np.array(_expand(case["seq_lens"], 0), dtype=np.int32)
        q = np.array(_expand(case["q_lens"], 0), dtype=np.int32)
        cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
        p, tok, nseg, n = oracle.plan(lens, cu, case["kv_heads"], g["num_sms"], g["seg_max"],
                                      g["tile_tokens"], case["plan_capacity"])
        assert p[0] == case["T"], case["name"]
        if "items" in case:
            assert list(p[1:1 + n]) == case["items"]
            assert n == len(case["items"])
            assert list(tok) == case["tok_nseg"]
        else:
            assert n == case["n_items"]
            assert set(nseg.tolist()) == {case["nseg_each"]}
            assert (tok == case["nseg_each"]).all()
        assert (p[1 + n:] == -1).all()


def _check_plan_invariants(lens, cu, kv_heads, num_sms, seg_max, p, tok, nseg, n):
    tiles = (lens.astype(np.int64) + TILE - 1) // TILE
    T = int(p[0])
    budget = num_sms // kv_heads
    segs = (tiles + T - 1) // T
    assert (segs == nseg).all()
    nonempty = int((tiles > 0).sum())
    fallback = nonempty > budget
    if not fallback:
        # the rule holds at T, and T is the smallest such
        assert segs.sum() <= budget and (segs.max() if len(segs) else 0) <= seg_max
        if T > 1:
            s2 = (tiles + T - 2) // (T - 1)
            assert s2.sum() > budget or s2.max() > seg_max
    else:
        assert T == max(1, int(tiles.max()))
        assert (segs == (tiles > 0)).all()
    # work list: every segment once, sequence-major, covering [0, L) with no empty segment
    items = p[1:1 + n]
    seq = items >> 16
    seg = items & 0xFFFF
    expect = [(s, g) for s in range(len(lens)) for g in range(int(segs[s]))]
    assert list(zip(seq.tolist(), seg.tolist())) == expect
    for s, g in expect:
        a, b = g * T * TILE, min((g + 1) * T * TILE, int(lens[s]))
        assert a < b
    assert (p[1 + n:] == -1).all()
    for s in range(len(lens)):
        assert (tok[cu[s]:cu[s + 1]] == segs[s]).all()


def test_plan_invariants_random(oracle):
    rng = np.random.default_rng(1234)
    for trial in range(300):
        bs = int(rng.integers(1, 300))
        kind = trial % 3
        if kind == 0:
            lens = rng.integers(0, 300_000, size=bs)
        elif kind == 1:
            lens = np.exp(rng.uniform(0, np.log(300_000), size=bs)).astype(np.int64)
            lens[rng.random(bs) < 0.1] = 0
        else:
            lens = rng.integers(0, 2_000, size=bs)
        lens = lens.astype(np.int32)
        q = rng.integers(1, 5, size=bs).astype(np.int32)
        cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
        kv = int(rng.choice([1, 2, 4, 8]))
        num_sms = int(rng.choice([148, 152, 256, 40]))
        seg_max = int(rng.choice([64, 16, 1]))
        cap = 1 + max(num_sms // kv, bs)
        p, tok, nseg, n = oracle.plan(lens, cu, kv, num_sms, seg_max, TILE, cap)
        _check_plan_invariants(lens, cu, kv, num_sms, seg_max, p, tok, nseg, n)


def test_plan_brute_force_tiny(oracle):
    """Exhaustive small batches: T equals the smallest t found by trying them all."""
    rng = np.random.default_rng(5)
    for _ in range(400):
        bs = int(rng.integers(1, 6))
        lens = rng.integers(0, 700, size=bs).astype(np.int32)
        cu = np.arange(bs + 1, dtype=np.int32)
        num_sms, kv, seg_max = int(rng.integers(1, 12)), 1, int(rng.integers(1, 5))
        p, tok, nseg, n = oracle.plan(lens, cu, kv, num_sms, seg_max, TILE, 1 + max(num_sms, bs))
        tiles = [(int(L) + TILE - 1) // TILE for L in lens]
        feasible = [t for t in range(1, max(tiles + [1]) + 1)
                    if sum(-(-x // t) for x in tiles) <= num_sms and max(-(-x // t) for x in tiles) <= seg_max]
        assert p[0] == (feasible[0] if feasible else max(tiles + [1]))


def test_plan_capacity_error(oracle):
    with pytest.raises(ValueError):
        oracle.plan(np.array([5000, 5000], np.int32), np.array([0, 1, 2], np.int32), 1, 148, 64, TILE, 3)


# --------------------------------------------------------------------------- attention

def _run(oracle, pr):
    out, lse = oracle.attention(*pr.oracle_args())
    return out.reshape(pr.num_tokens, pr.num_q_heads, pr.head_dim), lse.reshape(pr.num_tokens, pr.num_q_heads)


@pytest.mark.parametrize("kv_dtype", [KV_BF16, KV_FP8])
@pytest.mark.parametrize("causal", [1, 0])
def test_attention_matches_scipy_softmax(oracle, kv_dtype, causal):
    pr = build_problem([0, 1, 5, 17, 40], [1, 2, 4, 3, 4], 8, 2, head_dim=32, page=16,
                       kv_dtype=kv_dtype, k_scale=0.5, v_scale=0.25, causal=causal, seed=3)
    out, lse = _run(oracle, pr)
    ref, ref_lse = dense_reference(pr)
    assert np.max(np.abs(out - ref)) < 1e-12
    fin = np.isfinite(ref_lse)
    assert (np.isfinite(lse) == fin).all()
    assert np.max(np.abs(lse[fin] - ref_lse[fin])) < 1e-12


def test_v_one_gives_one(oracle):
    """Softmax rows sum to 1: with V = 1 every row that sees a key returns 1."""
    pr = build_problem([0, 1, 5, 17, 100], 4, 16, 2, vfun=lambda s, p, h, d: np.ones((len(p), len(d))), seed=4)
    out, lse = _run(oracle, pr)
    for s in range(pr.bs):
        for j in range(4):
            t = pr.cu_q[s] + j
            want = 1.0 if visible(pr, s, j) > 0 else 0.0
            assert np.all(out[t] == want) if want == 0 else np.max(np.abs(out[t] - 1)) < 1e-12


def test_k_zero_gives_mean_of_visible_v_causal(oracle):
    """K = 0 makes all scores equal; with V_p = p the output is the mean position
    (n-1)/2 over the visible keys, so an off-by-one in the causal limit shows."""
    pr = build_problem([10, 37, 3], 4, 4, 1, kfun=lambda s, p, h, d: np.zeros((len(p), len(d))),
                       vfun=lambda s, p, h, d: np.repeat(p[:, None].astype(float), len(d), 1), seed=5)
    out, _ = _run(oracle, pr)
    for s, L in enumerate(pr.seq_lens):
        for j in range(4):
            n = int(L) - 4 + j + 1
            t = pr.cu_q[s] + j
            want = (n - 1) / 2.0 if n > 0 else 0.0
            assert np.max(np.abs(out[t] - want)) < 1e-12, (s, j)


def test_single_key_returns_its_value(oracle):
    pr = build_problem([1, 4], [1, 4], 8, 2, seed=6)
    out, _ = _run(oracle, pr)
    for hq in range(8):
        assert np.array_equal(out[0, hq], pr.V[0][0, hq // 4])
        # sequence 1, token 0 sees only key 0 (L=4, q=4)
        assert np.array_equal(out[1, hq], pr.V[1][0, hq // 4])


def test_kv_head_mapping_is_contiguous_groups(oracle):
    """Query head hq reads KV head hq // G: give KV head h the constant V = h + 1."""
    pr = build_problem([50], 2, 12, 3, vfun=lambda s, p, h, d: np.full((len(p), len(d)), h + 1.0), seed=7)
    out, _ = _run(oracle, pr)
    for hq in range(12):
        assert np.max(np.abs(out[:, hq] - (hq // 4 + 1))) < 1e-12


def test_k_and_v_halves_are_not_swapped(oracle):
    """K = 0 and V = 3: the output is 3; reading V as K and K as V would give 0."""
    pr = build_problem([33], 1, 2, 1, kfun=lambda s, p, h, d: np.zeros((len(p), len(d))),
                       vfun=lambda s, p, h, d: np.full((len(p), len(d)), 3.0), seed=8)
    out, _ = _run(oracle, pr)
    assert np.max(np.abs(out - 3.0)) < 1e-12


def test_two_key_closed_form_with_fp8_scales(oracle):
    """Key 0 = 0, key 1 = 2 e_0 (fp8 code), q = a e_0: s_1 = sm_scale * k_scale * 2a, s_0 = 0.
    V_0 = 1, V_1 = 0 (codes): out = v_scale * 1 / (1 + exp(s_1))."""
    a, ks, vs = 3.0, 0.5, 0.25

    def kf(s, p, h, d):
        k = np.zeros((len(p), len(d)))
        k[p == 1, 0] = 2.0
        return k

    def vf(s, p, h, d):
        return np.where((p == 0)[:, None], 1.0, 0.0) * np.ones((len(p), len(d)))

    qf = lambda t, hq, d: np.where(d == 0, a, 0.0)
    pr = build_problem([2], 1, 1, 1, kv_dtype=KV_FP8, k_scale=ks, v_scale=vs, kfun=kf, vfun=vf, qfun=qf, seed=9)
    out, lse = _run(oracle, pr)
    s1 = pr.sm_scale * ks * 2 * a
    assert abs(out[0, 0, 0] - vs / (1 + math.exp(s1))) < 1e-14
    assert abs(lse[0, 0] - math.log(1 + math.exp(s1))) < 1e-14


def test_needle_dominates(oracle):
    """One key aligned with q and 40 scaled: softmax puts ~all weight on it."""
    def kf(s, p, h, d):
        k = np.zeros((len(p), len(d)))
        k[p == 123, :] = 40.0 / np.sqrt(128)
        return k
    qf = lambda t, hq, d: np.ones(len(d))
    pr = build_problem([300], 1, 2, 1, kfun=kf, qfun=qf, seed=10)
    out, _ = _run(oracle, pr)
    # score 40 for the needle, 0 elsewhere: the other 299 keys carry weight < 299 e^-40
    assert np.max(np.abs(out[0, 0] - pr.V[0][123, 0])) < 1e-12


def test_block_table_permutation_invariance(oracle):
    a = build_problem([70, 200, 3], 4, 16, 2, seed=11)
    b = repermute(a, seed=99)
    assert not np.array_equal(a.block_table, b.block_table)
    oa, _ = _run(oracle, a)
    ob, _ = _run(oracle, b)
    assert np.array_equal(oa, ob)


def test_zero_one_five_seventeen_token_sequences(oracle):
    """Verify q = 4 over L in {0, 1, 5, 17}: token j sees L - 4 + j + 1 keys, none when that is <= 0."""
    pr = build_problem([0, 1, 5, 17], 4, 8, 1, vfun=lambda s, p, h, d: np.repeat((p + 1.0)[:, None], len(d), 1),
                       kfun=lambda s, p, h, d: np.zeros((len(p), len(d))), seed=12)
    out, lse = _run(oracle, pr)
    for s, L in enumerate([0, 1, 5, 17]):
        for j in range(4):
            n = max(0, L - 3 + j)
            t = pr.cu_q[s] + j
            if n == 0:
                assert np.all(out[t] == 0) and np.all(np.isneginf(lse[t]))
            else:
                assert np.max(np.abs(out[t] - (n + 1) / 2.0)) < 1e-12


# --------------------------------------------------------------------------- split + merge identity

@pytest.mark.parametrize("kv_dtype", [KV_BF16, KV_FP8])
def test_split_equals_unsplit_for_plan_and_fixed(oracle, kv_dtype):
    pr = build_problem([0, 1, 5, 17, 700, 1333, 64, 257], [4, 4, 1, 2, 4, 3, 4, 1], 16, 2,
                       kv_dtype=kv_dtype, k_scale=0.5, v_scale=0.25, seed=13)
    ref, ref_lse = oracle.attention(*pr.oracle_args())
    # planned segments with a tight budget so long sequences split several ways
    p, tok, nseg, n = oracle.plan(pr.seq_lens, pr.cu_q, 2, 24, 64, TILE, 1 + 24)
    assert nseg.max() > 1
    for segs in (oracle.planned_segments(p, nseg), oracle.fixed_segments(pr.seq_lens, 4, TILE)):
        po, pm, pl, out, lse = oracle.attention_split(*pr.oracle_args(), segs[0], segs[1], TILE, 64)
        assert np.max(np.abs(out - ref)) < 1e-12
        fin = np.isfinite(ref_lse)
        assert np.max(np.abs(lse[fin] - ref_lse[fin])) < 1e-12
    # merging the float32-rounded partials with per-token counts from the plan
    po, pm, pl, out, lse = oracle.attention_split(*pr.oracle_args(), *oracle.planned_segments(p, nseg), TILE, 64)
    mo, ml = oracle.merge(po, pm, pl, tok, 0, pr.num_tokens, pr.num_q_heads, pr.head_dim, 64)
    assert np.max(np.abs(mo - ref)) < 1e-5
    fin = np.isfinite(ref_lse)
    assert np.max(np.abs(ml[fin] - ref_lse[fin])) < 1e-5


def test_merge_closed_forms(oracle):
    D, H, S = 4, 1, 8
    po = np.zeros((1, S, H, D), np.float32)
    pm = np.full((1, S, H), -np.inf, np.float32)
    pl = np.zeros((1, S, H), np.float32)
    # no segments -> 0, -inf
    out, lse = oracle.merge(po, pm, pl, np.array([0], np.int32), 0, 1, H, D, S)
    assert np.all(out == 0) and np.isneginf(lse[0])
    # one segment: out = o / l, lse = m + log l
    po[0, 0, 0] = [2, 4, 6, 8]
    pm[0, 0, 0] = 1.5
    pl[0, 0, 0] = 2.0
    out, lse = oracle.merge(po, pm, pl, np.array([1], np.int32), 0, 1, H, D, S)
    assert np.allclose(out[0], [1, 2, 3, 4], atol=0) and abs(lse[0] - (1.5 + math.log(2))) < 1e-12
    # two segments with equal mass e^{m} l: out is the average of o/l
    po[0, 1, 0] = [0, 0, 0, 0]
    pm[0, 1, 0] = 1.5 + math.log(2.0)
    pl[0, 1, 0] = 1.0
    out, lse = oracle.merge(po, pm, pl, np.array([2], np.int32), 0, 1, H, D, S)
    assert np.max(np.abs(out[0] - [0.5, 1, 1.5, 2])) < 1e-6
    # an empty segment (l = 0, m = -inf) next to a real one changes nothing
    out2, _ = oracle.merge(po, pm, pl, None, 3, 1, H, D, S)
    assert np.array_equal(out, out2)


def test_nan_in_unused_rows_never_reaches_results(oracle):
    pr = build_problem([17, 31, 1], [4, 1, 1], 8, 2, seed=14, garbage=np.nan)
    out, lse = oracle.attention(*pr.oracle_args())
    assert np.isfinite(out).all()


# --------------------------------------------------------------------------- workload recipe

def test_seeded_workloads_match_committed_configs():
    """The seeded generator still produces the committed lengths and shapes."""
    import sk_inputs as si
    with open(os.path.join(os.path.dirname(__file__), "..", "sk_inputs", "configs.json")) as f:
        committed = json.load(f)["workloads"]
    for c in committed:
        w = si.config(c["index"])
        assert w.name == c["name"] and w.bs == c["bs"]
        assert [int(x) for x in w.seq_lens] == c["seq_lens"]
        assert [int(x) for x in w.q_lens] == c["q_lens"]
        assert (w.num_q_heads, w.num_kv_heads, int(w.kv_bytes)) == (c["num_q_heads"], c["num_kv_heads"], c["kv_bytes"])
