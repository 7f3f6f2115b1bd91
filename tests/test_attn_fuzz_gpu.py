"""Seeded fuzz of attention + merge through the C ABI against the fp64 oracle.

Each case draws a small batch at random: 1..6 sequences of 0..2600 keys (page
tails and empty sequences included), 1..8 query tokens, GQA groups of 1..16
over 1..4 KV heads (so 1..128 rows per work item: every row tile and row
blocks), bf16 or e4m3 pages with random per-tensor scales, causal or not, and
the planned or the fixed split on a random SM budget.  Outputs and log-sum-exp
are compared element by element with the tolerances of the other parity tests
(max-abs 1e-2 for bf16 KV, 2e-2 for fp8 KV; lse 1e-3)."""
import math

import numpy as np
import pytest

from gpu_helpers import oracle_problem, problem_tensors, run_library, tol_for
from helpers import KV_BF16, KV_FP8, build_problem

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(seed):
    rng = np.random.default_rng(9000 + seed)
    bs = int(rng.integers(1, 7))
    lens = rng.integers(0, 2600, size=bs)
    lens[rng.random(bs) < 0.15] = 0                       # some empty sequences
    lens[rng.random(bs) < 0.15] = rng.integers(1, 17)     # and some shorter than a page
    q_lens = rng.integers(1, 9, size=bs)
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    fp8 = bool(rng.random() < 0.5)
    ks = float(rng.choice([0.5, 0.37, 1.0, 2.0])) if fp8 else 1.0
    vs = float(rng.choice([0.25, 0.61, 1.0])) if fp8 else 1.0
    causal = int(rng.random() < 0.8)
    sm_scale = float(rng.choice([1.0, 0.5, 2.0])) / math.sqrt(128)
    pr = build_problem(lens.tolist(), q_lens.tolist(), g * hkv, hkv, kv_dtype=KV_FP8 if fp8 else KV_BF16,
                       k_scale=ks, v_scale=vs, causal=causal, sm_scale=sm_scale, seed=seed)
    use_plan = bool(rng.random() < 0.7)
    num_sms = int(rng.choice([8, 24, 148]))
    return pr, use_plan, num_sms


@pytest.mark.parametrize("seed", range(40))
def test_attention_fuzz_elementwise(seed):
    pr, use_plan, num_sms = _case(seed)
    q, kv = problem_tensors(pr, DEV)
    r = run_library(pr, q, kv, use_plan=use_plan, num_sms=num_sms)
    assert r.status == 0
    ref, ref_lse = oracle_problem(pr)
    got = r.out.float().cpu().numpy()
    assert np.isfinite(got).all()
    err = float(np.max(np.abs(got - ref), initial=0.0))
    assert err <= tol_for(pr.kv_dtype), err
    lse = r.lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(lse), ~fin)
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) <= 1e-3
