"""Plan kernel vs the oracle's plan: bit-exact T, work list (with its -1 tail)
and per-token segment counts, on the five workloads, the small shapes and a
random fuzz of 2000 batches (and 400 more of at most 33 sequences)."""
import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
import sk_inputs as si
from oracle import oracle

pytestmark = pytest.mark.gpu


def _gpu_plan(lens, q_lens, kv_heads, num_sms, seg_max, cap=None):
    d = torch.device("cuda:0")
    lens = np.asarray(lens, np.int32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cap = cap or sk.plan_capacity(len(lens), kv_heads, num_sms)
    plan = torch.full((cap,), 12345, dtype=torch.int32, device=d)
    tok = torch.full((int(cu[-1]),), 777, dtype=torch.int32, device=d)
    sk.sk_plan_cache_reset()
    rc = sk.sk_build_plan(torch.as_tensor(lens, device=d), torch.as_tensor(cu, device=d), kv_heads,
                          plan, tok, num_sms, seg_max)
    assert rc == sk.SK_OK
    torch.cuda.synchronize()
    assert sk.sk_get_device_status() == 0
    return plan.cpu().numpy(), tok.cpu().numpy(), cu, cap


def _check(lens, q_lens, kv_heads, num_sms, seg_max):
    plan, tok, cu, cap = _gpu_plan(lens, q_lens, kv_heads, num_sms, seg_max)
    ref, ref_tok, _, _ = oracle.plan(np.asarray(lens, np.int32), cu, kv_heads, num_sms, seg_max,
                                     sk.sk_tile_tokens(), cap)
    np.testing.assert_array_equal(plan, ref)
    np.testing.assert_array_equal(tok, ref_tok)


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_plan_bit_exact_on_workloads(idx):
    w = si.config(idx)
    _check(w.seq_lens, w.q_lens, w.num_kv_heads, w.num_sms, w.seg_max)


def test_plan_bit_exact_on_small_shapes():
    for w in si.small_cases():
        _check(w.seq_lens, w.q_lens, w.num_kv_heads, w.num_sms, w.seg_max)


def test_plan_fuzz():
    rng = np.random.default_rng(99)
    for trial in range(2000):
        bs = int(rng.integers(1, 400)) if trial % 50 else int(rng.integers(1000, 32768))
        kind = trial % 4
        if kind == 0:
            lens = rng.integers(0, 300_000, size=bs)
        elif kind == 1:
            lens = np.exp(rng.uniform(0, np.log(300_000), size=bs)).astype(np.int64)
        elif kind == 2:
            lens = rng.integers(0, 3_000, size=bs)
        else:
            lens = np.zeros(bs, np.int64)
            lens[rng.integers(0, bs)] = int(rng.integers(1, 2_000_000))
        q = rng.integers(0, 5, size=bs)
        kv = int(rng.choice([1, 2, 4, 8, 16]))
        nsm = int(rng.choice([148, 152, 256, 20]))
        seg = int(rng.choice([64, 16, 1, 300]))
        _check(lens.astype(np.int32), q.astype(np.int32), kv, nsm, seg)


def test_plan_one_warp_search():
    """Batches of at most 32 sequences take the one-warp search (32 candidate T per
    round); 33 take bisection.  Wide length ranges (up to 16M keys; the oracle scans
    every T, so longer ones would take it minutes) make the search range long, so
    most cases run several rounds."""
    rng = np.random.default_rng(321)
    for trial in range(400):
        bs = 32 if trial % 10 == 0 else 33 if trial % 10 == 1 else int(rng.integers(1, 33))
        kind = trial % 3
        if kind == 0:
            lens = np.exp(rng.uniform(0, np.log(16_000_000), size=bs))
        elif kind == 1:
            lens = rng.integers(0, 2_000_000, size=bs)
        else:
            lens = np.full(bs, int(rng.integers(1, 16_000_000)))
            lens[rng.random(bs) < 0.3] = 0
        lens = lens.astype(np.int64)
        q = rng.integers(0, 4, size=bs)
        kv = int(rng.choice([1, 2, 4, 8]))
        nsm = int(rng.choice([148, 152, 40, 1000]))
        seg = int(rng.choice([64, 16, 1, 300, 4096]))
        _check(lens.astype(np.int32), q.astype(np.int32), kv, nsm, seg)


def test_plan_capacity_above_minimum_is_padded_with_minus_one():
    lens = np.array([5000, 70000, 3], np.int32)
    plan, tok, cu, cap = _gpu_plan(lens, [4, 4, 4], 2, 148, 64, cap=300)
    ref, _, _, _ = oracle.plan(lens, cu, 2, 148, 64, sk.sk_tile_tokens(), 300)
    np.testing.assert_array_equal(plan, ref)


def test_plan_degenerate_budgets_and_batches():
    """Fewer SMs than KV heads (a budget of 0 work items), an all-empty batch,
    a single sequence, and a batch at the shared-memory cache edge."""
    rng = np.random.default_rng(5)
    _check(np.array([900, 0, 77], np.int32), [1, 1, 1], 8, 4, 64)        # budget 0
    _check(np.array([0, 0, 0, 0], np.int32), [1, 0, 2, 1], 2, 148, 64)   # nothing to attend
    _check(np.array([123457], np.int32), [4], 2, 148, 64)                # bs 1
    for bs in (8192, 8193):
        lens = rng.integers(0, 50_000, size=bs).astype(np.int32)
        _check(lens, rng.integers(0, 3, size=bs).astype(np.int32), 2, 152, 64)
