"""Conditions only the device can see are reported through the status word,
and the affected work is skipped (no memory is touched out of bounds)."""
import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
import sk_inputs as si
from gpu_helpers import problem_tensors, run_library
from helpers import build_problem

pytestmark = pytest.mark.gpu
D = torch.device("cuda:0")


def test_out_of_range_block_id_is_reported_and_skipped():
    pr = build_problem([100, 40], 1, 8, 2, seed=51)
    q, kv = problem_tensors(pr, D)
    bad = pr.block_table.copy()
    bad[0, 2] = kv.shape[0] + 1000          # past the end of the cache
    bad[1, 0] = -5
    r = run_library(pr, q, kv, block_table=bad)
    assert r.status & sk.SK_DEV_BAD_BLOCK
    assert torch.isfinite(r.out.float()).all()
    # the context is still usable and a clean call reports nothing
    r2 = run_library(pr, q, kv)
    assert r2.status == 0


def test_query_length_above_bound_is_reported():
    pr = build_problem([100, 40], [2, 5], 8, 2, seed=52)
    q, kv = problem_tensors(pr, D)
    d = q.device
    lens = torch.as_tensor(pr.seq_lens, device=d)
    cu = torch.as_tensor(pr.cu_q, device=d)
    bt = torch.as_tensor(pr.block_table, device=d)
    nt = pr.num_tokens
    po = torch.zeros((nt, 64, 8, 128), dtype=torch.float32, device=d)
    pm = torch.zeros((nt, 64, 8), dtype=torch.float32, device=d)
    pl = torch.zeros((nt, 64, 8), dtype=torch.float32, device=d)
    sk.sk_get_device_status(clear=True)
    sk.sk_paged_decode_attn(q, kv, bt, lens, cu, None, po, pm, pl, max_q_len=3,
                            sm_scale=pr.sm_scale, num_sms=148)
    assert sk.sk_get_device_status(clear=True) & sk.SK_DEV_BAD_SEQ


def _partials(nt, hq, seg_max=64):
    return (torch.zeros((nt, seg_max, hq, 128), dtype=torch.float32, device=D),
            torch.zeros((nt, seg_max, hq), dtype=torch.float32, device=D),
            torch.zeros((nt, seg_max, hq), dtype=torch.float32, device=D))


def test_corrupted_query_offsets_are_reported():
    """cu_seqlens_q that runs backwards (sequence 1 would have -1 query tokens): the
    plan and the attention report it, skip that sequence and touch nothing outside
    their arrays; the next clean call reports nothing."""
    pr = build_problem([100, 40, 60], [3, 1, 1], 8, 2, seed=53)
    q, kv = problem_tensors(pr, D)
    lens = torch.as_tensor(pr.seq_lens, device=D)
    bt = torch.as_tensor(pr.block_table, device=D)
    bad_cu = torch.tensor([0, 3, 2, 5], dtype=torch.int32, device=D)
    assert q.shape[0] == 5
    plan = torch.full((sk.plan_capacity(3, 2, 148),), -7, dtype=torch.int32, device=D)
    tok = torch.zeros(5, dtype=torch.int32, device=D)
    po, pm, pl = _partials(5, 8)
    sk.sk_get_device_status(clear=True)
    sk.sk_plan_cache_reset()
    sk.sk_build_plan(lens, bad_cu, 2, plan, tok, 148, 64)
    torch.cuda.synchronize()
    assert sk.sk_get_device_status(clear=True) & sk.SK_DEV_BAD_SEQ
    sk.sk_paged_decode_attn(q, kv, bt, lens, bad_cu, plan, po, pm, pl, max_q_len=3,
                            sm_scale=pr.sm_scale, num_sms=148)
    assert sk.sk_get_device_status(clear=True) & sk.SK_DEV_BAD_SEQ
    assert torch.isfinite(po).all()
    r = run_library(pr, q, kv)
    assert r.status == 0


def test_sequence_longer_than_its_block_table_row_is_reported():
    """A length past block_table_stride * page: the item is skipped and reported."""
    pr = build_problem([100, 40], 1, 8, 2, seed=54)
    q, kv = problem_tensors(pr, D)
    bt = torch.as_tensor(pr.block_table, device=D)
    long_lens = torch.tensor([bt.shape[1] * 16 + 1, 40], dtype=torch.int32, device=D)
    cu = torch.as_tensor(pr.cu_q, device=D)
    po, pm, pl = _partials(pr.num_tokens, 8)
    sk.sk_get_device_status(clear=True)
    sk.sk_paged_decode_attn(q, kv, bt, long_lens, cu, None, po, pm, pl, max_q_len=1,
                            sm_scale=pr.sm_scale, num_sms=148)
    assert sk.sk_get_device_status(clear=True) & sk.SK_DEV_BAD_SEQ
    assert run_library(pr, q, kv).status == 0


def test_plan_entries_out_of_range_are_reported():
    """A caller-written plan naming a sequence past bs and a segment past seg_max:
    those items are skipped and reported; the valid item still runs."""
    pr = build_problem([100, 40], 1, 8, 2, seed=55)
    q, kv = problem_tensors(pr, D)
    lens = torch.as_tensor(pr.seq_lens, device=D)
    cu = torch.as_tensor(pr.cu_q, device=D)
    bt = torch.as_tensor(pr.block_table, device=D)
    cap = sk.plan_capacity(2, 2, 148)
    plan = torch.full((cap,), -1, dtype=torch.int32, device=D)
    plan[0] = 2                                   # two tiles per segment
    plan[1] = (5 << 16) | 0                       # sequence 5 of a batch of 2
    plan[2] = (0 << 16) | 70                      # segment 70 >= seg_max
    plan[3] = (1 << 16) | 0                       # sequence 1, segment 0: valid
    po, pm, pl = _partials(pr.num_tokens, 8)
    pl.fill_(-3.0)
    sk.sk_get_device_status(clear=True)
    sk.sk_paged_decode_attn(q, kv, bt, lens, cu, plan, po, pm, pl, max_q_len=1,
                            sm_scale=pr.sm_scale, num_sms=148)
    assert sk.sk_get_device_status(clear=True) & sk.SK_DEV_BAD_SEQ
    # the valid item wrote its rows: sequence 1 is token 1, segment 0, query heads 0..7
    assert torch.all(pl[1, 0] > 0)
    assert run_library(pr, q, kv).status == 0


def test_query_offsets_short_of_num_tokens_are_reported_and_the_tail_is_zero():
    """cu_seqlens_q ending before num_tokens: the plan reports it and gives the
    trailing tokens 0 segments, so the merge writes 0 (lse -inf) for them instead
    of blending partials nobody wrote."""
    pr = build_problem([100, 40], [2, 1], 8, 2, seed=57)
    q, kv = problem_tensors(pr, D)
    nt = pr.num_tokens + 2                       # two tokens past cu[bs]
    qx = torch.zeros((nt, 8, 128), dtype=torch.bfloat16, device=D)
    qx[:pr.num_tokens] = q
    lens = torch.as_tensor(pr.seq_lens, device=D)
    cu = torch.as_tensor(pr.cu_q, device=D)
    bt = torch.as_tensor(pr.block_table, device=D)
    plan = torch.empty(sk.plan_capacity(2, 2, 148), dtype=torch.int32, device=D)
    tok = torch.full((nt,), 9, dtype=torch.int32, device=D)
    po, pm, pl = _partials(nt, 8)
    po.fill_(float("nan"))
    pm.fill_(float("nan"))
    pl.fill_(float("nan"))
    out = torch.full((nt, 8, 128), float("nan"), dtype=torch.bfloat16, device=D)
    lse = torch.full((nt, 8), float("nan"), dtype=torch.float32, device=D)
    sk.sk_get_device_status(clear=True)
    sk.sk_plan_cache_reset()
    sk.sk_build_plan(lens, cu, 2, plan, tok, 148, 64)
    sk.sk_paged_decode_attn(qx, kv, bt, lens, cu, plan, po, pm, pl, max_q_len=2, sm_scale=pr.sm_scale,
                            num_sms=148)
    sk.sk_merge_segments(po, pm, pl, tok, out, lse)
    assert sk.sk_get_device_status(clear=True) & sk.SK_DEV_BAD_SEQ
    assert torch.equal(tok[pr.num_tokens:].cpu(), torch.zeros(2, dtype=torch.int32))
    assert torch.equal(out[pr.num_tokens:].float().cpu(), torch.zeros((2, 8, 128)))
    assert torch.isneginf(lse[pr.num_tokens:]).all()
    # the covered tokens are what a consistent call gives
    ref = run_library(pr, q, kv)
    assert ref.status == 0
    assert torch.equal(out[:pr.num_tokens], ref.out)


def test_fixed_split_reports_query_offsets_that_do_not_cover_the_tokens():
    pr = build_problem([100, 40], [2, 1], 8, 2, seed=58)
    q, kv = problem_tensors(pr, D)
    lens = torch.as_tensor(pr.seq_lens, device=D)
    bt = torch.as_tensor(pr.block_table, device=D)
    short_cu = torch.tensor([0, 2, 2], dtype=torch.int32, device=D)    # cu[bs] = 2 < 3 tokens
    po, pm, pl = _partials(pr.num_tokens, 8)
    sk.sk_get_device_status(clear=True)
    sk.sk_paged_decode_attn(q, kv, bt, lens, short_cu, None, po, pm, pl, max_q_len=2,
                            sm_scale=pr.sm_scale, num_sms=148)
    assert sk.sk_get_device_status(clear=True) & sk.SK_DEV_BAD_SEQ
    assert run_library(pr, q, kv, use_plan=False).status == 0


@pytest.mark.parametrize("hq, kv_dtype", [(32, si.KV_BF16), (16, si.KV_FP8), (32, si.KV_FP8)])
def test_bounded_wait_that_expires_is_reported_and_the_context_stays_usable(hq, kv_dtype):
    """The timeout path in an unchanged kernel: a wait limit of 0 cycles makes the
    attention kernel's abortable waits give up as soon as a copy or product is not
    already complete.  Every CTA then drains what it issued and exits; the status
    word carries SK_DEV_TIMEOUT, the C call reports SK_ERR_TIMEOUT, and the next
    call with the default limit is clean and bit-identical to one made before.
    Three kernel shapes: bf16 with 64 rows; e4m3 with 32 rows (a landing barrier per
    128-token half); e4m3 with 64 rows (four softmax groups, one S buffer)."""
    fp8 = kv_dtype == si.KV_FP8
    w = si.make_workload("timeout_4x60000_q4", [60000] * 4, 4, hq, 2, seed=59, kv_dtype=kv_dtype,
                         k_scale=0.5 if fp8 else 1.0, v_scale=0.25 if fp8 else 1.0)
    q = si.make_q(w, D)
    kv = si.make_kv(w, D)
    before = run_library(w, q, kv)
    assert before.status == 0
    lib = sk.lib()
    assert sk.sk_set_wait_limit(0) == 4000000000
    try:
        sk.sk_get_device_status(clear=True)
        lens = torch.as_tensor(w.seq_lens, device=D)
        cu = torch.as_tensor(w.cu_q, device=D)
        bt = torch.as_tensor(w.block_table, device=D)
        plan = torch.empty(sk.plan_capacity(w.bs, 2, 148), dtype=torch.int32, device=D)
        tok = torch.empty(w.num_tokens, dtype=torch.int32, device=D)
        po, pm, pl = _partials(w.num_tokens, hq)
        sk.sk_plan_cache_reset()
        sk.sk_build_plan(lens, cu, 2, plan, tok, 148, 64)
        for _ in range(3):                       # the calls return; nothing hangs
            sk.sk_paged_decode_attn(q, kv, bt, lens, cu, plan, po, pm, pl, max_q_len=4,
                                    sm_scale=w.sm_scale, num_sms=148, k_scale=w.k_scale, v_scale=w.v_scale)
        rc = lib.sk_get_device_status(None, 1)
        assert rc == sk.SK_ERR_TIMEOUT, rc
        assert lib.sk_last_device_status() & sk.SK_DEV_TIMEOUT
        assert b"expired" in lib.sk_last_error()
        # the binding returns the mask, timeout bit included
        sk.sk_paged_decode_attn(q, kv, bt, lens, cu, plan, po, pm, pl, max_q_len=4, sm_scale=w.sm_scale,
                                num_sms=148, k_scale=w.k_scale, v_scale=w.v_scale)
        assert sk.sk_get_device_status(clear=True) & sk.SK_DEV_TIMEOUT
    finally:
        sk.sk_set_wait_limit(-1)
    after = run_library(w, q, kv)
    assert after.status == 0
    assert torch.equal(after.out, before.out)
    assert torch.equal(after.lse, before.lse)
