"""Conditions only the device can see are reported through the status word,
and the affected work is skipped (no memory is touched out of bounds)."""
import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
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
