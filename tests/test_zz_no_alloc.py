"""The allocation-free entry point (sk_paged_decode_attention_static) against
the regular path.

It serves callers that cannot allocate device memory (a host engine that owns
all device memory and forbids plug-ins to call cudaMalloc, or a C caller with
no caching allocator that cannot pay for cudaMalloc inside a serving step):
the scratch between the kernels lives in the library's fixed device array.
Two calls in a row, with different batches, must each give exactly the bits of
the regular entry points (the same kernels run on the same plan), so nothing
left in the shared array by one call leaks into the next.  This file is
collected last."""
import pytest
import torch

import paged_split_kv_gb300 as sk
from gpu_helpers import problem_tensors
from helpers import KV_FP8, build_problem

pytestmark = pytest.mark.gpu
D = torch.device("cuda:0")


def _regular(pr, q, kv, use_plan):
    out, lse = sk.paged_decode_attention(
        q, kv, torch.as_tensor(pr.block_table, device=D), torch.as_tensor(pr.seq_lens, device=D),
        torch.as_tensor(pr.cu_q, device=D), max_q_len=int(pr.q_lens.max()), sm_scale=pr.sm_scale,
        num_sms=148, k_scale=pr.k_scale, v_scale=pr.v_scale, causal=bool(pr.causal), seg_max=16,
        use_plan=use_plan)
    return out, lse


def _static(pr, q, kv, use_plan):
    out = torch.full((pr.num_tokens, pr.num_q_heads, 128), float("nan"), dtype=torch.bfloat16, device=D)
    lse = torch.full((pr.num_tokens, pr.num_q_heads), float("nan"), dtype=torch.float32, device=D)
    rc = sk.sk_paged_decode_attention_static(
        q, kv, torch.as_tensor(pr.block_table, device=D), torch.as_tensor(pr.seq_lens, device=D),
        torch.as_tensor(pr.cu_q, device=D), out, lse, max_q_len=int(pr.q_lens.max()),
        sm_scale=pr.sm_scale, num_sms=148, k_scale=pr.k_scale, v_scale=pr.v_scale,
        causal=bool(pr.causal), seg_max=16, use_plan=use_plan)
    assert rc == sk.SK_OK
    return out, lse


def test_static_entry_matches_regular_path_two_calls_in_a_row():
    problems = [build_problem([0, 1, 17, 700, 3000, 64], [4, 4, 2, 4, 1, 3], 32, 2, seed=61),
                build_problem([5, 300, 1333], [1, 3, 4], 16, 2, kv_dtype=KV_FP8, k_scale=0.5,
                              v_scale=0.25, seed=62)]
    for use_plan in (True, False):
        for pr in problems:                       # two calls in a row share the static array
            q, kv = problem_tensors(pr, D)
            ref, ref_lse = _regular(pr, q, kv, use_plan)
            got, got_lse = _static(pr, q, kv, use_plan)
            torch.cuda.synchronize()
            assert sk.sk_get_device_status() == 0
            # the same kernels on the same plan and partial layout: the same bits
            assert torch.equal(got, ref), (got.float() - ref.float()).abs().max().item()
            assert torch.equal(got_lse, ref_lse)


def test_static_entry_rejects_calls_beyond_its_array():
    pr = build_problem([100], 4, 32, 2, seed=63)
    q, kv = problem_tensors(pr, D)
    big_nt = sk.sk_static_scratch_bytes() // (64 * 32 * 520) + 1
    qb = torch.zeros((big_nt, 32, 128), dtype=torch.bfloat16, device=D)
    out = torch.empty_like(qb)
    cu = torch.tensor([0, big_nt], dtype=torch.int32, device=D)
    with pytest.raises(sk.SkError, match="32 MiB"):
        sk.sk_paged_decode_attention_static(qb, kv, torch.as_tensor(pr.block_table, device=D),
                                            torch.as_tensor(pr.seq_lens, device=D), cu, out,
                                            max_q_len=big_nt, sm_scale=pr.sm_scale, num_sms=148,
                                            seg_max=64)
