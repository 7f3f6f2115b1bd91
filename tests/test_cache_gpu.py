"""Plan cache semantics (SGLang PR 39172, Accuracy Tests: 15 calls in one
forward -> 1 plan launch; reset -> recompute; an in-place seq_lens change or a
different tensor -> recompute; cached output bit-identical to uncached) and a
graph-captured 15-layer forward replayed with new lengths."""
import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
from gpu_helpers import problem_tensors
from helpers import build_problem
from oracle import oracle

pytestmark = pytest.mark.gpu
D = torch.device("cuda:0")


def _buffers(bs, nt, hkv, nsm=148):
    return (torch.empty(sk.plan_capacity(bs, hkv, nsm), dtype=torch.int32, device=D),
            torch.empty(nt, dtype=torch.int32, device=D))


def test_cache_semantics():
    lens = torch.tensor([119000, 5, 17, 4000], dtype=torch.int32, device=D)
    cu = torch.tensor([0, 4, 8, 12, 16], dtype=torch.int32, device=D)
    plan, tok = _buffers(4, 16, 2)
    sk.sk_plan_cache_reset()
    n0 = sk.sk_plan_launch_count()
    rcs = [sk.sk_build_plan(lens, cu, 2, plan, tok, 148) for _ in range(15)]
    assert rcs[0] == sk.SK_OK and all(rc == sk.SK_CACHED for rc in rcs[1:])
    assert sk.sk_plan_launch_count() - n0 == 1
    first = plan.clone()

    # reset -> recompute, same result
    sk.sk_plan_cache_reset()
    assert sk.sk_build_plan(lens, cu, 2, plan, tok, 148) == sk.SK_OK
    assert sk.sk_plan_launch_count() - n0 == 2
    assert torch.equal(plan, first)

    # an in-place change of seq_lens -> recompute with the new lengths
    lens[1] = 60000
    assert sk.sk_build_plan(lens, cu, 2, plan, tok, 148) == sk.SK_OK
    torch.cuda.synchronize()
    cu_np = cu.cpu().numpy()
    ref, _, _, _ = oracle.plan(lens.cpu().numpy(), cu_np, 2, 148, 64, 64, plan.numel())
    assert np.array_equal(plan.cpu().numpy(), ref)

    # a different tensor with the same values -> recompute
    lens2 = lens.clone()
    assert sk.sk_build_plan(lens2, cu, 2, plan, tok, 148) == sk.SK_OK

    # cached output bit-identical to an uncached build into fresh buffers
    plan_b, tok_b = _buffers(4, 16, 2)
    assert sk.sk_build_plan(lens2, cu, 2, plan, tok, 148) == sk.SK_CACHED
    assert sk.sk_build_plan(lens2, cu, 2, plan_b, tok_b, 148) == sk.SK_OK
    torch.cuda.synchronize()
    assert torch.equal(plan, plan_b) and torch.equal(tok, tok_b)


def test_graph_captured_forward_replays_with_new_lengths():
    """15 layers of attention + merge captured with one plan; replaying the graph
    after writing new lengths into the same tensor gives the eager result."""
    pr = build_problem([700, 3000, 5, 1], 4, 32, 2, seed=41)
    q, kv = problem_tensors(pr, D)
    bt = torch.as_tensor(pr.block_table, device=D)
    lens = torch.as_tensor(pr.seq_lens, device=D)
    cu = torch.as_tensor(pr.cu_q, device=D)
    layers = 15
    ws = {}
    outs = [torch.empty((pr.num_tokens, 32, 128), dtype=torch.bfloat16, device=D) for _ in range(layers)]
    lses = [torch.empty((pr.num_tokens, 32), dtype=torch.float32, device=D) for _ in range(layers)]

    def forward():
        sk.sk_plan_cache_reset()
        for i in range(layers):
            sk.paged_decode_attention(q, kv, bt, lens, cu, max_q_len=4, sm_scale=pr.sm_scale,
                                      num_sms=148, workspace=ws, out=outs[i], lse=lses[i],
                                      use_plan=True)

    forward()       # eager warm-up allocates the workspace
    torch.cuda.synchronize()
    eager = outs[0].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    n0 = sk.sk_plan_launch_count()
    with torch.cuda.graph(g, stream=s):
        forward()
    assert sk.sk_plan_launch_count() - n0 == 1       # one plan per forward, inside the graph
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], eager) and torch.equal(outs[14], eager)

    # new lengths written in place; the graph's plan kernel recomputes from them
    new_lens = np.array([690, 2999, 4, 1], dtype=np.int32)
    lens.copy_(torch.as_tensor(new_lens, device=D))
    g.replay()
    torch.cuda.synchronize()
    replayed = outs[7].clone()
    sk.sk_plan_cache_reset()
    fresh, _ = sk.paged_decode_attention(q, kv, bt, lens, cu, max_q_len=4, sm_scale=pr.sm_scale,
                                         num_sms=148, use_plan=True)
    torch.cuda.synchronize()
    assert torch.equal(replayed, fresh)
    assert not torch.equal(replayed, eager)
