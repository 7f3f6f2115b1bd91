"""Merge kernel vs the oracle's merge on synthetic partials, including empty
segments (l = 0, m = -inf) and tokens with no segment at all."""
import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("use_counts", [True, False])
def test_merge_matches_oracle(use_counts):
    rng = np.random.default_rng(3)
    nt, seg_max, hq, D = 37, 64, 8, 128
    po = rng.standard_normal((nt, seg_max, hq, D)).astype(np.float32)
    pm = rng.uniform(-20, 20, (nt, seg_max, hq)).astype(np.float32)
    pl = rng.uniform(0.5, 50, (nt, seg_max, hq)).astype(np.float32)
    po *= pl[..., None]        # o is un-normalised
    empty = rng.random((nt, seg_max, hq)) < 0.2
    pm[empty] = -np.inf
    pl[empty] = 0
    po[empty] = 0
    counts = rng.integers(0, seg_max + 1, size=nt).astype(np.int32)
    counts[3] = 0
    fixed = 11
    d = torch.device("cuda:0")
    t = lambda a: torch.as_tensor(a, device=d)
    out = torch.empty((nt, hq, D), dtype=torch.bfloat16, device=d)
    lse = torch.empty((nt, hq), dtype=torch.float32, device=d)
    sk.sk_merge_segments(t(po), t(pm), t(pl), t(counts) if use_counts else None, out, lse,
                         fixed_nseg=fixed)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.merge(po, pm, pl, counts if use_counts else None, fixed, nt, hq, D, seg_max)
    got = out.float().cpu().numpy().reshape(ref.shape)
    # out is bf16 rounded to nearest: within half a unit in the last place,
    # 2^-9 of |ref| (these synthetic outputs reach |x| ~ 8, beyond a fixed 1e-2)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)
    gl = lse.cpu().numpy().reshape(-1)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(gl), ~fin)
    assert np.max(np.abs(gl[fin] - ref_lse[fin])) <= 1e-4
