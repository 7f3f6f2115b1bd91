"""The serving step end to end on the GPU: this step's K/V written into the
paged cache by sk_reshape_and_cache, then plan + split-KV attention + merge
over that cache, against the oracle doing the same two steps.

Two writes: the whole history written at once (a prefill of the cache), then
each sequence's new query tokens appended (a verify step) and attended."""
import math

import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
from gpu_helpers import tol_for
from helpers import KV_BF16, KV_FP8, to_bf16_bits
from oracle import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PAGE, D = 16, 128


def _slots(bt, s, p0, p1):
    p = np.arange(p0, p1)
    return (bt[s, p // PAGE].astype(np.int64) * PAGE + p % PAGE)


@pytest.mark.parametrize("kv_dtype,ks,vs", [(KV_BF16, 1.0, 1.0), (KV_FP8, 0.5, 0.25), (KV_FP8, 0.3, 1.3)])
def test_write_then_attend(kv_dtype, ks, vs):
    rng = np.random.default_rng(50 + kv_dtype + int(ks * 10))
    hist = np.array([3000, 0, 17, 9000, 130], np.int32)    # keys already in the cache
    q_lens = np.array([4, 1, 3, 4, 2], np.int32)            # this step's tokens (appended)
    hq, hkv = 32, 2
    lens = hist + q_lens
    nblk = (lens + PAGE - 1) // PAGE
    nb = int(nblk.sum()) + 9
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(lens), int(nblk.max())), -1, np.int32)
    o = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[o:o + n]
        o += n
    d = torch.device(DEV)
    dt = torch.bfloat16 if kv_dtype == KV_BF16 else torch.uint8
    pages = torch.zeros((nb, hkv, PAGE, 2 * D), dtype=dt, device=d)
    ref_pages = np.zeros((nb, hkv, PAGE, 2 * D), np.uint16 if kv_dtype == KV_BF16 else np.uint8)

    def write(k_bits, v_bits, slots):
        kt = torch.as_tensor(k_bits.view(np.int16), device=d).view(torch.bfloat16)
        vt = torch.as_tensor(v_bits.view(np.int16), device=d).view(torch.bfloat16)
        assert sk.sk_reshape_and_cache(kt, vt, torch.as_tensor(slots, device=d), pages, k_scale=ks,
                                       v_scale=vs) == sk.SK_OK
        oracle.reshape_and_cache(k_bits, v_bits, slots, ref_pages, kv_dtype, ks, vs)

    # first write: the history of every sequence
    slots = np.concatenate([_slots(bt, s, 0, int(hist[s])) for s in range(len(lens))])
    kh = to_bf16_bits(rng.normal(0, 1, (len(slots), hkv, D)))
    vh = to_bf16_bits(rng.normal(0, 1, (len(slots), hkv, D)))
    write(kh, vh, slots)
    # second write: this step's tokens, appended after each history
    slots = np.concatenate([_slots(bt, s, int(hist[s]), int(lens[s])) for s in range(len(lens))])
    kn = to_bf16_bits(rng.normal(0, 1, (len(slots), hkv, D)))
    vn = to_bf16_bits(rng.normal(0, 1, (len(slots), hkv, D)))
    write(kn, vn, slots)
    torch.cuda.synchronize()
    assert sk.sk_get_device_status(clear=True) == 0
    got_pages = pages.cpu()
    got_pages = got_pages.view(torch.int16).numpy().view(np.uint16) if kv_dtype == KV_BF16 else got_pages.numpy()
    np.testing.assert_array_equal(got_pages, ref_pages)

    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q_bits = to_bf16_bits(rng.normal(0, 1, (int(cu[-1]), hq, D)))
    qt = torch.as_tensor(q_bits.view(np.int16), device=d).view(torch.bfloat16)
    scale = 1 / math.sqrt(D)
    out, lse = sk.paged_decode_attention(qt, pages, torch.as_tensor(bt, device=d), torch.as_tensor(lens, device=d),
                                         torch.as_tensor(cu, device=d), max_q_len=int(q_lens.max()), sm_scale=scale,
                                         num_sms=148, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert sk.sk_get_device_status(clear=True) == 0
    ref, ref_lse = oracle.attention(q_bits, ref_pages, kv_dtype, ks, vs, bt, PAGE, lens, cu, hq, hkv, D, scale, 1)
    got = out.float().cpu().numpy().reshape(-1, D)
    assert np.max(np.abs(got - ref)) <= tol_for(kv_dtype)
    fin = np.isfinite(ref_lse)
    got_lse = lse.cpu().numpy().reshape(-1)
    assert np.array_equal(np.isfinite(got_lse), fin)
    assert np.max(np.abs(got_lse[fin] - ref_lse[fin])) <= 1e-3
