"""KV write through the C ABI vs the oracle: the whole page array, bit for bit
(byte and index work), for bf16 and e4m3 pages.  Pages start filled with
random bytes so that a row written where it should not be, or left unwritten,
shows up.  The e4m3 path also runs every bf16 bit pattern (subnormals,
infinities, NaN) through two scales."""
import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
from helpers import KV_BF16, KV_FP8, to_bf16_bits
from oracle import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
D, PAGE = 128, 16


def _run(key_bits, val_bits, slots, pages0, kv_dtype, ks=1.0, vs=1.0):
    """GPU and oracle results for the same inputs (pages0 is not modified)."""
    d = torch.device(DEV)
    kt = torch.as_tensor(key_bits.view(np.int16), device=d).view(torch.bfloat16)
    vt = torch.as_tensor(val_bits.view(np.int16), device=d).view(torch.bfloat16)
    st = torch.as_tensor(slots, dtype=torch.int64, device=d)
    if kv_dtype == KV_BF16:
        pg = torch.as_tensor(pages0.view(np.int16), device=d).view(torch.bfloat16)
    else:
        pg = torch.as_tensor(pages0, device=d)
    sk.sk_get_device_status(clear=True)
    assert sk.sk_reshape_and_cache(kt, vt, st, pg, k_scale=ks, v_scale=vs) == sk.SK_OK
    torch.cuda.synchronize()
    status = sk.sk_get_device_status(clear=True)
    got = pg.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if kv_dtype == KV_BF16 else got.numpy()
    want = oracle.reshape_and_cache(key_bits, val_bits, slots, pages0.copy(), kv_dtype, ks, vs)
    return got, want, status


def _pages(rng, nb, hkv, kv_dtype):
    if kv_dtype == KV_BF16:
        return rng.integers(0, 1 << 16, size=(nb, hkv, PAGE, 2 * D), dtype=np.uint16)
    return rng.integers(0, 256, size=(nb, hkv, PAGE, 2 * D), dtype=np.uint8)


def _slots(rng, nt, nb, holes=3):
    s = rng.permutation(nb * PAGE)[:nt].astype(np.int64)
    s[rng.choice(nt, size=min(holes, nt), replace=False)] = -1
    return s


@pytest.mark.parametrize("kv_dtype,ks,vs", [(KV_BF16, 1.0, 1.0), (KV_FP8, 0.5, 0.25), (KV_FP8, 0.37, 1.7)])
@pytest.mark.parametrize("nt,hkv", [(1, 1), (37, 4), (300, 2), (5, 8)])
def test_small_writes_bit_exact(kv_dtype, ks, vs, nt, hkv):
    rng = np.random.default_rng(nt * 31 + hkv + kv_dtype)
    nb = max(2, (nt + PAGE - 1) // PAGE + 3)
    x = rng.normal(0, 1, (2, nt, hkv, D)) * np.exp(rng.uniform(-9, 7, (2, nt, hkv, 1)))
    kb, vb = to_bf16_bits(x[0]), to_bf16_bits(x[1])
    got, want, status = _run(kb, vb, _slots(rng, nt, nb), _pages(rng, nb, hkv, kv_dtype), kv_dtype, ks, vs)
    assert status == 0
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("ks,vs", [(1.0, 0.25), (0.37, 2.5)])
def test_every_bf16_pattern_through_e4m3(ks, vs):
    """65536 bf16 patterns as the K and V rows of 512 tokens, one KV head; the
    first pair of scales takes the power-of-two (multiply) path, the second the
    division path."""
    rng = np.random.default_rng(8)
    pat = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    kb = pat.reshape(512, 1, D)
    vb = rng.permutation(pat).reshape(512, 1, D)
    nb = 512 // PAGE + 2
    slots = rng.permutation(nb * PAGE)[:512].astype(np.int64)
    got, want, status = _run(kb, vb, slots, _pages(rng, nb, 1, KV_FP8), KV_FP8, ks, vs)
    assert status == 0
    nan_want = (want & 0x7F) == 0x7F
    assert np.array_equal((got & 0x7F) == 0x7F, nan_want)     # NaN exactly where the oracle has NaN
    np.testing.assert_array_equal(got[~nan_want], want[~nan_want])


def test_slot_past_the_end_is_skipped_and_flagged():
    rng = np.random.default_rng(9)
    nt, hkv, nb = 20, 2, 4
    kb = to_bf16_bits(rng.normal(0, 1, (nt, hkv, D)))
    vb = to_bf16_bits(rng.normal(0, 1, (nt, hkv, D)))
    slots = _slots(rng, nt, nb)
    slots[4] = nb * PAGE           # one past the last row
    slots[9] = 10 ** 12
    got, want, status = _run(kb, vb, slots, _pages(rng, nb, hkv, KV_BF16), KV_BF16)
    assert status == sk.SK_DEV_BAD_BLOCK
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("kv_dtype", [KV_BF16, KV_FP8])
def test_prefill_sized_write_bit_exact(kv_dtype):
    """A 4096-token chunk (8 KV heads) into a shuffled set of blocks."""
    rng = np.random.default_rng(10 + kv_dtype)
    nt, hkv = 4096 if kv_dtype == KV_BF16 else 1024, 8
    nb = nt // PAGE + 16
    kb = to_bf16_bits(rng.normal(0, 1, (nt, hkv, D)))
    vb = to_bf16_bits(rng.normal(0, 1, (nt, hkv, D)))
    got, want, status = _run(kb, vb, _slots(rng, nt, nb, holes=50), _pages(rng, nb, hkv, kv_dtype), kv_dtype,
                             0.5, 0.25)
    assert status == 0
    np.testing.assert_array_equal(got, want)
