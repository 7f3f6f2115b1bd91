"""Standard -> shuffled page conversion through the C ABI vs the oracle, bit for
bit (pure data movement), for bf16 and e4m3 pages: every block, a listed
subset with out-of-range ids (skipped and flagged), and outputs that start
with random bytes so that a unit written to the wrong place shows up."""
import numpy as np
import pytest
import torch

import paged_split_kv_gb300 as sk
from oracle import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(dtype, nb, h, ids, seed):
    rng = np.random.default_rng(seed)
    hi = 1 << 16 if dtype == np.uint16 else 256
    pages = rng.integers(0, hi, size=(nb, h, 16, 256), dtype=dtype)
    x = 16 // np.dtype(dtype).itemsize
    k0 = rng.integers(0, hi, size=(nb, h, 128 // x, 16, x), dtype=dtype)
    v0 = rng.integers(0, hi, size=(nb, h, 16 // x, 128, x), dtype=dtype)
    d = torch.device(DEV)

    def dev(a):
        t = torch.as_tensor(a.view(np.int16) if dtype == np.uint16 else a, device=d)
        return t.view(torch.bfloat16) if dtype == np.uint16 else t
    pg, kt, vt = dev(pages), dev(k0), dev(v0)
    it = None if ids is None else torch.as_tensor(np.asarray(ids, np.int32), device=d)
    sk.sk_get_device_status(clear=True)
    assert sk.sk_std_to_shuffled(pg, kt, vt, block_ids=it) == sk.SK_OK
    torch.cuda.synchronize()
    status = sk.sk_get_device_status(clear=True)

    def host(t):
        c = t.cpu()
        return c.view(torch.int16).numpy().view(np.uint16) if dtype == np.uint16 else c.numpy()
    kw, vw = oracle.std_to_shuffled(pages, block_ids=ids, k_shuf=k0.copy(), v_shuf=v0.copy())
    return host(kt), host(vt), kw, vw, status


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
@pytest.mark.parametrize("nb,h", [(1, 1), (7, 2), (64, 8)])
def test_all_blocks_bit_exact(dtype, nb, h):
    k, v, kw, vw, status = _case(dtype, nb, h, None, nb * 10 + h)
    assert status == 0
    np.testing.assert_array_equal(k, kw)
    np.testing.assert_array_equal(v, vw)


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
def test_listed_blocks_and_bad_ids(dtype):
    nb = 40
    ids = [3, 39, 0, 17, 40, -1, 1 << 30, 22]
    k, v, kw, vw, status = _case(dtype, nb, 4, ids, 5)
    assert status == sk.SK_DEV_BAD_BLOCK
    np.testing.assert_array_equal(k, kw)
    np.testing.assert_array_equal(v, vw)
