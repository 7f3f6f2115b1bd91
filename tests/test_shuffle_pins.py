"""Pins for the oracle's standard -> shuffled page conversion ([RFC] Proposed
Change, Convert).  The oracle is explicit index loops; it is checked against
NumPy's own reshape and transpose of the formula the page prints (a library
routine), against a bijection on unique values, against hand-placed spot
values, and for leaving unlisted blocks alone.  No GPU is needed."""
import numpy as np
import pytest


def _pages(rng, nb, h, dtype, d=128, n=16):
    hi = 1 << 16 if dtype == np.uint16 else 256
    return rng.integers(0, hi, size=(nb, h, n, 2 * d), dtype=dtype)


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
def test_matches_numpy_reshape_and_transpose(oracle, dtype):
    rng = np.random.default_rng(1)
    pages = _pages(rng, 5, 3, dtype)
    k, v = oracle.std_to_shuffled(pages)
    x = 16 // np.dtype(dtype).itemsize
    nb, h, n, d2 = pages.shape
    d = d2 // 2
    K, V = pages[..., :d], pages[..., d:]
    k_ref = K.reshape(nb, h, n, d // x, x).transpose(0, 1, 3, 2, 4)      # (H, D/x, N, x) per block
    v_ref = V.reshape(nb, h, n // x, x, d).transpose(0, 1, 2, 4, 3)      # (H, N/x, D, x) per block
    np.testing.assert_array_equal(k, k_ref)
    np.testing.assert_array_equal(v, v_ref)


@pytest.mark.parametrize("dtype", [np.uint16, np.uint8])
def test_every_element_lands_once(oracle, dtype):
    """Each (token, column) of a block's head gets a unique 12-bit label; for
    e4m3 bytes the low and high bytes of the label go through two runs and are
    put back together.  The outputs of each head hold every label once."""
    nb, h, n, d = 3, 2, 16, 128
    label = (np.arange(n)[:, None] * 2 * d + np.arange(2 * d)[None, :]).astype(np.uint16)   # < 4096
    if dtype == np.uint16:
        pages = np.broadcast_to(label, (nb, h, n, 2 * d)).copy()
        k, v = oracle.std_to_shuffled(pages)
        got_k, got_v = k.astype(np.uint32), v.astype(np.uint32)
    else:
        parts = []
        for shift in (0, 8):
            pages = np.broadcast_to((label >> shift) & 0xFF, (nb, h, n, 2 * d)).astype(np.uint8).copy()
            parts.append(oracle.std_to_shuffled(pages))
        got_k = parts[0][0].astype(np.uint32) | (parts[1][0].astype(np.uint32) << 8)
        got_v = parts[0][1].astype(np.uint32) | (parts[1][1].astype(np.uint32) << 8)
    for b in range(nb):
        for hh in range(h):
            both = np.concatenate([got_k[b, hh].ravel(), got_v[b, hh].ravel()])
            np.testing.assert_array_equal(np.sort(both), np.arange(n * 2 * d))


def test_spot_positions_bf16(oracle):
    pages = np.zeros((2, 2, 16, 256), np.uint16)
    pages[1, 0, 3, 10] = 111          # K, token 3, dim 10 -> k[1, 0, 10 // 8, 3, 10 % 8]
    pages[1, 1, 12, 128 + 77] = 222   # V, token 12, dim 77 -> v[1, 1, 12 // 8, 77, 12 % 8]
    k, v = oracle.std_to_shuffled(pages)
    assert k[1, 0, 1, 3, 2] == 111 and np.count_nonzero(k) == 1
    assert v[1, 1, 1, 77, 4] == 222 and np.count_nonzero(v) == 1


def test_spot_positions_fp8(oracle):
    pages = np.zeros((1, 1, 16, 256), np.uint8)
    pages[0, 0, 5, 40] = 9            # K, token 5, dim 40 -> k[0, 0, 40 // 16, 5, 40 % 16]
    pages[0, 0, 15, 128 + 3] = 7      # V, token 15, dim 3 -> v[0, 0, 0, 3, 15]
    k, v = oracle.std_to_shuffled(pages)
    assert k.shape == (1, 1, 8, 16, 16) and v.shape == (1, 1, 1, 128, 16)
    assert k[0, 0, 2, 5, 8] == 9 and np.count_nonzero(k) == 1
    assert v[0, 0, 0, 3, 15] == 7 and np.count_nonzero(v) == 1


def test_only_listed_blocks_are_written(oracle):
    rng = np.random.default_rng(2)
    pages = _pages(rng, 6, 2, np.uint16)
    k0 = rng.integers(0, 1 << 16, size=(6, 2, 16, 16, 8), dtype=np.uint16)
    v0 = rng.integers(0, 1 << 16, size=(6, 2, 2, 128, 8), dtype=np.uint16)
    k, v = oracle.std_to_shuffled(pages, block_ids=[4, 1, 99, -3], k_shuf=k0.copy(), v_shuf=v0.copy())
    full_k, full_v = oracle.std_to_shuffled(pages)
    for b in range(6):
        if b in (1, 4):
            np.testing.assert_array_equal(k[b], full_k[b])
            np.testing.assert_array_equal(v[b], full_v[b])
        else:
            np.testing.assert_array_equal(k[b], k0[b])
            np.testing.assert_array_equal(v[b], v0[b])
