"""Pins for the oracle's KV write step (standard pages, written through a slot
mapping) and its e4m3fn encoder.  The encoder is checked against the decoder
(itself pinned to the format definition), IEEE midpoints, saturation, and
PyTorch's own float8 cast where that cast is defined (|x| <= 464); the scatter
against a hand-written page image, untouched rows, and a round trip through
the oracle's attention on pages built by direct indexing.  No GPU is needed."""
import math

import numpy as np
import pytest
import torch

from helpers import KV_BF16, KV_FP8, bf16_bits_to_f64, to_bf16_bits


def _finite_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


# --------------------------------------------------------------------------- e4m3fn encoder

def test_encode_round_trips_every_finite_code(oracle):
    for c in _finite_codes():
        v = np.float32(oracle.e4m3fn_to_double(c))
        assert int(oracle.e4m3fn_encode(v)) == c, hex(c)


def test_encode_midpoints_go_to_the_even_code(oracle):
    for c in range(0x7E):                    # adjacent non-negative finite codes c, c + 1
        lo, hi = oracle.e4m3fn_to_double(c), oracle.e4m3fn_to_double(c + 1)
        mid = np.float32((lo + hi) / 2)      # at most 5 significant bits: exact in binary32
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert int(oracle.e4m3fn_encode(mid)) == even, hex(c)
        assert int(oracle.e4m3fn_encode(-mid)) == even | 0x80, hex(c)
        above = np.nextafter(mid, np.float32(np.inf))
        below = np.nextafter(mid, np.float32(-np.inf))
        assert int(oracle.e4m3fn_encode(above)) == c + 1, hex(c)
        assert int(oracle.e4m3fn_encode(below)) == c, hex(c)


def test_encode_saturates_and_keeps_nan(oracle):
    for x in (448.0, 460.0, 464.0, 470.0, 1e30, math.inf):
        assert int(oracle.e4m3fn_encode(np.float32(x))) == 0x7E, x
        assert int(oracle.e4m3fn_encode(np.float32(-x))) == 0xFE, x
    assert int(oracle.e4m3fn_encode(np.float32(math.nan))) == 0x7F
    assert int(oracle.e4m3fn_encode(np.float32(-0.0))) == 0x80
    assert int(oracle.e4m3fn_encode(np.float32(-1e-30))) == 0x80      # rounds to -0
    assert int(oracle.e4m3fn_encode(np.float32(2.0 ** -10))) == 0x00   # tie between 0 and 2^-9
    assert int(oracle.e4m3fn_encode(np.float32(3 * 2.0 ** -11))) == 0x01


def test_encode_matches_torch_cast_where_defined(oracle):
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-464, 464, 3000), rng.normal(0, 1, 3000) * 2.0 ** -7,
                        rng.normal(0, 4, 3000)]).astype(np.float32)
    want = torch.as_tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3fn_encode(x)
    np.testing.assert_array_equal(got, want)


def test_encode_is_monotone(oracle):
    x = np.linspace(-500, 500, 40001, dtype=np.float32)
    vals = np.array([oracle.e4m3fn_to_double(int(c)) for c in oracle.e4m3fn_encode(x)])
    assert np.all(np.diff(vals) >= 0)


# --------------------------------------------------------------------------- the scatter

def test_scatter_hand_example(oracle):
    """page 4, one KV head, head_dim 2: three tokens, slots 5, -1 and 0."""
    key = np.array([[[1, 2]], [[3, 4]], [[5, 6]]], np.uint16)
    val = np.array([[[11, 12]], [[13, 14]], [[15, 16]]], np.uint16)
    pages = np.full((3, 1, 4, 4), 7, np.uint16)
    oracle.reshape_and_cache(key, val, np.array([5, -1, 0]), pages, KV_BF16)
    want = np.full((3, 1, 4, 4), 7, np.uint16)
    want[1, 0, 1] = [1, 2, 11, 12]          # slot 5 = block 1, row 1: K then V
    want[0, 0, 0] = [5, 6, 15, 16]          # slot 0
    np.testing.assert_array_equal(pages, want)


def test_scatter_leaves_other_rows_and_bad_slots_alone(oracle):
    rng = np.random.default_rng(4)
    nt, hkv, d, page, nb = 40, 2, 8, 16, 6
    key = rng.integers(0, 1 << 16, size=(nt, hkv, d), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, size=(nt, hkv, d), dtype=np.uint16)
    slots = rng.permutation(nb * page)[:nt].astype(np.int64)
    slots[3] = -1
    slots[7] = nb * page + 5                # past the last block: ignored
    pages = rng.integers(0, 1 << 16, size=(nb, hkv, page, 2 * d), dtype=np.uint16)
    before = pages.copy()
    oracle.reshape_and_cache(key, val, slots, pages, KV_BF16)
    written = np.zeros((nb, page), bool)
    for t, s in enumerate(slots):
        if 0 <= s < nb * page:
            written[s // page, s % page] = True
            for h in range(hkv):
                np.testing.assert_array_equal(pages[s // page, h, s % page, :d], key[t, h])
                np.testing.assert_array_equal(pages[s // page, h, s % page, d:], val[t, h])
    untouched = ~written
    np.testing.assert_array_equal(pages.transpose(0, 2, 1, 3)[untouched], before.transpose(0, 2, 1, 3)[untouched])


@pytest.mark.parametrize("kv_dtype", [KV_BF16, KV_FP8])
def test_scatter_then_attention_equals_attention_on_directly_built_pages(oracle, kv_dtype):
    """Write every key of a small batch through the scatter into an empty cache,
    then run the oracle's attention on it; build the same cache by indexing in
    NumPy; the two attentions agree exactly."""
    rng = np.random.default_rng(11 + kv_dtype)
    seq_lens = np.array([37, 1, 70], np.int32)
    q_lens = np.array([2, 1, 3], np.int32)
    hq, hkv, d, page = 8, 2, 128, 16
    ks, vs = (0.5, 0.25) if kv_dtype == KV_FP8 else (1.0, 1.0)
    nblk = [int(-(-L // page)) for L in seq_lens]
    nb = sum(nblk) + 3
    perm = rng.permutation(nb)
    bt = np.full((len(seq_lens), max(nblk)), -1, np.int32)
    o = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[o:o + n]
        o += n
    toks = int(seq_lens.sum())
    key = to_bf16_bits(rng.normal(0, 1, (toks, hkv, d)))
    val = to_bf16_bits(rng.normal(0, 1, (toks, hkv, d)))
    slots = np.concatenate([bt[s, np.arange(L) // page] * page + np.arange(L) % page
                            for s, L in enumerate(seq_lens)]).astype(np.int64)
    dt = np.uint16 if kv_dtype == KV_BF16 else np.uint8
    via_scatter = np.zeros((nb, hkv, page, 2 * d), dt)
    oracle.reshape_and_cache(key, val, slots, via_scatter, kv_dtype, ks, vs)
    direct = np.zeros((nb, hkv, page, 2 * d), dt)
    t = 0
    for s, L in enumerate(seq_lens):
        for p in range(L):
            blk, off = bt[s, p // page], p % page
            for h in range(hkv):
                if kv_dtype == KV_BF16:
                    direct[blk, h, off, :d], direct[blk, h, off, d:] = key[t, h], val[t, h]
                else:
                    kx = (bf16_bits_to_f64(key[t, h]).astype(np.float32) / np.float32(ks)).astype(np.float32)
                    vx = (bf16_bits_to_f64(val[t, h]).astype(np.float32) / np.float32(vs)).astype(np.float32)
                    direct[blk, h, off, :d] = torch.as_tensor(kx).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    direct[blk, h, off, d:] = torch.as_tensor(vx).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            t += 1
    np.testing.assert_array_equal(via_scatter, direct)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = to_bf16_bits(rng.normal(0, 1, (int(cu[-1]), hq, d)))
    args = dict(kv_dtype=kv_dtype, k_scale=ks, v_scale=vs, block_table=bt, page=page, seq_lens=seq_lens,
                cu_q=cu, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, sm_scale=1 / math.sqrt(d), causal=1)
    a, la = oracle.attention(q, via_scatter, **args)
    b, lb = oracle.attention(q, direct, **args)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
