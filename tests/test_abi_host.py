"""Host-side checks of the C ABI that need no GPU: the library loads, every
function include/sk.h declares is exported, host arithmetic agrees with the
oracle, and invalid arguments are rejected before anything touches CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sklib():
    from paged_split_kv_gb300 import build as b
    b.build()
    import paged_split_kv_gb300 as sk
    return sk.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(sk_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(sklib):
    names = _declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(sklib, n), n


def test_tile_and_fixed_split_match_oracle(sklib, oracle):
    assert sklib.sk_tile_tokens() == 64
    for bs in range(1, 70):
        for kv in (1, 2, 4, 8):
            for nsm in (148, 152, 256):
                for seg_max in (64, 16):
                    assert sklib.sk_fixed_nseg(bs, kv, nsm, seg_max) == oracle.fixed_nseg(bs, kv, nsm, seg_max)


FAKE = ctypes.c_void_p(256)   # never dereferenced: validation runs first


def test_build_plan_rejects_bad_arguments_without_cuda(sklib):
    f = sklib.sk_build_plan
    # bs out of range
    assert f(FAKE, 0, FAKE, 0, 0, 4, 2, 148, 64, FAKE, 100, FAKE, None) == -1
    assert f(FAKE, 0, FAKE, 0, 40000, 4, 2, 148, 64, FAKE, 50000, FAKE, None) == -1
    # null plan
    assert f(FAKE, 0, FAKE, 0, 4, 4, 2, 148, 64, None, 100, FAKE, None) == -1
    # capacity below 1 + max(B, bs)
    assert f(FAKE, 0, FAKE, 0, 4, 4, 2, 148, 64, FAKE, 74, FAKE, None) == -2
    assert b"plan_capacity" in sklib.sk_last_error()
    # seg_max too large for the 16-bit segment field
    assert f(FAKE, 0, FAKE, 0, 4, 4, 2, 148, 70000, FAKE, 100, FAKE, None) == -1


def test_attention_rejects_bad_arguments_without_cuda(sklib):
    f = sklib.sk_paged_decode_attn
    base = dict(q=FAKE, kv=FAKE, dt=0, ks=1.0, vs=1.0, bt=FAKE, stride=10, nb=100, page=16,
                lens=FAKE, cu=FAKE, plan=FAKE, cap=75, bs=4, nt=16, mq=4, hq=32, hkv=2, d=128,
                scale=0.088, causal=1, nsm=148, seg=64, po=FAKE, pm=FAKE, pl=FAKE, st=None)

    def call(**kw):
        a = dict(base, **kw)
        return f(*a.values())

    assert call(d=64) == -3
    assert call(page=32) == -3
    assert call(hq=31) == -1
    assert call(dt=7) == -1
    assert call(cap=74) == -2
    assert call(bs=0) == -1
    assert call(q=None) == -1
    assert call(q=ctypes.c_void_p(264)) == -1          # not 16-byte aligned
    assert call(kv=ctypes.c_void_p(264)) == -1
    assert call(po=ctypes.c_void_p(264)) == -1         # the epilogue stores 16 bytes a lane
    assert call(scale=0.0) == -1
    assert call(dt=1, ks=0.0) == -1
    assert call(mq=0) == -1                            # tokens but no query length
    assert call(mq=5000) == -3                         # 16 x 5000 rows per work item: past the kernel's limit
    assert call(nb=1 << 30) == -3                      # 2^31 block-heads: past the tensor map


def test_merge_rejects_bad_arguments_without_cuda(sklib):
    f = sklib.sk_merge_segments
    assert f(FAKE, FAKE, FAKE, None, 65, 4, 8, 128, 64, FAKE, None, None) == -1
    assert f(FAKE, FAKE, FAKE, None, 1, 4, 8, 96, 64, FAKE, None, None) == -3
    assert f(None, FAKE, FAKE, None, 1, 4, 8, 128, 64, FAKE, None, None) == -1
    assert f(ctypes.c_void_p(264), FAKE, FAKE, None, 1, 4, 8, 128, 64, FAKE, None, None) == -1   # part_o % 16
    assert f(FAKE, FAKE, FAKE, None, 1, 4, 8, 128, 64, ctypes.c_void_p(260), None, None) == -1   # out % 8


def test_kv_write_rejects_bad_arguments_without_cuda(sklib):
    f = sklib.sk_reshape_and_cache

    def call(k=FAKE, v=FAKE, sm=FAKE, nt=4, h=2, d=128, pg=FAKE, dt=0, ks=1.0, vs=1.0, nb=8, page=16):
        return f(k, v, sm, nt, h, d, pg, dt, ks, vs, nb, page, None)
    assert call(d=64) == -3
    assert call(page=32) == -3
    assert call(dt=2) == -1
    assert call(nt=-1) == -1
    assert call(h=0) == -1
    assert call(nb=0) == -1
    assert call(dt=1, ks=0.0) == -1
    assert call(dt=1, vs=float("inf")) == -1
    assert call(k=None) == -1
    assert call(sm=None) == -1
    assert call(pg=ctypes.c_void_p(264)) == -1          # not 16-byte aligned
    assert call(nt=0, k=None, v=None, sm=None, pg=None) == 0   # nothing to write: no launch


def test_shuffle_rejects_bad_arguments_without_cuda(sklib):
    f = sklib.sk_std_to_shuffled

    def call(pg=FAKE, dt=0, ids=None, n=0, nb=8, h=2, d=128, page=16, k=FAKE, v=FAKE):
        return f(pg, dt, ids, n, nb, h, d, page, k, v, None)
    assert call(d=64) == -3
    assert call(page=8) == -3
    assert call(dt=3) == -1
    assert call(nb=0) == -1
    assert call(h=0) == -1
    assert call(ids=FAKE, n=-1) == -1
    assert call(pg=None) == -1
    assert call(v=ctypes.c_void_p(264)) == -1         # not 16-byte aligned
    assert call(ids=FAKE, n=0) == 0                   # empty id list: no launch


def test_python_binding_refuses_cpu_tensors(sklib):
    import torch
    import paged_split_kv_gb300 as sk
    with pytest.raises(ValueError):
        sk.sk_build_plan(torch.zeros(2, dtype=torch.int32), torch.zeros(3, dtype=torch.int32), 1,
                         torch.zeros(10, dtype=torch.int32), torch.zeros(2, dtype=torch.int32), 148)


def test_plan_capacity_is_computed_by_the_library(sklib, oracle):
    import paged_split_kv_gb300 as sk
    for bs in (1, 2, 16, 73, 74, 75, 128, 32767):
        for kv in (1, 2, 8):
            for nsm in (148, 152, 256):
                assert sklib.sk_plan_capacity(bs, kv, nsm) == 1 + max(nsm // kv, bs)
                assert sk.plan_capacity(bs, kv, nsm) == sklib.sk_plan_capacity(bs, kv, nsm)
    assert sklib.sk_plan_capacity(0, 2, 148) == -1
    assert sklib.sk_plan_capacity(40000, 2, 148) == -1
    assert sklib.sk_plan_capacity(4, 0, 148) == -1


def test_wait_limit_round_trip(sklib):
    default = sklib.sk_set_wait_limit(-1)
    assert default == 4000000000
    assert sklib.sk_set_wait_limit(0) == default
    assert sklib.sk_set_wait_limit(-1) == 0
    assert sklib.sk_set_wait_limit(-1) == default


def test_static_entry_rejects_sizes_that_would_wrap(sklib):
    """The scratch size of the allocation-free call is bounded by division, so a
    head count that would wrap the byte count is a capacity error, not a small
    size (checked before any CUDA call)."""
    f = sklib.sk_paged_decode_attention_static

    def call(nt=4, hq=32, hkv=2, seg=64, bs=1):
        return f(FAKE, FAKE, 0, 1.0, 1.0, FAKE, 10, 100, 16, FAKE, FAKE, 1, bs, nt, 4, hq, hkv, 128,
                 0.088, 1, 148, seg, FAKE, None, None)
    assert call(nt=1 << 20) == -2
    assert call(nt=0x7FFFFFFF, hq=0x40000000, hkv=1, seg=0xFFFF) == -2
    assert call(nt=2, hq=0x7FFFFFFE, hkv=1, seg=0xFFFF) == -2
    assert b"32 MiB" in sklib.sk_last_error()
    assert call(hq=0) == -1


def _cpu_batch(torch, nt=8, hq=8, hkv=2, d=128, bs=2, nb=4, stride=3, seg=4):
    return dict(q=torch.zeros((nt, hq, d), dtype=torch.bfloat16),
                kv=torch.zeros((nb, hkv, 16, 2 * d), dtype=torch.bfloat16),
                bt=torch.zeros((bs, stride), dtype=torch.int32),
                lens=torch.zeros(bs, dtype=torch.int32), cu=torch.zeros(bs + 1, dtype=torch.int32),
                po=torch.zeros((nt, seg, hq, d)), pm=torch.zeros((nt, seg, hq)), pl=torch.zeros((nt, seg, hq)),
                out=torch.zeros((nt, hq, d), dtype=torch.bfloat16), lse=torch.zeros((nt, hq)),
                tok=torch.zeros(nt, dtype=torch.int32))


def test_python_binding_checks_shapes_before_raw_pointers(sklib):
    """Every wrapper rejects a tensor whose shape would make a kernel read or write
    past it, before anything reaches the library (here on CPU tensors: the shape
    check comes before the device check)."""
    import torch
    import paged_split_kv_gb300 as sk

    def attn(b):
        return sk.sk_paged_decode_attn(b["q"], b["kv"], b["bt"], b["lens"], b["cu"], None, b["po"], b["pm"],
                                       b["pl"], max_q_len=4, sm_scale=0.1, num_sms=148)

    def static(b):
        return sk.sk_paged_decode_attention_static(b["q"], b["kv"], b["bt"], b["lens"], b["cu"], b["out"],
                                                   b["lse"], max_q_len=4, sm_scale=0.1, num_sms=148)

    def merge(b):
        return sk.sk_merge_segments(b["po"], b["pm"], b["pl"], b["tok"], b["out"], b["lse"])

    bad = {
        "kv last dim": dict(kv=torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16)),
        "cu entries": dict(cu=torch.zeros(4, dtype=torch.int32)),
        "block-table rows": dict(bt=torch.zeros((1, 3), dtype=torch.int32)),
        "head ratio": dict(kv=torch.zeros((4, 3, 16, 256), dtype=torch.bfloat16)),
    }
    for name, kw in bad.items():
        for fn in (attn, static):
            b = _cpu_batch(torch)
            b.update(kw)
            with pytest.raises(ValueError):
                fn(b)
    for name, kw in {"part_o": dict(po=torch.zeros((8, 4, 8, 64))), "part_m": dict(pm=torch.zeros((8, 3, 8))),
                     "part_l": dict(pl=torch.zeros((7, 4, 8)))}.items():
        b = _cpu_batch(torch)
        b.update(kw)
        with pytest.raises(ValueError, match=name):
            attn(b)
    for name, kw in {"out": dict(out=torch.zeros((8, 8, 64), dtype=torch.bfloat16)),
                     "lse": dict(lse=torch.zeros((8, 4))), "tok_nseg": dict(tok=torch.zeros(9, dtype=torch.int32)),
                     "part_m": dict(pm=torch.zeros((8, 4, 4)))}.items():
        b = _cpu_batch(torch)
        b.update(kw)
        with pytest.raises(ValueError, match=name):
            merge(b)
    for name, kw in {"out": dict(out=torch.zeros((7, 8, 128), dtype=torch.bfloat16)),
                     "lse": dict(lse=torch.zeros((8, 9)))}.items():
        b = _cpu_batch(torch)
        b.update(kw)
        with pytest.raises(ValueError, match=name):
            static(b)
    with pytest.raises(ValueError, match="cu_seqlens_q"):
        sk.sk_build_plan(torch.zeros(2, dtype=torch.int32), torch.zeros(2, dtype=torch.int32), 1,
                         torch.zeros(10, dtype=torch.int32), torch.zeros(2, dtype=torch.int32), 148)
    # well-shaped CPU tensors get as far as the device check
    for fn in (attn, static, merge):
        with pytest.raises(ValueError, match="CUDA"):
            fn(_cpu_batch(torch))
