"""Every OCP e4m3fn code through the fp8 paths of the GPU kernels.

V path: sequences of one key whose V row holds the codes; the output of a
single visible key is that key's V, so it must equal v_scale * decode(code)
exactly (every e4m3 value times a power-of-two scale is a bf16 value), and
NaN for the NaN code.
K path: for each code c, two keys with K_0 = 0 and K_1 = c e_0, V_0 = 0 and
V_1 = 1, so the output is sigmoid(sm_scale * k_scale * q_0 * decode(c)) *
v_scale, compared with the oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import oracle_problem, problem_tensors, run_library
from helpers import KV_FP8, build_problem

pytestmark = pytest.mark.gpu
D = "cuda:0"


def _decoded_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_all_codes_through_v():
    vals = _decoded_codes()

    def vf(s, p, h, d):
        return np.repeat(vals[128 * s + d][None, :], len(p), 0)

    def kf(s, p, h, d):
        return np.zeros((len(p), len(d)))
    v_scale = 0.25
    pr = build_problem([1, 1], 1, 2, 1, kv_dtype=KV_FP8, k_scale=0.5, v_scale=v_scale, kfun=kf, vfun=vf, seed=71)
    q, kv = problem_tensors(pr, D)
    got = run_library(pr, q, kv, use_plan=True).out.float().cpu().numpy()   # [2 tokens, 2 heads, 128]
    for s in range(2):
        want = v_scale * vals[128 * s: 128 * s + 128]
        row = got[s, 0]
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(row), nan), s
        assert np.array_equal(row[~nan], want[~nan].astype(np.float32)), s


def test_all_codes_through_k():
    vals = _decoded_codes()
    finite = [c for c in range(256) if np.isfinite(vals[c])]

    def kf(s, p, h, d):
        k = np.zeros((len(p), len(d)))
        k[p == 1, 0] = vals[finite[s]]
        return k

    def vf(s, p, h, d):
        return np.where((p == 1)[:, None], 1.0, 0.0) * np.ones((len(p), len(d)))

    qf = lambda t, hq, d: np.where(d == 0, 2.0, 0.0)
    pr = build_problem([2] * len(finite), 1, 1, 1, kv_dtype=KV_FP8, k_scale=0.5, v_scale=0.25,
                       kfun=kf, vfun=vf, qfun=qf, seed=72)
    q, kv = problem_tensors(pr, D)
    got = run_library(pr, q, kv, use_plan=True).out.float().cpu().numpy()
    ref, _ = oracle_problem(pr)
    assert np.max(np.abs(got - ref)) <= 2e-3
    # the output is monotone in the code's value: catches a sign or byte-order slip
    order = np.argsort([vals[c] for c in finite], kind="stable")
    w = got[order, 0, 0]
    assert np.all(np.diff(w) >= -1e-3)
