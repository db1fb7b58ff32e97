"""merge_state / merge_states on the GPU against the oracle's merge operator."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import dev, f64

pytestmark = pytest.mark.gpu


def _tol(dtype, ref):
    # fp32 math; the output rounding of 16-bit types dominates
    if dtype == "f32":
        return 2e-5 + 2e-6 * np.abs(ref)
    if dtype == "f16":
        return 1e-4 + 2.0 ** -10 * np.abs(ref)
    return 1e-4 + 2.0 ** -8 * np.abs(ref)


def _check(got_v, got_s, ref_v, ref_s, dtype):
    gv = got_v.float().cpu().numpy().astype(np.float64)
    gs = got_s.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(gs), np.isneginf(ref_s))
    fin = ~np.isneginf(ref_s)
    assert np.all(np.abs(gs[fin] - ref_s[fin]) <= 1e-5 + 1e-6 * np.abs(ref_s[fin]))
    assert np.all(np.isfinite(gv))
    assert np.all(np.abs(gv - ref_v) <= _tol(dtype, ref_v))


def _states(T, H, D, dtype, seed, n=None, empty_frac=0.0):
    rng = np.random.default_rng(seed)
    shape_s = (T, H) if n is None else (T, n, H)
    shape_v = shape_s + (D,)
    s = rng.uniform(-10, 10, size=shape_s).astype(np.float32)
    if empty_frac:
        s[rng.random(shape_s) < empty_frac] = -np.inf
    v = workloads.normal(shape_v, seed, 7, dtype)
    return v, s


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("T,H,D", [(1, 1, 128), (37, 5, 128), (100, 3, 64), (9, 2, 256), (13, 7, 32)])
def test_merge_state_small(dtype, T, H, D):
    va, sa = _states(T, H, D, dtype, 1, empty_frac=0.2)
    vb, sb = _states(T, H, D, dtype, 2, empty_frac=0.2)
    ref_v, ref_s = oracle.merge2(f64(va), sa, f64(vb), sb)
    got_v, got_s = pkc.merge_state(dev(va), dev(sa), dev(vb), dev(sb))
    torch.cuda.synchronize()
    _check(got_v, got_s, ref_v, ref_s, dtype)


def test_merge_state_in_place():
    va, sa = _states(64, 4, 128, "f32", 3)
    vb, sb = _states(64, 4, 128, "f32", 4)
    ref_v, ref_s = oracle.merge2(f64(va), sa, f64(vb), sb)
    ta, tsa = dev(va), dev(sa)
    pkc.merge_state(ta, tsa, dev(vb), dev(sb), v_out=ta, s_out=tsa)
    torch.cuda.synchronize()
    _check(ta, tsa, ref_v, ref_s, "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 5, 16])
def test_merge_states_small(dtype, n):
    v, s = _states(29, 3, 128, dtype, 5, n=n, empty_frac=0.25)
    ref_v, ref_s = oracle.merge_n(np.moveaxis(f64(v), 1, 0), np.moveaxis(s, 1, 0))
    got_v, got_s = pkc.merge_states(dev(v), dev(s))
    torch.cuda.synchronize()
    _check(got_v, got_s, ref_v, ref_s, dtype)


def test_merge_state_full_workload():
    w = workloads.workload("merge")
    got_v, got_s = pkc.merge_state(dev(w["v_a"]), dev(w["s_a"]), dev(w["v_b"]), dev(w["s_b"]))
    torch.cuda.synchronize()
    ref_v, ref_s = oracle.merge2(f64(w["v_a"]), w["s_a"], f64(w["v_b"]), w["s_b"])
    _check(got_v, got_s, ref_v, ref_s, "f32")


def test_merge_states_full_workload_every_token():
    """16-ary merge of 4096 tokens x 32 heads: every (token, head) row, the
    oracle taken over blocks of 256 tokens to bound its float64 memory."""
    w = workloads.workload("merge")
    got_v, got_s = pkc.merge_states(dev(w["v_n"]), dev(w["s_n"]))
    torch.cuda.synchronize()
    got_v, got_s = got_v.cpu(), got_s.cpu()
    T = w["v_n"].shape[0]
    for t0 in range(0, T, 256):
        sl = slice(t0, min(T, t0 + 256))
        ref_v, ref_s = oracle.merge_n(np.moveaxis(f64(w["v_n"][sl]), 1, 0),
                                      np.moveaxis(w["s_n"][sl], 1, 0))
        _check(got_v[sl], got_s[sl], ref_v, ref_s, "f32")
