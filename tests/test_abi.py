"""C ABI checks that need no GPU: the library loads, exports every symbol
that include/pkc.h declares, rejects bad arguments before touching the
device, and its host-side plan equals the oracle's plan bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from paged_kv_cascade_gb300 import build as pkc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    pkc_build.build()
    return pkc.lib()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "pkc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkc_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), f"{n} declared in pkc.h but not exported"
        assert n in pkc.SIGNATURES, f"{n} has no Python binding"
    assert set(pkc.SIGNATURES) == set(names)


def test_version_and_error_string(L):
    assert L.pkc_version() >= 100
    assert isinstance(L.pkc_last_error(), bytes)


def test_bad_arguments_are_rejected_without_a_device(L):
    fake = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x100000)
    # head_dim 64 is valid but unsupported
    rc = L.pkc_paged_decode_state(fake, fake, fake, fake, 4, fake, 2, 8, 8, 64, 16, 10, 1.0,
                                  None, ws, 1 << 20, fake, fake, 1, None)
    assert rc == 2 and b"head_dim" in L.pkc_last_error()
    # heads not a multiple
    rc = L.pkc_paged_decode_state(fake, fake, fake, fake, 4, fake, 2, 6, 4, 128, 16, 10, 1.0,
                                  None, ws, 1 << 20, fake, fake, 1, None)
    assert rc == 1
    # workspace too small
    rc = L.pkc_paged_decode_state(fake, fake, fake, fake, 4, fake, 2, 8, 8, 128, 16, 10, 1.0,
                                  None, ws, 16, fake, fake, 1, None)
    assert rc == 3
    # misaligned workspace
    rc = L.pkc_paged_decode_state(fake, fake, fake, fake, 4, fake, 2, 8, 8, 128, 16, 10, 1.0,
                                  None, ctypes.c_void_p(0x100010), 1 << 20, fake, fake, 1, None)
    assert rc == 3
    # bad dtype for attention
    rc = L.pkc_cascade_decode(fake, fake, fake, None, None, 1, fake, fake, fake, 4, fake, 2, 8,
                              8, 128, 16, 10, 1.0, None, ws, 1 << 20, fake, fake, 0, None)
    assert rc == 1
    # n_states 0
    rc = L.pkc_merge_states(fake, fake, fake, fake, 4, 0, 2, 128, 0, None)
    assert rc == 1
    # a plan made for another batch size
    buf = pkc.plan([5, 6, 7], 4)
    rc = L.pkc_paged_decode_state(fake, fake, fake, fake, 4, fake, 2, 8, 8, 128, 16, 10, 1.0,
                                  ctypes.c_void_p(buf.ctypes.data), ws, 1 << 24, fake, fake, 1,
                                  None)
    assert rc == 7 and b"plan" in L.pkc_last_error()


def test_fp8_decode_and_kernel_switch_reject_bad_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x100000)
    args = [fake, fake, fake, fake, 4, fake, 2, 8, 8, 128, 16, 10, 1.0]
    # scales must be finite and positive
    for ks, vs in [(0.0, 1.0), (1.0, -2.0), (float("nan"), 1.0), (1.0, float("inf"))]:
        rc = L.pkc_paged_decode_state_fp8(*args, ks, vs, None, ws, 1 << 20, fake, fake, None)
        assert rc == 1 and b"scale" in L.pkc_last_error()
    # page size 12 (not a power of two) is valid but unsupported for fp8
    rc = L.pkc_paged_decode_state_fp8(fake, fake, fake, fake, 4, fake, 2, 8, 8, 128, 12, 10,
                                      1.0, 1.0, 1.0, None, ws, 1 << 20, fake, fake, None)
    assert rc == 2 and b"page_size" in L.pkc_last_error()
    # one KV head with 4-slot pages: a slice is less than one swizzle atom
    rc = L.pkc_paged_decode_state_fp8(fake, fake, fake, fake, 4, fake, 2, 2, 1, 128, 4, 10,
                                      1.0, 1.0, 1.0, None, ws, 1 << 20, fake, fake, None)
    assert rc == 2
    # head_dim 64 is unsupported here too
    rc = L.pkc_paged_decode_state_fp8(fake, fake, fake, fake, 4, fake, 2, 8, 8, 64, 16, 10,
                                      1.0, 1.0, 1.0, None, ws, 1 << 20, fake, fake, None)
    assert rc == 2
    for bad in (-1, 3, 7):
        assert L.pkc_set_decode_kernel(bad) == 1
    for ok in (1, 2, 0):  # leaves the automatic choice set
        assert L.pkc_set_decode_kernel(ok) == 0
    for bad in (-1, 2):
        assert L.pkc_set_decode_schedule(bad) == 1
    for ok in (0, 1):  # leaves the dynamic schedule set
        assert L.pkc_set_decode_schedule(ok) == 0
    assert L.pkc_last_launch_blocks(None, None) == 1
    assert L.pkc_set_prefix_ctas(-1) == 1
    for ok in (40, 0):  # leaves the automatic prefix block count set
        assert L.pkc_set_prefix_ctas(ok) == 0


def test_append_kv_rejects_bad_arguments(L):
    fake = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x100000)
    args = (fake, fake, fake, fake, fake, 4, fake, None, 2, 8)
    assert L.pkc_append_kv(*args, 64, 16, 10, 1, ws, 1 << 20, None) == 2   # head_dim
    assert L.pkc_append_kv(*args, 128, 16, 10, 0, ws, 1 << 20, None) == 1  # fp32 cache
    assert L.pkc_append_kv(*args, 128, 0, 10, 1, ws, 1 << 20, None) == 1   # page_size
    assert L.pkc_append_kv(*args, 128, 16, 10, 1, ws, 16, None) == 3       # workspace
    mis = ctypes.c_void_p(0x1008)
    assert L.pkc_append_kv(mis, fake, fake, fake, fake, 4, fake, None, 2, 8, 128, 16, 10, 1,
                           ws, 1 << 20, None) == 1                         # alignment
    assert L.pkc_append_kv(*args[:8], 0, 8, 128, 16, 10, 1, ws, 1 << 20, None) == 0  # empty


def test_workspace_size_matches_documented_layout(L):
    def al(x):
        return (x + 255) // 256 * 256
    B, H, D, C, S = 7, 32, 128, 148, 3
    words = pkc.plan_words(B, C)
    # status, plan, suffix states, chunk partials, arrival counters, prefix splits
    want = 256 + al(4 * words) + al(4 * B * H * D) + al(4 * B * H) + al(4 * 2 * C * H * D) \
        + al(4 * 2 * C * H) + al(4 * B * H) + S * (al(4 * B * H * D) + al(4 * B * H))
    assert pkc.workspace_size(B, H, C, S) == want
    assert pkc.workspace_size(B, H, 0, 0) == 256 + al(4 * B * H * D) + al(4 * B * H) + al(4 * B * H)


def _compare_plans(kv, C, T=1, qo=None, alpha=1.0, beta=1.0):
    ref = oracle.plan_ref(qo if qo is not None else [1] * len(kv), kv, T, C, alpha, beta)
    got = pkc.plan_dict(pkc.plan(kv, C, tile_q=T, qo_len=qo, alpha=alpha, beta=beta))
    assert got["header"]["MAGIC"] == pkc.PLAN_MAGIC
    assert got["kv_chunk"] == ref["kv_chunk"]
    assert got["work"] == [tuple(w) for w in ref["work"]]
    assert got["cta_work"] == ref["cta_work"]
    assert got["partial"] == ref["partial"]
    assert got["split_units"] == ref["split_units"]
    assert got["empty_units"] == ref["empty_units"]
    assert got["cta_cost"] == ref["cta_cost"]
    assert got["n_partials"] == ref["n_partials"]
    assert got["unit_req"] == [u[0] for u in ref["units"]]
    assert got["unit_qtile"] == [u[1] for u in ref["units"]]
    assert got["unit_n_chunks"] == [len(c) for c in ref["unit_chunks"]]
    # the step-4 order and its records (the dynamic decode's queue)
    assert got["order"] == ref["order"]
    assert got["order_rec"] == [(ref["work"][w][0], ref["work"][w][1], ref["work"][w][2], ref["partial"][w])
                                for w in ref["order"]]
    return got


@pytest.mark.parametrize("seed", range(25))
def test_plan_equals_oracle_random(L, seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 300))
    kv = rng.integers(0, 20000, size=n).tolist()
    if seed % 5 == 0:
        kv[: n // 3] = [0] * (n // 3)
    C = int(rng.integers(1, 300))
    T = int(rng.choice([1, 1, 1, 4, 128]))
    qo = None if T == 1 else rng.integers(1, 400, size=n).tolist()
    _compare_plans(kv, C, T, qo, float(rng.choice([1.0, 0.25, 3.0])), float(rng.choice([1.0, 2.0])))


def test_plan_equals_oracle_on_every_workload(L):
    for name in ["tiny_cascade", "paged_decode", "cascade_long_prompt", "gqa_cascade_lb"]:
        w = workloads.WORKLOADS[name]
        lens = workloads.suffix_lengths(w["suffix"], w["batch"], np.random.default_rng(w["seed"]))
        _compare_plans(lens.tolist(), w.get("num_ctas", 148), 1, None,
                       w.get("alpha", 1.0), w.get("beta", 1.0))
        if name == "gqa_cascade_lb":  # over 148 CTAs, the values the oracle's plan tests pin
            got = _compare_plans(lens.tolist(), 148, 1, None, w["alpha"], w["beta"])
            assert got["kv_chunk"] == 2974 and len(got["split_units"]) == 37


def test_plan_is_deterministic(L):
    a = pkc.plan(list(range(100)), 17)
    b = pkc.plan(list(range(100)), 17)
    assert np.array_equal(a, b)


def test_plan_rejects_bad_input(L):
    with pytest.raises(pkc.PkcError):
        pkc.plan([3, -1], 4)
    with pytest.raises(pkc.PkcError):
        pkc.plan([3, 1], 0)


def test_binding_refuses_negative_prefix_block_count():
    with pytest.raises(ValueError):
        pkc.set_prefix_ctas(-1)


def test_binding_refuses_host_tensors_before_any_call():
    """The binding passes raw pointers down: host tensors (or tensors of the
    wrong shape or dtype) are refused in Python, before the library is called."""
    import torch
    q = torch.zeros(2, 8, 128, dtype=torch.float16)
    kc = torch.zeros(4, 16, 2, 128, dtype=torch.float16)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    sl = torch.zeros(2, dtype=torch.int32)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        pkc.paged_decode_state(q, kc, kc, bt, sl, 0.1, ws)
    with pytest.raises(TypeError, match="dtype"):
        pkc.merge_state(torch.zeros(2, 2, 128, dtype=torch.int32), None, None, None)
    with pytest.raises(ValueError, match="shape"):
        pkc.merge_states(torch.zeros(2, 128), None)
