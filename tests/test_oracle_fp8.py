"""Pins of the oracle's FP8 (e4m3) KV cache path (CPU only).

The pages ask for an fp8 KV cache with fp16 queries and outputs (MLSys'25
notes, appendix F) without fixing the format; the oracle decodes OCP E4M3
("e4m3fn") codes and applies one scale per tensor.  Pinned here against
the library's own float8_e4m3fn conversion (all 256 codes), closed-form
values of the format, and invariants of where the scales enter.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads


def _oracle_decode(c):
    return oracle.decode_scalar(int(c), oracle.E4M3)


def _e4m3_ok(decode):
    """The checks a decoder must pass: closed forms and the library cast."""
    closed = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0,
              0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x40: 2.0,
              0x3C: 1.5, 0x77: 240.0, 0x78: 256.0}
    for c, v in closed.items():
        if decode(c) != v:
            return False
    if not (math.isnan(decode(0x7F)) and math.isnan(decode(0xFF))):
        return False
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = lib.to(torch.float64).numpy()
    mine = np.array([decode(c) for c in range(256)])
    same_nan = np.array_equal(np.isnan(ref), np.isnan(mine))
    return bool(same_nan and np.array_equal(ref[~np.isnan(ref)], mine[~np.isnan(mine)]))


def test_e4m3_decoder_matches_closed_forms_and_library_cast():
    assert _e4m3_ok(_oracle_decode)
    assert math.copysign(1.0, _oracle_decode(0x80)) == -1.0  # negative zero


def test_e4m3_decoder_mutants_are_caught():
    def make(bias=7, sub_shift=-9, nan_all=False):
        def dec(c):
            s, e, f = (c >> 7) & 1, (c >> 3) & 15, c & 7
            if e == 15 and (nan_all or f == 7):
                m = math.nan
            elif e == 0:
                m = math.ldexp(f, sub_shift)
            else:
                m = math.ldexp(f + 8, e - bias - 3)
            return -m if s else m
        return dec
    assert _e4m3_ok(make())  # the mutants' own skeleton is right
    assert not _e4m3_ok(make(bias=8))
    assert not _e4m3_ok(make(sub_shift=-10))
    assert not _e4m3_ok(make(nan_all=True))  # e5m2-style special values


def _fp8_problem(**kw):
    cfg = dict(batch=3, hq=8, hkv=2, d=128, dtype="f16", kv_dtype="e4m3",
               prefix_lens=[], prefix_groups=[], suffix=("list", [19, 1, 40]),
               page_size=16, seed=5, k_scale=0.5, v_scale=1.25)
    cfg.update(kw)
    return workloads.make_problem(**cfg)


def _args(p, **over):
    a = dict(sm_scale=p["sm_scale"], num_kv_heads=p["num_kv_heads"], k_cache=p["k_cache"],
             v_cache=p["v_cache"], block_table=p["block_table"],
             cache_seqlens=p["cache_seqlens"], page_size=p["page_size"],
             k_scale=p["k_scale"], v_scale=p["v_scale"])
    a.update(over)
    return a


def test_fp8_cache_equals_f32_cache_of_the_scaled_values():
    # The library cast decodes the codes; the scales 0.5 and 1.25 keep every
    # scaled value exact in float32, so the float32 path must agree exactly
    # (up to float64 summation order, which is the same).
    p = _fp8_problem()
    dec = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    k32 = dec(p["k_cache"]) * np.float32(p["k_scale"])
    v32 = dec(p["v_cache"]) * np.float32(p["v_scale"])
    q32 = p["q"].astype(np.float32)
    o, lse = oracle.attention_rows(p["q"], **_args(p))
    o2, lse2 = oracle.attention_rows(q32, **_args(p, k_cache=k32, v_cache=v32, k_scale=1.0,
                                                  v_scale=1.0))
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def test_k_scale_is_a_score_scale_and_v_scale_an_output_scale():
    p = _fp8_problem(k_scale=1.0, v_scale=1.0)
    base_o, base_lse = oracle.attention_rows(p["q"], **_args(p))
    o, lse = oracle.attention_rows(p["q"], **_args(p, k_scale=2.0))
    o2, lse2 = oracle.attention_rows(p["q"], **_args(p, sm_scale=2.0 * p["sm_scale"]))
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)
    assert np.abs(o - base_o).max() > 1e-3  # the scale does change the scores
    o3, lse3 = oracle.attention_rows(p["q"], **_args(p, v_scale=3.0))
    np.testing.assert_allclose(o3, 3.0 * base_o, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(lse3, base_lse)


def test_fp8_single_token_row_is_that_token():
    # one cached token: O = v_scale * e4m3(v), LSE = the single scaled score
    p = _fp8_problem(suffix=("list", [1, 1, 1]))
    o, lse = oracle.attention_rows(p["q"], **_args(p))
    g = p["q"].shape[1] // p["num_kv_heads"]
    for r, (b, h) in enumerate((b, h) for b in range(3) for h in range(8)):
        page = p["block_table"][b, 0]
        kc, vc = p["k_cache"][page, 0, h // g], p["v_cache"][page, 0, h // g]
        v = np.array([_oracle_decode(c) for c in vc]) * p["v_scale"]
        k = np.array([_oracle_decode(c) for c in kc]) * p["k_scale"]
        s = p["sm_scale"] * float(np.dot(p["q"][b, h].astype(np.float64), k))
        np.testing.assert_allclose(o[r], v, rtol=0, atol=1e-15)
        assert abs(lse[r] - s) < 1e-12


def test_scales_on_a_16bit_cache_are_refused():
    p = workloads.make_problem(batch=1, hq=2, hkv=2, d=128, dtype="f16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", [3]), page_size=16, seed=1)
    with pytest.raises(AssertionError):
        oracle.attention_rows(p["q"], **_args(p, k_scale=2.0))
    with pytest.raises(ValueError):
        workloads.make_problem(batch=1, hq=2, hkv=2, d=128, dtype="bf16", kv_dtype="e4m3",
                               prefix_lens=[], prefix_groups=[], suffix=("list", [3]),
                               page_size=16, seed=1)
