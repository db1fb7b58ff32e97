"""Shared helpers for the GPU parity tests: host arrays -> device tensors,
oracle references for whole problems or sampled rows, and the tolerances.

Tolerances (fp16 / bf16 attention outputs, fp32 accumulation): O max-abs
error <= 2e-3 and LSE max-abs error <= 1e-3 against the float64 oracle.
"""
import json
import math
import os

import numpy as np
import torch

import oracle

O_TOL = 2e-3
LSE_TOL = 1e-3


def dev(a, device="cuda"):
    """numpy host array -> torch device tensor (uint16 arrays hold bf16 bits)."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_device(p, device="cuda"):
    out = {}
    for k in ("q", "k_prefix", "v_prefix", "k_cache", "v_cache", "block_table", "cache_seqlens"):
        out[k] = dev(p[k], device)
    return out


def workspace_for(pkc, p, num_ctas=0, prefix_splits=None, device="cuda"):
    B, Hq, _ = p["q"].shape
    if prefix_splits is None:
        prefix_splits = 64 if p.get("k_prefix") is not None else 0
    nbytes = pkc.workspace_size(B, Hq, num_ctas, prefix_splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    pkc.workspace_init(ws)
    return ws


def oracle_args(p, prefix=True, suffix=True):
    a = dict(sm_scale=p["sm_scale"], num_kv_heads=p["num_kv_heads"])
    if prefix and p.get("k_prefix") is not None:
        a.update(k_prefix=p["k_prefix"], v_prefix=p["v_prefix"],
                 prefix_kv_indptr=p["prefix_kv_indptr"],
                 prefix_req_indptr=p["prefix_req_indptr"])
    if suffix:
        a.update(k_cache=p["k_cache"], v_cache=p["v_cache"], block_table=p["block_table"],
                 cache_seqlens=p["cache_seqlens"], page_size=p["page_size"],
                 k_scale=p.get("k_scale", 1.0), v_scale=p.get("v_scale", 1.0))
    return a


def sample_rows(B, Hq, n, seed=0):
    """n distinct (request, head) rows, always including the corners."""
    rng = np.random.default_rng(seed)
    total = B * Hq
    idx = set(rng.choice(total, size=min(n, total), replace=False).tolist())
    idx |= {0, total - 1, Hq - 1, (B - 1) * Hq}
    idx = np.array(sorted(i for i in idx if i < total))
    return np.stack([idx // Hq, idx % Hq], axis=1).astype(np.int32)


MANTISSA_BITS = {torch.float16: 10, torch.bfloat16: 7, torch.float32: 23}


def half_ulp(x, dtype):
    """Half a unit in the last place of `dtype` at |x| (normal range)."""
    m = MANTISSA_BITS[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -14)))
    return 0.5 * 2.0 ** (e - m)


def compare(o_dev, lse_dev, o_ref, lse_ref, rows=None, o_tol=O_TOL, lse_tol=LSE_TOL):
    """Max-abs errors of device outputs [B, Hq, D] / [B, Hq] vs oracle rows.

    O passes when |O - O_ref| <= o_tol + half an ulp of the output dtype at
    O_ref: the arithmetic error allowed (2e-3) plus the final rounding to
    fp16 / bf16, which no output of that type can avoid.  Returns the
    largest O error beyond that rounding, and the largest LSE error.
    """
    out_dtype = o_dev.dtype
    o = o_dev.float().cpu().numpy().astype(np.float64)
    lse = lse_dev.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        o = o[rows[:, 0], rows[:, 1]]
        lse = lse[rows[:, 0], rows[:, 1]]
    else:
        o = o.reshape(-1, o.shape[-1])
        lse = lse.reshape(-1)
    assert np.all(np.isfinite(o)), "non-finite O"
    empty_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty_ref), "empty-state rows differ"
    excess = np.abs(o - o_ref) - half_ulp(o_ref, out_dtype)
    o_err = float(max(0.0, np.max(excess))) if o.size else 0.0
    fin = ~empty_ref
    lse_err = float(np.max(np.abs(lse[fin] - lse_ref[fin]))) if fin.any() else 0.0
    o_raw = float(np.max(np.abs(o - o_ref))) if o.size else 0.0
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0],
           "rows": int(o.shape[0]), "o_raw_max_abs": o_raw, "o_err_beyond_rounding": o_err,
           "lse_max_abs": lse_err, "o_tol": o_tol, "lse_tol": lse_tol}
    # shown by pytest -rP / -s, and appended to PKC_PARITY_LOG when set
    print("parity " + json.dumps(rec))
    log = os.environ.get("PKC_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps(rec) + "\n")
    assert o_err <= o_tol, (f"O max-abs error beyond output rounding {o_err:.3e} > {o_tol} "
                            f"(raw max-abs {o_raw:.3e})")
    assert lse_err <= lse_tol, f"LSE max-abs error {lse_err:.3e} > {lse_tol}"
    return o_err, lse_err


def f64(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def scale_of(d):
    return 1.0 / math.sqrt(d)
