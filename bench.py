#!/usr/bin/env python
"""Cascade decode benchmark: µs/step and effective KV GB/s on GB300.

One step = one pass of the whole hot path over one batch of decode queries:
the host plan (load-balanced KV chunks over CTAs), its upload, the prefix
states on the tensor cores, the paged suffix decode, and the contraction +
merge into the final O / LSE.  Inputs are resident in HBM before timing.

Default workload "gqa_cascade_lb": batch 256, 32 query / 8 KV heads x 128,
bf16, page size 16, 4 shared prefixes of 8192 tokens (64 requests each),
suffix lengths clip(rint(lognormal(7, 1)), 16, 16384) (440,093 tokens at
seed 5), plan over 148 CTAs with alpha = beta = 1.  One step reads 1.94 GB,
more than the 129 MB L2, so no flush is needed between steps.

Prints one JSON line (rank 0).  `--impl reference` times the float64 CPU
oracle instead, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["pkc", "reference"], default="pkc")
    ap.add_argument("--workload", default="gqa_cascade_lb",
                    choices=["gqa_cascade_lb", "cascade_long_prompt", "tiny_cascade",
                             "paged_decode", "paged_decode_gqa", "paged_decode_fp8", "merge",
                             "gqa_cascade_3level", "gqa_cascade_paged_prefix"],
                    help="cascade workloads time the whole step; 'paged_decode*' time the "
                         "non-cascade decode (fp16 MHA, fp16 GQA, fp8-KV GQA) and 'merge' the "
                         "binary / 16-ary merge kernels (auxiliary lines)")
    ap.add_argument("--decode-kernel", choices=["auto", "simt", "mma"], default="auto",
                    help="paged-decode kernel for a 16-bit cache (auto: tensor cores for "
                         "grouped heads)")
    ap.add_argument("--decode-schedule", choices=["dynamic", "static"], default="dynamic",
                    help="planned decode: blocks take the plan's chunks from a shared "
                         "longest-first queue (dynamic) or run their CTA's plan list (static)")
    ap.add_argument("--num-ctas", type=int, default=None,
                    help="CTAs of the host plan (default: the workload's)")
    ap.add_argument("--prefix-ctas", type=int, default=0,
                    help="thread blocks of the prefix stage (0: automatic, pkc_set_prefix_ctas)")
    ap.add_argument("--batch", type=int, default=None,
                    help="keep only the first N requests (and their prefix groups); "
                         "a smaller case of the same workload, for profiling")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value, dist, device):
    """Largest `value` over all ranks (every rank gets it); the value itself
    when running alone.  Used for the timed region: the job is as slow as its
    slowest replica."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step, steps, world, elapsed_s):
    """Whole-job effective throughput: every replica processes the same
    per-GPU workload (weak scaling), so N replicas move N times the bytes in
    the slowest replica's time."""
    return world * bytes_per_step * steps / elapsed_s / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def host_plan(pkc, lens, num_ctas, cfg, out=None):
    """The step's host plan, or None where the workload decodes without one
    (one block per (request, KV-head group), scheduled by the hardware)."""
    if not num_ctas:
        return None
    return pkc.plan(lens, num_ctas, alpha=cfg["alpha"], beta=cfg["beta"], out=out)


def upload_plan(pkc, buf, ws, stream=None):
    if buf is not None:
        pkc.plan_upload(buf, ws, stream=stream)


def workload_cfg(name, batch=None):
    cfg = dict(workloads.WORKLOADS[name])
    cfg.setdefault("num_ctas", 148)
    if not cfg.get("plan", True):
        cfg["num_ctas"] = 0
    cfg.setdefault("alpha", 1.0)
    cfg.setdefault("beta", 1.0)
    if batch is not None and batch < cfg["batch"]:
        lens, groups, left = [], [], batch
        for L, g in zip(cfg["prefix_lens"], cfg["prefix_groups"]):
            if left <= 0:
                break
            lens.append(L)
            groups.append(min(g, left))
            left -= g
        cfg.update(batch=batch, prefix_lens=lens, prefix_groups=groups)
    return cfg


def make_workload(name, batch=None):
    cfg = workload_cfg(name, batch)
    return cfg, workloads.make_problem(**cfg)


def kv_bytes_per_token(p):
    return 2 * p["num_kv_heads"] * p["q"].shape[2] * p["q"].dtype.itemsize


def kernel_source_sha(src_file):
    """First 16 hex digits of sha256 over a kernel's source file and the
    library's headers it includes (any change to them invalidates a record)."""
    import hashlib
    csrc = os.path.join(ROOT, "paged_kv_cascade_gb300", "csrc")
    h = hashlib.sha256()
    for name in [src_file] + sorted(f for f in os.listdir(csrc) if f.endswith((".h", ".cuh"))):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def kernel_traffic(kernel, workload):
    """Per-launch DRAM bytes from a committed ncu summary, if its recorded
    source hash matches the current kernel source and it was recorded on
    this workload; else None."""
    import hashlib
    src_file = {"paged_decode_kernel": "decode.cu", "paged_decode_mma_kernel": "decode_mma.cu",
                "prefix_state_kernel": "prefix.cu"}.get(kernel)
    summ = os.path.join(ROOT, "profiles", f"{kernel}_traffic.md")
    if not src_file or not os.path.exists(summ):
        return None
    sha = kernel_source_sha(src_file)
    rec = {}
    for line in open(summ):
        if line.startswith("traffic_record:"):
            for kv in line.split(":", 1)[1].split():
                k, _, v = kv.partition("=")
                rec[k] = v
    if rec.get("source_sha") != sha or rec.get("workload") != workload:
        return None
    try:
        return {"bytes_per_launch": float(rec["dram_bytes_per_launch"]),
                "workload": rec["workload"], "scaled": rec.get("scaled", "no")}
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", f"pkc_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def gpu_smi_id(torch, local):
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[local] if vis else local


def cpu_oracle_sample(p, target_s, rows_total_cap=None, n_threads=0):
    """Time the oracle on a bounded sample of (request, head) rows (all host
    cores, or n_threads)."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from pkc_testing import oracle_args
    B, Hq, _ = p["q"].shape
    args = oracle_args(p)
    threads = n_threads or oracle.max_threads()
    rng = np.random.default_rng(123)
    order = rng.permutation(B * Hq)
    n = min(32, B * Hq)
    rows = np.stack([order[:n] // Hq, order[:n] % Hq], 1).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attention_rows(p["q"], rows=rows, n_threads=n_threads, **args)
    t_cal = time.perf_counter() - t0
    n2 = int(min(B * Hq, max(n, n * target_s / max(t_cal, 1e-6))))
    rows = np.stack([order[:n2] // Hq, order[:n2] % Hq], 1).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attention_rows(p["q"], rows=rows, n_threads=n_threads, **args)
    t = time.perf_counter() - t0
    return n2, B * Hq, t, threads


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg, p = make_workload(args.workload, args.batch)
    eff = workloads.effective_bytes(p)
    per_step_s = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    times, fracs = [], []
    n_rows = total = threads = 0
    for i in range(args.warmup + args.steps):
        n_rows, total, t, threads = cpu_oracle_sample(p, per_step_s)
        if i >= args.warmup:
            times.append(t)
            fracs.append(n_rows / total)
    # seconds for one full step, extrapolated from each sampled fraction
    full = [t / f for t, f in zip(times, fracs)]
    ms = 1e3 * sum(full) / len(full)
    value = eff / (ms / 1e3) / 1e9
    line = {
        "impl": "reference",
        "metric": "cascade decode effective KV throughput",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "batch": cfg["batch"],
                   "num_qo_heads": cfg["hq"], "num_kv_heads": cfg["hkv"], "head_dim": cfg["d"],
                   "page_size": cfg["page_size"], "prefix_lens": cfg["prefix_lens"],
                   "suffix_tokens": int(p["cache_seqlens"].sum()), "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_rows} of {total} (request, head) rows per step, "
                                   "extrapolated to the full step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_region(torch, fn, steps, warmup):
    """Mean ms of fn() over `steps` launches, CUDA events on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_aux(args):
    """Auxiliary single-kernel lines: merge kernels, non-cascade decode."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cascade_gb300 as pkc
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from pkc_testing import dev, to_device
    hbm_peak, _, peak_kind = load_peaks()
    K, W = max(args.steps, 3), max(args.warmup, 3)
    if args.workload == "merge":
        w = workloads.workload("merge")
        va, sa, vb, sb = dev(w["v_a"]), dev(w["s_a"]), dev(w["v_b"]), dev(w["s_b"])
        vn, sn = dev(w["v_n"]), dev(w["s_n"])
        vo, so = torch.empty_like(va), torch.empty_like(sa)
        T, H, D = va.shape
        n = vn.shape[1]
        ms2 = time_region(torch, lambda: pkc.merge_state(va, sa, vb, sb, vo, so), K, W)
        msn = time_region(torch, lambda: pkc.merge_states(vn, sn, vo, so), K, W)
        b2 = 3 * T * H * (D + 1) * 4       # read 2 states, write 1
        bn = (n + 1) * T * H * (D + 1) * 4  # read n states, write 1
        line = {"metric": "merge_state effective HBM throughput", "unit": "GB/s",
                "value": b2 / (ms2 / 1e3) / 1e9, "us": 1e3 * ms2, "bytes": b2,
                "frac": b2 / (ms2 / 1e3) / 1e9 / hbm_peak,
                "n_ary": {"n": n, "value": bn / (msn / 1e3) / 1e9, "us": 1e3 * msn, "bytes": bn,
                          "frac": bn / (msn / 1e3) / 1e9 / hbm_peak},
                "peak": hbm_peak, "peak_source": f"{peak_kind} hbm_gbs", "steps": K, "warmup": W,
                "dtype": "f32", "data": "synthetic",
                "config": {"workload": "merge", "tokens": T, "heads": H, "head_dim": D,
                           "l2": "inputs larger than L2 (203 MB / 1.15 GB)"}}
    else:  # paged_decode*: non-cascade decode through the plan
        cfg = workload_cfg(args.workload)
        if args.num_ctas is not None:
            cfg["num_ctas"] = args.num_ctas
        p = workloads.make_problem(**cfg)
        d = to_device(p)
        fp8 = p["kv_dtype"] == "e4m3"
        pkc.set_decode_kernel(args.decode_kernel)
        pkc.set_decode_schedule(args.decode_schedule)
        B, Hq, D = p["q"].shape
        C = cfg["num_ctas"]
        ws = torch.empty(pkc.workspace_size(B, Hq, C, 0), dtype=torch.uint8, device="cuda")
        pkc.workspace_init(ws)
        buf = pkc.plan(p["cache_seqlens"], C)
        pkc.plan_upload(buf, ws)
        o = torch.empty_like(d["q"])
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        if fp8:
            call = lambda: pkc.paged_decode_state_fp8(
                d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"],
                p["sm_scale"], ws, k_scale=p["k_scale"], v_scale=p["v_scale"], plan_buf=buf,
                o=o, lse=lse)
        else:
            call = lambda: pkc.paged_decode_state(
                d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"],
                p["sm_scale"], ws, plan_buf=buf, o=o, lse=lse)
        ms = time_region(torch, call, K, W)
        if pkc.device_status(ws) != 0:
            raise RuntimeError("device status not OK")
        eff = workloads.effective_bytes(p)
        line = {"metric": "paged decode (non-cascade) effective KV throughput", "unit": "GB/s",
                "value": eff / (ms / 1e3) / 1e9, "us": 1e3 * ms, "bytes": eff,
                "frac": eff / (ms / 1e3) / 1e9 / hbm_peak, "peak": hbm_peak,
                "peak_source": f"{peak_kind} hbm_gbs", "steps": K, "warmup": W,
                "dtype": cfg["dtype"], "data": "synthetic",
                "config": {"workload": args.workload, "batch": B, "num_qo_heads": Hq,
                           "num_kv_heads": p["num_kv_heads"], "kv_dtype": p["kv_dtype"],
                           "kv_tokens": int(p["cache_seqlens"].sum()), "num_ctas": C,
                           "decode_kernel": "mma" if fp8 else args.decode_kernel,
                           "decode_schedule": args.decode_schedule,
                           "launches": "decode + contraction"}}
    print(json.dumps(line), flush=True)


def run_cascade_variant(args):
    """Auxiliary cascade lines: the three-level cascade, and the two-level
    cascade with its prefixes read in place from the page pool (timed beside
    the contiguous-prefix call on the same tokens)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cascade_gb300 as pkc
    pkc.set_prefix_ctas(args.prefix_ctas)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from pkc_testing import dev, to_device
    hbm_peak, _, peak_kind = load_peaks()
    K, W = max(args.steps, 3), max(args.warmup, 3)
    paged = args.workload == "gqa_cascade_paged_prefix"
    cfg = workload_cfg("gqa_cascade_lb" if paged else args.workload)
    if args.num_ctas is not None:
        cfg["num_ctas"] = args.num_ctas
    p = workloads.make_problem(**cfg)
    d = to_device(p)
    B, Hq, D = p["q"].shape
    C = cfg["num_ctas"]
    ws = torch.empty(pkc.workspace_size(B, Hq, C, 64), dtype=torch.uint8, device="cuda")
    pkc.workspace_init(ws)
    buf = pkc.plan(p["cache_seqlens"], C)
    pkc.plan_upload(buf, ws)
    o = torch.empty_like(d["q"])
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    eff = workloads.effective_bytes(p)
    extra = {}
    if paged:
        kc, vc, pages, page_indptr = workloads.pool_prefixes(p, 5, poison=False)
        kc, vc, pages = dev(kc), dev(vc), dev(pages)
        ind = p["prefix_req_indptr"]
        ranges = [(int(ind[j]), int(ind[j + 1])) for j in range(len(ind) - 1)]
        call = lambda: pkc.cascade_decode_paged_prefix(
            d["q"], pages, page_indptr, p["prefix_kv_indptr"], ranges, kc, vc, d["block_table"],
            d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf, o=o, lse=lse)
        ms_contig = time_region(torch, lambda: pkc.cascade_decode(
            d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], p["prefix_req_indptr"],
            d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws,
            plan_buf=buf, o=o, lse=lse), K, W)
        extra = {"contiguous_prefix_us": 1e3 * ms_contig,
                 "contiguous_prefix_value": eff / (ms_contig / 1e3) / 1e9}
        metric = "cascade decode effective KV throughput, prefix read from the page pool"
    else:
        ranges = cfg["prefix_ranges"]
        call = lambda: pkc.cascade_decode_multilevel(
            d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], ranges, d["k_cache"],
            d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf,
            o=o, lse=lse)
        metric = "three-level cascade decode effective KV throughput"
    ms = time_region(torch, call, K, W)
    if pkc.device_status(ws) != 0:
        raise RuntimeError("device status not OK")
    line = {"metric": metric, "unit": "GB/s", "value": eff / (ms / 1e3) / 1e9, "us": 1e3 * ms,
            "bytes": eff, "frac": eff / (ms / 1e3) / 1e9 / hbm_peak, "peak": hbm_peak,
            "peak_source": f"{peak_kind} hbm_gbs", "steps": K, "warmup": W, "dtype": cfg["dtype"],
            "data": "synthetic", "launch": "direct (prefix, decode, contraction)",
            "config": {"workload": args.workload, "batch": B, "num_qo_heads": Hq,
                       "num_kv_heads": p["num_kv_heads"], "prefix_lens": cfg["prefix_lens"],
                       "prefix_ranges": ranges, "suffix_tokens": int(p["cache_seqlens"].sum()),
                       "num_ctas": C}}
    line.update(extra)
    print(json.dumps(line), flush=True)


def run_e2e(torch, pkc, p, d, cfg, eff, steps, num_ctas, world, dist):
    """Effective GB/s through the public API with host buffers.

    Every step copies its inputs (q, block table, lengths, plan) in from
    pinned host memory, runs the cascade (replayed from a CUDA graph), and
    copies O and LSE back; the host reads each step's result.  Two buffer
    sets alternate so the host prepares step i+1 while the GPU runs step i;
    a set is reused only after its previous result has been read.
    """
    B, Hq, D = p["q"].shape
    words = pkc.plan_words(B, num_ctas) if num_ctas else 1
    q_h = torch.from_numpy(p["q"].view(np.int16) if p["q"].dtype == np.uint16 else p["q"]).pin_memory()
    bt_h = torch.from_numpy(p["block_table"]).pin_memory()
    sl_h = torch.from_numpy(p["cache_seqlens"]).pin_memory()
    stream = torch.cuda.Stream()
    copy_stream = torch.cuda.Stream()  # inputs in
    out_stream = torch.cuda.Stream()   # results out
    sets = []
    for _ in range(2):
        st = {"q": torch.empty_like(d["q"]), "bt": torch.empty_like(d["block_table"]),
              "sl": torch.empty_like(d["cache_seqlens"]),
              "ws": torch.empty(pkc.workspace_size(B, Hq, num_ctas, 64), dtype=torch.uint8,
                                device=d["q"].device),
              "o": torch.empty_like(d["q"]),
              "lse": torch.empty((B, Hq), dtype=torch.float32, device=d["q"].device),
              "plan": torch.empty(words, dtype=torch.int32).pin_memory(),
              "o_h": torch.empty(d["q"].shape, dtype=d["q"].dtype).pin_memory(),
              "lse_h": torch.empty((B, Hq), dtype=torch.float32).pin_memory(),
              "done": torch.cuda.Event(), "copied": torch.cuda.Event(), "ran": torch.cuda.Event(),
              "pending": False}
        pkc.workspace_init(st["ws"])
        sets.append(st)

    def qview(t):
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t

    def enqueue(st):
        # inputs go in on their own stream so they overlap the other set's run
        buf = host_plan(pkc, sl_h.numpy(), num_ctas, cfg, out=st["plan"].numpy())
        with torch.cuda.stream(copy_stream):
            qview(st["q"]).copy_(q_h, non_blocking=True)
            st["bt"].copy_(bt_h, non_blocking=True)
            st["sl"].copy_(sl_h, non_blocking=True)
            upload_plan(pkc, buf, st["ws"], stream=copy_stream)
            st["copied"].record(copy_stream)
        stream.wait_event(st["copied"])
        return buf

    with torch.cuda.stream(stream):
        for st in sets:  # capture one graph per buffer set
            buf = enqueue(st)

            def run(st=st, buf=buf):
                pkc.cascade_decode(st["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                   p["prefix_req_indptr"], d["k_cache"], d["v_cache"], st["bt"],
                                   st["sl"], p["sm_scale"], st["ws"], plan_buf=buf, o=st["o"],
                                   lse=st["lse"], stream=stream)
            run()
            stream.synchronize()
            st["graph"] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(st["graph"], stream=stream):
                run()
        checksum = 0.0

        def step(i):
            nonlocal checksum
            st = sets[i & 1]
            if st["pending"]:  # read this set's previous result before reusing it
                st["done"].synchronize()
                checksum += float(st["lse_h"][0, 0])
            enqueue(st)
            st["graph"].replay()
            # the result goes out on its own copy stream, overlapping the
            # other set's step on the compute stream and its input copies
            st["ran"].record(stream)
            out_stream.wait_event(st["ran"])
            with torch.cuda.stream(out_stream):
                st["o_h"].copy_(st["o"], non_blocking=True)
                st["lse_h"].copy_(st["lse"], non_blocking=True)
                st["done"].record(out_stream)
            st["pending"] = True

        def drain():
            nonlocal checksum
            for st in sets:
                if st["pending"]:
                    st["done"].synchronize()
                    checksum += float(st["lse_h"][0, 0])
                    st["pending"] = False

        for i in range(4):
            step(i)
        drain()
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        for i in range(steps):
            step(i)
        drain()
        t = reduce_max(time.perf_counter() - t0, dist, d["q"].device)
    for st in sets:
        if pkc.device_status(st["ws"]) != 0:
            raise RuntimeError("device status not OK after the e2e run")
    h2d = q_h.numel() * q_h.element_size() + bt_h.numel() * 4 + sl_h.numel() * 4 + (words * 4 if num_ctas else 0)
    d2h = sets[0]["o_h"].numel() * sets[0]["o_h"].element_size() + sets[0]["lse_h"].numel() * 4
    return {"value": whole_job_gbs(eff, steps, world, t), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": 1e3 * t / steps, "steps": steps,
            "note": "pinned host inputs in, O/LSE out and read every step; two buffer sets "
                    "alternate, inputs in and results out on two copy streams, so host work "
                    "and copies overlap the other set's step"}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload in ("gqa_cascade_3level", "gqa_cascade_paged_prefix"):
        run_cascade_variant(args)
        return
    if args.workload == "merge" or args.workload.startswith("paged_decode"):
        run_aux(args)
        return
    import torch
    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    if dist is None or rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()
    import paged_kv_cascade_gb300 as pkc
    pkc.set_decode_kernel(args.decode_kernel)
    pkc.set_decode_schedule(args.decode_schedule)
    pkc.set_prefix_ctas(args.prefix_ctas)

    cfg, p = make_workload(args.workload, args.batch)
    if args.num_ctas is not None:
        cfg["num_ctas"] = args.num_ctas
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from pkc_testing import to_device
    d = to_device(p, f"cuda:{local}")
    B, Hq, D = p["q"].shape
    num_ctas = cfg["num_ctas"]
    lens = p["cache_seqlens"]
    ws = torch.empty(pkc.workspace_size(B, Hq, num_ctas, 64), dtype=torch.uint8, device=d["q"].device)
    pkc.workspace_init(ws)
    words = pkc.plan_words(B, num_ctas) if num_ctas else 1
    pinned = [torch.empty(words, dtype=torch.int32).pin_memory() for _ in range(2)]
    plan_np = [t.numpy() for t in pinned]
    o = torch.empty_like(d["q"])
    lse = torch.empty((B, Hq), dtype=torch.float32, device=d["q"].device)

    host_plan_s = []
    # A pinned plan buffer is rewritten only after the previous upload from
    # it has run on the GPU (the host runs ahead of the device).
    uploaded = [torch.cuda.Event(), torch.cuda.Event()]

    def step(i):
        uploaded[i & 1].synchronize()
        t0 = time.perf_counter()
        buf = host_plan(pkc, lens, num_ctas, cfg, out=plan_np[i & 1])
        host_plan_s.append(time.perf_counter() - t0)
        upload_plan(pkc, buf, ws)
        uploaded[i & 1].record()
        pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                           p["prefix_req_indptr"], d["k_cache"], d["v_cache"], d["block_table"],
                           d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf, o=o, lse=lse)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    status = pkc.device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status after warm-up: {pkc.STATUS_NAMES.get(status, status)}")
    host_plan_s.clear()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for e in ev:  # torch creates the CUDA event on first record
        for x in e:
            x.record()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_smi_id(torch, local))
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    start.record()
    for i in range(K):
        pkc.set_stage_events(ev[i])
        step(i)
    end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    elapsed_ms = reduce_max(start.elapsed_time(end), dist, d["q"].device)
    status = pkc.device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status after timing: {pkc.STATUS_NAMES.get(status, status)}")

    stage_ms = {
        "prefix_state": statistics.mean(e[0].elapsed_time(e[1]) for e in ev),
        "paged_decode": statistics.mean(e[1].elapsed_time(e[2]) for e in ev),
        "contraction": statistics.mean(e[2].elapsed_time(e[3]) for e in ev),
    }
    eff = workloads.effective_bytes(p)
    direct_ms_per_step = elapsed_ms / K

    hbm_peak, tf_peak, peak_kind = load_peaks()
    kvb = kv_bytes_per_token(p)
    suffix_tokens = int(lens.sum())
    prefix_tokens = int(p["prefix_kv_indptr"][-1])
    dominant = max(stage_ms, key=stage_ms.get)
    if dominant == "prefix_state":
        alg_bytes = prefix_tokens * kvb
        unit_desc = f"{kvb} B per shared-prefix token x {prefix_tokens} tokens"
    else:
        dominant = "paged_decode"
        alg_bytes = suffix_tokens * kvb
        unit_desc = f"{kvb} B per suffix token x {suffix_tokens} tokens"
    achieved = alg_bytes / (stage_ms[dominant] / 1e3) / 1e9
    # the decode kernel the library picks (pkc_set_decode_kernel semantics)
    G = Hq // p["num_kv_heads"]
    mma = args.decode_kernel == "mma" or (args.decode_kernel == "auto" and G >= 2)
    kernel_name = {"prefix_state": "prefix_state_kernel"}.get(
        dominant, "paged_decode_mma_kernel" if mma else "paged_decode_kernel")
    tr = kernel_traffic(kernel_name, args.workload if args.batch is None else None)
    # prefix stage on the tensor cores: FLOPs 4*D per (row, prefix token)
    rows_per_prefix = np.diff(p["prefix_req_indptr"]) * (Hq // p["num_kv_heads"])
    prefix_flops = float(4 * D * np.sum(rows_per_prefix * np.diff(p["prefix_kv_indptr"])) *
                         p["num_kv_heads"])

    # ---- the same step with the device work replayed from a CUDA graph ----
    # The plan still runs on the host and is uploaded every step (outside the
    # graph); the captured cascade call reads it from its workspace.  Two
    # workspaces and two graphs alternate, so that step i+1's plan upload (on
    # a copy stream) overlaps step i's device work; a workspace's plan is
    # overwritten only after the graph that read it has run.
    graph = None
    try:
        gstream, cstream = torch.cuda.Stream(), torch.cuda.Stream()
        gplan = [torch.empty(words, dtype=torch.int32).pin_memory() for _ in range(2)]
        gplan_np = [t.numpy() for t in gplan]
        gws = [ws, torch.empty_like(ws)]
        pkc.workspace_init(gws[1])
        gdone = [torch.cuda.Event(), torch.cuda.Event()]      # graph s has run
        uploaded = [torch.cuda.Event(), torch.cuda.Event()]   # plan s is on the GPU
        graphs = []
        with torch.cuda.stream(gstream):
            for sidx in range(2):
                gbuf = host_plan(pkc, lens, num_ctas, cfg, out=gplan_np[sidx])

                def g_run(sidx=sidx, gbuf=gbuf):
                    pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                       p["prefix_req_indptr"], d["k_cache"], d["v_cache"],
                                       d["block_table"], d["cache_seqlens"], p["sm_scale"], gws[sidx],
                                       plan_buf=gbuf, o=o, lse=lse, stream=gstream)

                upload_plan(pkc, gbuf, gws[sidx], stream=gstream)
                g_run()
                gstream.synchronize()
                cg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(cg, stream=gstream):
                    g_run()
                graphs.append(cg)
            for e in gdone + uploaded:
                e.record(gstream)
            gstream.synchronize()

            def g_step(i):
                sidx = i & 1
                uploaded[sidx].synchronize()  # the pinned plan buffer is free again
                b = host_plan(pkc, lens, num_ctas, cfg, out=gplan_np[sidx])
                cstream.wait_event(gdone[sidx])  # the graph that read this plan has run
                upload_plan(pkc, b, gws[sidx], stream=cstream)
                uploaded[sidx].record(cstream)
                gstream.wait_event(uploaded[sidx])
                graphs[sidx].replay()
                gdone[sidx].record(gstream)

            for i in range(max(3, args.warmup)):
                g_step(i)
            gstream.synchronize()
            if dist is not None:
                dist.barrier()
            ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ga.record(gstream)
            for i in range(K):
                g_step(i)
            gb.record(gstream)
            gstream.synchronize()
            if dist is not None:
                dist.barrier()
            # Single replays with and without an L2 flush (a 256 MB write)
            # before each, timed alone: the median step with a cold L2 and
            # with whatever the previous step left in it.
            flush = torch.empty((256 << 20) // 4, dtype=torch.int32, device=d["q"].device)
            n_iso = min(K, 50)
            iso = {}
            for flushed in (True, False):
                evs = []
                for i in range(n_iso):
                    if flushed:
                        flush.fill_(i)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(gstream)
                    graphs[i & 1].replay()
                    e1.record(gstream)
                    evs.append((e0, e1))
                gstream.synchronize()
                iso[flushed] = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
        g_ms = reduce_max(ga.elapsed_time(gb), dist, d["q"].device)
        graph = {"value": whole_job_gbs(eff, K, world, g_ms / 1e3), "unit": "GB/s",
                 "us_per_step": 1e3 * g_ms / K,
                 "note": "host plan + upload each step (on a copy stream, two workspaces "
                         "alternating), device work replayed from a CUDA graph",
                 "isolated_replay_us_median": {"l2_flushed": iso[True], "unflushed": iso[False],
                                               "flush_bytes": 256 << 20, "replays": n_iso}}
        if pkc.device_status(gws[0]) != 0 or pkc.device_status(gws[1]) != 0:
            raise RuntimeError("device status after graph replay")
    except RuntimeError:
        raise
    except Exception as exc:  # graph capture unavailable: report why
        graph = {"unavailable": str(exc)[:200]}
    clocks = sampler.stop()
    # Headline: the graph-replayed step (how the pages run it: plan per step
    # on the CPU, the captured run replayed); the directly launched,
    # event-instrumented run gives the per-stage times.
    if graph and "us_per_step" in graph:
        mode, ms_per_step = "cuda_graph", graph["us_per_step"] / 1e3
    else:
        mode, ms_per_step = "direct", direct_ms_per_step
    value = whole_job_gbs(eff, 1, world, ms_per_step / 1e3)

    # ---- e2e through host buffers ----
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(torch, pkc, p, d, cfg, eff, args.e2e_steps, num_ctas, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_rows, total, t, threads = cpu_oracle_sample(p, args.cpu_seconds)
        full_s = t / (n_rows / total)
        n1, _, t1, _ = cpu_oracle_sample(p, args.cpu_seconds / 2, n_threads=1)
        cpu = {"value": eff / full_s / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{n_rows} of {total} (request, head) rows of one step in {t:.1f} s, "
                         "extrapolated to the full step",
               "single_thread": {"value": eff / (t1 / (n1 / total)) / 1e9, "unit": "GB/s", "cores": 1,
                                 "sample": f"{n1} of {total} rows in {t1:.1f} s"}}

    if rank == 0:
        line = {
            "metric": "cascade decode effective KV throughput",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_step": 1e3 * ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg["dtype"], "data": "synthetic",
            "config": {"workload": args.workload, "batch": B, "num_qo_heads": Hq,
                       "num_kv_heads": p["num_kv_heads"], "head_dim": D,
                       "page_size": cfg["page_size"], "prefix_lens": cfg["prefix_lens"],
                       "suffix_tokens": suffix_tokens,
                       "num_ctas": num_ctas or None,
                       "plan": "host plan over num_ctas CTAs" if num_ctas else
                               "none: one decode block per (request, KV-head group)",
                       "effective_bytes_per_step": eff,
                       "l2": "inputs larger than L2 (one step reads %.2f GB)" % (eff / 1e9),
                       "launch": mode, "decode_kernel": args.decode_kernel,
                       "decode_schedule": args.decode_schedule if num_ctas else None,
                       "prefix_ctas": args.prefix_ctas or "auto",
                       "parallelism": f"replicas x{world}"},
            "stage_split": dict(zip(("prefix_blocks", "decode_blocks"), pkc.last_launch_blocks())),
            "direct_us_per_step": 1e3 * direct_ms_per_step,
            "hbm_fraction": value / world / hbm_peak,
            "stages_us": {k: 1e3 * v for k, v in stage_ms.items()},
            "host_plan_us": 1e6 * statistics.mean(host_plan_s) if host_plan_s else None,
            "roofline": {"kernel": kernel_name, "stage": dominant, "bound": "hbm", "achieved": achieved,
                         "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": alg_bytes, "per_unit": unit_desc,
                         "traffic": tr["bytes_per_launch"] if tr else None},
            "prefix_tensor": {"flops_per_launch": prefix_flops,
                              "tflops": prefix_flops / (stage_ms["prefix_state"] / 1e3) / 1e12,
                              "peak_tflops": tf_peak, "peak_source": f"{peak_kind} bf16_tflops"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "graph": graph,
            "gpu_launches": 3 * K,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
