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

Prints one JSON line (rank 0).  Besides the headline step it carries, timed
in the same process with their own clock records: the pages' static CTA
assignment next to the default dynamic queue, and (`configs`) every other
workload of the set -- the tiny cascade, the binary and 16-ary merge, the
non-cascade paged decode, the long-prompt cascade with the non-cascade
decode of the same problem, the fp8-KV decode, the three-level and the
paged-prefix cascades, and a batch / prefix / suffix sweep of cascade
against non-cascade decode.  `--workload X` prints X's entry alone.
`--impl reference` times the float64 CPU oracle instead, on bounded samples
of the same workload.
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
                    help="headline cascade workload (gqa_cascade_lb, cascade_long_prompt, "
                         "tiny_cascade), or one other workload printed alone: 'paged_decode*' "
                         "(fp16 MHA, fp16 GQA, fp8-KV GQA), 'merge', the 3-level and "
                         "paged-prefix cascades")
    ap.add_argument("--decode-kernel", choices=["auto", "simt", "mma"], default="auto",
                    help="paged-decode kernel for a 16-bit cache (auto: tensor cores for "
                         "grouped heads)")
    ap.add_argument("--decode-schedule", choices=["dynamic", "static"], default="dynamic",
                    help="planned decode: blocks take the plan's chunks from a shared "
                         "longest-first queue (dynamic) or run their CTA's plan list (static)")
    ap.add_argument("--contraction", choices=["fused", "separate", "separate_plain"], default="separate",
                    help="split states contracted inside the attention kernels (fused) or by a "
                         "standalone contraction kernel after them")
    ap.add_argument("--cascade-small", type=int, default=16,
                    help="largest rows per KV head of a prefix group for the one-launch "
                         "small-batch cascade (0: never; pkc_set_cascade_small)")
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
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' entries (`configs`) in the headline line")
    ap.add_argument("--no-ab", action="store_true",
                    help="skip the schedule and contraction comparisons (profiling runs)")
    ap.add_argument("--config-seconds", type=float, default=0.5,
                    help="least timed device time per workload entry")
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


def line_config(name, cfg, p, num_ctas, args, world, extra=None):
    """The `config` object of a JSON line: the same keys for both arms."""
    B, Hq, D = p["q"].shape
    c = {"workload": name, "batch": B, "num_qo_heads": Hq, "num_kv_heads": p["num_kv_heads"],
         "head_dim": D, "page_size": cfg["page_size"], "prefix_lens": list(cfg["prefix_lens"]),
         "suffix_tokens": int(p["cache_seqlens"].sum()), "num_ctas": num_ctas or None,
         "plan": "host plan over num_ctas CTAs" if num_ctas else
                 "none: one decode block per (request, KV-head group)",
         "effective_bytes_per_step": workloads.effective_bytes(p),
         "l2": ("inputs larger than L2 (one step reads %.2f GB)" % (workloads.effective_bytes(p) / 1e9)
                if workloads.effective_bytes(p) > 129e6 else
                "inputs fit in L2 (%.1f MB), no flush: a launch-bound workload, read in us" %
                (workloads.effective_bytes(p) / 1e6)),
         "parallelism": f"replicas x{world}"}
    if extra:
        c.update(extra)
    return c


def run_reference(args):
    """The reference arm: the float64 CPU oracle, as it stands, on the host
    cores.  Each timed step computes a bounded sample of the step's
    (request, head) rows; `value` is the rows' share of the step's effective
    bytes over the measured time, and `ms_per_step` the measured time of the
    sampled step (not an extrapolation)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg, p = make_workload(args.workload, args.batch)
    if args.num_ctas is not None:
        cfg["num_ctas"] = args.num_ctas
    eff = workloads.effective_bytes(p)
    # the whole --steps/--warmup run within about 100 s of oracle time
    per_step_s = max(0.5, min(10.0, 100.0 / max(1, args.steps + args.warmup)))
    times, fracs = [], []
    n_rows = total = threads = 0
    for i in range(args.warmup + args.steps):
        n_rows, total, t, threads = cpu_oracle_sample(p, per_step_s)
        if i >= args.warmup:
            times.append(t)
            fracs.append(n_rows / total)
    secs = sum(times)
    value = sum(eff * f for f in fracs) / secs / 1e9
    ms = 1e3 * secs / len(times)
    line = {
        "impl": "reference",
        "metric": "cascade decode effective KV throughput",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(args.workload, cfg, p, cfg["num_ctas"], args, world),
        "impl_config": {"step": "a sample of the step's (request, head) rows, every prefix and "
                                "suffix token of each, float64 on the host cores"},
        "sample_fraction": statistics.mean(fracs),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_rows} of {total} (request, head) rows per step, "
                                   f"{args.steps} timed steps; value = the sampled rows' share "
                                   "of the effective bytes over the measured time"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class GraphStepper:
    """One step = host plan + its upload + the device work replayed from a
    CUDA graph (how the pages run it: the plan per step on the CPU, copied
    in asynchronously, the captured run replayed).

    Two workspaces and two captured graphs alternate.  The plan of step i+1
    is computed and uploaded (on a copy stream) while step i runs, so the
    device never waits for the host; a workspace's plan is overwritten only
    after the graph that read it has run, and a pinned plan buffer only
    after its previous upload has run.  With no plan, a step is one replay.

    run(workspace, plan_buf, stream) issues the device work of one step.
    """

    def __init__(self, torch, pkc, run, lens, num_ctas, cfg, ws_bytes, device):
        self.torch, self.pkc, self.lens, self.num_ctas, self.cfg = torch, pkc, lens, num_ctas, cfg
        self.stream, self.cstream = torch.cuda.Stream(device), torch.cuda.Stream(device)
        words = pkc.plan_words(len(lens), num_ctas) if num_ctas else 1
        self.pinned = [torch.empty(words, dtype=torch.int32).pin_memory() for _ in range(2)]
        self.plan_np = [t.numpy() for t in self.pinned]
        self.ws = [torch.empty(ws_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
        for w in self.ws:
            pkc.workspace_init(w)
        self.done = [torch.cuda.Event(), torch.cuda.Event()]
        self.uploaded = [torch.cuda.Event(), torch.cuda.Event()]
        self.graphs = []
        with torch.cuda.stream(self.stream):
            for s in range(2):
                buf = host_plan(pkc, lens, num_ctas, cfg, out=self.plan_np[s])
                upload_plan(pkc, buf, self.ws[s], stream=self.stream)
                run(self.ws[s], buf, self.stream)  # eager first: kernels loaded, maps built
                self.stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    run(self.ws[s], buf, self.stream)
                self.graphs.append(g)
        for e in self.done + self.uploaded:
            e.record(self.stream)
        self.stream.synchronize()
        self.i = 0
        self._prepare(0)

    def _prepare(self, i):
        if not self.num_ctas:
            return
        s = i & 1
        self.uploaded[s].synchronize()
        buf = host_plan(self.pkc, self.lens, self.num_ctas, self.cfg, out=self.plan_np[s])
        self.cstream.wait_event(self.done[s])
        upload_plan(self.pkc, buf, self.ws[s], stream=self.cstream)
        self.uploaded[s].record(self.cstream)

    def step(self):
        s = self.i & 1
        with self.torch.cuda.stream(self.stream):
            if self.num_ctas:
                self.stream.wait_event(self.uploaded[s])
            self.graphs[s].replay()
            self.done[s].record(self.stream)
        self._prepare(self.i + 1)
        self.i += 1

    def status_ok(self):
        return all(self.pkc.device_status(w) == 0 for w in self.ws)


def time_loop(ctx, fn, stream, min_steps, min_seconds=None):
    """Mean ms per call of fn() (which issues its work on `stream`), timed
    with CUDA events on that stream over max(min_steps, enough calls for
    min_seconds), with nvidia-smi clock samples taken meanwhile.  Warm-up
    keeps the GPU busy for ~0.3 s first, so the samples are taken under load."""
    torch = ctx.torch
    min_seconds = ctx.config_seconds if min_seconds is None else min_seconds
    sampler = ClockSampler(ctx.gpu_id)
    sampler.start()
    for _ in range(max(3, ctx.warmup)):
        fn()
    stream.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    stream.synchronize()
    t1 = max(a.elapsed_time(b) / 1e3, 1e-6)
    for _ in range(int(math.ceil(0.3 / t1))):
        fn()
    n = max(min_steps, int(math.ceil(min_seconds / t1)))
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    stream.synchronize()
    clocks = sampler.stop()
    return a.elapsed_time(b) / n, n, clocks


def _gbs(nbytes, ms):
    return nbytes / (ms / 1e3) / 1e9


def _entry(ctx, nbytes, ms, steps, clocks, **kw):
    e = {"us_per_step": 1e3 * ms, "value": _gbs(nbytes, ms), "unit": "GB/s",
         "frac": _gbs(nbytes, ms) / ctx.hbm_peak, "effective_bytes": int(nbytes), "steps": steps,
         "clocks": clocks}
    e.update(kw)
    return e


def cascade_call(pkc, name, p, d, extra):
    """run(ws, plan_buf, stream) for a cascade workload, writing into
    preallocated O / LSE."""
    torch = extra["torch"]
    B, Hq, _ = d["q"].shape
    o = torch.empty_like(d["q"])
    lse = torch.empty((B, Hq), dtype=torch.float32, device=d["q"].device)
    if name == "gqa_cascade_3level":
        ranges = extra["cfg"]["prefix_ranges"]
        return lambda ws, buf, st: pkc.cascade_decode_multilevel(
            d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], ranges, d["k_cache"],
            d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf,
            o=o, lse=lse, stream=st)
    if name == "gqa_cascade_paged_prefix":
        pool_k, pool_v, pages, page_indptr = extra["pool"]
        ind = p["prefix_req_indptr"]
        ranges = [(int(ind[j]), int(ind[j + 1])) for j in range(len(ind) - 1)]
        return lambda ws, buf, st: pkc.cascade_decode_paged_prefix(
            d["q"], pages, page_indptr, p["prefix_kv_indptr"], ranges, pool_k, pool_v,
            d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf, o=o, lse=lse,
            stream=st)
    return lambda ws, buf, st: pkc.cascade_decode(
        d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], p["prefix_req_indptr"],
        d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws,
        plan_buf=buf, o=o, lse=lse, stream=st)


def stage_times(ctx, run, ws, buf, steps):
    """Per-stage times (prefix, decode, contraction), launched one after the
    other with stage events on the current stream; plan uploaded once."""
    torch, pkc = ctx.torch, ctx.pkc
    stream = torch.cuda.current_stream()
    upload_plan(pkc, buf, ws, stream=stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in ev:  # torch creates the CUDA event on its first record
        for x in e:
            x.record(stream)
    for _ in range(3):
        run(ws, buf, stream)
    for e in ev:
        pkc.set_stage_events(e)
        run(ws, buf, stream)
    torch.cuda.synchronize()
    if pkc.device_status(ws) != 0:
        raise RuntimeError("device status not OK in the stage-timed run")
    names = ("prefix_state", "paged_decode", "contraction")
    return {k: 1e3 * statistics.mean(e[i].elapsed_time(e[i + 1]) for e in ev)
            for i, k in enumerate(names)}


def measure_cascade(ctx, name, stage_steps=10):
    """A cascade workload, graph-replayed steps with the plan per step, plus
    its stage times launched one after the other."""
    torch, pkc = ctx.torch, ctx.pkc
    from pkc_testing import dev, to_device
    paged = name == "gqa_cascade_paged_prefix"
    cfg, p = make_workload("gqa_cascade_lb" if paged else name)
    d = to_device(p, ctx.device)
    extra = {"torch": torch, "cfg": cfg}
    if paged:
        kc, vc, pages, page_indptr = workloads.pool_prefixes(p, 5, poison=False)
        extra["pool"] = (dev(kc, ctx.device), dev(vc, ctx.device), dev(pages, ctx.device), page_indptr)
        del kc, vc
    run = cascade_call(pkc, name, p, d, extra)
    B, Hq, _ = p["q"].shape
    C = cfg["num_ctas"]
    ws_bytes = pkc.workspace_size(B, Hq, C, 64)
    gs = GraphStepper(torch, pkc, run, p["cache_seqlens"], C, cfg, ws_bytes, ctx.device)
    ms, n, clocks = time_loop(ctx, gs.step, gs.stream, ctx.steps)
    if not gs.status_ok():
        raise RuntimeError(f"{name}: device status not OK")
    split = dict(zip(("prefix_blocks", "decode_blocks"), pkc.last_launch_blocks()))
    buf = host_plan(pkc, p["cache_seqlens"], C, cfg)
    torch.cuda.synchronize()  # the stepper's last plan upload has landed
    stages = stage_times(ctx, run, gs.ws[0], buf, stage_steps)
    eff = workloads.effective_bytes(p)
    kvb = kv_bytes_per_token(p)
    entry = _entry(ctx, eff, ms, n, clocks, launch="cuda_graph (host plan + upload per step)",
                   stages_us_serial=stages, stage_split=split, num_ctas=C or None,
                   prefix_tokens=int(p["prefix_kv_indptr"][-1]),
                   suffix_tokens=int(p["cache_seqlens"].sum()))
    if not C:  # an unplanned step is one launch: also time it among others in one graph
        entry["in_multi_call_graph"] = multi_call_graph_time(ctx, run, gs.ws[0], 20)
    entry["prefix_stage_gbs_serial"] = _gbs(int(p["prefix_kv_indptr"][-1]) * kvb,
                                            stages["prefix_state"] / 1e3)
    entry["decode_stage_gbs_serial"] = _gbs(int(p["cache_seqlens"].sum()) * kvb,
                                            stages["paged_decode"] / 1e3)
    return entry, (cfg, p, d, gs)


def multi_call_graph_time(ctx, run, ws, calls):
    """µs per call with `calls` unplanned calls captured in one CUDA graph,
    the way a model's per-layer attention calls are captured into one
    decode-step graph: the kernel with its launch gap inside a graph,
    without the cost of launching a graph per call.  Same inputs and outputs
    every call."""
    torch = ctx.torch
    st = torch.cuda.Stream(ctx.device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        run(ws, None, st)
        st.synchronize()
        with torch.cuda.graph(g, stream=st):
            for _ in range(calls):
                run(ws, None, st)
        ms, n, clocks = time_loop(ctx, g.replay, st, max(10, ctx.steps // calls))
    if ctx.pkc.device_status(ws) != 0:
        raise RuntimeError("multi-call graph: device status not OK")
    return {"calls_per_graph": calls, "us_per_call": 1e3 * ms / calls, "graph_replays": n,
            "clocks": clocks}


def noncascade_pool(torch, d, p):
    """Device-side non-cascade form of a single-prefix cascade problem: the
    prefix's pages appended to the cache pool (one copy, shared by every
    request) and every block table row listing them ahead of the request's
    own pages."""
    ps = p["page_size"]
    Lp = int(p["prefix_kv_indptr"][-1])
    assert Lp % ps == 0 and len(p["prefix_kv_indptr"]) == 2
    P0 = d["k_cache"].shape[0]
    npre = Lp // ps
    shape = (npre,) + tuple(d["k_cache"].shape[1:])
    kc = torch.cat([d["k_cache"], d["k_prefix"].reshape(shape)])
    vc = torch.cat([d["v_cache"], d["v_prefix"].reshape(shape)])
    B = d["q"].shape[0]
    pre = torch.arange(P0, P0 + npre, dtype=torch.int32, device=kc.device).expand(B, npre)
    bt = torch.cat([pre, d["block_table"]], dim=1).contiguous()
    lens = (d["cache_seqlens"] + Lp).contiguous()
    return kc, vc, bt, lens


def measure_noncascade(ctx, p, d, casc_ms, steps=None):
    """The pages' non-cascade baseline on the same problem: one paged decode
    over prefix + suffix per request (pkc_paged_decode_state), the prefix
    pages shared through the block tables.  Plan over 148 CTAs, uploaded
    once; direct launches."""
    torch, pkc = ctx.torch, ctx.pkc
    kc, vc, bt, lens = noncascade_pool(torch, d, p)
    lens_h = lens.cpu().numpy()
    B, Hq, _ = d["q"].shape
    C = 148
    buf = pkc.plan(lens_h, C)
    ws = torch.empty(pkc.workspace_size(B, Hq, C, 0), dtype=torch.uint8, device=ctx.device)
    pkc.workspace_init(ws)
    pkc.plan_upload(buf, ws)
    o = torch.empty_like(d["q"])
    lse = torch.empty((B, Hq), dtype=torch.float32, device=ctx.device)
    stream = torch.cuda.current_stream()
    call = lambda: pkc.paged_decode_state(d["q"], kc, vc, bt, lens, p["sm_scale"], ws,
                                          plan_buf=buf, o=o, lse=lse)
    ms, n, clocks = time_loop(ctx, call, stream, steps or ctx.steps)
    if pkc.device_status(ws) != 0:
        raise RuntimeError("non-cascade decode: device status not OK")
    eff = workloads.effective_bytes(p)
    read = int(lens_h.sum()) * kv_bytes_per_token(p)
    del kc, vc
    return {"us_per_step": 1e3 * ms, "value": _gbs(eff, ms), "unit": "GB/s",
            "kv_bytes_read": read, "kv_read_gbs": _gbs(read, ms),
            "kv_read_frac": _gbs(read, ms) / ctx.hbm_peak, "steps": n, "clocks": clocks,
            "num_ctas": C, "launch": "direct (decode + contraction), plan uploaded once",
            "cascade_speedup": ms / casc_ms}


def measure_decode(ctx, name):
    """Non-cascade paged decode of a workload through its plan (graph-replayed
    steps with the plan per step)."""
    torch, pkc = ctx.torch, ctx.pkc
    from pkc_testing import to_device
    cfg = workload_cfg(name)
    p = workloads.make_problem(**cfg)
    d = to_device(p, ctx.device)
    fp8 = p["kv_dtype"] == "e4m3"
    B, Hq, _ = p["q"].shape
    C = cfg["num_ctas"]
    o = torch.empty_like(d["q"])
    lse = torch.empty((B, Hq), dtype=torch.float32, device=ctx.device)
    if fp8:
        run = lambda ws, buf, st: pkc.paged_decode_state_fp8(
            d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"],
            p["sm_scale"], ws, k_scale=p["k_scale"], v_scale=p["v_scale"], plan_buf=buf,
            o=o, lse=lse, stream=st)
    else:
        run = lambda ws, buf, st: pkc.paged_decode_state(
            d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"],
            p["sm_scale"], ws, plan_buf=buf, o=o, lse=lse, stream=st)
    gs = GraphStepper(torch, pkc, run, p["cache_seqlens"], C, cfg,
                      pkc.workspace_size(B, Hq, C, 0), ctx.device)
    ms, n, clocks = time_loop(ctx, gs.step, gs.stream, ctx.steps)
    if not gs.status_ok():
        raise RuntimeError(f"{name}: device status not OK")
    eff = workloads.effective_bytes(p)
    G = Hq // p["num_kv_heads"]
    kernel = "paged_decode_mma_kernel" if (fp8 or G >= 2) else "paged_decode_kernel"
    return _entry(ctx, eff, ms, n, clocks, launch="cuda_graph (host plan + upload per step)",
                  kernel=kernel, kv_dtype=p["kv_dtype"], num_ctas=C,
                  kv_tokens=int(p["cache_seqlens"].sum()), launches="decode + contraction")


def measure_merge(ctx):
    torch, pkc = ctx.torch, ctx.pkc
    from pkc_testing import dev
    w = workloads.workload("merge")
    va, sa, vb, sb = (dev(w[k], ctx.device) for k in ("v_a", "s_a", "v_b", "s_b"))
    vn, sn = dev(w["v_n"], ctx.device), dev(w["s_n"], ctx.device)
    vo, so = torch.empty_like(va), torch.empty_like(sa)
    T, H, D = va.shape
    n = vn.shape[1]
    stream = torch.cuda.current_stream()
    ms2, k2, c2 = time_loop(ctx, lambda: pkc.merge_state(va, sa, vb, sb, vo, so), stream, ctx.steps)
    msn, kn, cn = time_loop(ctx, lambda: pkc.merge_states(vn, sn, vo, so), stream, ctx.steps)
    b2 = 3 * T * H * (D + 1) * 4
    bn = (n + 1) * T * H * (D + 1) * 4
    return {"binary": _entry(ctx, b2, ms2, k2, c2, kernel="merge2_kernel", launch="direct"),
            "n_ary": _entry(ctx, bn, msn, kn, cn, kernel="mergen_kernel", n_states=n, launch="direct"),
            "tokens": T, "heads": H, "head_dim": D, "dtype": "f32"}


def measure_sweep(ctx):
    """The pages' trend (blog "Cascade Inference", "Evaluation"): the gain of
    the cascade over the non-cascade decode grows with the shared prefix and
    the batch and shrinks as the unique suffix grows.  32 heads x 128, fp16,
    page size 16, N(0,1) inputs drawn on the device; both arms planned over
    148 CTAs with the plan uploaded once, direct launches."""
    torch, pkc = ctx.torch, ctx.pkc
    points = [(128, 32768, 256), (32, 32768, 256), (256, 32768, 256), (128, 2048, 256),
              (128, 8192, 256), (128, 32768, 1024), (128, 32768, 4096)]
    out = []
    gen = torch.Generator(device=ctx.device)
    H, D, ps = 32, 128, 16
    for B, Lp, Ls in points:
        gen.manual_seed(1000 + B + Lp + Ls)
        npre, nsuf = Lp // ps, B * (Ls // ps)
        pool_k = torch.randn((npre + nsuf, ps, H, D), generator=gen, device=ctx.device).half()
        pool_v = torch.randn((npre + nsuf, ps, H, D), generator=gen, device=ctx.device).half()
        q = torch.randn((B, H, D), generator=gen, device=ctx.device).half()
        perm = torch.randperm(nsuf, generator=gen, device=ctx.device).to(torch.int32) + npre
        bt_s = perm.view(B, Ls // ps).contiguous()
        lens_s = torch.full((B,), Ls, dtype=torch.int32, device=ctx.device)
        k_pre = pool_k[:npre].reshape(Lp, H, D)
        v_pre = pool_v[:npre].reshape(Lp, H, D)
        kv_ind, req_ind = np.array([0, Lp], np.int32), np.array([0, B], np.int32)
        scale = 1.0 / math.sqrt(D)
        C = 148
        lens_h = np.full(B, Ls, np.int32)
        buf = pkc.plan(lens_h, C)
        ws = torch.empty(pkc.workspace_size(B, H, C, 64), dtype=torch.uint8, device=ctx.device)
        pkc.workspace_init(ws)
        pkc.plan_upload(buf, ws)
        o = torch.empty_like(q)
        lse = torch.empty((B, H), dtype=torch.float32, device=ctx.device)
        stream = torch.cuda.current_stream()
        ms_c, n_c, clk_c = time_loop(ctx, lambda: pkc.cascade_decode(
            q, k_pre, v_pre, kv_ind, req_ind, pool_k, pool_v, bt_s, lens_s, scale, ws,
            plan_buf=buf, o=o, lse=lse), stream, 5, 0.25)
        bt_n = torch.cat([torch.arange(npre, dtype=torch.int32, device=ctx.device).expand(B, npre),
                          bt_s], dim=1).contiguous()
        lens_n = lens_s + Lp
        buf_n = pkc.plan(np.full(B, Lp + Ls, np.int32), C)
        ws_n = torch.empty(pkc.workspace_size(B, H, C, 0), dtype=torch.uint8, device=ctx.device)
        pkc.workspace_init(ws_n)
        pkc.plan_upload(buf_n, ws_n)
        ms_n, n_n, clk_n = time_loop(ctx, lambda: pkc.paged_decode_state(
            q, pool_k, pool_v, bt_n, lens_n, scale, ws_n, plan_buf=buf_n, o=o, lse=lse),
            stream, 3, 0.25)
        if pkc.device_status(ws) != 0 or pkc.device_status(ws_n) != 0:
            raise RuntimeError("sweep: device status not OK")
        kvb = 2 * H * D * 2
        eff = (Lp + B * Ls) * kvb + 2 * B * H * D * 2 + B * H * 4
        out.append({"batch": B, "prefix": Lp, "suffix": Ls, "cascade_us": 1e3 * ms_c,
                    "cascade_gbs": _gbs(eff, ms_c), "non_cascade_us": 1e3 * ms_n,
                    "non_cascade_kv_read_gbs": _gbs(B * (Lp + Ls) * kvb, ms_n),
                    "speedup": ms_n / ms_c, "steps": [n_c, n_n],
                    "sm_mhz": [c.get("sm_mhz") if c else None for c in (clk_c, clk_n)],
                    "reasons": sorted(set((clk_c or {}).get("reasons", []) +
                                          (clk_n or {}).get("reasons", [])))})
        del pool_k, pool_v, q, ws, ws_n, bt_n, k_pre, v_pre
        torch.cuda.empty_cache()
    return out


class Ctx:
    pass


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


HEADLINE_WORKLOADS = ("gqa_cascade_lb", "cascade_long_prompt", "tiny_cascade")


def make_ctx(args, torch, pkc, local):
    ctx = Ctx()
    ctx.torch, ctx.pkc, ctx.args = torch, pkc, args
    ctx.steps, ctx.warmup = max(1, args.steps), args.warmup
    ctx.config_seconds = args.config_seconds
    ctx.hbm_peak, ctx.tf_peak, ctx.peak_kind = load_peaks()
    ctx.gpu_id = gpu_smi_id(torch, local)
    ctx.device = f"cuda:{local}"
    return ctx


def run_single(ctx, args, world):
    """`--workload` other than a headline cascade: that workload's entry as
    its own line (same measurement as in the headline line's `configs`)."""
    name = args.workload
    if name == "merge":
        e = measure_merge(ctx)
        head = e["binary"]
        metric = "merge_state effective HBM throughput"
    elif name.startswith("paged_decode"):
        e = head = measure_decode(ctx, name)
        metric = "paged decode (non-cascade) effective KV throughput"
    else:
        e, _ = measure_cascade(ctx, name)
        head = e
        metric = "cascade decode effective KV throughput"
    line = {"metric": metric, "value": head["value"], "unit": "GB/s", "n_gpus": world,
            "steps": head["steps"], "warmup": args.warmup, "ms_per_step": head["us_per_step"] / 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "data": "synthetic", "config": {"workload": name}, "entry": e,
            "clocks": head.get("clocks"), "peak": ctx.hbm_peak,
            "peak_source": f"{ctx.peak_kind} hbm_gbs"}
    print(json.dumps(line), flush=True)


def measure_configs(ctx):
    """Every workload of the benchmark set, each timed in this process with
    its own clock record.  Slow to set up (host input generation), fast to
    time."""
    torch = ctx.torch
    out = {}

    def long_prompt():
        e, (cfg, p, d, gs) = measure_cascade(ctx, "cascade_long_prompt")
        e["non_cascade"] = measure_noncascade(ctx, p, d, e["us_per_step"] / 1e3)
        return e

    jobs = [("tiny_cascade", lambda: measure_cascade(ctx, "tiny_cascade")[0]),
            ("merge", lambda: measure_merge(ctx)),
            ("paged_decode", lambda: measure_decode(ctx, "paged_decode")),
            ("cascade_long_prompt", long_prompt),
            ("paged_decode_fp8", lambda: measure_decode(ctx, "paged_decode_fp8")),
            ("gqa_cascade_3level", lambda: measure_cascade(ctx, "gqa_cascade_3level")[0]),
            ("gqa_cascade_paged_prefix", lambda: measure_cascade(ctx, "gqa_cascade_paged_prefix")[0]),
            ("cascade_vs_non_cascade_sweep", lambda: measure_sweep(ctx))]
    for name, job in jobs:
        # A failing entry is reported as such; it does not take the headline
        # line with it.  A device status other than OK raises inside.
        try:
            out[name] = job()
        except Exception as exc:  # noqa: BLE001
            out[name] = {"error": f"{type(exc).__name__}: {str(exc)[:300]}"}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
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
    pkc.set_contraction(args.contraction)
    pkc.set_cascade_small(args.cascade_small)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from pkc_testing import to_device
    ctx = make_ctx(args, torch, pkc, local)
    if args.workload not in HEADLINE_WORKLOADS:
        run_single(ctx, args, world)
        if dist is not None:
            dist.destroy_process_group()
        return

    cfg, p = make_workload(args.workload, args.batch)
    if args.num_ctas is not None:
        cfg["num_ctas"] = args.num_ctas
    d = to_device(p, ctx.device)
    B, Hq, D = p["q"].shape
    num_ctas = cfg["num_ctas"]
    lens = p["cache_seqlens"]
    run = cascade_call(pkc, args.workload, p, d, {"torch": torch, "cfg": cfg})
    ws_bytes = pkc.workspace_size(B, Hq, num_ctas, 64)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=ctx.device)
    pkc.workspace_init(ws)
    words = pkc.plan_words(B, num_ctas) if num_ctas else 1
    pinned = [torch.empty(words, dtype=torch.int32).pin_memory() for _ in range(2)]
    plan_np = [t.numpy() for t in pinned]

    # ---- directly launched steps with per-stage events (stages one after
    # the other: the stage events keep the prefix on the caller's stream) ----
    host_plan_s = []
    uploaded = [torch.cuda.Event(), torch.cuda.Event()]

    def step(i):
        uploaded[i & 1].synchronize()  # the pinned buffer's previous upload ran
        t0 = time.perf_counter()
        buf = host_plan(pkc, lens, num_ctas, cfg, out=plan_np[i & 1])
        host_plan_s.append(time.perf_counter() - t0)
        upload_plan(pkc, buf, ws)
        uploaded[i & 1].record()
        run(ws, buf, torch.cuda.current_stream())

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    status = pkc.device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status after warm-up: {pkc.STATUS_NAMES.get(status, status)}")
    host_plan_s.clear()
    K = ctx.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for e in ev:  # torch creates the CUDA event on first record
        for x in e:
            x.record()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(ctx.gpu_id)
    sampler.start()
    torch.cuda.synchronize()
    start.record()
    for i in range(K):
        pkc.set_stage_events(ev[i])
        step(i)
    end.record()
    torch.cuda.synchronize()
    direct_ms_per_step = start.elapsed_time(end) / K
    status = pkc.device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status after timing: {pkc.STATUS_NAMES.get(status, status)}")
    stage_ms = {
        "prefix_state": statistics.mean(e[0].elapsed_time(e[1]) for e in ev),
        "paged_decode": statistics.mean(e[1].elapsed_time(e[2]) for e in ev),
        "contraction": statistics.mean(e[2].elapsed_time(e[3]) for e in ev),
    }

    # ---- the headline: exactly K graph-replayed steps (host plan + upload
    # per step, overlapping the previous step's device work) ----
    gs = GraphStepper(torch, pkc, run, lens, num_ctas, cfg, ws_bytes, ctx.device)
    for _ in range(max(3, args.warmup)):
        gs.step()
    gs.stream.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ga.record(gs.stream)
    for _ in range(K):
        gs.step()
    gb.record(gs.stream)
    gs.stream.synchronize()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    g_ms = reduce_max(ga.elapsed_time(gb), dist, d["q"].device)
    # Single replays with and without an L2 flush (a 256 MB write) before
    # each, timed alone: the median step with a cold L2, and with what the
    # previous step left in it.
    flush = torch.empty((256 << 20) // 4, dtype=torch.int32, device=ctx.device)
    n_iso = min(max(K, 20), 50)
    iso = {}
    with torch.cuda.stream(gs.stream):
        for flushed in (True, False):
            evs = []
            for i in range(n_iso):
                if flushed:
                    flush.fill_(i)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(gs.stream)
                gs.step()
                e1.record(gs.stream)
                evs.append((e0, e1))
            gs.stream.synchronize()
            iso[flushed] = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
    del flush
    clocks = sampler.stop()
    if not gs.status_ok():
        raise RuntimeError("device status after the graph-replayed steps")
    split = dict(zip(("prefix_blocks", "decode_blocks"), pkc.last_launch_blocks()))

    # ---- the pages' own CTA assignment (the plan's static CTA lists) ----
    schedules = None
    if num_ctas and world == 1 and not args.no_ab:
        pkc.set_decode_schedule("static" if args.decode_schedule == "dynamic" else "dynamic")
        gs2 = GraphStepper(torch, pkc, run, lens, num_ctas, cfg, ws_bytes, ctx.device)
        ms2, n2, clk2 = time_loop(ctx, gs2.step, gs2.stream, K)
        if not gs2.status_ok():
            raise RuntimeError("device status after the other schedule")
        other = "static" if args.decode_schedule == "dynamic" else "dynamic"
        split2 = dict(zip(("prefix_blocks", "decode_blocks"), pkc.last_launch_blocks()))
        pkc.set_decode_schedule(args.decode_schedule)
        ms1, n1, clk1 = time_loop(ctx, gs.step, gs.stream, K)
        schedules = {
            args.decode_schedule: {"us_per_step": 1e3 * ms1, "steps": n1, "clocks": clk1,
                                   "stage_split": split},
            other: {"us_per_step": 1e3 * ms2, "steps": n2, "clocks": clk2, "stage_split": split2},
            "note": "graph-replayed steps timed back to back; static = each decode block runs "
                    "its CTA's list from the host plan's min-cost priority queue; dynamic = "
                    "blocks take the same plan's chunks from a longest-first device queue"}
        del gs2

    # ---- where the split states are contracted: inside the attention
    # kernels (fused) or by the standalone contraction kernel after them ----
    contractions = None
    if world == 1 and not args.no_ab:
        contractions = {}
        for mode in ("separate", "separate_plain", "fused"):
            if mode == args.contraction:
                continue
            pkc.set_contraction(mode)
            gs3 = GraphStepper(torch, pkc, run, lens, num_ctas, cfg, ws_bytes, ctx.device)
            ms3, n3, clk3 = time_loop(ctx, gs3.step, gs3.stream, K)
            if not gs3.status_ok():
                raise RuntimeError(f"device status after contraction mode {mode}")
            contractions[mode] = {"us_per_step": 1e3 * ms3, "steps": n3, "clocks": clk3}
            del gs3
        pkc.set_contraction(args.contraction)
        ms4, n4, clk4 = time_loop(ctx, gs.step, gs.stream, K)
        contractions[args.contraction] = {"us_per_step": 1e3 * ms4, "steps": n4, "clocks": clk4}
        contractions["note"] = ("graph-replayed steps timed back to back; separate = contraction kernel "
                                "after both stages, launched as the decode's programmatic dependent; "
                                "separate_plain = the same launched plainly; fused = the kernel writing "
                                "a (request, KV head)'s last source merges it (no contraction launch)")

    eff = workloads.effective_bytes(p)
    ms_per_step = g_ms / K
    value = whole_job_gbs(eff, 1, world, ms_per_step / 1e3)
    hbm_peak, tf_peak, peak_kind = ctx.hbm_peak, ctx.tf_peak, ctx.peak_kind
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
    G = Hq // p["num_kv_heads"]
    mma = args.decode_kernel == "mma" or (args.decode_kernel == "auto" and G >= 2)
    kernel_name = {"prefix_state": "prefix_state_kernel"}.get(
        dominant, "paged_decode_mma_kernel" if mma else "paged_decode_kernel")
    tr = kernel_traffic(kernel_name, args.workload if args.batch is None else None)
    rows_per_prefix = np.diff(p["prefix_req_indptr"]) * G
    prefix_flops = float(4 * D * np.sum(rows_per_prefix * np.diff(p["prefix_kv_indptr"])) *
                         p["num_kv_heads"])

    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(torch, pkc, p, d, cfg, eff, args.e2e_steps, num_ctas, world, dist)
    del gs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

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

    configs = None
    if world == 1 and not args.no_configs and args.batch is None:
        configs = measure_configs(ctx)

    if rank == 0:
        line = {
            "metric": "cascade decode effective KV throughput",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_step": 1e3 * ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg["dtype"], "data": "synthetic",
            "config": line_config(args.workload, cfg, p, num_ctas, args, world),
            "impl_config": {
                "launch": "cuda_graph", "decode_kernel": args.decode_kernel,
                "contraction": args.contraction,
                "decode_schedule": args.decode_schedule if num_ctas else None,
                "prefix_ctas": args.prefix_ctas or "auto",
                "step": "host plan + plan upload + prefix states + paged decode + contraction"},
            "stage_split": split,
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
            "graph": {"isolated_replay_us_median": {"l2_flushed": iso[True], "unflushed": iso[False],
                                                    "flush_bytes": 256 << 20, "replays": n_iso}},
            "decode_schedules": schedules,
            "contractions": contractions,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": (2 if args.contraction == "fused" else 3) * K,
            "clocks": clocks,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
