"""Benchmark of the fused AllToAll + MXFP8 block-scaled GEMM (libmxa2a) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME_OR_INDEX] [--path fused|unfused]

A step is one pass of the whole hot path (B-scale pack + the fused staging /
block-scaled GEMM kernel [+ split-K reduce]) over one batch of synthetic
inputs already resident in HBM.  Before every step the L2 is flushed (a write
of twice its size); the flush sits outside the per-step CUDA events, which are
recorded on the launch stream around the library call.  Rank 0 prints one
JSON line.

With N > 1 (torchrun), every rank runs its own replica on its own GPU (the
path has no cross-GPU exchange on a one-GPU-per-box pool: the R segments are
local buffers); ranks are barrier-aligned, the slowest rank's time counts and
``value`` is the job's total TFLOP/s ("scaling": "weak").

``--impl reference`` times the CPU oracle (exact integer accumulation, the
correctness reference) on the host cores instead, on a bounded sample of the
same workload, and prints the same line with ``"impl": "reference"``.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused MXFP8 a2a-GEMM TFLOP/s and % of roofline (1 GB300)"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = 3          # the largest problem: 8 segments, 8192 x 8192 x 8192
CONFIG_WORKLOADS = (1, 2, 3, 4)   # the tensor-bound and the HBM-bound problems reported beside it
ABLATION_WORKLOAD = 1         # the 2048 x 4096 x 4096 problem: the ring limits it the most
FP8_OVER_BF16 = 2.0           # nominal dense fp8 : bf16 tensor rate (4.5 : 2.25 PFLOP/s)
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["mxgemm.cu", "kernels.cuh", "ptx.cuh", "atoms.cuh"]


# ----------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max_sum(t_local: float, work_local: float, device=None):
    """(max over ranks of t, sum over ranks of work) with torch.distributed;
    identity when no process group is initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return t_local, work_local
    t = torch.tensor([t_local], dtype=torch.float64, device=device)
    w = torch.tensor([work_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(w, op=dist.ReduceOp.SUM)
    return float(t.item()), float(w.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "all_mxfp8_block_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary,
    or None when there is none or the kernel sources changed since."""
    path = os.path.join(ROOT, "profiles", f"mxgemm_fused_{workload_name}.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    m_h = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    if not m_t or not m_h or m_h.group(1) != kernel_source_hash():
        return None
    return int(m_t.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open(f"/tmp/mxa2a_clocks_{os.getpid()}.csv", "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period), "-i", str(self.gpu)],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.out:
            self.out.close()

    def summary(self):
        if self.proc is None or not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


def roofline_terms(w, p_tflops: float, bw_gbs: float):
    t_flop = w.flops / (p_tflops * 1e12)
    t_bytes = w.bytes_alg / (bw_gbs * 1e9)
    return max(t_flop, t_bytes), ("tensor" if t_flop >= t_bytes else "hbm")


# ----------------------------------------------------------------------------- oracle (CPU) arm
def time_oracle(w, x, seconds: float = 12.0, max_rows: int | None = None):
    """Time the CPU oracle on rows 0..r-1 of C (all columns, full K), r grown
    until one call takes about `seconds`.  Returns (TFLOP/s, rows, secs, cores)."""
    import oracle
    rows = 8
    cores = os.cpu_count() or 1
    while True:
        t0 = time.perf_counter()
        oracle.gemm(x["A_seg"], x["A_scale_seg"], x["B"], x["B_scale"], rows=list(range(rows)))
        dt = time.perf_counter() - t0
        cap = w.M if max_rows is None else min(w.M, max_rows)
        if dt >= seconds * 0.5 or rows >= cap:
            return 2.0 * rows * w.N * w.K / dt / 1e12, rows, dt, cores
        rows = min(cap, max(rows + 1, int(rows * min(8.0, seconds / max(dt, 1e-3)))))


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from all_mxfp8_block_gb300 import inputs
    import oracle
    oracle.build()
    x = inputs.make_inputs(w)
    # size one step to roughly 1.5 s of oracle work
    _, rows, dt, cores = time_oracle(w, x, seconds=1.5)
    for _ in range(args.warmup):
        oracle.gemm(x["A_seg"], x["A_scale_seg"], x["B"], x["B_scale"], rows=list(range(rows)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm(x["A_seg"], x["A_scale_seg"], x["B"], x["B_scale"], rows=list(range(rows)))
    total = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    value = flops * args.steps / total / 1e12
    sample = f"rows 0..{rows - 1} of C ({rows} x {w.N} outputs, full K={w.K}) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64-exact",
        "data": "synthetic",
        "config": {"workload": w.name, "R": w.R, "M": w.M, "kPerRank": w.kPerRank, "K": w.K, "N": w.N,
                   "commMSize": w.commMSize, "buffer_num": w.buffer_num, "seed": w.seed,
                   "path": "cpu oracle", "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def time_tiny_graph(dev, runs: int = 200):
    """The smallest workload is launch-latency bound: time it back to back as
    eager library calls and as replays of one CUDA graph holding the call (no
    L2 flush; CUDA events around all runs), after checking the replay
    reproduces the eager bits."""
    import torch
    from all_mxfp8_block_gb300 import inputs, mxa2a
    w0 = inputs.workload(0)
    x0 = inputs.make_inputs(w0)
    dA = [a.to(dev) for a in x0["A_seg"]]
    dS = [s.to(dev) for s in x0["A_scale_seg"]]
    dB, dBs = x0["B"].to(dev), x0["B_scale"].to(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    C = torch.empty((w0.M, w0.N), dtype=torch.int16, device=dev)
    with mxa2a.Plan(w0.R, w0.M, w0.kPerRank, w0.N, w0.commMSize, w0.buffer_num) as plan:
        plan.set_option(mxa2a.MXA2A_OPT_SPLIT_K, 1)
        out = {"workload": w0.name, "runs": runs, "splits": 1,
               "timer": "CUDA events around the runs, back to back, no L2 flush"}
        with torch.cuda.stream(side):
            for _ in range(10):
                plan.run(dA, dS, dB, dBs, C, side)
            side.synchronize()
            eager_bits = C.clone()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(side)
            for _ in range(runs):
                plan.run(dA, dS, dB, dBs, C, side)
            e1.record(side)
            side.synchronize()
            out["eager_us_per_run"] = e0.elapsed_time(e1) * 1e3 / runs
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            plan.run(dA, dS, dB, dBs, C, side)
        C.zero_()
        g.replay()
        torch.cuda.synchronize(dev)
        out["replay_matches_eager"] = bool(torch.equal(C, eager_bits))
        with torch.cuda.stream(side):
            e0.record(side)
            for _ in range(runs):
                g.replay()
            e1.record(side)
            side.synchronize()
        out["graph_us_per_run"] = e0.elapsed_time(e1) * 1e3 / runs
        out["tflops_graph"] = 2.0 * w0.M * w0.N * w0.K / (out["graph_us_per_run"] * 1e-6) / 1e12
    return out


def time_siblings(dev, stream, flush, flush_bytes, steps, warmup, with_allreduce=True):
    """Mean ms per call of the sibling operators' fused and unfused paths on
    their benchmark workloads (AllGather + GEMM: 4 blocks of 512 rows, K = N =
    4096; GEMM + ReduceScatter and, with_allreduce, GEMM + AllReduce: rank 1 of
    4, 2048 x 4096 x 4096), each call after an L2 flush, CUDA events around
    each call."""
    import torch
    from all_mxfp8_block_gb300 import inputs, mxa2a

    def timed(call):
        for _ in range(warmup):
            mxa2a.mxa2a_l2_flush(flush, flush_bytes, stream)
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize(dev)
        for i in range(steps):
            mxa2a.mxa2a_l2_flush(flush, flush_bytes, stream)
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in ev) / steps

    bf16_tf, _, _ = measured_peaks()
    peak = bf16_tf * FP8_OVER_BF16
    out = {}
    w = inputs.AG_WORKLOADS[1]
    x = inputs.make_allgather_inputs(w)
    A = [a.to(dev) for a in x["A_blk"]]
    S = [s.to(dev) for s in x["A_scale_blk"]]
    B, Bs = x["B"].to(dev), x["B_scale"].to(dev)
    C = torch.empty((w.M, w.N), dtype=torch.int16, device=dev)
    with mxa2a.AllGatherPlan(w.R, w.rowsPerRank, w.K, w.N, w.commMSize, w.buffer_num) as p:
        res = {path + "_ms": timed(lambda fn=fn: fn(A, S, B, Bs, C, stream))
               for path, fn in (("fused", p.run), ("unfused", p.run_unfused), ("direct", p.run_direct))}
        st = p.status()
        if st["code"] != 0:
            raise RuntimeError(f"device status after the all-gather timing: {st}")
    tf = w.flops / (res["fused_ms"] / 1e3) / 1e12
    out["allgather_gemm"] = {"workload": w.name, "R": w.R, "rowsPerRank": w.rowsPerRank, "K": w.K, "N": w.N,
                             "commMSize": w.commMSize, "buffer_num": w.buffer_num, **res, "value": tf,
                             "unit": UNIT, "roofline_frac": tf / peak, "steps": steps}
    del A, S, B, Bs, C
    w = inputs.RS_WORKLOADS[1]
    x = inputs.make_reduce_scatter_inputs(w)
    A, S, B, Bs = (x[k].to(dev) for k in ("A", "A_scale", "B", "B_scale"))
    recv = [None if r is None else r.to(dev) for r in x["recv"]]
    send = [None if j == w.rank else torch.empty((w.rows, w.N), dtype=torch.int16, device=dev)
            for j in range(w.R)]
    o = torch.empty((w.rows, w.N), dtype=torch.int16, device=dev)
    with mxa2a.ReduceScatterPlan(w.R, w.rank, w.M, w.K, w.N) as p:
        res = {path + "_ms": timed(lambda fn=fn: fn(A, S, B, Bs, recv, send, o, stream))
               for path, fn in (("fused", p.run), ("unfused", p.run_unfused))}
        st = p.status()
        if st["code"] != 0:
            raise RuntimeError(f"device status after the reduce-scatter timing: {st}")
    tf = w.flops / (res["fused_ms"] / 1e3) / 1e12
    out["gemm_reduce_scatter"] = {"workload": w.name, "R": w.R, "rank": w.rank, "M": w.M, "K": w.K, "N": w.N,
                                  **res, "value": tf, "unit": UNIT, "roofline_frac": tf / peak, "steps": steps}
    del A, S, B, Bs, recv, send, o
    if not with_allreduce:
        return out
    w = inputs.AR_WORKLOADS[1]
    x = inputs.make_allreduce_inputs(w)
    A, S, B, Bs = (x[k].to(dev) for k in ("A", "A_scale", "B", "B_scale"))
    recv = [None if r is None else r.to(dev) for r in x["recv"]]
    pub = torch.empty((w.M, w.N), dtype=torch.int16, device=dev)
    o = torch.empty((w.M, w.N), dtype=torch.int16, device=dev)
    with mxa2a.AllReducePlan(w.R, w.rank, w.M, w.K, w.N) as p:
        res = {path + "_ms": timed(lambda fn=fn: fn(A, S, B, Bs, recv, pub, o, stream))
               for path, fn in (("fused", p.run), ("unfused", p.run_unfused))}
        st = p.status()
        if st["code"] != 0:
            raise RuntimeError(f"device status after the all-reduce timing: {st}")
    tf = w.flops / (res["fused_ms"] / 1e3) / 1e12
    out["gemm_allreduce"] = {"workload": w.name, "R": w.R, "rank": w.rank, "M": w.M, "K": w.K, "N": w.N,
                             **res, "value": tf, "unit": UNIT, "roofline_frac": tf / peak, "steps": steps}
    return out


def run_siblings_only(args):
    """The sibling operators alone (for profiling them): each path `warmup`
    calls, then `steps` timed calls, in the order AllGather + GEMM fused,
    unfused, direct, GEMM + ReduceScatter fused, unfused, GEMM + AllReduce
    fused, unfused."""
    import torch
    from all_mxfp8_block_gb300 import build as mxbuild
    from all_mxfp8_block_gb300 import mxa2a
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    mxbuild.build()
    mxa2a.load()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_bytes = max(2 * l2, 64 << 20) // 16 * 16
    flush = torch.zeros(flush_bytes // 4, dtype=torch.int32, device=dev)
    res = time_siblings(dev, torch.cuda.current_stream(dev), flush, flush_bytes, args.steps, args.warmup)
    print(json.dumps({"siblings": res, "steps": args.steps, "warmup": args.warmup}), flush=True)
    return 0


def _device_inputs(x, dev):
    return ([a.to(dev) for a in x["A_seg"]], [s.to(dev) for s in x["A_scale_seg"]],
            x["B"].to(dev), x["B_scale"].to(dev))


def make_timed_loop(dev, stream, flush, flush_bytes, ws):
    """timed(fn, args, steps, warmup, sampler) -> per-step ms: every step after
    an L2 flush (outside the events), CUDA events on the launch stream around
    the library call; ranks barrier-aligned around the timed region."""
    import torch
    import torch.distributed as dist
    from all_mxfp8_block_gb300 import mxa2a

    def timed(fn, fargs, steps, warmup, sampler=None):
        for _ in range(warmup):
            mxa2a.mxa2a_l2_flush(flush, flush_bytes, stream)
            fn(*fargs, stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ctx = sampler if sampler is not None else _Null()
        with ctx:
            for i in range(steps):
                mxa2a.mxa2a_l2_flush(flush, flush_bytes, stream)
                ev[i][0].record(stream)
                fn(*fargs, stream)
                ev[i][1].record(stream)
            torch.cuda.synchronize(dev)
        if ws > 1:
            dist.barrier()
        return [a.elapsed_time(b) for a, b in ev]
    return timed


def roofline_of(w, step_s, kernel_s):
    """t_roof = max(2MNK / MXFP8 peak, bytes_alg / HBM); the fraction of the
    bound's peak the fused kernel reaches, and t_roof / t_step."""
    bf16_tf, hbm, _ = measured_peaks()
    p_fp8 = bf16_tf * FP8_OVER_BF16
    t_roof, bound = roofline_terms(w, p_fp8, hbm)
    if bound == "tensor":
        achieved, peak, unit = w.flops / kernel_s / 1e12, p_fp8, "TFLOP/s"
    else:
        achieved, peak, unit = w.bytes_alg / kernel_s / 1e9, hbm, "GB/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "t_roof_us": t_roof * 1e6, "roofline_pct": 100.0 * t_roof / step_s}


def time_config(dev, timed, w, steps, warmup):
    """One problem size: fused step, fused kernel (the library's events around
    the GEMM launch), unfused step; the roofline fraction of the fused kernel."""
    import torch
    from all_mxfp8_block_gb300 import inputs, mxa2a
    x = inputs.make_inputs(w)
    dA, dS, dB, dBs = _device_inputs(x, dev)
    C = torch.empty((w.M, w.N), dtype=torch.int16, device=dev)
    with mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num) as plan:
        plan.set_option(mxa2a.MXA2A_OPT_RECORD_EVENTS, min(4096, steps))
        fused = timed(plan.run, (dA, dS, dB, dBs, C), steps, warmup)
        kern = plan.kernel_times(min(4096, steps))
        plan.set_option(mxa2a.MXA2A_OPT_RECORD_EVENTS, 0)
        unfused = timed(plan.run_unfused, (dA, dS, dB, dBs, C), steps, warmup)
        st = plan.status()
        if st["code"] != 0:
            raise RuntimeError(f"device status after timing {w.name}: {st}")
        info = {"splits": plan.get_option(mxa2a.MXA2A_INFO_SPLITS),
                "cta_pair": plan.get_option(mxa2a.MXA2A_INFO_CTA_PAIR),
                "cta_pair_unfused": plan.get_option(mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED),
                "tail_split": plan.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT),
                "tail_split_unfused": plan.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT_UNFUSED)}
    return summarize_config(w, fused, kern, unfused, steps, info)


def summarize_config(w, fused_ms, kern_ms, unfused_ms, steps, info):
    f = statistics.mean(fused_ms) * 1e-3
    k = statistics.mean(kern_ms) * 1e-3 if kern_ms else f
    u = statistics.mean(unfused_ms) * 1e-3
    rf = roofline_of(w, f, k)
    return {"workload": w.name, "steps": steps, "fused_step_us": f * 1e6, "fused_kernel_us": k * 1e6,
            "unfused_step_us": u * 1e6, "fused_faster": f < u, "fused_tflops": w.flops / f / 1e12,
            "bound": rf["bound"], "frac": rf["frac"], "frac_unit": rf["unit"], "achieved": rf["achieved"],
            "peak": rf["peak"], "roofline_pct": rf["roofline_pct"], "t_roof_us": rf["t_roof_us"], **info}


def time_credit_ablation(dev, timed, steps, warmup, skew_ns):
    """The staging-protocol ablation on the problem the ring limits most:
    per-(slot, segment) credits against the whole-step protocol, each with and
    without slowed copies on every 4th CTA."""
    import torch
    from all_mxfp8_block_gb300 import inputs, mxa2a
    w = inputs.workload(ABLATION_WORKLOAD)
    x = inputs.make_inputs(w)
    dA, dS, dB, dBs = _device_inputs(x, dev)
    C = torch.empty((w.M, w.N), dtype=torch.int16, device=dev)
    out = {"workload": w.name, "skew_ns": skew_ns, "steps": steps,
           "what": "fused ms per step; skew: the copy workers of every 4th CTA wait skew_ns before each copy task"}
    with mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num) as plan:
        if plan.get_option(mxa2a.MXA2A_INFO_CTA_PAIR):
            plan.set_option(mxa2a.MXA2A_OPT_CTA_PAIR, 0)   # the protocol options live in the single-CTA kernel
        for sc, name in ((0, "per_segment"), (1, "whole_step")):
            for skew in (0, skew_ns):
                plan.set_option(mxa2a.MXA2A_OPT_STEP_CREDITS, sc)
                plan.set_option(mxa2a.MXA2A_OPT_COPY_SKEW_NS, skew)
                ms = timed(plan.run, (dA, dS, dB, dBs, C), steps, warmup)
                out[name + ("_skew_ms" if skew else "_ms")] = statistics.mean(ms)
        st = plan.status()
        if st["code"] != 0:
            raise RuntimeError(f"device status after the credit ablation: {st}")
    return out


def time_e2e(dev, stream, plan, x, w, steps, warmup, ws):
    """End to end through mxa2a_run_host with pinned host buffers (host
    wall clock per step: the copies in, the run, the copy of C out, the stream
    sync), and beside it the host link alone: the same bytes moved by one
    pinned cudaMemcpyAsync per buffer, timed the same way."""
    import torch
    import torch.distributed as dist
    hA = [a.pin_memory() for a in x["A_seg"]]
    hS = [s.pin_memory() for s in x["A_scale_seg"]]
    hB, hBs = x["B"].pin_memory(), x["B_scale"].pin_memory()
    hC = torch.empty((w.M, w.N), dtype=torch.int16).pin_memory()
    for _ in range(warmup):
        plan.run_host(hA, hS, hB, hBs, hC, stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        plan.run_host(hA, hS, hB, hBs, hC, stream)
        stream.synchronize()
    t_e2e = time.perf_counter() - t0
    if ws > 1:
        dist.barrier()
    t_e2e_max, fl = reduce_max_sum(t_e2e, float(w.flops) * steps, dev if ws > 1 else None)
    h2d = sum(a.numel() for a in hA) + sum(s.numel() for s in hS) + hB.numel() + hBs.numel()
    d2h = hC.numel() * 2
    # the link alone: device buffers of the same sizes, one async copy per buffer
    srcs = hA + hS + [hB, hBs]
    dsts = [torch.empty_like(h, device=dev) for h in srcs]
    dC = torch.empty((w.M, w.N), dtype=torch.int16, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for d, h in zip(dsts, srcs):
                d.copy_(h, non_blocking=True)
            hC.copy_(dC, non_blocking=True)
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            for d, h in zip(dsts, srcs):
                d.copy_(h, non_blocking=True)
            hC.copy_(dC, non_blocking=True)
            stream.synchronize()
        t_link = time.perf_counter() - t0
    t_link_max, _ = reduce_max_sum(t_link, 0.0, dev if ws > 1 else None)
    link_gbs = (h2d + d2h) * steps / t_link_max / 1e9
    return {"value": fl / t_e2e_max / 1e12, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "timer": "host wall clock per step (h2d copies + run + d2h copy + stream sync)", "steps": steps,
            "us_per_step": t_e2e_max / steps * 1e6,
            "link_us_per_step": t_link_max / steps * 1e6, "link_gbs": link_gbs,
            "link_frac": t_link_max / t_e2e_max,
            "link_what": "the same h2d + d2h bytes as one pinned cudaMemcpyAsync per buffer, nothing else; "
                         "link_frac = link-only time / end-to-end time"}


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    from all_mxfp8_block_gb300 import build as mxbuild
    from all_mxfp8_block_gb300 import inputs, mxa2a

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        mxbuild.build()
    if ws > 1:
        dist.barrier()
    mxa2a.load()

    x = inputs.make_inputs(w)
    dA, dS, dB, dBs = _device_inputs(x, dev)
    C = torch.empty((w.M, w.N), dtype=torch.int16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_bytes = max(2 * l2, 64 << 20) // 16 * 16
    flush = torch.zeros(flush_bytes // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    timed = make_timed_loop(dev, stream, flush, flush_bytes, ws)

    plan = mxa2a.Plan(w.R, w.M, w.kPerRank, w.N, w.commMSize, w.buffer_num)
    plan.set_option(mxa2a.MXA2A_OPT_RECORD_EVENTS, min(4096, max(1, args.steps)))
    if args.split:
        plan.set_option(mxa2a.MXA2A_OPT_SPLIT_K, args.split)
    if args.single_cta:
        plan.set_option(mxa2a.MXA2A_OPT_CTA_PAIR, 0)
    if args.cta_pair:
        plan.set_option(mxa2a.MXA2A_OPT_CTA_PAIR, 1)
    if args.group_m:
        plan.set_option(mxa2a.MXA2A_OPT_GROUP_M, args.group_m)
    run = plan.run if args.path == "fused" else plan.run_unfused
    fargs = (dA, dS, dB, dBs, C)

    sampler = ClockSampler(local)
    step_ms = timed(run, fargs, args.steps, args.warmup, sampler)
    launches_per_run = plan.get_option(mxa2a.MXA2A_INFO_LAUNCHES)
    kern_ms = plan.kernel_times(min(4096, args.steps))
    plan.set_option(mxa2a.MXA2A_OPT_RECORD_EVENTS, 0)
    st = plan.status()
    if st["code"] != 0:
        raise RuntimeError(f"device status after the timed region: {st}")
    clocks = sampler.summary()

    # the other variant, same caliber, for the fused-vs-unfused comparison
    other = plan.run_unfused if args.path == "fused" else plan.run
    other_steps = min(args.steps, args.other_steps)
    other_ms = timed(other, fargs, other_steps, args.warmup)
    # the direct-read ablation: A read in place, no exchange (same caliber)
    # (the direct read runs on the single-CTA kernel only)
    direct_ms = None
    if not plan.get_option(mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED):
        direct_ms = timed(plan.run_direct, fargs, other_steps, args.warmup)
    st = plan.status()
    if st["code"] != 0:
        raise RuntimeError(f"device status after the comparison paths: {st}")

    t_local = sum(step_ms) / 1e3
    t_max, flops_total = reduce_max_sum(t_local, float(w.flops) * args.steps, dev if ws > 1 else None)
    value = flops_total / t_max / 1e12
    ms_per_step = t_max / args.steps * 1e3

    # end to end through the C ABI with pinned host buffers (copies in the timed
    # region), with the host link's own time for the same bytes beside it
    e2e = None
    if not args.no_e2e:
        e2e = time_e2e(dev, stream, plan, x, w, min(args.steps, 50), max(3, args.warmup), ws)

    # every problem size, fused and unfused, same caliber (the headline's own numbers reused)
    configs = None
    if not args.no_configs:
        configs = {}
        fused_ms = step_ms if args.path == "fused" else other_ms
        unfused_ms = other_ms if args.path == "fused" else step_ms
        for idx in CONFIG_WORKLOADS:
            wc = inputs.workload(idx)
            if wc.name == w.name:
                info = {"splits": plan.get_option(mxa2a.MXA2A_INFO_SPLITS),
                        "cta_pair": plan.get_option(mxa2a.MXA2A_INFO_CTA_PAIR),
                        "cta_pair_unfused": plan.get_option(mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED),
                        "tail_split": plan.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT),
                        "tail_split_unfused": plan.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT_UNFUSED)}
                configs[wc.name] = summarize_config(wc, fused_ms, kern_ms if args.path == "fused" else [],
                                                    unfused_ms, args.steps, info)
            else:
                configs[wc.name] = time_config(dev, timed, wc, min(args.steps, args.config_steps), args.warmup)

    # the staging protocol ablation (fused) on the problem the ring limits most
    credit_ablation = None
    if args.path == "fused" and not args.no_ablation:
        credit_ablation = time_credit_ablation(dev, timed, min(other_steps, 200), args.warmup, args.skew_ns)

    # the sibling fused operators, same caliber
    siblings = None
    if not args.no_siblings:
        siblings = time_siblings(dev, stream, flush, flush_bytes, min(other_steps, 200), args.warmup,
                                 with_allreduce=args.with_allreduce)

    # the smallest workload, latency-bound: eager calls vs CUDA-graph replay
    tiny_graph = None
    if rank == 0 and not args.no_graph:
        try:
            tiny_graph = time_tiny_graph(dev)
        except Exception as e:   # reported, not fatal: the headline line stands on its own
            tiny_graph = {"error": str(e).splitlines()[0][:200]}

    bf16_tf, hbm, peak_src = measured_peaks()
    p_fp8 = bf16_tf * FP8_OVER_BF16
    t_roof, bound = roofline_terms(w, p_fp8, hbm)
    kern_avg_s = (sum(kern_ms) / len(kern_ms) / 1e3) if kern_ms else None
    if bound == "tensor":
        achieved = w.flops / kern_avg_s / 1e12 if kern_avg_s else None
        peak, r_unit = p_fp8, "TFLOP/s"
        peak_note = f"{peak_src} bf16 {bf16_tf:.0f} TFLOP/s (burst) x nominal fp8:bf16 ratio 2"
    else:
        achieved = w.bytes_alg / kern_avg_s / 1e9 if kern_avg_s else None
        peak, r_unit = hbm, "GB/s"
        peak_note = f"{peak_src} HBM copy bandwidth"

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0

    cpu = None
    if not args.no_cpu_baseline:
        tf, rows, dt, cores = time_oracle(w, x, seconds=args.cpu_seconds)
        cpu = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"rows 0..{rows - 1} of C ({rows} x {w.N} outputs, full K={w.K}), one call, "
                         f"{dt:.1f} s wall"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8", "data": "synthetic",
        "config": {"workload": w.name, "R": w.R, "M": w.M, "kPerRank": w.kPerRank, "K": w.K, "N": w.N,
                   "commMSize": w.commMSize, "buffer_num": w.buffer_num, "seed": w.seed,
                   "path": args.path, "parallelism": "replicas" if ws > 1 else "single",
                   "splits": plan.get_option(mxa2a.MXA2A_INFO_SPLITS),
                   "tail_split": plan.get_option(mxa2a.MXA2A_INFO_TAIL_SPLIT if args.path == "fused"
                                                 else mxa2a.MXA2A_INFO_TAIL_SPLIT_UNFUSED),
                   "cta_pair": plan.get_option(mxa2a.MXA2A_INFO_CTA_PAIR if args.path == "fused"
                                               else mxa2a.MXA2A_INFO_CTA_PAIR_UNFUSED),
                   "grid": plan.get_option(mxa2a.MXA2A_INFO_GRID_FUSED if args.path == "fused"
                                           else mxa2a.MXA2A_INFO_GRID_UNFUSED),
                   "raster_group_m": plan.get_option(mxa2a.MXA2A_INFO_GROUP_FUSED if args.path == "fused"
                                                     else mxa2a.MXA2A_INFO_GROUP_UNFUSED),
                   "l2": f"flushed before every step ({flush_bytes >> 20} MiB write, 2x L2), outside the events",
                   "timer": "CUDA events on the launch stream around each library call"},
        "roofline_pct": 100.0 * t_roof / (ms_per_step / 1e3),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": r_unit,
                     "frac": (achieved / peak) if achieved else None,
                     "traffic": profiled_traffic(w.name),
                     "kernel": "mxgemm_kernel<fused>" if args.path == "fused" else "mxgemm_kernel<unfused>",
                     "kernel_ms_avg": kern_avg_s * 1e3 if kern_avg_s else None,
                     "peak_note": peak_note, "t_roof_us": t_roof * 1e6, "hbm_gbs": hbm},
        "unfused" if args.path == "fused" else "fused": {
            "ms_per_step": sum(other_ms) / len(other_ms), "steps": other_steps,
            "value": w.flops / (sum(other_ms) / len(other_ms) / 1e3) / 1e12},
        "direct_read": None if direct_ms is None else {
            "ms_per_step": sum(direct_ms) / len(direct_ms), "steps": other_steps,
            "value": w.flops / (sum(direct_ms) / len(direct_ms) / 1e3) / 1e12,
            "what": "A read in place from the segments (no staging ring, no pack): the exchange's cost"},
        "configs": configs,
        "credit_ablation": credit_ablation,
        "siblings": siblings,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(args.steps * (1 + launches_per_run)),
        "clocks": clocks,
        "tiny_graph": tiny_graph,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    plan.destroy()
    return 0


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=str(DEFAULT_WORKLOAD))
    ap.add_argument("--shape", default="",
                    help="R,M,kPerRank,N,commMSize,buffer_num[,seed]: a synthetic problem of these sizes instead of "
                         "--workload (the benchmark problems' input recipe), e.g. a smaller case to profile")
    ap.add_argument("--path", choices=["fused", "unfused"], default="fused")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph timing of the smallest workload")
    ap.add_argument("--no-ablation", action="store_true", help="skip the staging-protocol ablation timings")
    ap.add_argument("--no-siblings", action="store_true", help="skip the sibling operators' timings")
    ap.add_argument("--with-allreduce", action="store_true",
                    help="also time GEMM + AllReduce (one-shot) among the sibling operators")
    ap.add_argument("--no-configs", action="store_true", help="skip the other problem sizes' timings")
    ap.add_argument("--config-steps", type=int, default=200, help="timed steps per other problem size")
    ap.add_argument("--other-steps", type=int, default=500,
                    help="timed steps of the unfused and direct-read comparison paths")
    ap.add_argument("--only-siblings", action="store_true",
                    help="time only the sibling operators (one JSON line of their timings, not the benchmark line)")
    ap.add_argument("--skew-ns", type=int, default=4000, help="copy delay of every 4th CTA in the ablation")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--split", type=int, default=0, help="force the K split of both paths (0 = automatic)")
    ap.add_argument("--single-cta", action="store_true", help="never use the CTA-pair kernel")
    ap.add_argument("--cta-pair", action="store_true", help="use the CTA-pair kernel where the shape allows it")
    ap.add_argument("--group-m", type=int, default=0, help="largest unfused raster group in m-tiles (0 = library default)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from all_mxfp8_block_gb300 import inputs
    if args.shape:
        v = [int(s) for s in args.shape.split(",")]
        if len(v) not in (6, 7):
            ap.error("--shape wants R,M,kPerRank,N,commMSize,buffer_num[,seed]")
        R, M, ka, N, cm, bn = v[:6]
        w = inputs.Workload(f"r{R}_m{M}_k{R * ka}_n{N}", R, M, ka, N, cm, bn, v[6] if len(v) == 7 else 0)
    else:
        w = inputs.workload(int(args.workload)) if args.workload.isdigit() else inputs.workload(args.workload)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.only_siblings:
        return run_siblings_only(args)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
