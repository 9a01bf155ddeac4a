"""RMSNorm throughput on GB300: achieved HBM GB/s of forward, fused residual-add
forward and backward, bf16, against the HBM roofline.

One step = the whole path once on the three full-size workloads:
  forward    16384 x 8192  bf16 (bf16 gamma, writes y and fp32 rstd)
  fused add  32768 x 4096  bf16 (h = r + x over r, y; 0.1 % outliers in r, x)
  backward   16384 x 8192  bf16 (fp32 gamma, saved rstd; dx and fp32 dgamma)
value = algorithmic HBM bytes of the step / device time of the step.  Every
operand is at least 256 MiB, larger than the 126 MiB L2, so no flush is
needed between steps.  Launch with torchrun for N > 1: every rank runs the
same workload on its own GPU (independent replicas, weak scaling) and the
slowest rank's time counts.

--impl reference times the double-precision CPU oracle on the same step
(bounded row samples of each workload), on this host's cores.
--sweep prints one line per workload of the shape sweep (and the three step
workloads) instead: back-to-back launches rotating over enough operand copies
that no launch finds its operands in L2.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RMSNorm fwd/fused-add/bwd achieved HBM GB/s and % of GB300 peak (bf16, M x N)"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
STEP_WORKLOADS = ("fwd_bf16_m16384_n8192", "fadd_bf16_m32768_n4096", "bwd_bf16_m16384_n8192")
LAUNCHES_PER_OP = {"fwd": 1, "fused_add": 1, "bwd": 2}


def esize(dt):
    return 4 if dt == "f32" else 2


def alg_bytes(wl, rows=None) -> int:
    """Bytes the operation must move: activations per row, plus gamma (and
    dgamma) once per call; the dgamma workspace is not counted."""
    M = wl.M if rows is None else rows
    sx, sw, N = esize(wl.x_dtype), esize(wl.w_dtype), wl.N
    rstd = 4 * M if (wl.store_rstd and wl.op != "bwd") else 0
    if wl.op in ("fwd", "fwd_strided"):   # strided: only the rows move, not the gaps
        return M * N * 2 * sx + N * sw + rstd
    if wl.op == "fused_add":
        return M * N * 4 * sx + N * sw + rstd
    if wl.op == "fused_add_bwd":   # h, dy, dres in; dh out; dgamma in the weight dtype
        return M * N * 4 * sx + 4 * M + N * sw + N * sw
    if wl.op == "ln_fwd":    # x in, y out; gamma and beta; mean and rstd out
        return M * N * 2 * sx + 2 * N * sw + 8 * M
    if wl.op == "ln_bwd":    # x, dy, mean, rstd in; dx out; dgamma and dbeta out (fp32)
        return M * N * 3 * sx + 8 * M + N * sw + 8 * N
    if wl.op in ("fwd_fp8", "fused_add_fp8", "fwd_nvfp4", "fused_add_nvfp4"):
        # x (fused: r and x in, h out), then codes and scales out
        act = M * N * (3 if wl.op.startswith("fused") else 1) * sx
        codes = M * N + 4 * M if "fp8" in wl.op else M * N // 2 + M * N // 16
        return act + codes + N * sw + rstd
    return M * N * 3 * sx + 4 * M + N * sw + 4 * N


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The files the step's kernels are compiled from: the forward and fused-add
# register kernels, the staged backward and its stage 2, and what they include.
STEP_KERNEL_SOURCES = ("rmsnorm_fwd.cu", "rmsnorm_fwd_common.cuh", "rmsnorm_staged.cu",
                       "rmsnorm_ring.cuh", "rmsnorm_device.cuh", "rmsnorm_internal.h")


def source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_wise_normalization_02_gb300", "csrc")
    for f in STEP_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(op: str, variant: str):
    """DRAM bytes per launch of an op from the committed ncu summary, or None
    when the summary is missing, was taken on other kernel sources, or on
    another variant than the one the dispatch picks now."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_hash") != source_hash() or d.get("variants", {}).get(op) != variant:
        return None
    v = d.get("per_launch_bytes", {}).get(op)
    return int(v) if v is not None else None


# ------------------------------------------------------------------ ranks

def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time (all ranks get it)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes: int, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every rank moves step_bytes per step (replicas)."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while it runs."""

    QUERY = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid=None, period_ms=50):
        self.proc = None
        self.uuid = (device_uuid or "").lower().replace("gpu-", "")
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               f"-lms={period_ms}"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        self.lines = []

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        uuids = {ln.split(",")[0].strip().lower() for ln in self.lines}
        for ln in self.lines:
            f = [c.strip() for c in ln.split(",")]
            if len(uuids) > 1 and self.uuid and not f[0].lower().endswith(self.uuid):
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names[1:], f[5:9]):
                if v.lower().startswith("active") or v == "0x1":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, world):
    import torch

    import __graft_entry__
    import row_wise_normalization_02_gb300 as rn
    import seeded_inputs as si

    __graft_entry__.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    wls = [si.WORKLOADS[n] for n in STEP_WORKLOADS]

    def to_dev(a):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        return t.to(dev)

    ops = []
    host = []
    for wl in wls:
        inp = si.make_inputs(wl)
        d = {k: to_dev(v) for k, v in inp.items()}
        act = torch.int16 if wl.x_dtype == "bf16" else torch.float32
        M, N, eps = wl.M, wl.N, float(np.float32(wl.eps))
        if wl.op == "fwd":
            d["y"] = torch.empty((M, N), dtype=act, device=dev)
            d["rstd"] = torch.empty(M, dtype=torch.float32, device=dev)

            def launch(d=d, wl=wl, M=M, N=N, eps=eps):
                rn.rmsnorm_fwd(d["x"], d["gamma"], d["y"], d["rstd"], M, N, eps, wl.x_dtype,
                               wl.w_dtype, stream)

            def launch_rows(r0, m, d=d, wl=wl, N=N, eps=eps):
                rn.rmsnorm_fwd(d["x"][r0:r0 + m], d["gamma"], d["y"][r0:r0 + m],
                               d["rstd"][r0:r0 + m], m, N, eps, wl.x_dtype, wl.w_dtype, stream)
            outs = ("y", "rstd")
            ins = ("x", "gamma")
        elif wl.op == "fused_add":
            d["y"] = torch.empty((M, N), dtype=act, device=dev)

            def launch(d=d, wl=wl, M=M, N=N, eps=eps):
                rn.rmsnorm_fused_add_fwd(d["x"], d["residual"], d["gamma"], d["y"], None, M, N,
                                         eps, wl.x_dtype, wl.w_dtype, stream)

            def launch_rows(r0, m, d=d, wl=wl, N=N, eps=eps):
                rn.rmsnorm_fused_add_fwd(d["x"][r0:r0 + m], d["residual"][r0:r0 + m], d["gamma"],
                                         d["y"][r0:r0 + m], None, m, N, eps, wl.x_dtype,
                                         wl.w_dtype, stream)
            outs = ("residual", "y")
            ins = ("x", "residual", "gamma")
        else:
            d["dx"] = torch.empty((M, N), dtype=act, device=dev)
            d["dgamma"] = torch.empty(N, dtype=torch.float32, device=dev)
            d["rstd"] = torch.empty(M, dtype=torch.float32, device=dev)
            ws = rn.rmsnorm_bwd_workspace_size(M, N, wl.x_dtype, wl.w_dtype)
            d["ws"] = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
            # saved rstd of this x, from the forward kernel (outside timing)
            ytmp = torch.empty((M, N), dtype=act, device=dev)
            with torch.cuda.stream(stream):
                rn.rmsnorm_fwd(d["x"], d["gamma"], ytmp, d["rstd"], M, N, eps, wl.x_dtype,
                               wl.w_dtype, stream)
            stream.synchronize()
            del ytmp

            def launch(d=d, wl=wl, M=M, N=N, eps=eps, ws=ws):
                rn.rmsnorm_bwd(d["dy"], d["x"], d["rstd"], d["gamma"], d["dx"], d["dgamma"],
                               d["ws"], ws, M, N, eps, wl.x_dtype, wl.w_dtype, stream)
            def launch_rows(r0, m, launch=launch):
                launch()
            outs = ("dx", "dgamma")
            ins = ("x", "dy", "rstd", "gamma")
        plan = rn.rmsnorm_describe_plan({"fwd": 0, "fused_add": 1, "bwd": 2}[wl.op], M, N,
                                        wl.x_dtype, wl.w_dtype)
        ops.append(dict(wl=wl, d=d, launch=launch, launch_rows=launch_rows, outs=outs, ins=ins,
                        plan=plan, bytes=alg_bytes(wl)))
        host.append(inp)
    torch.cuda.synchronize()

    copy_gbs = inrun_copy_gbs(dev, stream)
    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for _ in range(W):
            for op in ops:
                op["launch"]()
    stream.synchronize()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    # timed region 1: K steps back to back, nothing between the launches, so
    # each kernel's launch overlaps the previous one (programmatic dependent
    # launch) as it would in a model
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for i in range(K):
            for op in ops:
                op["launch"]()
        t_end.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if sampler:
        sampler.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    # timed region 2: each op alone, K calls back to back in 5 rounds, one
    # event pair around each round (no events between the launches, so the
    # launch overlap of consecutive calls stays as in region 1): the op's
    # steady rate, as in --sweep
    step_bytes = sum(op["bytes"] for op in ops)
    ms_per_step = total_ms / K
    value = job_gbs(step_bytes, ms_per_step, world)
    peak, peak_src = measured_peak()
    rounds = 5
    per_round = max(1, K // rounds)
    per_op = {}
    for op in ops:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(rounds)]
        with torch.cuda.stream(stream):
            for a, b in ev:
                a.record(stream)
                for _ in range(per_round):
                    op["launch"]()
                b.record(stream)
        stream.synchronize()
        times = [a.elapsed_time(b) / per_round for a, b in ev]
        avg = statistics.median(times)
        gbs = op["bytes"] / (avg * 1e-3) / 1e9
        wl = op["wl"]
        per_op[wl.op] = {"workload": wl.name, "avg_us": round(avg * 1e3, 2),
                         "rounds_us": [round(t * 1e3, 2) for t in times],
                         "min_us": round(min(times) * 1e3, 2), "gbs": round(gbs, 1),
                         "frac_of_measured_peak": round(gbs / peak, 4),
                         "rows_per_s": round(wl.M / (avg * 1e-3), 1),
                         "alg_bytes": op["bytes"], "launches": LAUNCHES_PER_OP[wl.op],
                         "variant": op["plan"]}
    dom = max(per_op, key=lambda k: per_op[k]["avg_us"])
    d = per_op[dom]
    roofline = {"bound": "hbm", "achieved": d["gbs"], "peak": peak, "unit": "GB/s",
                "frac": round(d["gbs"] / peak, 4), "traffic": ncu_traffic(dom, d["variant"]),
                "kernel": f"{dom} ({d['workload']}, {d['variant']})",
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src ==
                "measured" else "fallback 6800 GB/s"}

    # ---- end to end through the C ABI with pinned host buffers: every step
    # copies each op's inputs in and its outputs out.  Three streams overlap
    # host->device copies, kernels and device->host copies; the forward and the
    # fused add (row-independent) go in row chunks so a chunk computes while
    # the next one arrives.  The backward is one call (dgamma sums all rows).
    Ke = max(3, min(K, args.e2e_steps))
    pin = []
    h2d = d2h = 0
    for op, inp in zip(ops, host):
        hin = {k: torch.from_numpy(inp[k].view(np.int16) if inp[k].dtype == np.uint16
                                   else inp[k]).pin_memory() for k in op["ins"] if k in inp}
        if "rstd" in op["ins"]:
            hin["rstd"] = op["d"]["rstd"].cpu().pin_memory()
        hout = {k: torch.empty_like(op["d"][k], device="cpu").pin_memory() for k in op["outs"]}
        h2d += sum(t.numel() * t.element_size() for t in hin.values())
        d2h += sum(t.numel() * t.element_size() for t in hout.values())
        pin.append((hin, hout))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    chunks = max(1, args.e2e_chunks)

    def row_chunks(wl):
        if wl.op == "bwd":
            return [(0, wl.M)]
        step_rows = -(-wl.M // chunks)
        return [(r, min(step_rows, wl.M - r)) for r in range(0, wl.M, step_rows)]

    def copy_rows(dst, src, key, r0, m, wl):
        if key in ("gamma",) or (key == "rstd" and wl.op == "bwd"):
            if r0 == 0:
                dst.copy_(src, non_blocking=True)
        elif key == "rstd":
            dst[r0:r0 + m].copy_(src[r0:r0 + m], non_blocking=True)
        else:
            dst[r0:r0 + m].copy_(src[r0:r0 + m], non_blocking=True)

    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    done = [None] * len(ops)       # last device->host copy of each op's previous step
    e0.record(s_in)
    t_host = time.perf_counter()
    for _ in range(Ke):
        for j, (op, (hin, hout)) in enumerate(zip(ops, pin)):
            wl = op["wl"]
            if done[j] is not None:
                s_in.wait_event(done[j])     # its buffers are free again
            for r0, m in row_chunks(wl):
                with torch.cuda.stream(s_in):
                    for k, t in hin.items():
                        copy_rows(op["d"][k], t, k, r0, m, wl)
                    arrived = torch.cuda.Event()
                    arrived.record(s_in)
                stream.wait_event(arrived)
                with torch.cuda.stream(stream):
                    op["launch_rows"](r0, m)
                    computed = torch.cuda.Event()
                    computed.record(stream)
                s_out.wait_event(computed)
                with torch.cuda.stream(s_out):
                    for k, t in hout.items():
                        if k == "dgamma":
                            t.copy_(op["d"][k], non_blocking=True)
                        else:
                            t[r0:r0 + m].copy_(op["d"][k][r0:r0 + m], non_blocking=True)
                    out_done = torch.cuda.Event()
                    out_done.record(s_out)
            done[j] = out_done
    for ev_done in done:
        s_in.wait_event(ev_done)
    e1.record(s_in)
    host_ms = (time.perf_counter() - t_host) * 1e3 / Ke   # enqueueing, not waiting
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / Ke, world, dev)

    # the host link's bound for these bytes: the same copies, whole tensors,
    # with no kernels and no dependencies (copy in and copy out at once).  The
    # fused add's residual is both input and output: its copy out reads y (same
    # size) so that the two directions never touch the same buffer.
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    c0.record(s_in)
    s_out.wait_event(c0)
    for _ in range(Ke):
        for op, (hin, hout) in zip(ops, pin):
            with torch.cuda.stream(s_in):
                for k, t in hin.items():
                    op["d"][k].copy_(t, non_blocking=True)
            with torch.cuda.stream(s_out):
                for k, t in hout.items():
                    t.copy_(op["d"]["y" if k == "residual" else k], non_blocking=True)
    s_in.wait_stream(s_out)
    c1.record(s_in)
    torch.cuda.synchronize()
    copy_ms = c0.elapsed_time(c1) / Ke
    e2e = {"value": round(job_gbs(step_bytes, e2e_ms, world), 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
           "ms_per_step": round(e2e_ms, 3), "pinned": True,
           "pipeline": f"3 streams (copy in / kernels / copy out), fwd and fused add in "
                       f"{chunks} row chunks",
           "copy_bound_ms_per_step": round(copy_ms, 3),
           "host_enqueue_ms_per_step": round(host_ms, 3),
           "frac_of_copy_bound": round(copy_ms / e2e_ms, 4),
           "copy_bound": "the same host<->device copies alone (no kernels, no dependencies, "
                         "both directions at once), timed on this GPU"}

    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "rmsnorm step: fwd bf16 16384x8192 (+rstd) + fused-add bf16 "
                                   "32768x4096 + bwd bf16 16384x8192 (fp32 gamma, dgamma)",
                       "step_alg_bytes": step_bytes,
                       "l2": "inputs larger than L2 (every operand >= 256 MiB; L2 126 MiB)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "frac_of_measured_peak": round(value / world / peak, 4),
            "frac_of_nominal_7900": round(value / world / NOMINAL_HBM_GBS, 4),
            "inrun_copy_gbs": round(copy_gbs, 1),
            "frac_of_inrun_copy": round(value / world / copy_gbs, 4),
            "roofline": roofline, "ops": per_op, "e2e": e2e,
            "gpu_launches": K * sum(LAUNCHES_PER_OP[op["wl"].op] for op in ops),
            "gpu_launches_per_op_region": {op["wl"].op: per_round * rounds *
                                           LAUNCHES_PER_OP[op["wl"].op] for op in ops},
            "timing": {"value": "CUDA events around K back-to-back steps on the launching stream",
                       "ops": "per op: CUDA events around 5 rounds of K/5 back-to-back calls "
                              "of that op alone; median round"},
            "clocks": sampler.summary() if sampler else None}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


# ------------------------------------------------------------------ oracle

def _oracle_step(samples):
    """Run the oracle once over the sampled rows of the three workloads."""
    import oracle
    t0 = time.perf_counter()
    done = 0
    for wl, inp in samples:
        eps = float(np.float32(wl.eps))
        if wl.op == "fwd":
            oracle.fwd(inp["x"], inp["gamma"], eps, wl.x_dtype, wl.w_dtype, want64=False)
        elif wl.op == "fused_add":
            oracle.fused_add_fwd(inp["x"], inp["residual"], inp["gamma"], eps, wl.x_dtype,
                                 wl.w_dtype, want64=False)
        else:
            oracle.bwd(inp["dy"], inp["x"], inp["rstd"], inp["gamma"], eps, wl.x_dtype,
                       wl.w_dtype, want64=False)
        done += alg_bytes(wl, rows=inp["x"].shape[0])
    return time.perf_counter() - t0, done


def _oracle_step_threads(samples, threads):
    """The same step over `threads` row blocks of every workload at once: the
    oracle's C calls release the interpreter lock, so the blocks run on that
    many host cores (the oracle itself unchanged)."""
    from concurrent.futures import ThreadPoolExecutor
    blocks = []
    for wl, inp in samples:
        M = inp["x"].shape[0]
        edges = np.linspace(0, M, min(threads, M) + 1).astype(int)
        for a, b in zip(edges[:-1], edges[1:]):
            if b > a:
                part = {k: (v[a:b] if k in ("x", "residual", "dy", "rstd") else v)
                        for k, v in inp.items()}
                blocks.append((wl, part))
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda blk: _oracle_step([blk]), blocks))
    t = time.perf_counter() - t0
    # the bytes of the whole sample (per-call terms such as gamma counted once)
    return t, sum(alg_bytes(wl, rows=inp["x"].shape[0]) for wl, inp in samples)


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _samples(rows_fraction):
    import oracle
    import seeded_inputs as si
    out = []
    for n in STEP_WORKLOADS:
        wl = si.WORKLOADS[n]
        rows = max(1, int(wl.M * rows_fraction))
        inp = si.make_inputs(wl, rows=rows)
        if wl.op == "bwd":
            inp["rstd"] = oracle.fwd(inp["x"], inp["gamma"], float(np.float32(wl.eps)),
                                     wl.x_dtype, wl.w_dtype, want64=False)["rstd"]
        out.append((wl, inp))
    return out


def cpu_baseline(target_s=12.0):
    """The oracle as it stands (single-threaded C, double precision) on a
    bounded row sample of each workload of the step, scaled to GB/s."""
    probe = _samples(1 / 256)
    t, b = _oracle_step(probe)
    frac = min(1.0, max(1 / 256, target_s / max(t, 1e-6) / 256))
    samples = _samples(frac)
    t, b = _oracle_step(samples)
    n = host_threads()
    tn, bn = _oracle_step_threads(samples, n)
    rows = {wl.name: inp["x"].shape[0] for wl, inp in samples}
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(t, 2),
            "sample": "first rows of each step workload: " +
                      ", ".join(f"{k} {v} rows" for k, v in rows.items()),
            "all_cores": {"value": round(bn / tn / 1e9, 4), "cores": n,
                          "seconds": round(tn, 2),
                          "how": "the same sample in row blocks on that many threads"}}


def run_reference(args):
    """Reference arm: the oracle on all the host cores (row blocks on as many
    threads), K timed steps after W warm-up steps, each step a bounded row
    sample of the three workloads."""
    budget_s = 120.0
    n = host_threads()
    probe = _samples(1 / 512)
    t, _ = _oracle_step_threads(probe, n)
    per_step = budget_s / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1 / 16384, per_step / max(t, 1e-6) / 512))
    samples = _samples(frac)
    for _ in range(args.warmup):
        _oracle_step_threads(samples, n)
    tot_t = tot_b = 0.0
    for _ in range(args.steps):
        t, b = _oracle_step_threads(samples, n)
        tot_t += t
        tot_b += b
    value = tot_b / tot_t / 1e9
    rows = {wl.name: inp["x"].shape[0] for wl, inp in samples}
    sample = "first rows of each step workload: " + ", ".join(f"{k} {v} rows"
                                                             for k, v in rows.items())
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "rmsnorm step: fwd bf16 16384x8192 (+rstd) + fused-add bf16 "
                                   "32768x4096 + bwd bf16 16384x8192 (fp32 gamma, dgamma)",
                       "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n,
                             "kind": "oracle", "sample": sample + f", in row blocks on {n} "
                                                                  "threads"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ sweep

def _op_code(op):
    return {"fwd": 0, "fused_add": 1, "bwd": 2, "fused_add_bwd": 3, "fwd_strided": 4,
            "fwd_fp8": 5, "fused_add_fp8": 6, "fwd_nvfp4": 7, "fused_add_nvfp4": 8,
            "ln_fwd": 9, "ln_bwd": 10}[op]


def device_sets(wl, inp, dev, l2_bytes, rn):
    """Device copies of one workload's operands, repeated until the rotation
    covers at least 3 x L2 (so every launch reads operands that are not in L2)
    -- one set when a single call already streams that much."""
    import torch
    per_set = alg_bytes(wl)
    nsets = 1 if per_set >= 3 * l2_bytes else min(64, -(-3 * l2_bytes // per_set))
    act = torch.int16 if wl.x_dtype == "bf16" else torch.float32
    host = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v)
            for k, v in inp.items()}
    M, N = wl.M, wl.N
    off = dict(wl.offsets)

    def placed(k, v):
        # an operand `off[k]` bytes past a 16-byte boundary: a view into a
        # slightly larger buffer (allocations start on 256 bytes)
        if not off.get(k):
            return v.to(dev)
        e = v.element_size()
        assert off[k] % e == 0
        buf = torch.empty(v.numel() + 16 // e, dtype=v.dtype, device=dev)
        view = buf[off[k] // e: off[k] // e + v.numel()].view(v.shape)
        view.copy_(v.to(dev))
        return view

    sets = []
    for _ in range(nsets):
        d = {k: placed(k, v) for k, v in host.items()}
        if wl.op.startswith("ln_"):
            d["y"] = torch.empty((M, N), dtype=act, device=dev)
            d["mean"] = torch.empty(M, dtype=torch.float32, device=dev)
            d["dgamma"] = torch.empty(N, dtype=torch.float32, device=dev)
            d["dbeta"] = torch.empty(N, dtype=torch.float32, device=dev)
        elif "fp8" in wl.op:
            d["q"] = torch.empty((M, N), dtype=torch.uint8, device=dev)
            d["qs"] = torch.empty(M, dtype=torch.float32, device=dev)
        elif "nvfp4" in wl.op:
            d["q"] = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
            d["qs"] = torch.empty((M, N // 16), dtype=torch.uint8, device=dev)
        elif wl.op != "fwd_strided":   # the strided forward writes in place
            yoff = off.get("dx" if wl.op in ("bwd", "fused_add_bwd") else "y", 0)
            if yoff:   # an output placed off 16 bytes, like `placed`
                e = torch.empty((), dtype=act).element_size()
                buf = torch.empty(M * N + 16 // e, dtype=act, device=dev)
                d["y"] = buf[yoff // e: yoff // e + M * N].view(M, N)
            else:
                d["y"] = torch.empty((M, N), dtype=act, device=dev)
        d["rstd"] = torch.empty(M, dtype=torch.float32, device=dev)
        if wl.op == "bwd":
            d["dgamma"] = torch.empty(N, dtype=torch.float32, device=dev)
        if wl.op == "fused_add_bwd":
            d["dgamma"] = torch.empty(N, dtype=torch.int16 if wl.w_dtype == "bf16"
                                      else torch.float32, device=dev)
        sets.append(d)
    return sets


def make_launch(wl, d, stream, rn):
    """A closure that enqueues one call of the workload's op on `stream`."""
    M, N, eps = wl.M, wl.N, float(np.float32(wl.eps))
    if wl.op == "fwd":
        return lambda: rn.rmsnorm_fwd(d["x"], d["gamma"], d["y"],
                                      d["rstd"] if wl.store_rstd else None, M, N, eps,
                                      wl.x_dtype, wl.w_dtype, stream)
    if wl.op == "fused_add":
        return lambda: rn.rmsnorm_fused_add_fwd(d["x"], d["residual"], d["gamma"], d["y"],
                                                d["rstd"] if wl.store_rstd else None, M, N,
                                                eps, wl.x_dtype, wl.w_dtype, stream)
    if wl.op == "ln_fwd":
        return lambda: rn.layernorm_fwd(d["x"], d["gamma"], d["beta"], d["y"], d["mean"],
                                        d["rstd"], M, N, eps, wl.x_dtype, wl.w_dtype, stream)
    if wl.op == "ln_bwd":      # mean and rstd: the (untimed) forward's, saved in the set
        import torch
        lws = rn.layernorm_bwd_workspace_size(M, N, wl.x_dtype, wl.w_dtype)
        d["lws"] = torch.empty(max(16, lws), dtype=torch.uint8, device=d["x"].device)
        return lambda: rn.layernorm_bwd(d["dy"], d["x"], d["mean"], d["rstd"], d["gamma"],
                                        d["y"], d["dgamma"], d["dbeta"], d["lws"], lws, M, N,
                                        eps, wl.x_dtype, wl.w_dtype, stream)
    if "fp8" in wl.op:
        return lambda: rn.rmsnorm_fwd_fp8(d["x"], d.get("residual"), d["gamma"], d["q"], d["qs"],
                                          d["rstd"] if wl.store_rstd else None, M, N, eps,
                                          wl.x_dtype, wl.w_dtype, stream)
    if "nvfp4" in wl.op:
        return lambda: rn.rmsnorm_fwd_nvfp4(d["x"], d.get("residual"), d["gamma"],
                                            wl.global_scale, d["q"], d["qs"],
                                            d["rstd"] if wl.store_rstd else None, M, N, eps,
                                            wl.x_dtype, wl.w_dtype, stream)
    if wl.op == "fwd_strided":   # the q slice of each token, normalised in place
        st, H = wl.stride_token, wl.heads
        return lambda: rn.rmsnorm_fwd_strided(d["x"], st, N, d["gamma"], d["x"], st, N,
                                              d["rstd"] if wl.store_rstd else None, M // H, H,
                                              N, eps, wl.x_dtype, wl.w_dtype, stream)
    ws = rn.rmsnorm_bwd_workspace_size(M, N, wl.x_dtype, wl.w_dtype)
    import torch
    d["ws"] = torch.empty(max(16, ws), dtype=torch.uint8, device=d["x"].device)
    if wl.op == "fused_add_bwd":   # dres (the residual set) is overwritten with dh
        return lambda: rn.rmsnorm_fused_add_bwd(d["dy"], d["x"], d["rstd"], d["gamma"],
                                                d["residual"], d["dgamma"], wl.w_dtype, d["ws"],
                                                ws, M, N, eps, wl.x_dtype, wl.w_dtype, stream)
    return lambda: rn.rmsnorm_bwd(d["dy"], d["x"], d["rstd"], d["gamma"], d["y"], d["dgamma"],
                                  d["ws"], ws, M, N, eps, wl.x_dtype, wl.w_dtype, stream)


def time_rotation(launches, steps, warmup, stream):
    """Average device time (ms) per launch of `steps` back-to-back launches
    cycling through the operand sets, after `warmup` untimed ones: one event
    pair around the whole batch, so the number is steady-state throughput
    (inter-kernel gaps included, no per-launch event overhead)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(warmup):
            launches[i % len(launches)]()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            launches[(warmup + i) % len(launches)]()
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b) / steps


def plan_layout(wl):
    """The layout argument of rmsnorm_describe_plan for a workload's operand
    offsets: True (all on 16 bytes), "mixed" (inputs off outputs that agree)
    or False (outputs that disagree: the scalar kernel)."""
    if not wl.offsets:
        return True
    off = dict(wl.offsets)
    outs = {"fwd": ["y"], "fused_add": ["residual", "y"], "bwd": ["dx"],
            "fused_add_bwd": ["residual"]}.get(wl.op, ["y"])
    return "mixed" if len({off.get(k, 0) % 16 for k in outs}) == 1 else False


def time_graph(launches, calls, reps, stream):
    """Device time (ms) per call of `calls` back-to-back launches captured once
    in a CUDA graph (so no host work between them: the GPU-side cost of a call,
    which the eager rotation hides when the host enqueues slower than the GPU
    runs); median of `reps` replays, CUDA events around each."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(len(launches)):
            launches[i]()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(calls):
            launches[i % len(launches)]()
    ms = []
    with torch.cuda.stream(stream):
        g.replay()
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b) / calls)
    del g
    return statistics.median(ms)


def inrun_copy_gbs(dev, stream, nbytes=1 << 30, reps=10):
    """Device-to-device copy bandwidth measured in this run (cudaMemcpyAsync of
    a 1 GiB buffer; read + write bytes, the convention of the measured peak)."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    src.fill_(1)
    with torch.cuda.stream(stream):
        for _ in range(2):
            dst.copy_(src, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
    stream.synchronize()
    ms = a.elapsed_time(b) / reps
    del src, dst
    torch.cuda.empty_cache()
    return 2 * nbytes / (ms * 1e-3) / 1e9


def run_sweep(args):
    import torch

    import __graft_entry__
    import row_wise_normalization_02_gb300 as rn
    import seeded_inputs as si

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    peak, _ = measured_peak()
    copy_gbs = inrun_copy_gbs(dev, stream)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    names = args.workloads.split(",") if args.workloads else [
        n for n, w in si.WORKLOADS.items()
        if set(w.tags) & {"sweep", "headline", "next", "mixed", "wide"}]
    for name in names:
        wl = si.WORKLOADS[name]
        inp = si.make_inputs(wl)
        sets = device_sets(wl, inp, dev, l2, rn)
        # saved statistics for the backward (untimed forward, default variant
        # even when RMSNORM_FORCE_VARIANT names a backward-only one)
        forced = os.environ.pop("RMSNORM_FORCE_VARIANT", None)
        if forced is not None:
            rn.rmsnorm_reload_debug_env()
        for d in sets:
            if wl.op == "ln_bwd":
                gam = d["gamma"]
                rn.layernorm_fwd(d["x"], gam, None, d["y"], d["mean"], d["rstd"], wl.M, wl.N,
                                 float(np.float32(wl.eps)), wl.x_dtype, wl.w_dtype, stream)
                continue
            if wl.op not in ("bwd", "fused_add_bwd"):
                break
            rn.rmsnorm_fwd(d["x"], d["gamma"], d["y"], d["rstd"], wl.M, wl.N,
                           float(np.float32(wl.eps)), wl.x_dtype, wl.w_dtype, stream)
        torch.cuda.synchronize()
        if forced is not None:
            os.environ["RMSNORM_FORCE_VARIANT"] = forced
            rn.rmsnorm_reload_debug_env()
        launches = [make_launch(wl, d, stream, rn) for d in sets]
        us = [time_rotation(launches, args.steps, args.warmup, stream) * 1e3
              for _ in range(args.rounds)]
        med = statistics.median(us)
        byts = alg_bytes(wl)
        graph = {}
        if args.graph:
            calls = max(len(launches), min(args.steps, 200))
            g_us = time_graph(launches, calls, args.rounds, stream) * 1e3
            graph = {"graph_us_per_call": round(g_us, 2),
                     "graph_frac_of_measured_peak": round(byts / g_us / 1e3 / peak, 4),
                     "graph": f"{calls} calls captured in one CUDA graph, median of "
                              f"{args.rounds} replays"}
        print(json.dumps({"workload": name, "op": wl.op, "M": wl.M, "N": wl.N,
                          "variant": rn.rmsnorm_describe_plan(
                              _op_code(wl.op), wl.M, wl.N, wl.x_dtype, wl.w_dtype,
                              plan_layout(wl)),
                          "us_per_call": round(med, 2), "rounds_us": [round(u, 2) for u in us],
                          "min_us": round(min(us), 2),
                          "spread": round((max(us) - min(us)) / med, 4),
                          "interference": (max(us) - min(us)) / med > 0.10,
                          "gbs": round(byts / med / 1e3, 1),
                          "frac_of_measured_peak": round(byts / med / 1e3 / peak, 4),
                          "inrun_copy_gbs": round(copy_gbs, 1),
                          "frac_of_inrun_copy": round(byts / med / 1e3 / copy_gbs, 4),
                          "rows_per_s": round(wl.M / med * 1e6, 1), "alg_bytes": byts,
                          "l2": f"rotation over {len(sets)} operand set(s) "
                                f">= 3 x L2, back-to-back launches",
                          "timer": "CUDA events around each round of back-to-back calls; "
                                   "median of rounds", **graph}), flush=True)
        del sets, launches
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--workloads", default="")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-chunks", type=int, default=8)
    ap.add_argument("--rounds", type=int, default=5, help="--sweep: timed rounds per workload")
    ap.add_argument("--graph", action="store_true",
                    help="--sweep: also time the calls captured in a CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.sweep:
        run_sweep(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
