#!/usr/bin/env python
"""Benchmark of the fused NF4 dequantise-and-multiply (forward + input gradient).

One step = the whole hot path over one batch: the forward y = x W^T and the input
gradient grad_x = grad_y W of the seven projections of a Llama-3.1-8B-shaped layer
(q, k, v, o, gate, up, down) at M = 512 tokens, NF4 with double-quantised absmax,
as 8 launches: q/k/v and gate/up each as one multi-product launch per direction
(the products become ready together in a layer), o and down alone.
Weights ~ N(0, 0.02) and activations ~ N(0, 1) are seeded synthetic stand-ins for
the checkpoint; three replicas of the quantised weights rotate across steps so the
weights read by a step (337 MB in total) are never L2-resident from the step before.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead
on a bounded sample of the same workload.  Multi-GPU (torchrun): independent
replicas, one per GPU; value = work of all ranks / max time over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NF4 fwd+dgrad TFLOP/s vs M (1–8192); % of bf16 TC peak / % HBM BW at small M"
WORKLOAD = ("llama3.1-8b projection set (q,k,v,o 4096x4096; k,v 1024x4096; gate,up 14336x4096; "
            "down 4096x14336) at M=512, NF4 blocksize 64 + double-quant absmax, fwd + dgrad")
M_HEAD = 512
REPLICAS = 3
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_SRC = os.path.join(ROOT, "bit_nf4_quantized_linear_gb300", "csrc", "nf4_gemm.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "nf4_gemm_traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1500)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--single", default=None,
                   help="profiling case: one projection of the workload (q,k,v,o,gate,up,down)")
    p.add_argument("--m", type=int, default=M_HEAD, help="tokens of the --single case")
    p.add_argument("--reps", type=int, default=3, help="fwd+dgrad pairs of the --single case")
    p.add_argument("--stream-k", choices=["auto", "off", "force"], default="auto",
                   help="schedule of the fused kernel (library default: auto)")
    p.add_argument("--weight-prefetch", choices=["on", "off"], default="on",
                   help="declare the weights frozen so kernels may read them before the "
                        "previous kernel on the stream has finished (library default: off)")
    return p.parse_args()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value over all ranks (step time of the slowest replica)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: the work of every replica over the slowest replica's time."""
    return flops_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


def flops_per_step(M: int) -> float:
    from bit_nf4_quantized_linear_gb300 import synth
    return sum(2.0 * 2.0 * M * N * K for _, K, N in synth.LLAMA8B_PROJ)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            def pick(*keys):
                for k in keys:
                    if k in d and isinstance(d[k], (int, float)):
                        return float(d[k])
                return None
            hbm = pick("hbm_gbs")
            bf = pick("bf16_tflops")
            bfs = pick("bf16_tflops_sustained") or bf
            if hbm and bf:
                return {"hbm_gbs": hbm, "bf16_tflops": bf, "bf16_tflops_sustained": bfs}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def gemm_src_sha() -> str:
    with open(GEMM_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_per_launch():
    """DRAM bytes per launch of the fused kernel from a committed ncu summary, only
    while the kernel source is the one the counters were taken on."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        if d.get("kernel_src_sha") == gemm_src_sha():
            return d.get("bytes_per_launch_headline")
    except Exception:
        pass
    return None


class _Nvml:
    """Minimal ctypes view of NVML (NVIDIA's management library): SM clock,
    its maximum, power draw and the active clock-event (throttle) reasons of one
    device.  Read-only; nothing here changes a device setting."""

    # clock-event reason bits of nvml.h, named as nvidia-smi reports them
    REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8 | 0x80), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40))

    def __init__(self, uuid: str | None, index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        rc = 1
        if uuid:
            rc = self.lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        v = ctypes.c_uint(0)
        self.max_mhz = float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(v)) == 0 \
            and v.value else None

    def sample(self):
        c = self.c
        clk, mw, rs = c.c_uint(0), c.c_uint(0), c.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(clk)) != 0:  # NVML_CLOCK_SM
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(mw))
        self.reasons_fn(self.h, c.byref(rs))
        return float(clk.value), mw.value / 1000.0, int(rs.value)


class ClockSampler:
    """SM clock and throttle reasons sampled while the timed region runs: NVML read
    every millisecond from a thread (so a region of a few milliseconds still gets
    samples), else nvidia-smi every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, uuid: str | None = None):
        self.gpu = gpu_index
        self.uuid = uuid
        self.proc = None
        self.nvml = None
        self.samples = []
        self.source = None

    def __enter__(self):
        import threading
        try:
            self.nvml = _Nvml(self.uuid, self.gpu)
            self.source = "nvml 1 ms"
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.stop = threading.Event()

            def loop():
                while not self.stop.is_set():
                    r = self.nvml.sample()
                    if r is not None:
                        self.samples.append(r)
                    time.sleep(0.001)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi 100 ms"
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.nvml is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            return
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons, power = [], None, set(), []
        if self.nvml is not None:
            mx = self.nvml.max_mhz
            for clk, w, rs in self.samples:
                sm.append(clk)
                power.append(w)
                for name, bit in _Nvml.REASONS:
                    if rs & bit:
                        reasons.add(name)
        else:
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in (self.out or "").splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": self.source}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
               "samples": len(sm), "source": self.source}
        if power:
            out["power_w_max"] = max(power)
        return out


# ------------------------------------------------------------------ workload --

def make_weights(dev, replicas: int):
    """Quantised weights of the seven projections (seeded), plus replicas that are
    byte copies in separate buffers."""
    import torch
    import bit_nf4_quantized_linear_gb300 as nf4
    from bit_nf4_quantized_linear_gb300 import synth
    g = synth.generator(0)
    base = []
    for name, K, N in synth.LLAMA8B_PROJ:
        w32 = synth.weight(N, K, g).to(dev)
        base.append(nf4.quantize(w32, double_quant=True))
        del w32
    torch.cuda.synchronize()
    sets = [base]
    for _ in range(replicas - 1):
        cp = []
        for w in base:
            # (codebooks shared, as among the base weights: a multi-product launch
            # takes one codebook)
            cp.append(nf4.NF4Weight(w.packed.clone(), None, w.absmax_q.clone(),
                                    w.nested_absmax.clone(), w.nested_offset.clone(),
                                    w.code4, w.code8, w.N, w.K, True))
        sets.append(cp)
    return sets, g


# Projections that take one launch each way: q, k and v (ready together: one input
# in the forward, their output gradients together in the backward), o, gate and up,
# down.  A group of more than one runs as a multi-product launch
# (nf4_linear_fwd_multi / nf4_linear_dgrad_multi): the same products and outputs,
# one grid.
LAUNCH_GROUPS = [(0, 1, 2), (3,), (4, 5), (6,)]


def run_group(ops, grp, ws, xs, gys, ys, gxs, fwd=True, dgrad=True):
    if len(grp) == 1:
        j = grp[0]
        if fwd:
            ops.linear_fwd(xs[j], ws[j], out=ys[j])
        if dgrad:
            ops.linear_dgrad(gys[j], ws[j], out=gxs[j])
        return
    if fwd:
        ops.linear_fwd_multi([xs[j] for j in grp], [ws[j] for j in grp], outs=[ys[j] for j in grp])
    if dgrad:
        ops.linear_dgrad_multi([gys[j] for j in grp], [ws[j] for j in grp], outs=[gxs[j] for j in grp])


def make_acts(g, M, dev):
    from bit_nf4_quantized_linear_gb300 import synth
    xs, gys = [], []
    for _, K, N in synth.LLAMA8B_PROJ:
        xs.append(synth.activation(M, K, g))
        gys.append(synth.activation(M, N, g))
    return [x.to(dev) for x in xs], [y.to(dev) for y in gys], xs, gys


def run_ours(args, rank, world, local_rank):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import bit_nf4_quantized_linear_gb300 as nf4
    from bit_nf4_quantized_linear_gb300 import ops, synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    nf4.device_check()
    nf4.device_status(clear=True)
    ops.set_weight_prefetch(args.weight_prefetch == "on")  # frozen weights may be read early
    ops.set_stream_k({"off": 0, "auto": 1, "force": 2}[args.stream_k])
    sets, g = make_weights(dev, REPLICAS)
    xs, gys, xs_host, gys_host = make_acts(g, M_HEAD, dev)
    ys = [torch.empty(M_HEAD, w.N, dtype=torch.bfloat16, device=dev) for w in sets[0]]
    gxs = [torch.empty(M_HEAD, w.K, dtype=torch.bfloat16, device=dev) for w in sets[0]]
    weight_bytes = sum(w.nbytes() for w in sets[0])
    stream = torch.cuda.current_stream()

    def step(i):
        ws = sets[i % REPLICAS]
        for grp in LAUNCH_GROUPS:
            run_group(ops, grp, ws, xs, gys, ys, gxs)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # The timed region: exactly args.steps steps, nothing else on the stream.
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0 = nf4.path_counters()["total"]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "") or None
    with ClockSampler(local_rank, uuid) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = nf4.path_counters()["total"] - c0
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_step = ms / args.steps
    flops = flops_per_step(M_HEAD)
    value = job_throughput(flops, world, ms_step)

    # Dominant kernel: the fused tcgen05 product kernel (forward and input-gradient
    # instances).  A separate pass after the timed region brackets every launch with
    # CUDA events on the launching stream (events between launches stop the next
    # kernel from starting early, so each launch runs alone): achieved = algorithmic
    # flops per launch / mean launch duration, against the burst peak.
    n_ev = max(5, min(args.steps, 40))
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in LAUNCH_GROUPS]
           for _ in range(n_ev)]
    for i in range(n_ev):
        for gi, grp in enumerate(LAUNCH_GROUPS):
            e = evs[i][gi]
            ws_i = sets[i % REPLICAS]
            e[0].record(stream)
            run_group(ops, grp, ws_i, xs, gys, ys, gxs, dgrad=False)
            e[1].record(stream)
            e[2].record(stream)
            run_group(ops, grp, ws_i, xs, gys, ys, gxs, fwd=False)
            e[3].record(stream)
    torch.cuda.synchronize()
    launch_ms, launch_flops = [], []
    for i in range(n_ev):
        for gi, grp in enumerate(LAUNCH_GROUPS):
            e = evs[i][gi]
            fl = sum(2.0 * M_HEAD * synth.LLAMA8B_PROJ[j][2] * synth.LLAMA8B_PROJ[j][1] for j in grp)
            launch_ms += [e[0].elapsed_time(e[1]), e[2].elapsed_time(e[3])]
            launch_flops += [fl] * 2
    mean_ms = sum(launch_ms) / len(launch_ms)
    mean_flops = sum(launch_flops) / len(launch_flops)
    # Per launch of the step (each run alone between events), mean over the pass.
    per_launch = {}
    names = [p[0] for p in synth.LLAMA8B_PROJ]
    for gi, grp in enumerate(LAUNCH_GROUPS):
        tag = "+".join(names[j] for j in grp)
        for d, off in (("fwd", 0), ("dgrad", 1)):
            v = [launch_ms[(i * len(LAUNCH_GROUPS) + gi) * 2 + off] for i in range(n_ev)]
            per_launch[f"{tag} {d}"] = round(sum(v) / len(v) * 1e3, 2)
    achieved = mean_flops / (mean_ms * 1e-3) / 1e12
    pk, pk_src = peaks()
    peak = pk["bf16_tflops"]
    status = nf4.device_status()

    # End to end through the public API: each step copies that step's inputs from
    # pinned host memory and reads its results back.  All inputs of a step (x and
    # grad_y of the seven projections) sit in one pinned buffer and go over in one
    # copy, the results in one copy back (few host calls per step, so the host does
    # not bound it); the copies run on two copy streams ordered with events, so
    # step i + 1's inputs arrive and step i - 1's results leave while step i
    # computes, and two device buffer sets alternate between steps.
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    in_shapes = [tuple(t.shape) for t in xs_host] + [tuple(t.shape) for t in gys_host]
    out_shapes = [tuple(y.shape) for y in ys] + [tuple(x.shape) for x in gxs]
    n_in = sum(a * b for a, b in in_shapes)
    n_out = sum(a * b for a, b in out_shapes)
    in_h = torch.empty(n_in, dtype=torch.bfloat16).pin_memory()
    off = 0
    for t in list(xs_host) + list(gys_host):
        in_h[off:off + t.numel()].copy_(t.reshape(-1))
        off += t.numel()
    out_h = torch.empty(n_out, dtype=torch.bfloat16).pin_memory()
    h2d, d2h = n_in * 2, n_out * 2

    def views(flat, shapes):
        vs, o = [], 0
        for a, b in shapes:
            vs.append(flat[o:o + a * b].view(a, b))
            o += a * b
        return vs

    nproj = len(sets[0])
    bufs = []
    for _ in range(2):
        fin = torch.empty(n_in, dtype=torch.bfloat16, device=dev)
        fout = torch.empty(n_out, dtype=torch.bfloat16, device=dev)
        vin, vout = views(fin, in_shapes), views(fout, out_shapes)
        bufs.append((fin, fout, vin[:nproj], vin[nproj:], vout[:nproj], vout[nproj:]))
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        b = i & 1
        fin, fout, xb, gyb, yb, gxb = bufs[b]
        ws = sets[i % REPLICAS]
        with torch.cuda.stream(up_s):
            if used[b]:
                up_s.wait_event(ev_done[b])  # the last step on this set read its inputs
            fin.copy_(in_h, non_blocking=True)
            ev_in[b].record(up_s)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])  # the last step's results on this set have left
        for grp in LAUNCH_GROUPS:
            run_group(ops, grp, ws, xb, gyb, yb, gxb)
        ev_done[b].record(stream)
        with torch.cuda.stream(down_s):
            down_s.wait_event(ev_done[b])
            out_h.copy_(fout, non_blocking=True)
            ev_out[b].record(down_s)
        used[b] = True

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(ev_out[(e2e_steps - 1) & 1])  # the last results are on the host before the clock stops
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    e2e_val = job_throughput(flops, world, e2e_ms)

    sweep = grouped = storage8 = f16 = stack = None
    if rank == 0 and world == 1 and not args.no_sweep:
        sweep = run_sweep(dev, pk)
        grouped = run_grouped(dev, pk)
        storage8 = run_storage8(dev, pk)
        f16 = run_storage8(dev, pk, (("nf4_f16", "nf4", "f16"),))
        stack = run_stack(dev, pk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(target_s=12.0)

    out = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights quantised to NF4, N(0,1) bf16 activations)",
        "config": {
            "workload": WORKLOAD, "M": M_HEAD, "flops_per_step": flops,
            "nf4_weight_bytes": weight_bytes,
            "l2": f"inputs larger than L2: {REPLICAS} rotating weight replicas, "
                  f"{REPLICAS * weight_bytes / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB",
            "parallelism": f"replicas x{world}",
            "weight_prefetch": ("on (frozen weights: kernels read them before the dependency "
                                "on the previous kernel resolves)") if args.weight_prefetch == "on"
                               else "off",
            "stream_k": args.stream_k,
            "launches": "q/k/v and gate/up as multi-product launches (one grid per group and "
                        "direction, outputs separate), o and down alone: 8 launches per step",
        },
        "roofline": {
            "kernel": "nf4_gemm_kernel (fused tcgen05 fwd + dgrad launches of the step, per launch)",
            "bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "peak_kind": f"bf16 dense burst (launches timed alone), of {pk_src}",
            "traffic": traffic_per_launch(), "launches_timed": len(launch_ms),
            "mean_launch_ms": round(mean_ms, 5),
            "launch_us": per_launch,
            "timing": "separate pass after the timed region, CUDA events around each launch",
        },
        "e2e": {"value": round(e2e_val, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "copies": "one pinned host buffer of the step's inputs and one of its results, "
                          "one H2D and one D2H copy per step on two copy streams overlapping the "
                          "products of the neighbouring steps (event-ordered, two device buffer sets)"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "device_status": status,
    }
    if sweep is not None:
        out["m_sweep_4096"] = sweep
    if grouped is not None:
        out["grouped_olmoe"] = grouped
    if storage8 is not None:
        out["storage_8bit_4096"] = storage8
    if f16 is not None:
        out["f16_compute_4096"] = f16
    if stack is not None:
        out["config5_stack"] = stack
    if cpu is not None:
        out["cpu_baseline"] = cpu
    if sweep is not None:
        # Compact summaries last on the line, where a truncated log keeps them: the
        # K = N = 4096 curve as [M, us fwd, us dgrad, TFLOP/s, fraction of the burst
        # tensor peak, fraction of HBM on weight bytes], then the expert and stack rows.
        summ = {"cols": ["M", "us_fwd", "us_dgrad", "tflops", "frac_tc", "frac_hbm"],
                "rows": [[r["M"], r["us_fwd"], r["us_dgrad"], r["tflops"], r["frac_tc"], r["frac_hbm"]]
                         for r in sweep]}
        if grouped is not None:
            summ["grouped_olmoe_tflops"] = grouped["tflops"]
            summ["grouped_olmoe_weight_gbs"] = grouped["weight_gbs"]
        if stack is not None:
            summ["config5_stack_ms"] = stack["ms_per_step"]
            summ["config5_stack_tflops"] = stack["tflops_products"]
        out["m_sweep_4096_summary"] = summ
    return out


def run_sweep(dev, pk):
    """K = N = 4096 NF4 (double quant) fwd + dgrad across M; each point is a CUDA
    graph of R back-to-back fwd+dgrad pairs over R weight replicas (R * weight bytes
    >= 4 x L2 at small M), replayed after warm-up."""
    import torch
    import bit_nf4_quantized_linear_gb300 as nf4
    from bit_nf4_quantized_linear_gb300 import ops, synth
    N = K = 4096
    g = synth.generator(1)
    base = nf4.quantize(synth.weight(N, K, g).to(dev), double_quant=True)
    wbytes = base.nbytes()
    res = []
    for M in synth.M_SWEEP:
        R = max(2, min(64, int(4 * L2_BYTES / wbytes) + 1)) if M <= 128 else (8 if M <= 2048 else 4)
        reps = [base] + [nf4.NF4Weight(base.packed.clone(), None, base.absmax_q.clone(),
                                       base.nested_absmax.clone(), base.nested_offset.clone(),
                                       base.code4, base.code8, N, K, True) for _ in range(R - 1)]
        x = synth.activation(M, K, g).to(dev)
        gy = synth.activation(M, N, g).to(dev)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        gx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        wsz = max(ops.workspace_size(1, M, N, K), ops.workspace_size(2, M, N, K), 16)
        wsb = torch.empty(wsz, dtype=torch.uint8, device=dev)
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for w in reps[:2]:
                ops.linear_fwd(x, w, out=y, ws=wsb)
                ops.linear_dgrad(gy, w, out=gx, ws=wsb)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        def timed(ops_list):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                for w in reps:
                    for op in ops_list:
                        op(w)
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize()
            times = []
            for _ in range(10):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                graph.replay()
                b.record()
                b.synchronize()
                times.append(a.elapsed_time(b) / R)
            del graph
            return statistics.median(times) * 1e-3  # seconds per call group
        fwd = lambda w: ops.linear_fwd(x, w, out=y, ws=wsb)
        bwd = lambda w: ops.linear_dgrad(gy, w, out=gx, ws=wsb)
        nf4.reset_path_counters()
        fwd(base)
        pf = [k for k, v in nf4.path_counters().items() if v and k not in ("total", "splitk_reduce")]
        nf4.reset_path_counters()
        bwd(base)
        pd = [k for k, v in nf4.path_counters().items() if v and k not in ("total", "splitk_reduce")]
        t_f = timed([fwd])
        t_d = timed([bwd])
        t = t_f + t_d
        # single-launch latency: one forward call between events on an idle stream
        # (launch overhead included; the graphs above hide it)
        singles = []
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                a.record()
                fwd(base)
                b.record()
            b.synchronize()
            singles.append(a.elapsed_time(b) * 1e3)
        t_single = statistics.median(singles)
        # comparison arms in the same session: dense bf16 cuBLAS (same shape, a dense
        # weight per replica) and dequantise-then-matmul (the unfused design)
        dense = [nf4.dequantize(w) for w in reps[:max(2, min(R, int(4 * L2_BYTES / (2 * N * K)) + 1))]]
        Rd = len(dense)
        def timed_dense(fn):
            with torch.cuda.stream(s):  # library handles are created outside the capture
                fn(dense[0])
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                for wd in dense:
                    fn(wd)
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize()
            times = []
            for _ in range(10):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                graph.replay()
                b.record()
                b.synchronize()
                times.append(a.elapsed_time(b) / Rd)
            del graph
            return statistics.median(times) * 1e-3
        t_cub = timed_dense(lambda wd: (torch.matmul(x, wd.t(), out=y), torch.matmul(gy, wd, out=gx)))
        wtmp = torch.empty(N, K, dtype=torch.bfloat16, device=dev)
        def deq_linear(w):
            ops.dequantize(w, out=wtmp)
            torch.matmul(x, wtmp.t(), out=y)
            ops.dequantize(w, out=wtmp)
            torch.matmul(gy, wtmp, out=gx)
        with torch.cuda.stream(s):
            deq_linear(base)
        torch.cuda.synchronize()
        t_deq = timed([deq_linear])
        del dense, wtmp
        tfl = 4.0 * M * N * K / t / 1e12
        gbs = 2.0 * wbytes / t / 1e9
        res.append({"M": M, "us_per_fwd_dgrad": round(t * 1e6, 2), "us_fwd": round(t_f * 1e6, 2),
                    "us_dgrad": round(t_d * 1e6, 2), "tflops": round(tfl, 2),
                    "frac_tc": round(tfl / pk["bf16_tflops"], 4),
                    "weight_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                    "fwd_weight_gbs": round(wbytes / t_f / 1e9, 1),
                    "dgrad_weight_gbs": round(wbytes / t_d / 1e9, 1),
                    "replicas": R, "path_fwd": pf, "path_dgrad": pd,
                    "single_launch_fwd_us": round(t_single, 2),
                    "cublas_dense_bf16_us": round(t_cub * 1e6, 2),
                    "dequant_then_matmul_us": round(t_deq * 1e6, 2)})
        del reps, x, gy, y, gx, wsb
        torch.cuda.empty_cache()
    return res


def run_storage8(dev, pk, variants=(("int8", "int8", "bf16"), ("fp8", "fp8", "bf16"))):
    """Storage / dtype variants at K = N = 4096, double-quant statistics: one-byte
    storage ("int8" dynamic map, "fp8" e4m3 levels) and the fp16 compute dtype; fwd +
    dgrad through the fused kernel, each point a CUDA graph of back-to-back calls over
    weight replicas (>= 4 x L2 at small M)."""
    import torch
    import bit_nf4_quantized_linear_gb300 as nf4
    from bit_nf4_quantized_linear_gb300 import ops, synth
    N = K = 4096
    out = {}
    for name, qt, adt in variants:
        adt = torch.float16 if adt == "f16" else torch.bfloat16
        g = synth.generator(2)
        base = nf4.quantize(synth.weight(N, K, g).to(dev), double_quant=True, quant_type=qt)
        wbytes = base.nbytes()
        rows = []
        for M in (1, 16, 512, 4096):
            R = max(2, min(32, int(4 * L2_BYTES / wbytes) + 1)) if M <= 16 else 4
            reps = [base] + [nf4.NF4Weight(base.packed.clone(), None, base.absmax_q.clone(),
                                           base.nested_absmax.clone(), base.nested_offset.clone(),
                                           base.code4, base.code8, N, K, True) for _ in range(R - 1)]
            x = synth.activation(M, K, g).float().to(adt).to(dev)
            gy = synth.activation(M, N, g).float().to(adt).to(dev)
            y = torch.empty(M, N, dtype=adt, device=dev)
            gx = torch.empty(M, K, dtype=adt, device=dev)
            wsz = max(ops.workspace_size(1, M, N, K), ops.workspace_size(2, M, N, K), 16)
            wsb = torch.empty(wsz, dtype=torch.uint8, device=dev)
            s = torch.cuda.Stream(dev)
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                for w in reps[:2]:
                    ops.linear_fwd(x, w, out=y, ws=wsb)
                    ops.linear_dgrad(gy, w, out=gx, ws=wsb)
            torch.cuda.synchronize()
            ts = []
            for op in (lambda w: ops.linear_fwd(x, w, out=y, ws=wsb),
                       lambda w: ops.linear_dgrad(gy, w, out=gx, ws=wsb)):
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=s):
                    for w in reps:
                        op(w)
                for _ in range(3):
                    graph.replay()
                torch.cuda.synchronize()
                times = []
                for _ in range(10):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    graph.replay()
                    b.record()
                    b.synchronize()
                    times.append(a.elapsed_time(b) / R)
                ts.append(statistics.median(times) * 1e-3)
                del graph
            t = ts[0] + ts[1]
            tfl = 4.0 * M * N * K / t / 1e12
            gbs = 2.0 * wbytes / t / 1e9
            rows.append({"M": M, "us_fwd": round(ts[0] * 1e6, 2), "us_dgrad": round(ts[1] * 1e6, 2),
                         "tflops": round(tfl, 2), "frac_tc": round(tfl / pk["bf16_tflops"], 4),
                         "weight_gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4)})
            del reps, x, gy, y, gx, wsb
            torch.cuda.empty_cache()
        out[name] = {"weight_bytes": wbytes, "rows": rows}
    return out


def run_grouped(dev, pk):
    """OLMoE-shaped experts (64 experts, hidden 2048, intermediate 1024, 512 tokens,
    top-8 routing from seeded uniform logits): grouped forward + input gradient of
    the gate, up and down stacks, each a CUDA graph over weight replicas."""
    import torch
    import bit_nf4_quantized_linear_gb300 as nf4
    from bit_nf4_quantized_linear_gb300 import ops, synth
    c = synth.OLMOE
    E, H, I = c["experts"], c["hidden"], c["inter"]
    g = synth.generator(4)
    row_token, offsets = synth.routing(c["tokens"], E, c["topk"], g)
    T = int(offsets[-1])
    offs = offsets.to(dev)
    out = {"workload": "olmoe experts: 64 x (gate, up 2048->1024; down 1024->2048), "
                       "512 tokens top-8 (4096 rows), NF4 double quant, grouped fwd + grad_x",
           "rows": T}
    total_t, total_fl, total_b = 0.0, 0.0, 0.0
    for name, N_e, K in (("gate", I, H), ("up", I, H), ("down", H, I)):
        base = nf4.quantize(synth.weight(E * N_e, K, g).to(dev), double_quant=True)
        wbytes = base.nbytes()
        R = max(2, min(8, int(4 * L2_BYTES / wbytes) + 1))
        reps = [base] + [nf4.NF4Weight(base.packed.clone(), None, base.absmax_q.clone(),
                                       base.nested_absmax.clone(), base.nested_offset.clone(),
                                       base.code4, base.code8, base.N, base.K, True) for _ in range(R - 1)]
        x = synth.activation(T, K, g).to(dev)
        gy = synth.activation(T, N_e, g).to(dev)
        y = torch.empty(T, N_e, dtype=torch.bfloat16, device=dev)
        gx = torch.empty(T, K, dtype=torch.bfloat16, device=dev)
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for w in reps[:2]:
                ops.grouped_fwd(x, offs, w, E, out=y)
                ops.grouped_dgrad(gy, offs, w, E, out=gx)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for w in reps:
                ops.grouped_fwd(x, offs, w, E, out=y)
                ops.grouped_dgrad(gy, offs, w, E, out=gx)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b) / R)
        t = statistics.median(times) * 1e-3
        fl = 4.0 * T * N_e * K
        out[name] = {"us_fwd_dgrad": round(t * 1e6, 2), "tflops": round(fl / t / 1e12, 2),
                     "weight_gbs": round(2 * wbytes / t / 1e9, 1)}
        total_t += t
        total_fl += fl
        total_b += 2 * wbytes
        del graph, reps, x, gy, y, gx
        torch.cuda.empty_cache()
    out["tflops"] = round(total_fl / total_t / 1e12, 2)
    out["frac_tc"] = round(total_fl / total_t / 1e12 / pk["bf16_tflops"], 4)
    out["weight_gbs"] = round(total_b / total_t / 1e9, 1)

    # Forward of the expert MLP's first half, h = silu(x Wg^T) * (x Wu^T) * routing
    # weight: the fused epilogue over the interleaved gate/up weight, against two
    # grouped products and the same steps in torch (the unfused form).
    gate = synth.weight(E * I, H, g)
    up = synth.weight(E * I, H, g)
    wgu = nf4.quantize(nf4.interleave_gate_up(gate, up, E).to(dev), double_quant=True)
    wg = nf4.quantize(gate.to(dev), double_quant=True)
    wu = nf4.quantize(up.to(dev), double_quant=True)
    x = synth.activation(T, H, g).to(dev)
    rw = torch.rand(T, generator=g).to(dev)
    h = torch.empty(T, I, dtype=torch.bfloat16, device=dev)
    yg = torch.empty(T, I, dtype=torch.bfloat16, device=dev)
    yu = torch.empty(T, I, dtype=torch.bfloat16, device=dev)
    def fused():
        ops.grouped_fwd(x, offs, wgu, E, out=h, row_scale=rw, swiglu=True)
    def unfused():
        ops.grouped_fwd(x, offs, wg, E, out=yg)
        ops.grouped_fwd(x, offs, wu, E, out=yu)
        h.copy_(torch.nn.functional.silu(yg.float()) * yu.float() * rw[:, None])
    def time_graph(fn, reps=8):
        s2 = torch.cuda.Stream(dev)
        s2.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s2):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s2):
            for _ in range(reps):
                fn()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b) / reps)
        del graph
        return statistics.median(ts) * 1e-3
    t_f, t_u = time_graph(fused), time_graph(unfused)
    out["swiglu_gate_up_fwd"] = {"us_fused_epilogue": round(t_f * 1e6, 2),
                                 "us_unfused_torch_glue": round(t_u * 1e6, 2),
                                 "tflops_fused": round(2.0 * T * 2 * I * H / t_f / 1e12, 2)}

    # The top-k combine of the down projection's rows ([T, H] -> [tokens, H]) and its
    # backward, over 16 row buffers (268 MB > L2) in turn.  Bytes: rows in, tokens
    # out, the route table (forward); the reverse (backward).
    tokens, topk = c["tokens"], c["topk"]
    tr = ops.route_rows(row_token.to(dev), tokens, topk)
    nbuf = 16
    rows_b = [synth.activation(T, H, g).to(dev) for _ in range(nbuf)]
    grads_b = [synth.activation(tokens, H, g).to(dev) for _ in range(nbuf)]
    comb = torch.empty(tokens, H, dtype=torch.bfloat16, device=dev)
    grows = torch.empty(T, H, dtype=torch.bfloat16, device=dev)  # every row is routed once
    state = {"i": 0}
    def combine():
        ops.moe_combine(rows_b[state["i"] % nbuf], tr, out=comb)
        state["i"] += 1
    def combine_bwd():
        ops.moe_combine_bwd(grads_b[state["i"] % nbuf], tr, T, out=grows)
        state["i"] += 1
    t_c, t_cb = time_graph(combine, reps=nbuf), time_graph(combine_bwd, reps=nbuf)
    b_c = 2 * T * H + 2 * tokens * H + 4 * tokens * topk
    out["topk_combine"] = {"rows": T, "tokens": tokens, "H": H,
                           "us_fwd": round(t_c * 1e6, 2), "gbs_fwd": round(b_c / t_c / 1e9, 1),
                           "us_bwd": round(t_cb * 1e6, 2), "gbs_bwd": round(b_c / t_cb / 1e9, 1),
                           "frac_hbm_fwd": round(b_c / t_c / 1e9 / pk["hbm_gbs"], 4)}
    return out


def run_stack(dev, pk, layers_n: int = 8, M: int = 4096, reps: int = 3):
    """The 32B-class layer stack (hidden 5120, intermediate 27648, k/v 1024, M = 4096,
    eight layers of NF4 double-quant weights) under non-reentrant checkpointing with
    each layer's quantised tensors copied into one of two recycled slot sets inside
    its checkpointed region; one step = forward, recompute and input gradients of the
    whole stack (h = x / rms(x) s; a = h + o(q(h)); kv = mean(k(h) v(h));
    z = silu(gate(a)) up(a); out = a + down(z)).  TFLOP/s counts the products only: three passes of 2 M N K
    per projection (forward, recompute, input gradient)."""
    import itertools
    import torch
    import torch.nn.functional as F
    from torch.utils.checkpoint import checkpoint
    import bit_nf4_quantized_linear_gb300 as nf4
    from bit_nf4_quantized_linear_gb300 import ops, synth
    g = torch.Generator(device=dev)
    g.manual_seed(60)
    layers = []
    for _ in range(layers_n):
        layer = {}
        for name, K, N in synth.QWEN32B_PROJ:
            layer[name] = nf4.quantize(torch.randn(N, K, generator=g, device=dev) * synth.WEIGHT_STD,
                                       double_quant=True)
        layers.append(layer)
    torch.cuda.empty_cache()
    slot_sets = [{n: [None if t is None else torch.empty_like(t) for t in w.tensors()]
                  for n, w in layers[0].items()} for _ in range(2)]
    turn = itertools.cycle(range(2))

    def load(layer):
        dst = slot_sets[next(turn)]
        out = {}
        for n, w in layer.items():
            for b, t in zip(dst[n], w.tensors()):
                if b is not None:
                    b.copy_(t)
            out[n] = ops.NF4Weight.from_tensors(tuple(dst[n]), w.N, w.K, w.double_quant)
        return out

    H = synth.QWEN32B_PROJ[0][1]
    x0 = torch.randn(M, H, generator=g, device=dev).to(torch.bfloat16)
    scales = [(1 + 0.01 * torch.randn(H, generator=g, device=dev)).to(torch.bfloat16)
              .requires_grad_(True) for _ in range(layers_n)]

    def block(i):
        def run(x, s):
            w = load(layers[i])
            p = lambda t, n: nf4.nf4_linear(t, w[n])
            xf = x.float()
            h = (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + 1e-6) * s.float()).to(torch.bfloat16)
            a = h + p(p(h, "q"), "o")
            kv = (p(h, "k").float() * p(h, "v").float()).mean()
            z = F.silu(p(a, "gate")) * p(a, "up")
            return a + p(z, "down"), kv
        return run

    def step():
        x = x0.clone().requires_grad_(True)
        h, kvs = x, 0.0
        for i in range(layers_n):
            h, kv = checkpoint(block(i), h, scales[i], use_reentrant=False)
            kvs = kvs + kv
        (h.float().pow(2).mean() + kvs).backward()

    step()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e-3)
    t = statistics.median(times)
    flops = 3.0 * layers_n * sum(2.0 * M * N * K for _, K, N in synth.QWEN32B_PROJ)
    per_layer = sum(w.nbytes() for w in layers[0].values())
    del layers, slot_sets
    torch.cuda.empty_cache()
    return {"workload": "qwen2.5-32b-shaped stack: 8 layers x (q,o 5120^2; k,v 1024x5120; gate,up "
                        "27648x5120; down 5120x27648), M=4096, checkpointed, 2 recycled slot sets",
            "nf4_bytes_per_layer": per_layer, "ms_per_step": round(t * 1e3, 3),
            "tflops_products": round(flops / t / 1e12, 1),
            "frac_tc": round(flops / t / 1e12 / pk["bf16_tflops"], 4)}


# ------------------------------------------------------------- CPU oracle --

def oracle_workload():
    """The headline workload for the CPU oracle (untimed setup): the seven
    projections quantised by the oracle, and the activations / output gradients."""
    import oracle
    from oracle import codebooks as ocb
    from bit_nf4_quantized_linear_gb300 import synth
    g = synth.generator(0)
    code4, code8 = ocb.nf4_code4(), ocb.dynamic_code8()
    states = []
    for _, K, N in synth.LLAMA8B_PROJ:
        states.append(oracle.quantize(synth.weight(N, K, g).numpy(), code4, 64, True, code8, 256))
    xs = [synth.activation(M_HEAD, K, g) for _, K, N in synth.LLAMA8B_PROJ]
    gys = [synth.activation(M_HEAD, N, g) for _, K, N in synth.LLAMA8B_PROJ]
    return states, xs, gys


def cpu_baseline(target_s: float = 12.0, workload=None):
    """The CPU oracle as it stands, on a bounded sample of the headline workload:
    all seven projections dequantised by the oracle, then S token rows of the
    forward and S rows of the input gradient of each.  `value` is the sample's own
    throughput (the flops of the rows computed over the time the whole sample took,
    dequantisation included); the time a full 512-row step would take is reported
    beside it as an estimate."""
    import numpy as np
    import oracle
    from bit_nf4_quantized_linear_gb300 import synth
    states, xs, gys = workload if workload is not None else oracle_workload()
    bits = lambda t: t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    wbs = [oracle.dequantize(st, "bf16") for st in states]
    t_deq = time.perf_counter() - t0
    # calibrate the row count on one row per projection and direction
    t0 = time.perf_counter()
    for j in range(len(wbs)):
        oracle.linear_fwd(bits(xs[j]), wbs[j], rows=[0])
        oracle.linear_dgrad(bits(gys[j]), wbs[j], rows=[0])
    t_one = time.perf_counter() - t0
    S = int(max(1, min(64, (target_s - t_deq) / max(t_one, 1e-6))))
    rows = np.arange(S, dtype=np.int64)
    t0 = time.perf_counter()
    for j in range(len(wbs)):
        oracle.linear_fwd(bits(xs[j]), wbs[j], rows=rows)
        oracle.linear_dgrad(bits(gys[j]), wbs[j], rows=rows)
    t_rows = time.perf_counter() - t0
    t_sample = t_deq + t_rows
    sample_flops = sum(2.0 * 2.0 * S * N * K for _, K, N in synth.LLAMA8B_PROJ)
    return {"value": sample_flops / t_sample / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "scaled": False,
            "sample": f"7 projections dequantised ({t_deq:.2f} s) + {S} of {M_HEAD} token rows of "
                      f"fwd and of dgrad ({t_rows:.2f} s); value = flops of those rows / "
                      f"{t_sample:.2f} s",
            "rows_timed": S, "s_per_sample": t_sample, "sample_flops": sample_flops,
            "full_step_estimate_s": t_deq + (M_HEAD / S) * t_rows}


def run_single(args):
    """One projection, `reps` forward + input-gradient pairs, timed with events (a
    small case for profilers)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import bit_nf4_quantized_linear_gb300 as nf4
    from bit_nf4_quantized_linear_gb300 import ops, synth
    dev = torch.device("cuda", 0)
    ops.set_stream_k({"off": 0, "auto": 1, "force": 2}[args.stream_k])
    shapes = {n: (K, N) for n, K, N in synth.LLAMA8B_PROJ}
    K, N = shapes[args.single]
    g = synth.generator(0)
    w = nf4.quantize(synth.weight(N, K, g).to(dev), double_quant=True)
    x = synth.activation(args.m, K, g).to(dev)
    gy = synth.activation(args.m, N, g).to(dev)
    tf, td = [], []
    for _ in range(args.reps):
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record()
        ops.linear_fwd(x, w)
        b.record()
        ops.linear_dgrad(gy, w)
        c.record()
        c.synchronize()
        tf.append(a.elapsed_time(b))
        td.append(b.elapsed_time(c))
    fl = 2.0 * args.m * N * K
    return {"single": args.single, "M": args.m, "N": N, "K": K, "ms_fwd": tf, "ms_dgrad": td,
            "tflops_fwd_last": fl / (tf[-1] * 1e-3) / 1e12, "tflops_dgrad_last": fl / (td[-1] * 1e-3) / 1e12,
            "device_status": nf4.device_status()}


def run_reference(args, rank, world):
    """The oracle timed on the host cores (rank 0 only): up to three warm-up and
    three timed steps, each a bounded sample of the headline workload, about a
    minute in all whatever --steps / --warmup ask for; the line reports the steps
    actually run, the time one sample step took (ms_per_step) and its throughput."""
    if rank != 0:
        return None
    steps = max(1, min(args.steps, 3))
    warm = max(0, min(args.warmup, 3))
    target = max(2.0, min(8.0, 48.0 / (steps + warm)))
    wl = oracle_workload()
    for _ in range(warm):
        cpu_baseline(target_s=target, workload=wl)
    vals, times = [], []
    last = None
    for _ in range(steps):
        last = cpu_baseline(target_s=target, workload=wl)
        vals.append(last["value"])
        times.append(last["s_per_sample"])
    v = statistics.median(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": statistics.median(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_HEAD, "flops_per_step": flops_per_step(M_HEAD),
                   "step": f"a bounded sample of the workload: {last['rows_timed']} of {M_HEAD} "
                           "token rows per projection and direction, after dequantising all seven",
                   "sample_flops_per_step": last["sample_flops"],
                   "full_step_estimate_ms": last["full_step_estimate_s"] * 1e3},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"], "scaled": False},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.single:
        print(json.dumps(run_single(args)), flush=True)
        return
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
