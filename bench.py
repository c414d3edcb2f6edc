#!/usr/bin/env python3
"""Benchmark of the MoE expert layer on GB300.

One step = one pass of the whole layer: dispatch plan, training forward
(gather, gate_up GEMM + clamped GLU, down GEMM + routing weight, combine) and
backward (both dgrads with the activation backward, d(topk weights), both
fp32 weight gradients, dX combine), on the dispatch-and-combine workload
(T=8192 tokens, H=I=2880, 128 experts, top-4, clamped GLU, bf16).  Inputs are
seeded synthetic data resident in HBM; the 6.4 GB of expert weights exceed
the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
instead (the reference arm: there is no reference implementation to run).

Run: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch one process per GPU with torch.distributed.run; every rank
runs an independent replica (weak scaling, no data-path collective).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD = "clamped_glu_fwd"

# ---------------------------------------------------------------- accounting


def layer_flops(r):
    """Forward 2*Tk*3*H*I, backward twice that (useful work only)."""
    fwd = 2.0 * r.T * r.k * 3 * r.H * r.I
    return fwd, 2.0 * fwd


def layer_bytes(r, e_active):
    """Algorithmic bytes of the layer: what the method must move.
    forward : x + y + active-expert weights + routing ids/weights
    backward: dy + x + dx + active weights + saved pre-activations (bf16
              equivalent) + fp32 weight gradients of every expert + routing"""
    es = 2 if r.dtype == "bf16" else 4
    Tk = r.T * r.k
    w_act = e_active * 3.0 * r.H * r.I * es
    routing = Tk * 8.0
    fwd = 2.0 * r.T * r.H * es + w_act + routing
    bwd = 3.0 * r.T * r.H * es + w_act + Tk * 2.0 * r.I * es + r.E * 3.0 * r.H * r.I * 4 + routing
    return fwd, bwd


def kernel_work(r, e_active):
    """Per-launch algorithmic FLOPs and compulsory bytes of each kernel kind:
    its operands and outputs once each, at their stored precision, useful rows
    only.  The saved pre-activations count at their stored width (fp16 for the
    clamped GLU with bf16 storage and an fp16 clamp limit, else fp32); the
    weight gradients' computed operands (dH1, w*a) count once, without the
    bf16 remainder some experts carry for precision."""
    es = 2 if r.dtype == "bf16" else 4
    T, H, I, E, k = r.T, r.H, r.I, r.E, r.k
    Tk = T * k
    h1 = 2 if (es == 2 and r.act == 1 and float(np.float16(r.limit)) == r.limit
               and abs(r.limit) <= 32768) else 4
    wgu = e_active * H * 2.0 * I * es
    wd = e_active * I * H * es
    return {
        "gather_rows": (0.0, T * H * es + Tk * H * es),
        "gemm_fwd_gate_up_act": (4.0 * Tk * H * I, Tk * H * es + wgu + Tk * I * es + Tk * 2 * I * h1),
        "gemm_fwd_down_scale": (2.0 * Tk * I * H, Tk * I * es + wd + Tk * H * 4),
        "combine": (0.0, Tk * H * 4.0 + T * H * es),
        "gemm_dgrad_down_act_bwd": (2.0 * Tk * H * I,
                                    Tk * H * es + wd + Tk * 2 * I * h1 + Tk * 3 * I * es),
        "gemm_wgrad_down": (2.0 * Tk * I * H, Tk * I * es + Tk * H * es + E * I * H * 4.0),
        "gemm_dgrad_gate_up": (4.0 * Tk * I * H, Tk * 2 * I * es + wgu + Tk * H * 4),
        "gemm_wgrad_gate_up": (4.0 * Tk * H * I, Tk * H * es + Tk * 2 * I * es + E * H * 2.0 * I * 4),
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(key)
                if isinstance(v, dict):
                    v = v.get("value")
                if v is not None:
                    out[key] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "dispatch_gemm_combine_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(kernel):
    """Per-launch DRAM bytes of `kernel` on this workload from a committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "%s_%s.txt" % (kernel, WORKLOAD))
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if "=" in line and not line.startswith("#"):
            a, b = line.split("=", 1)
            kv[a.strip()] = b.strip()
    if kv.get("source_hash") != csrc_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- ranks


def max_over_ranks(v, world, dist=None, device="cpu"):
    """Largest value of v over all ranks (the slowest rank sets the time)."""
    if world == 1 or dist is None:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step, world, ms_per_step):
    """Whole-job TFLOP/s: every rank runs its own replica of the step."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)

    def summary(self):
        return summarize_clocks(self.lines)


def summarize_clocks(lines):
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle leg


class _HostExperts(dict):
    """Some experts' weights in host fp64, keyed by expert id; len() is the
    number of experts of the layer (the oracle sizes its outputs by it)."""

    def __init__(self, d, n_experts):
        super().__init__(d)
        self.n_experts = n_experts

    def __len__(self):
        return self.n_experts


class OracleSample:
    """A bounded sample of a workload for timing the fp64 oracle on the host:
    the first tokens of the case, as many as touch at most `max_experts`
    experts.  Everything the oracle reads (those tokens' rows and routing and
    the touched experts' weights) is converted to host fp64 once, here, so a
    timed pass runs the oracle's arithmetic only.  The cpu_baseline leg and
    the reference arm both use this sample, so their per-token rates agree."""

    def __init__(self, case, max_experts=16):
        import numpy as np
        r = case.recipe
        self.r = r
        idx_all = case.topk_idx.cpu().numpy().astype(np.int64)
        n = 0
        while n < r.T and len(np.unique(idx_all[:n + 1])) <= max_experts:
            n += 1
        self.n_max = max(1, n)
        self.idx = idx_all[:self.n_max]
        used = sorted(set(int(e) for e in np.unique(self.idx)))
        self.wgu = _HostExperts({e: case.w_gate_up[e].double().cpu().numpy() for e in used}, r.E)
        self.wd = _HostExperts({e: case.w_down[e].double().cpu().numpy() for e in used}, r.E)
        self.x = case.x[:self.n_max].double().cpu().numpy()
        self.w = case.topk_w[:self.n_max].double().cpu().numpy()
        self.dy = case.dy[:self.n_max].double().cpu().numpy()

    def experts(self, n):
        import numpy as np
        return sorted(set(int(e) for e in np.unique(self.idx[:n])))

    def step(self, n):
        """One fp64 oracle pass (forward + backward) over the first n sampled
        tokens; returns its wall time in seconds."""
        import oracle
        r = self.r
        ex = self.experts(n)
        t0 = time.perf_counter()
        oracle.moe_forward(self.x[:n], self.idx[:n], self.w[:n], self.wgu, self.wd, r.act,
                           r.limit, r.alpha)
        oracle.moe_backward(self.dy[:n], self.x[:n], self.idx[:n], self.w[:n], self.wgu, self.wd,
                            r.act, r.limit, r.alpha, experts=ex)
        return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def cpu_baseline(case, target_s):
    """The oracle timed on the host cores over OracleSample's tokens, repeated
    until about target_s seconds of CPU work have been timed."""
    smp = OracleSample(case)
    n = smp.n_max
    t1 = smp.step(n)
    reps = max(1, int(round(target_s / max(t1, 1e-3))))
    t = sum(smp.step(n) for _ in range(reps))
    fs = layer_flops(case.recipe.scaled(T=n))
    return {"value": round(reps * (fs[0] + fs[1]) / t / 1e12, 5), "unit": "TFLOP/s",
            "cores": cpu_cores(), "kind": "oracle",
            "sample": "fp64 numpy oracle on %s: fwd+bwd over the first %d of %d tokens (the "
                      "prefix touching at most 16 experts; their weights in host fp64 before the "
                      "clock), %d passes, %.1f s" % (cpu_model(), n, case.recipe.T, reps, t)}


def stats_ms(samples):
    """Median, p10 and p90 of per-call times in ms."""
    xs = sorted(samples)

    def q(p):
        if not xs:
            return None
        pos = p * (len(xs) - 1)
        lo = int(pos)
        hi = min(lo + 1, len(xs) - 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (pos - lo)

    return {"median": round(q(0.5), 4), "p10": round(q(0.1), 4), "p90": round(q(0.9), 4),
            "n": len(xs)}


def timed_calls(fn, n, stream):
    """Run fn n times on `stream` with an event pair around each call; returns
    the per-call device times in ms."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]


# ---------------------------------------------------------------- other configs

# The workloads reported beside the bench line: the SwiGLU forward and
# backward shapes and the load-imbalance sweep on the backward shape.
CONFIG_RUNS = [("swiglu_fwd", None), ("swiglu_bwd", None)] + \
    [("zipf_sweep", T) for T in (512, 2048, 8192, 16384)]


def measure_configs(synth, LayerRunner, stream, P, BW, peak_src, n_calls=10, warm=2):
    """Per workload: training forward, inference forward and backward, each
    timed per call (median, p10, p90 over n_calls after `warm` untimed
    calls), with each half's fraction of its roofline max(FLOPs / P, bytes /
    BW) at the median."""
    import torch
    from dispatch_gemm_combine_gb300 import MOE_BF16
    res = {}
    for name, T in CONFIG_RUNS:
        r = synth.RECIPES[name]
        if T is not None:
            r = r.scaled(T=T)
        case = synth.make_case(r, device="cuda")
        run = LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, MOE_BF16, r.limit, r.alpha)
        a = (case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)

        def fwd(inference=False):
            run.plan(case.topk_idx)
            run.forward(*a, inference=inference)

        def bwd():
            run.backward(case.dy, *a)

        for _ in range(warm):
            fwd()
            bwd()
        fc = timed_calls(fwd, n_calls, stream)
        ic = timed_calls(lambda: fwd(True), n_calls, stream)
        fwd()   # the saved context of a training forward for the backward calls
        bc = timed_calls(bwd, n_calls, stream)
        run.check()
        e_active = int((run.plan_t["counts"] > 0).sum().item())
        zero, ratio = synth.routing_stats(case.topk_idx, r.E)
        f_fwd, f_bwd = layer_flops(r)
        b_fwd, b_bwd = layer_bytes(r, e_active)

        def part(calls, flops, byts):
            m = statistics.median(calls)
            roof = max(flops / P, byts / BW) * 1e3
            return {"ms": stats_ms(calls), "tflops": round(flops / (m * 1e-3) / 1e12, 1),
                    "frac": round(roof / m, 4), "bound": "tensor" if flops / P > byts / BW else "hbm"}

        key = name if T is None else "%s_T%d" % (name, T)
        fp = part(fc, f_fwd, b_fwd)
        bp = part(bc, f_bwd, b_bwd)
        res[key] = {"workload": workload_name(name, r), "fwd": fp,
                    "fwd_inference": part(ic, f_fwd, b_fwd), "bwd": bp,
                    "step_ms": round(fp["ms"]["median"] + bp["ms"]["median"], 4),
                    "tflops": round((f_fwd + f_bwd) / ((fp["ms"]["median"] + bp["ms"]["median"])
                                                       * 1e-3) / 1e12, 1),
                    "experts_active": e_active, "experts_empty_frac": round(zero, 3),
                    "hottest_over_mean": round(ratio, 2)}
        del run, case, a
        torch.cuda.empty_cache()
    res["peaks"] = "%s: P = %.1f TFLOP/s sustained bf16, BW = %.1f GB/s" % (peak_src, P / 1e12,
                                                                           BW / 1e9)
    return res


# ---------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target length of the oracle sample (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload table of the other synthetic configs")
    ap.add_argument("--tokens", type=int, default=None,
                    help="run the workload at this many tokens (the load-imbalance sweep's T "
                         "values); the bench line itself uses the workload's own T")
    ap.add_argument("--gate-up-layout", choices=["concat", "interleaved"], default="concat",
                    help="column layout of w_gate_up (the same random weights either way)")
    ap.add_argument("--experts", type=int, default=None,
                    help="profiling case: use this many experts and scale the tokens so each "
                         "expert keeps the workload's rows (not a bench line)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    import torch
    import synth

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, torch, synth)

    import torch.distributed as dist
    from dispatch_gemm_combine_gb300 import moe_kernel_launch_count, moe_profile_enable, moe_profile_read
    from dispatch_gemm_combine_gb300.runner import LayerRunner
    from dispatch_gemm_combine_gb300 import MOE_BF16, MOE_FP32

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    r = synth.RECIPES[args.workload]
    if args.tokens:
        r = r.scaled(T=args.tokens)
    if args.experts:
        r = r.scaled(E=args.experts, T=max(1, r.T * args.experts // r.E))
    case = synth.make_case(r, device="cuda")
    dt = MOE_BF16 if r.dtype == "bf16" else MOE_FP32
    layout = 1 if args.gate_up_layout == "interleaved" else 0
    run = LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, dt, r.limit, r.alpha, gate_up_layout=layout)
    stream = torch.cuda.current_stream()

    def step():
        run.plan(case.topk_idx)
        run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
        run.backward(case.dy, case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    run.check()

    def barrier():
        if world > 1:
            dist.barrier()

    def ranks_max(v):
        return max_over_ranks(v, world, dist if world > 1 else None, "cuda")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.6)
    # ---- timed region: K steps, device time with CUDA events on the stream
    barrier()
    torch.cuda.synchronize()
    n0 = moe_kernel_launch_count()
    # one event before the first step and one after each step (same stream):
    # the whole region gives the mean, the gaps give per-step percentiles
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    launches = moe_kernel_launch_count() - n0
    clocks.stop()
    ms = ranks_max(evs[0].elapsed_time(evs[-1])) / args.steps
    step_stats = stats_ms([evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)])
    run.check()

    # ---- per-kernel times (separate pass, library event timer on the same stream)
    moe_profile_enable(True)
    moe_profile_read()
    nprof = max(3, min(args.steps, 20))
    for _ in range(nprof):
        step()
    torch.cuda.synchronize()
    prof = moe_profile_read()
    moe_profile_enable(False)

    # ---- fwd / bwd split: per-call device times (median, p10, p90)
    def timed(fn, n):
        return statistics.mean(timed_calls(fn, n, stream))

    n_split = max(3, min(args.steps, 20))
    fwd_calls = timed_calls(lambda: (run.plan(case.topk_idx),
                                     run.forward(case.x, case.topk_idx, case.topk_w,
                                                 case.w_gate_up, case.w_down)), n_split, stream)
    bwd_calls = timed_calls(lambda: run.backward(case.dy, case.x, case.topk_idx, case.topk_w,
                                                 case.w_gate_up, case.w_down), n_split, stream)
    # inference-mode forward: no context saved for a backward
    inf_calls = timed_calls(lambda: (run.plan(case.topk_idx),
                                     run.forward(case.x, case.topk_idx, case.topk_w,
                                                 case.w_gate_up, case.w_down, inference=True)),
                            n_split, stream)
    fwd_ms = statistics.median(fwd_calls)
    bwd_ms = statistics.median(bwd_calls)
    # the memory-lean backward: no saved context, recomputed inside
    run.backward(case.dy, case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down,
                 recompute=True)
    bwd_re_ms = statistics.median(timed_calls(
        lambda: run.backward(case.dy, case.x, case.topk_idx, case.topk_w, case.w_gate_up,
                             case.w_down, recompute=True), n_split, stream))
    # the layer's forward output for the e2e check below (the inference
    # forward above left the same y)
    # ---- end to end: pinned host inputs in, per-token results out, every step.
    # As a training input pipeline runs it: a copy stream brings step i+1's
    # inputs in and step i's results out while step i+1 computes, with two sets
    # of device buffers (a second runner) so that no copy touches a buffer a
    # running step uses.  Every step still moves its whole inputs and results
    # across the host link; the timed region runs from the first input copy to
    # the last result copy.
    runs = [run, LayerRunner(r.T, r.H, r.I, r.E, r.k, r.act, dt, r.limit, r.alpha,
                             gate_up_layout=layout)]
    h_in = {n: getattr(case, n).cpu().pin_memory() for n in ("x", "topk_idx", "topk_w", "dy")}
    d_in = [{n: torch.empty_like(getattr(case, n)) for n in h_in} for _ in runs]
    h_out = [{"y": torch.empty(run.y.shape, dtype=run.y.dtype).pin_memory(),
              "dx": torch.empty(run.dx.shape, dtype=run.dx.dtype).pin_memory(),
              "d_topk_w": torch.empty(run.d_topk_w.shape, dtype=torch.float32).pin_memory()}
             for _ in runs]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())
    copy = torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event() for _ in runs]
    in_ready, computed, out_done = ev(), ev(), ev()

    def e2e_steps(n):
        """n end-to-end steps; returns their mean time in ms."""
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        copy.wait_event(t0)

        def bring_in(i):
            b = i % 2
            with torch.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(computed[b])        # step i-2 has read these buffers
                for name in h_in:
                    d_in[b][name].copy_(h_in[name], non_blocking=True)
                in_ready[b].record(copy)

        bring_in(0)
        for i in range(n):
            b, R = i % 2, runs[i % 2]
            if i + 1 < n:
                bring_in(i + 1)
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(out_done[b])          # step i-2's results have left
            d = d_in[b]
            R.plan(d["topk_idx"])
            R.forward(d["x"], d["topk_idx"], d["topk_w"], case.w_gate_up, case.w_down)
            R.backward(d["dy"], d["x"], d["topk_idx"], d["topk_w"], case.w_gate_up, case.w_down)
            computed[b].record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(computed[b])
                h_out[b]["y"].copy_(R.y, non_blocking=True)
                h_out[b]["dx"].copy_(R.dx, non_blocking=True)
                h_out[b]["d_topk_w"].copy_(R.d_topk_w, non_blocking=True)
                out_done[b].record(copy)
        stream.wait_event(out_done[(n - 1) % 2])
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    e2e_steps(3)
    n_e2e = max(3, args.steps)   # as many steps as the device-only figure, at the same clocks
    barrier()
    e2e_ms = ranks_max(e2e_steps(n_e2e))
    for R in runs:
        R.check()
    # the results that came back are the layer's (same inputs every step)
    assert torch.equal(h_out[(n_e2e - 1) % 2]["dx"], run.dx.cpu())

    # ---- the expert-parallel path on this one rank (§8(f) row 4): its
    # exchanges are identities here, so this times its own steps (two row
    # gathers, the owner-side layer at k = 1, the fp32 combine and the host
    # round trip of the counts each forward makes) against the fused layer,
    # and checks that it returns the same y and dx bit for bit
    from dispatch_gemm_combine_gb300.expert_parallel import CudaOps, ExpertParallelMoE
    run.plan(case.topk_idx)
    y_ref = run.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down).clone()
    dx_ref = run.backward(case.dy, case.x, case.topk_idx, case.topk_w, case.w_gate_up,
                          case.w_down)[0].clone()
    ep = ExpertParallelMoE(r.E, r.k, CudaOps(r.H, r.I, r.act, dt, r.limit, r.alpha,
                                             gate_up_layout=layout))

    def ep_step():
        ep.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
        return ep.backward(case.dy)

    ep_step()
    ep_y = ep.forward(case.x, case.topk_idx, case.topk_w, case.w_gate_up, case.w_down)
    ep_dx = ep.backward(case.dy)[0]
    ep_same = bool(torch.equal(ep_y, y_ref) and torch.equal(ep_dx, dx_ref))
    ep_calls = timed_calls(ep_step, max(3, min(args.steps, 10)), stream)
    del ep, ep_y, ep_dx, y_ref, dx_ref
    torch.cuda.empty_cache()

    # ---- accounting
    e_active = int((run.plan_t["counts"] > 0).sum().item())

    # ---- the router step before the layer (not part of the layer metric):
    # fp32 logits [T, E] -> top-k ids, softmax weights and the plan (it
    # overwrites the runner's plan, so it runs after the layer's accounting)
    g = torch.Generator(device="cuda").manual_seed(r.seed)
    logits = torch.randn(r.T, r.E, device="cuda", generator=g)
    r_idx = torch.empty((r.T, r.k), dtype=torch.int32, device="cuda")
    r_w = torch.empty((r.T, r.k), dtype=torch.float32, device="cuda")
    for _ in range(3):
        run.route(logits, r_idx, r_w)
    route_ms = timed(lambda: run.route(logits, r_idx, r_w), 50)
    run.check()
    f_fwd, f_bwd = layer_flops(r)
    b_fwd, b_bwd = layer_bytes(r, e_active)
    peaks, peak_src = load_peaks()
    P = peaks["bf16_tflops_sustained"] * 1e12
    BW = peaks["hbm_gbs"] * 1e9
    step_flops = f_fwd + f_bwd
    value = job_throughput(step_flops, world, ms)

    # dominant kernel and its roofline
    work = kernel_work(r, e_active)
    per_kernel = {}
    for name, (tot, cnt) in prof.items():
        if cnt:
            per_kernel[name] = {"ms_per_launch": tot / cnt, "launches": cnt,
                                "share": None}
    tot_ms = sum(v["ms_per_launch"] * v["launches"] for v in per_kernel.values())
    for v in per_kernel.values():
        v["share"] = v["ms_per_launch"] * v["launches"] / tot_ms if tot_ms else None
    dom = max(per_kernel, key=lambda n: per_kernel[n]["ms_per_launch"] * per_kernel[n]["launches"])
    dflops, dbytes = work.get(dom, (0.0, 0.0))
    dsec = per_kernel[dom]["ms_per_launch"] * 1e-3
    tensor_bound = dflops / P > dbytes / BW
    if tensor_bound:
        achieved, peak, unit = dflops / dsec / 1e12, P / 1e12, "TFLOP/s"
    else:
        achieved, peak, unit = dbytes / dsec / 1e9, BW / 1e9, "GB/s"
    roofline = {"kernel": dom, "bound": "tensor" if tensor_bound else "hbm",
                "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": committed_traffic(dom),
                "algorithmic": dflops if tensor_bound else dbytes,
                "peak_source": peak_src + (" sustained bf16" if tensor_bound else " hbm")}
    for name, v in per_kernel.items():
        fl, by = work.get(name, (0.0, 0.0))
        s = v["ms_per_launch"] * 1e-3
        v["tflops"] = round(fl / s / 1e12, 1) if fl else None
        v["gbs"] = round(by / s / 1e9, 1) if by else None
        v["ms_per_launch"] = round(v["ms_per_launch"], 4)
        v["share"] = round(v["share"], 4) if v["share"] is not None else None

    def layer_part(ms_, flops, byts):
        roof = max(flops / P, byts / BW) * 1e3
        return {"ms": round(ms_, 4), "tflops": round(flops / (ms_ * 1e-3) / 1e12, 1),
                "roofline_ms": round(roof, 4), "frac": round(roof / ms_, 4),
                "bound": "tensor" if flops / P > byts / BW else "hbm",
                "algorithmic_bytes": byts, "flops": flops}

    out = {
        "metric": "MoE layer ms & TFLOP/s, % of bf16 tensor roofline (fwd and bwd)",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": r.dtype,
        "data": "synthetic",
        "config": {"workload": workload_name(args.workload, r),
                   "T": r.T, "H": r.H, "I": r.I, "E": r.E, "k": r.k, "seed": r.seed,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "gate_up_layout": args.gate_up_layout,
                   "l2": "no flush: %.1f GB of expert weights per step exceed the 129 MB L2"
                         % (r.E * 3 * r.H * r.I * case.w_down.element_size() / 1e9)},
        "step_ms": step_stats,
        "layer": {"fwd": dict(layer_part(fwd_ms, f_fwd, b_fwd), **{"calls": stats_ms(fwd_calls)}),
                  "fwd_inference": dict(layer_part(statistics.median(inf_calls), f_fwd, b_fwd),
                                        **{"calls": stats_ms(inf_calls)}),
                  "bwd": dict(layer_part(bwd_ms, f_bwd, b_bwd), **{"calls": stats_ms(bwd_calls)}),
                  "bwd_recompute_ms": round(bwd_re_ms, 4),
                  "timing": "fwd = plan + training forward (saves the context), fwd_inference = "
                            "plan + forward without it, bwd = backward from the saved context; "
                            "ms and frac use the median call"},
        "roofline": roofline,
        "kernels": per_kernel,
        "e2e": {"value": round(job_throughput(step_flops, world, e2e_ms), 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipeline": "pinned-host copies on a copy stream: step i+1's inputs in and step "
                            "i's results out while the GPU computes (two buffer sets)"},
        "gpu_launches": int(launches),
        "router": {"ms": round(route_ms, 4), "what": "moe_route: fp32 logits [T,E] -> top-%d ids, "
                   "softmax weights and the dispatch plan (outside the layer metric)" % r.k},
        "expert_parallel": {"ranks": 1, "ms": stats_ms(ep_calls),
                            "overhead_vs_layer": round(statistics.median(ep_calls) /
                                                       (fwd_ms + bwd_ms) - 1.0, 4),
                            "bitwise_equal_to_layer": ep_same,
                            "what": "ExpertParallelMoE fwd+bwd on one rank (exchanges are "
                                    "identities): plan, row gathers, the owner-side layer at "
                                    "k = 1, fp32 combine, one host read of the counts"},
        "clocks": clocks.summary(),
        "experts_active": e_active,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    if not args.no_configs and args.tokens is None and args.experts is None:
        # the other synthetic workloads, each on its own buffers (the bench
        # workload's are released first)
        del runs, d_in, run, case
        torch.cuda.empty_cache()
        out["configs"] = measure_configs(synth, LayerRunner, stream, P, BW, peak_src)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()
    return 0


def workload_name(name, r):
    act = "clamped GLU (%.1f, %g)" % (r.limit, r.alpha) if r.act == 1 else "SwiGLU"
    return "%s fwd+bwd: T=%d H=%d I=%d E=%d top-%d %s" % (name, r.T, r.H, r.I, r.E, r.k, act)


def run_reference(args, torch, synth):
    """Reference arm: the fp64 oracle on the host cores, each step a bounded
    token sample of the same workload (OracleSample: the prefix of tokens that
    touches at most 16 experts, their weights in host fp64 before the steps),
    as many of those tokens as fit about two minutes for all steps."""
    r = synth.RECIPES[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = synth.make_case(r, device=dev)
    smp = OracleSample(case)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    t1 = smp.step(1)
    n_tok = max(1, min(smp.n_max, int(per_step / max(t1, 1e-3))))
    for _ in range(args.warmup):
        smp.step(n_tok)
    t = sum(smp.step(n_tok) for _ in range(args.steps))
    fs = layer_flops(r.scaled(T=n_tok))
    value = args.steps * (fs[0] + fs[1]) / t / 1e12
    sample = ("fp64 numpy oracle on %s: fwd+bwd over the first %d of %d tokens per step (%d "
              "experts' weights, in host fp64 before the steps)"
              % (cpu_model(), n_tok, r.T, len(smp.experts(n_tok))))
    out = {
        "metric": "MoE layer ms & TFLOP/s, % of bf16 tensor roofline (fwd and bwd)",
        "value": round(value, 5), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * t / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": workload_name(args.workload, r), "sample_tokens": n_tok},
        "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())
