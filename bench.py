#!/usr/bin/env python
"""Throughput of the grouped MXFP8 MoE expert MLP (route + forward + backward)
on GB300, through the library's C ABI.

One step = one pass of the whole path over one batch: top-k routing, permute,
weight and activation quantisation, gate-up GEMM with fused ScaledSwiGLU and
re-quantisation, down GEMM, combine, then the backward (dy quantisation,
dgrad-down with fused dSwiGLU, wgrad-down, dgrad-gate-up, wgrad-gate-up,
combine dx, dprobs).  Default workload: one Mixtral-8x7B MoE layer
(T=16384 tokens = batch 4 x seq 4096, H=4096, I=14336, E=8, top-2), seeded
synthetic inputs.

  value   : GEMM TFLOP/s of the whole step (18*R*H*I per step), inputs resident
            in HBM, timed with CUDA events on the launching stream.
  e2e     : the same metric with inputs copied host->device and y, dx copied
            back each step (pinned host buffers), through the C ABI.
  roofline: the dominant kernel, timed live per launch with events around its
            stage call, against the MXFP8 peak: the higher of 2 x the measured
            burst dense bf16 rate and this GPU's MXFP8 MMA-only loop
            (mxg_bench_mxfp8_mma_peak), measured in the same run.
  workloads: the Zipf-skewed Mixtral layer and the fine-grained 64-expert
            top-8 layer, timed the same way (device-resident), with their
            routing balance.
  cpu_baseline: the CPU oracle on a bounded sample of the same workload.

--impl reference runs that CPU oracle as the reference arm.
Multi-GPU (torchrun): every rank runs an independent replica (the path does
not exchange data); value = all ranks' work / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped MoE MLP fwd+bwd TFLOP/s & tokens/s; % of MXFP8 tensor-core peak"
FALLBACK_BF16_SUSTAINED = 1700.0     # TFLOP/s, used only without a measured peaks file
FALLBACK_HBM = 6800.0                # GB/s

# CPU sample of the workload for the oracle: the first T_S tokens, all experts,
# full hidden size, the intermediate dimension cut to its first I_S columns.
CPU_SAMPLE_TOKENS = 512
CPU_SAMPLE_I = 2048          # the reported cpu_baseline (~10-30 s of host work: ~10 s on 16 Grace cores)
CPU_SAMPLE_I_REF = 256       # per step of the reference arm (K + W steps within a few minutes)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-router", action="store_true", help="skip timing the router front end")
    ap.add_argument("--no-workloads", action="store_true", help="skip timing the skew and fine-grained workloads")
    ap.add_argument("--no-accum", action="store_true",
                    help="skip timing gradient-accumulation micro-batches (weight cache + fp32 main_grad)")
    ap.add_argument("--precision", choices=["mxfp8", "bf16", "fp8"], default="mxfp8",
                    help="bf16: the like-for-like BF16 grouped MLP; fp8: per-tensor FP8 (one scale per expert "
                         "tensor) instead of the MXFP8 path")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": FALLBACK_BF16_SUSTAINED, "hbm_gbs": FALLBACK_HBM}, "fallback"


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip() == "Active":
                    reasons.add(n)
        loaded = [s for s in sm if s > 0.5 * (max(sm) if sm else 1)]
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle --
def cpu_sample_inputs(inp, wl, i_cut=CPU_SAMPLE_I):
    import torch
    T_s, I_s, I = min(CPU_SAMPLE_TOKENS, wl.T), min(i_cut, wl.I), wl.I
    wgu = torch.cat([inp["w_gate_up"][:, :I_s], inp["w_gate_up"][:, I:I + I_s]], 1)
    return {"logits": inp["logits"][:T_s].numpy(), "x": inp["x"][:T_s].double().numpy(),
            "w_gate_up": wgu.double().numpy(), "w_down": inp["w_down"][:, :, :I_s].double().numpy(),
            "dy": inp["dy"][:T_s].double().numpy(), "T": T_s, "I": I_s}


def cpu_sample_run(s, k, quant=True):
    from oracle import moe
    ids, probs = moe.route_topk(s["logits"], k)
    ctx = moe.mlp_fwd(s["x"], ids, probs, s["w_gate_up"], s["w_down"], quant=quant)
    moe.mlp_bwd(ctx, s["dy"])


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(inp, wl, reps: int = 1, quant: bool | str = True) -> dict:
    s = cpu_sample_inputs(inp, wl)
    flops = 18.0 * s["T"] * wl.k * wl.H * s["I"]
    t0 = time.perf_counter()
    for _ in range(reps):
        cpu_sample_run(s, wl.k, quant)
    dt = (time.perf_counter() - t0) / reps
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"fwd+bwd of the first {s['T']} tokens, all {wl.E} experts, H={wl.H}, intermediate cut to "
                      f"its first {s['I']} columns ({flops / 1e9:.1f} GFLOP, {dt:.1f} s), fp64 numpy oracle",
            "seconds": dt}


# ------------------------------------------------------------------- GPU --
def code_hash(path: str) -> str:
    """sha256 (16 hex digits) of a source file's code: `//` comments, trailing
    blanks and empty lines are left out, so a comment edit keeps a profile valid
    while any change to the code itself invalidates it."""
    lines = []
    for ln in open(path, encoding="utf-8").read().splitlines():
        code = re.sub(r"//.*$", "", ln) if '"' not in ln else ln
        code = code.rstrip()
        if code:
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def traffic_for(stage: str, workload: str) -> int | None:
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current source of the kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    src = os.path.join(ROOT, "mxfp8_grouped_gemm_gb300", "csrc", d.get("source", "gemm.cu"))
    h = code_hash(src) if os.path.exists(src) else None
    e = d.get("entries", {}).get(f"{workload}/{stage}")
    if not e or e.get("source_sha") != h:
        return None
    return int(e["bytes_per_launch"])


def max_over_ranks(times_ms, world, device=None):
    """Per-rank step times -> the slowest rank's (replicas run in lock step from
    the barrier, so the job's time is the maximum)."""
    if world == 1:
        return [float(t) for t in times_ms]
    import torch
    t = torch.tensor([float(x) for x in times_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(flops_per_replica_step, ms, world):
    """Whole-job TFLOP/s: every replica does a full step of work per step time."""
    return world * flops_per_replica_step / (ms * 1e-3) / 1e12


def mma_peak(m, dev, stream, steps: int = 20000, reps: int = 5) -> dict:
    """The MXFP8 MMA-only loop (mxg_bench_mxfp8_mma_peak): best of `reps`
    launches, each timed with events on the launching stream."""
    import torch
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):
        m.mxg_bench_mxfp8_mma_peak(steps, st, stream)
    best, flops = 0.0, 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        flops = m.mxg_bench_mxfp8_mma_peak(steps, st, stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        best = max(best, flops / (a.elapsed_time(b) * 1e-3) / 1e12)
    if int(st.item()) != 0:
        raise SystemExit(f"bench: MMA peak loop status {m.status_string(int(st.item()))}")
    return {"tflops": round(best, 1), "flop_per_launch": flops,
            "how": f"one CTA per SM, {steps} steps of four 128x256x32 block-scaled E4M3 MMAs on resident "
                   f"operands (scale factors copied into TMEM per stage), best of {reps} launches"}


def split_stats(split) -> dict:
    """Routing balance of one step: rows per expert."""
    import numpy as np
    split = np.asarray(split)
    nz = split[split > 0]
    return {"min": int(split.min()), "max": int(split.max()), "mean": round(float(split.mean()), 1),
            "zeros": int((split == 0).sum()), "max_over_mean": round(float(split.max() / split.mean()), 3),
            "not_multiple_of_128": int((nz % 128 != 0).sum())}


def time_router(m, x, k: int, E: int, dev, stream, reps: int = 20) -> dict:
    """The router front end on the workload's tokens, outside the MLP step:
    logits on the tensor cores + route (fwd), the same fused with the permute
    (fwd_permute), and the backward; events on the stream."""
    import torch

    import synthetic
    T, H = x.shape
    peaks, _ = load_peaks()
    w_r = synthetic.random_bf16((E, H), 4242, std=0.02).to(dev)
    dprobs = torch.randn(T, k, device=dev, generator=torch.Generator(device=dev).manual_seed(5))
    dx_r = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
    st_r = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_r = torch.empty(m.mxg_router_bwd_workspace_bytes(T, H, E, k), dtype=torch.uint8, device=dev)
    dw_r = torch.empty((E, H), dtype=torch.float32, device=dev)
    lo, ri, rp = m.mxg_router_fwd(x, w_r, k)
    # the calls are recorded in CUDA graphs and the replays timed: each call
    # is a few tens of microseconds of GPU work, shorter than its host-side
    # launch path, so back-to-back eager calls would time the host
    fp_out = m.mxg_router_fwd_permute(x, w_r, k, st_r)
    graphs = []
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        for _ in range(2):       # warm-up (module loading, function attributes) before capture
            m.mxg_router_fwd(x, w_r, k, logits=lo, ids=ri, probs=rp)
            m.mxg_router_bwd(x, w_r, ri, rp, dprobs, dx_r, st_r, dw_router=dw_r, workspace=ws_r)
    torch.cuda.synchronize(dev)
    for call in (lambda: m.mxg_router_fwd(x, w_r, k, logits=lo, ids=ri, probs=rp),
                 lambda: m.mxg_router_fwd_permute(x, w_r, k, st_r),
                 lambda: m.mxg_router_bwd(x, w_r, ri, rp, dprobs, dx_r, st_r, dw_router=dw_r, workspace=ws_r)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                call()
        graphs.append(g)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record(stream)
    for i, g in enumerate(graphs):
        g.replay()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    del fp_out
    if int(st_r.item()) != 0:
        raise SystemExit(f"bench: router status {m.status_string(int(st_r.item()))}")
    f_ms, fp_ms, b_ms = (ev[i].elapsed_time(ev[i + 1]) / reps for i in range(3))
    # algorithmic bytes: fwd reads x (and W_r), writes logits, ids, probs; bwd
    # reads probs, dprobs, ids, x, reads and writes dx, writes dW_r
    fb = T * H * 2 + E * H * 2 + T * E * 4 + T * k * 8
    bb = T * k * 12 + T * H * 2 + 2 * T * H * 2 + E * H * 4
    flops = 2.0 * T * H * E
    return {"T": T, "H": H, "E": E, "k": k, "fwd_ms": round(f_ms, 4), "fwd_permute_ms": round(fp_ms, 4),
            "bwd_ms": round(b_ms, 4), "fwd_gbs": round(fb / (f_ms * 1e-3) / 1e9, 1),
            "fwd_frac_of_hbm": round(fb / (f_ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]), 3),
            "fwd_tflops": round(flops / (f_ms * 1e-3) / 1e12, 1),
            "fwd_frac_of_bf16": round(flops / (f_ms * 1e-3) / 1e12 / float(peaks["bf16_tflops"]), 4),
            "bwd_gbs": round(bb / (b_ms * 1e-3) / 1e9, 1), "note": "not part of the MLP step"}


def time_workload(m, name: str, steps: int, warmup: int, dev, stream, precision: str, p_mx: float) -> dict:
    """One more workload through the same calls as the main step (device-resident
    inputs, route + forward + backward per step, events on the stream)."""
    import torch

    import synthetic
    wl = synthetic.WORKLOADS[name]
    inp = synthetic.make_inputs(wl)
    if "dy" not in inp:
        inp["dy"] = synthetic.random_bf16((wl.T, wl.H), 77)
    layer = m.GroupedMLP(wl.T, wl.H, wl.I, wl.E, wl.k, device=dev, precision=precision)
    d = {n: v.to(dev) for n, v in inp.items() if isinstance(v, torch.Tensor)}

    def step():
        ids, probs = layer.route(d["logits"])
        layer.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"])
        layer.backward(d["dy"])
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    if layer.status() != 0:
        raise SystemExit(f"bench: {name} device status {m.status_string(layer.status())}")
    ms = a.elapsed_time(b) / steps
    router = time_router(m, d["x"], wl.k, wl.E, dev, stream) if wl.H % 128 == 0 else None
    flops = wl.gemm_flops(True)
    tf = flops / (ms * 1e-3) / 1e12
    out = {"workload": workload_config(wl, precision, 1)["workload"], "ms_per_step": round(ms, 4),
           "tflops": round(tf, 2), "tokens_per_s": round(wl.T / (ms * 1e-3), 1), "frac_of_mxfp8_peak": round(tf / p_mx, 4),
           "steps": steps, "warmup": warmup, "split_sizes": split_stats(layer.split_sizes.cpu().numpy()),
           "router": router}
    del layer, d
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world):
    import numpy as np
    import torch

    import mxfp8_grouped_gemm_gb300 as m
    import synthetic
    from mxfp8_grouped_gemm_gb300 import build as libbuild

    libbuild.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    if not m.mxg_device_supported():
        raise SystemExit("bench: current device is not sm_103 (GB300)")
    wl = synthetic.WORKLOADS[args.workload]
    inp = synthetic.make_inputs(wl)
    if "dy" not in inp:
        inp["dy"] = synthetic.random_bf16((wl.T, wl.H), 77)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    layer = m.GroupedMLP(T, H, I, E, k, device=dev, precision=args.precision)
    d = {n: v.to(dev) for n, v in inp.items() if isinstance(v, torch.Tensor)}
    stream = torch.cuda.current_stream(dev)

    def step_full():
        ids, probs = layer.route(d["logits"])
        layer.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"])
        layer.backward(d["dy"])

    peak_mma = mma_peak(m, dev, stream) if args.precision != "bf16" else None
    for _ in range(args.warmup):
        step_full()
    torch.cuda.synchronize(dev)
    if layer.status() != 0:
        raise SystemExit(f"bench: device status {m.status_string(layer.status())}")

    # ---- device-resident timed region: every stage bracketed by events ----
    stages = ["route"] + [f"fwd.{s}" for s in m.FWD_STAGES] + [f"bwd.{s}" for s in m.BWD_STAGES]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    launches0 = m.mxg_launch_count()
    for s in range(args.steps):
        e = evs[s]
        e[0].record(stream)
        ids, probs = layer.route(d["logits"])
        e[1].record(stream)
        i = 2
        for st in range(len(m.FWD_STAGES)):
            layer.forward(d["x"], ids, probs, d["w_gate_up"], d["w_down"], stage=st)
            e[i].record(stream)
            i += 1
        for st in range(len(m.BWD_STAGES)):
            layer.backward(d["dy"], stage=st)
            e[i].record(stream)
            i += 1
    torch.cuda.synchronize(dev)
    launches = (m.mxg_launch_count() - launches0) / args.steps
    if world > 1:
        torch.distributed.barrier()
    total_ms = evs[0][0].elapsed_time(evs[-1][-1])
    stage_ms = {st: statistics.mean(evs[s][j].elapsed_time(evs[s][j + 1]) for s in range(args.steps))
                for j, st in enumerate(stages)}

    # ---- end to end through the C ABI with host buffers ----
    # Every step copies its inputs (x, logits, dy) from pinned host memory and
    # its results (y, dx) back.  Copies run on their own streams with double
    # buffering, so step i+1's inputs upload and step i's results download while
    # step i computes; the timed region spans the first upload to the last
    # download.
    e2e = None
    if not args.no_e2e:
        names = ("logits", "x", "dy")
        pin = {n: inp[n].pin_memory() for n in names}
        dev_in = [{n: torch.empty_like(d[n]) for n in names} for _ in range(2)]
        dev_out = [(torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                    torch.empty((T, H), dtype=torch.bfloat16, device=dev)) for _ in range(2)]
        host_out = [(torch.empty((T, H), dtype=torch.bfloat16).pin_memory(),
                     torch.empty((T, H), dtype=torch.bfloat16).pin_memory()) for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = 2 * T * H * 2
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        loaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        stored = [torch.cuda.Event() for _ in range(2)]
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        ea.record(up)
        for i in range(args.steps):
            b = i % 2
            if i >= 2:
                up.wait_event(computed[b])           # step i-2 is done reading these inputs
            with torch.cuda.stream(up):
                for n in names:
                    dev_in[b][n].copy_(pin[n], non_blocking=True)
            loaded[b].record(up)
            stream.wait_event(loaded[b])
            if i >= 2:
                stream.wait_event(stored[b])         # step i-2's results have been downloaded
            ids, probs = layer.route(dev_in[b]["logits"], stream=stream)
            layer.forward(dev_in[b]["x"], ids, probs, d["w_gate_up"], d["w_down"], stream=stream, y=dev_out[b][0])
            layer.backward(dev_in[b]["dy"], stream=stream, dx=dev_out[b][1])
            computed[b].record(stream)
            down.wait_event(computed[b])
            with torch.cuda.stream(down):
                host_out[b][0].copy_(dev_out[b][0], non_blocking=True)
                host_out[b][1].copy_(dev_out[b][1], non_blocking=True)
            stored[b].record(down)
        eb.record(down)
        torch.cuda.synchronize(dev)
        e2e_ms = ea.elapsed_time(eb) / args.steps
        e2e = {"ms": e2e_ms, "h2d": h2d, "d2h": d2h}
    # ---- router front end (logits GEMM H -> E + route, and its backward), on
    # the same tokens, outside the MLP step: reported beside it ----
    router = None
    if not args.no_router and H % 128 == 0:
        router = time_router(m, d["x"], k, E, dev, stream)
    # ---- gradient accumulation (MXFP8 path): the weights quantised once into
    # a weight cache per optimizer step, then micro-batches whose weight
    # gradients are added into fp32 main_grad buffers; reported beside the step
    accum = None
    if args.precision == "mxfp8" and not args.no_accum:
        mg = (torch.zeros((E, 2 * I, H), dtype=torch.float32, device=dev),
              torch.zeros((E, H, I), dtype=torch.float32, device=dev))

        def microbatch():
            ids_, probs_ = layer.route(d["logits"])
            layer.forward(d["x"], ids_, probs_)
            layer.backward(d["dy"], main_grad=mg)
        layer.quantize_weights(d["w_gate_up"], d["w_down"])
        for _ in range(2):
            microbatch()
        def microbatch_bf16_dw():
            ids_, probs_ = layer.route(d["logits"])
            layer.forward(d["x"], ids_, probs_)
            layer.backward(d["dy"])
        reps = max(3, min(args.steps, 10))
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        layer.quantize_weights(d["w_gate_up"], d["w_down"])
        ev[1].record(stream)
        for _ in range(reps):
            microbatch()
        ev[2].record(stream)
        for _ in range(reps):
            microbatch_bf16_dw()
        ev[3].record(stream)
        wg = [m.BWD_STAGES.index("wgrad_down"), m.BWD_STAGES.index("wgrad_gate_up")]
        for _ in range(reps):
            layer.backward(d["dy"], stage=wg[0], main_grad=mg)
        ev[4].record(stream)
        for _ in range(reps):
            layer.backward(d["dy"], stage=wg[1], main_grad=mg)
        ev[5].record(stream)
        torch.cuda.synchronize(dev)
        q_ms = ev[0].elapsed_time(ev[1])
        mb_ms, mb16_ms = ev[1].elapsed_time(ev[2]) / reps, ev[2].elapsed_time(ev[3]) / reps
        accum = {"quantize_weights_ms": round(q_ms, 4),
                 "ms_per_microbatch": round(mb_ms, 4),
                 "tflops_per_microbatch": round(wl.gemm_flops(True) / (mb_ms * 1e-3) / 1e12, 2),
                 "ms_per_microbatch_bf16_dw": round(mb16_ms, 4),
                 "wgrad_main_grad_ms": {"wgrad_down": round(ev[3].elapsed_time(ev[4]) / reps, 4),
                                        "wgrad_gate_up": round(ev[4].elapsed_time(ev[5]) / reps, 4)},
                 "note": "weights quantised once per optimizer step (weight cache); each micro-batch runs "
                         "route, forward and backward with dW added into fp32 main_grad (bf16_dw: dW written "
                         "in bf16 instead); not the step above"}
    clk = clocks.stop()
    if layer.status() != 0:
        raise SystemExit(f"bench: device status {m.status_string(layer.status())}")

    ms, e2e_ms = max_over_ranks([total_ms / args.steps, e2e["ms"] if e2e else 0.0], world, dev)
    if e2e:
        e2e["ms"] = e2e_ms
    flops = wl.gemm_flops(True)
    value = job_throughput(flops, ms, world)
    split = layer.split_sizes.cpu().numpy()

    peaks, peaks_kind = load_peaks()
    # the tensor roofline of the computing dtype.  The kernels are timed inside
    # a region of well under a second, so the burst figures apply: for MXFP8 the
    # higher of 2 x the measured burst bf16 (the nominal fp8/bf16 ratio) and the
    # MMA-only loop measured above; for the BF16 path the measured burst bf16
    ratio = 1.0 if args.precision == "bf16" else 2.0
    p_bf = ratio * float(peaks["bf16_tflops"])
    p_sus = ratio * float(peaks["bf16_tflops_sustained"])
    if peak_mma is not None and peak_mma["tflops"] > p_bf:
        p_mx = peak_mma["tflops"]
        p_src = f"MXFP8 MMA-only loop on this GPU in this run ({peak_mma['tflops']} TFLOP/s; " \
                f"2 x {peaks_kind} burst dense bf16 = {p_bf:.1f})"
    else:
        p_mx = p_bf
        p_src = (f"2 x " if ratio == 2.0 else "") + f"{peaks_kind} burst dense bf16 ({peaks['bf16_tflops']} TFLOP/s)"
    R = T * k
    stage_flops = {"fwd.gate_up": 4.0 * R * H * I, "fwd.down": 2.0 * R * H * I, "bwd.dgrad_down": 2.0 * R * H * I,
                   "bwd.wgrad_down": 2.0 * R * H * I, "bwd.dgrad_gate_up": 4.0 * R * H * I,
                   "bwd.wgrad_gate_up": 4.0 * R * H * I}
    dom = max(stage_ms, key=lambda s_: stage_ms[s_])
    if dom in stage_flops:
        ach = stage_flops[dom] / (stage_ms[dom] * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": round(ach, 1), "peak": round(p_mx, 1),
                "unit": "TFLOP/s", "frac": round(ach / p_mx, 4), "traffic": traffic_for(dom, args.workload),
                "peak_source": p_src, "frac_of_2x_burst_bf16": round(ach / p_bf, 4),
                "frac_of_2x_sustained_bf16": round(ach / p_sus, 4)}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": None, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": None, "traffic": None}
    gemm_ms = sum(stage_ms[s_] for s_ in stage_flops)
    gemm_kernels = {"peak_tflops": round(p_mx, 1), "peak_source": p_src,
                    **{s_: {"ms": round(stage_ms[s_], 4), "tflops": round(f / (stage_ms[s_] * 1e-3) / 1e12, 1),
                            "frac": round(f / (stage_ms[s_] * 1e-3) / 1e12 / p_mx, 4),
                            "frac_of_2x_burst_bf16": round(f / (stage_ms[s_] * 1e-3) / 1e12 / p_bf, 4)}
                       for s_, f in stage_flops.items()}}
    # memory-bound kernels against the measured copy bandwidth: algorithmic
    # bytes (each input read once, each output written once) / CUDA-event time
    mx = lambda n: n + n // 32                                  # E4M3 codes + E8M0 scales
    # algorithmic bytes: every input read once, every output written once,
    # unpadded rows (the padding rows the kernels also write are not credited)
    hbm_bytes = {
        "fwd.quant_weights": 2 * E * 3 * H * I + 2 * mx(E * 3 * H * I),   # bf16 in, two orientations out
        "fwd.quant_x": 2 * T * H + 2 * mx(R * H),                           # x once, row + token-column MX out
        "bwd.quant_dy": 2 * T * H + 2 * mx(R * H),
        "fwd.combine": 2 * R * H + 2 * T * H,                              # k rows in, one row out
        "bwd.combine_dx": 2 * R * H + 2 * T * H,
    }
    if args.precision != "mxfp8":       # the quantise stages move other bytes on the bf16 / fp8 paths
        hbm_bytes = {s_: v for s_, v in hbm_bytes.items() if "combine" in s_}
    else:                               # the MXFP8 path's combines run inside the down / dgrad-gate-up epilogues
        hbm_bytes = {s_: v for s_, v in hbm_bytes.items() if "combine" not in s_}
    hbm = {s_: {"ms": round(stage_ms[s_], 4), "bytes": int(b), "gbs": round(b / (stage_ms[s_] * 1e-3) / 1e9, 1),
                "frac": round(b / (stage_ms[s_] * 1e-3) / 1e9 / float(peaks["hbm_gbs"]), 3),
                "frac_of_8tbs": round(b / (stage_ms[s_] * 1e-3) / 8e12, 3)}
           for s_, b in hbm_bytes.items()}
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if args.precision == "bf16" else "e4m3", "data": "synthetic",
        "config": workload_config(wl, args.precision, world),
        "tokens_per_s": round(world * T / (ms * 1e-3), 1),
        "gemm_tflops": round(world * flops / (gemm_ms * 1e-3) / 1e12, 2),
        ("frac_of_bf16_peak" if args.precision == "bf16" else "frac_of_mxfp8_peak"): round(value / world / p_mx, 4),
        "peak_tflops": round(p_mx, 1),
        "peak_source": p_src,
        "stages_ms": {s_: round(v, 4) for s_, v in stage_ms.items()},
        "split_sizes": split_stats(split),
        "roofline": roof,
        "gemm_kernels": gemm_kernels,
        "hbm_kernels": {"peak_gbs": float(peaks["hbm_gbs"]), "peak_source": f"{peaks_kind} copy", **hbm},
        "gpu_launches": int(round(launches)),
        "clocks": clk,
    }
    if peak_mma is not None:
        res["mma_peak"] = peak_mma
    if router:
        res["router"] = router
    if accum:
        res["accumulation"] = accum
    if e2e:
        res["e2e"] = {"value": round(world * flops / (e2e["ms"] * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                      "ms_per_step": round(e2e["ms"], 4), "h2d_bytes_per_step": e2e["h2d"],
                      "d2h_bytes_per_step": e2e["d2h"]}
    # the other two large workloads, timed the same way (not part of `value`)
    if world == 1 and not args.no_workloads and args.workload == "mixtral":
        res["workloads"] = {n: time_workload(m, n, max(3, min(args.steps, 10)), 3, dev, stream, args.precision, p_mx)
                            for n in ("skew", "fine")}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(inp, wl, quant={"mxfp8": True, "bf16": False, "fp8": "fp8"}[args.precision])
    return res


def workload_config(wl, precision: str, world: int) -> dict:
    """The `config` object of the JSON line (both arms report the same one)."""
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    name = (f"{wl.name}: Mixtral-8x7B MoE layer T={T} H={H} I={I} E={E} top-{k}" if wl.name == "mixtral"
            else f"{wl.name}: T={T} H={H} I={I} E={E} top-{k}")
    return {"workload": name, "precision": precision, "tokens_per_step": T,
            "gemm_flops_per_step": wl.gemm_flops(True),
            "l2": "no flush: every step streams > 10 GB (weights 2.8 GB) through HBM, inputs > L2",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args):
    import synthetic
    wl = synthetic.WORKLOADS[args.workload]
    inp = synthetic.make_inputs(wl)
    if "dy" not in inp:
        inp["dy"] = synthetic.random_bf16((wl.T, wl.H), 77)
    s = cpu_sample_inputs(inp, wl, CPU_SAMPLE_I_REF)
    flops = 18.0 * s["T"] * wl.k * wl.H * s["I"]
    for _ in range(args.warmup):
        cpu_sample_run(s, wl.k)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_sample_run(s, wl.k)
    dt = (time.perf_counter() - t0) / args.steps
    value = flops / dt / 1e12
    sample = (f"each step: fwd+bwd of the first {s['T']} tokens, all {wl.E} experts, H={wl.H}, intermediate cut "
              f"to its first {s['I']} columns ({flops / 1e9:.1f} GFLOP), fp64 numpy CPU oracle")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, "mxfp8", 1),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
