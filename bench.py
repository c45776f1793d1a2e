#!/usr/bin/env python3
"""Benchmark of the fused feed-forward block on GB300, one JSON line on stdout.

Step = one forward of the GeGLU feed-forward block at 70B-class size
(T=8192 tokens, D=8192, H=28672: gate+up dual GEMM with the gelu_tanh(g)*u epilogue, then
the down GEMM) through the C ABI, inputs resident in HBM. The weights (1.41 GB) are far
larger than L2, so every step streams them from HBM again. Extra keys report the other
workloads (GPT-2-small GeGLU, the 4096-wide MLP at 4096 tokens and at 1 token, the small
fused block, the single Linear), the dominant kernel's roofline, an end-to-end number with
host buffers, and the oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs under torch.distributed.run: every rank runs its own replica of the step on its
own GPU (weak scaling, no collective in the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused MLP fwd TFLOP/s & % BF16 peak; batch-1 latency µs & % HBM GB/s"
HEADLINE = "geglu_8192x8192x28672"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=150)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-extras", action="store_true", help="headline only")
    p.add_argument("--cpu-sample-rows", type=int, default=0)
    p.add_argument("--profile-kernel", default=None,
                   choices=["gate_up", "down", "geglu", "mlp_up", "mlp", "mlp_decode", "linear",
                            "moe"],
                   help="profiling aid: launch one entry point --launches times on random "
                        "inputs of --shape and exit (no timing, no JSON)")
    p.add_argument("--shape", default="8192,8192,8192", help="T,D,H for --profile-kernel")
    p.add_argument("--launches", type=int, default=3)
    p.add_argument("--tiles", default="auto", choices=["auto", "single", "pair"],
                   help="tile-kernel policy for --profile-kernel")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------- distributed

class Dist:
    def __init__(self, n):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world != n and n > 1:
            raise SystemExit(f"--gpus {n} but WORLD_SIZE={self.world}: launch with torchrun")

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float, device=None) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------------- our arm

def run_ours(args, dist: Dist):
    import numpy as np
    import torch

    import feed_forward_gemm_gb300 as fm
    import synth

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    dist.init("nccl")
    fm.load()
    stream = torch.cuda.current_stream(dev)

    def up(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    def events_time(fn, iters):
        """ms per iteration of fn() over `iters` calls, CUDA events on the launching stream."""
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for _ in range(iters):
            fn()
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / iters

    # ---------------- headline workload: inputs resident in HBM
    w = synth.WORKLOADS[HEADLINE]
    t = w.generate()
    x, Wg, Wu, Wd = up(t["x"]), up(t["Wg"]), up(t["Wu"]), up(t["Wd"])
    y = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
    ws_bytes = fm.fmlp_geglu_workspace_size(w.T, w.D, w.H)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    m = ws.view(torch.bfloat16).view(w.T, w.H)

    def step():
        fm.fmlp_geglu(x, Wg, Wu, Wd, y, w.T, w.D, w.H, ws, ws_bytes, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fm.fmlp_device_status(stream) != fm.FMLP_OK:
        raise SystemExit(f"device status after warm-up: {fm.fmlp_last_error()}")

    clocks = ClockSampler(dist.local)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize(dev)
    ms = events_time(step, args.steps)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clk = clocks.stop()
    ms_max = dist.max(ms, dev)
    flops = w.flops()
    value = dist.world * flops / (ms_max * 1e-3) / 1e12

    # ---------------- the step's two kernels as separate calls, CUDA events between them
    # (the dominant kernel's roofline); these legs add up to this loop's time per iteration,
    # which is the step's without the programmatic overlap between the two kernels
    gu_flops = 2 * 2 * w.T * w.D * w.H

    def gate_up():
        fm.fmlp_geglu_gate_up(x, Wg, Wu, m, w.T, w.D, w.H, stream)

    def down():
        fm.fmlp_linear_bias(m, Wd, None, y, w.T, w.H, w.D, stream)
    for _ in range(2):
        gate_up()
        down()
    legs_iters = max(3, args.steps)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(legs_iters)]
    clocks_legs = ClockSampler(dist.local)
    clocks_legs.start()
    torch.cuda.synchronize(dev)
    for e in evs:
        e[0].record(stream)
        gate_up()
        e[1].record(stream)
        down()
        e[2].record(stream)
    torch.cuda.synchronize(dev)
    clk_legs = clocks_legs.stop()
    gu_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    down_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    pk, pk_src = peaks()
    gu_tflops = gu_flops / (gu_ms * 1e-3) / 1e12
    roofline = {
        "kernel": "gate+up dual GEMM with the gelu_tanh(g)*u epilogue ("
                  + fm.fmlp_describe_plan("gate_up", w.T, w.D, w.H) + ")",
        "bound": "tensor", "achieved": round(gu_tflops, 1), "peak": pk["bf16_tflops"],
        "unit": "TFLOP/s", "frac": round(gu_tflops / pk["bf16_tflops"], 4),
        "peak_source": f"{pk_src} bf16 burst (kernel timed alone)",
        "traffic": traffic_for("gemm_tc_geglu", gu_flops),
        "algorithmic_flops_per_launch": gu_flops, "ms_per_launch": round(gu_ms, 4),
        "down_gemm": {"plan": fm.fmlp_describe_plan("linear", w.T, w.H, w.D),
                      "ms_per_launch": round(down_ms, 4),
                      "tflops": round(2 * w.T * w.D * w.H / (down_ms * 1e-3) / 1e12, 1)},
        "legs": {"gate_up_ms": round(gu_ms, 4), "down_ms": round(down_ms, 4),
                 "sum_ms": round(gu_ms + down_ms, 4), "step_ms": round(ms_max, 4),
                 "iterations": legs_iters, "clocks": clk_legs,
                 "method": "each iteration: event, gate/up call, event, down call, event"},
    }
    torch.cuda.synchronize(dev)
    if fm.fmlp_device_status(stream) != fm.FMLP_OK:
        raise SystemExit(f"device status after timing: {fm.fmlp_last_error()}")

    # ---------------- end to end through the C ABI with host buffers
    # Every step copies its x from pinned host memory and its y back. Copies run on their own
    # streams into double-buffered device tensors, so step i's copies overlap the compute of
    # its neighbours, as a serving loop would run; each step's copies and compute are all
    # inside the timed region.
    x_host = torch.from_numpy(t["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = [torch.empty((w.T, w.D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    y_dev = [torch.empty_like(y) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):   # start with every buffer free
        ev_used[b].record(stream)
        ev_out[b].record(stream)

    def e2e_step(i):
        b = i % 2
        h2d.wait_event(ev_used[b])            # step i-2's compute is done with x_dev[b]
        with torch.cuda.stream(h2d):
            x_dev[b].copy_(x_host, non_blocking=True)
        ev_in[b].record(h2d)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])          # step i-2's result has left y_dev[b]
        fm.fmlp_geglu(x_dev[b], Wg, Wu, Wd, y_dev[b], w.T, w.D, w.H, ws, ws_bytes, stream)
        ev_used[b].record(stream)
        d2h.wait_event(ev_used[b])
        with torch.cuda.stream(d2h):
            y_host[b].copy_(y_dev[b], non_blocking=True)
        ev_out[b].record(d2h)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_iters = max(6, args.steps // 2)
    dist.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    t_start.record(h2d)
    for i in range(e2e_iters):
        e2e_step(i)
    stream.wait_stream(d2h)
    t_end.record(stream)
    t_end.synchronize()
    wall_ms = (time.perf_counter() - t0) * 1e3 / e2e_iters
    e2e_ms = max(t_start.elapsed_time(t_end) / e2e_iters, wall_ms)
    e2e_ms = dist.max(e2e_ms, dev)
    e2e = {"value": round(dist.world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": y_host[0].numel() * 2,
           "ms_per_step": round(e2e_ms, 4),
           "method": "pinned host x -> device, fmlp_geglu, y -> pinned host every step; copies on "
                     "their own streams, double-buffered, overlapping neighbouring steps"}
    del x_host, y_host, x_dev, y_dev

    cpu = None
    oracle_check = None
    timed_s = ms_max * args.steps / 1e3
    peak_key, peak_basis = bf16_peak_basis(timed_s)
    y_rows = y.view(torch.int16).cpu().numpy().view(np.uint16)
    del x, Wg, Wu, Wd, y, ws
    torch.cuda.empty_cache()
    if dist.rank == 0:
        cpu, ref_rows = cpu_baseline(t, w, args.cpu_sample_rows)
        oracle_check = error_stats(np, y_rows[:ref_rows.shape[0]], ref_rows,
                                   f"the first {ref_rows.shape[0]} token rows (the CPU "
                                   "baseline's sample)")

    extras = {}
    if not args.no_extras:
        extras = run_extras(fm, synth, torch, np, dev, stream, events_time, pk)

    launches_per_step = 2
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64/Box-Muller; x~N(0,1), W~U(+-1/sqrt(in)))",
        "config": {"workload": f"{HEADLINE}: GeGLU FFN T=8192 D=8192 H=28672, bias-free, "
                               "gelu_tanh, bf16 in / fp32 acc / bf16 out",
                   "T": w.T, "D": w.D, "H": w.H, "flops_per_step": flops,
                   "l2": "inputs larger than L2 (1.41 GB of weights streamed per step)",
                   "parallelism": f"replicas x{dist.world} (one block per GPU, no collective)"},
        "roofline": roofline,
        "pct_bf16_peak": round(value / dist.world / pk[peak_key], 4),
        "pct_bf16_peak_basis": f"{pk_src} {peak_basis} bf16 (the timed region is "
                               f"{timed_s:.2f} s long)",
        "cpu_baseline": cpu,
        "oracle": oracle_check,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "workloads": extras,
    }
    dist.barrier()
    dist.close()
    return out


def traffic_for(name: str, units):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[name]
        from feed_forward_gemm_gb300 import _build
        if e.get("source_fingerprint") != _build.kernel_fingerprint():
            return None
        return e["dram_bytes_per_launch"]
    except Exception:
        return None


def bf16_peak_basis(timed_s: float):
    """Which measured bf16 peak a whole-step fraction is quoted against: the sustained one
    (a seconds-long loop under the power cap) once the timed region lasts a second or more,
    else the burst one."""
    return ("bf16_tflops_sustained", "sustained") if timed_s >= 1.0 else ("bf16_tflops", "burst")


def error_stats(np, got_bits, ref_bits, what):
    """Oracle agreement of a timed configuration: max |y - ref|, relative Frobenius error and
    the largest difference in bf16 units in the last place, over `what`."""
    y = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (ref_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nr = float(np.linalg.norm(r))
    ulp = np.abs(got_bits.astype(np.int32) - ref_bits.astype(np.int32))
    return {"max_abs": float(np.abs(y - r).max()),
            "frob_rel": float(np.linalg.norm(y - r) / nr) if nr > 0 else None,
            "max_ulp": int(ulp.max()), "mismatch_bits": int((got_bits != ref_bits).sum()),
            "checked": what}


def run_extras(fm, synth, torch, np, dev, stream, events_time, pk):
    """The other workloads, each timed alone with CUDA events (device-resident inputs), each
    with its oracle agreement (all rows, or a seeded sample of rows for the large ones)."""
    import oracle
    out = {}
    pick = np.random.default_rng(99)

    def up(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    def host(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def cold_time(fn, iters):
        """ms per call of fn() with L2 flushed (256 MB written) before every call; only the
        call itself sits between the two events."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(iters)]
        fn()
        torch.cuda.synchronize(dev)
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    # GPT-2-small-shaped GeGLU FFN
    w = synth.WORKLOADS["geglu_8192x768x3072"]
    t = w.generate()
    x, Wg, Wu, Wd = up(t["x"]), up(t["Wg"]), up(t["Wu"]), up(t["Wd"])
    y = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
    wsb = fm.fmlp_geglu_workspace_size(w.T, w.D, w.H)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ms = cold_time(lambda: fm.fmlp_geglu(x, Wg, Wu, Wd, y, w.T, w.D, w.H, ws, wsb, stream), 30)
    kernels = fm.fmlp_describe_plan("geglu", w.T, w.D, w.H)
    # the same block as two launches (gate/up, then down), which the plan does not choose here
    fm.fmlp_test_two_stage(-1)
    try:
        ms_two = cold_time(
            lambda: fm.fmlp_geglu(x, Wg, Wu, Wd, y, w.T, w.D, w.H, ws, wsb, stream), 30)
    finally:
        fm.fmlp_test_two_stage(0)
    fm.fmlp_geglu(x, Wg, Wu, Wd, y, w.T, w.D, w.H, ws, wsb, stream)
    torch.cuda.synchronize(dev)
    rows = np.sort(pick.choice(w.T, 256, replace=False))
    out[w.name] = {"ms": round(ms, 4), "tflops": round(w.flops() / (ms * 1e-3) / 1e12, 1),
                   "frac_bf16_burst": round(w.flops() / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                   "plan": fm.fmlp_geglu_plan(w.T, w.D, w.H), "kernels": kernels,
                   "ms_two_launches": round(ms_two, 4),
                   "l2": "flushed before every call (median of 30)",
                   "oracle": error_stats(np, host(y)[rows], oracle.geglu(
                       t["x"], t["Wg"], t["Wu"], t["Wd"], rows=rows), "256 seeded rows")}
    del x, Wg, Wu, Wd, y, ws

    # 4096-wide Linear -> GELU(erf) -> Linear with biases at 4096 tokens
    w = synth.WORKLOADS["mlp_4096_t4096"]
    t = w.generate()
    d = {k: up(v) for k, v in t.items()}
    y = torch.empty((w.T, w.Dout), dtype=torch.bfloat16, device=dev)
    wsb = fm.fmlp_mlp_gelu_workspace_size(w.T, w.D, w.H, w.Dout)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    rows = np.sort(pick.choice(w.T, 256, replace=False))
    for name, mode in ((w.name, fm.FMLP_GELU_ERF), (w.name + "_relu", fm.FMLP_RELU)):
        def mlp(mode=mode):
            fm.fmlp_mlp_gelu(d["x"], d["W1"], d["b1"], d["W2"], d["b2"], y, w.T, w.D, w.H,
                             w.Dout, mode, ws, wsb, stream)
        ms = cold_time(mlp, 30)
        om = oracle.GELU_ERF if mode == fm.FMLP_GELU_ERF else oracle.RELU
        out[name] = {"ms": round(ms, 4), "tflops": round(w.flops() / (ms * 1e-3) / 1e12, 1),
                     "frac_bf16_burst": round(w.flops() / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
                                              4),
                     "activation": "gelu_erf" if mode == fm.FMLP_GELU_ERF else "relu",
                     "plan": fm.fmlp_mlp_gelu_plan(w.T, w.D, w.H, w.Dout),
                     "l2": "flushed before every call (median of 30)",
                     "oracle": error_stats(np, host(y)[rows], oracle.mlp_gelu(
                         t["x"], t["W1"], t["b1"], t["W2"], t["b2"], gelu_mode=om, rows=rows),
                         "256 seeded rows")}
    del d, y, ws

    # mixture of experts: 8 GeGLU experts (D 4096, H 14336, Mixtral-shaped), 16384 routed token
    # rows in uneven groups, both GEMM stages one launch each over all experts
    w = synth.MOE_WORKLOADS["moe_geglu_8x4096x14336"]
    t = w.generate()
    off = w.offsets()
    xm, Wgm, Wum, Wdm = (up(t[k]) for k in ("x", "Wg", "Wu", "Wd"))
    offm = torch.tensor(off, dtype=torch.int32, device=dev)
    ym = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
    wsm = torch.empty(fm.fmlp_moe_geglu_workspace_size(w.T, w.D, w.H), dtype=torch.uint8,
                      device=dev)

    def moe():
        fm.fmlp_moe_geglu(xm, offm, Wgm, Wum, Wdm, ym, w.T, w.D, w.H, w.E, wsm, wsm.numel(),
                          stream)
    for _ in range(3):
        moe()
    ms = events_time(moe, 10)
    fl = w.flops()
    rows = np.sort(np.concatenate([off[e] + pick.choice(off[e + 1] - off[e], 32, replace=False)
                                   for e in range(w.E)]))
    out[w.name] = {
        "ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
        "frac_bf16_burst": round(fl / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
        "tokens_per_expert": list(w.counts), "kernel": "grouped CTA-pair tcgen05, one launch per stage",
        "l2": "inputs larger than L2 (2.8 GB of expert weights)",
        "oracle": error_stats(np, host(ym)[rows], oracle.moe_geglu(
            t["x"], off, t["Wg"], t["Wu"], t["Wd"], rows=rows), "32 seeded rows per expert")}
    del xm, Wgm, Wum, Wdm, offm, ym, wsm, t

    # the 4096-wide MLP at 1..128 tokens: weights rotate through 5 copies (336 MB > 2x L2)
    w = synth.WORKLOADS["mlp_4096_t1"]
    sets, host_sets = [], []
    for r in range(5):
        t = w.generate(replica=r)
        host_sets.append(t)
        sets.append({k: up(v) for k, v in t.items()})
    wbytes = 2 * (w.D * w.H + w.H * w.Dout)
    xall = rne_normal_rows(np, synth, 128, w.D)
    for T in (1, 2, 4, 16, 64, 128):
        xT = up(xall[:T]) if T > 1 else None
        yT = torch.empty((T, w.Dout), dtype=torch.bfloat16, device=dev)
        wsbT = fm.fmlp_mlp_gelu_workspace_size(T, w.D, w.H, w.Dout)
        wsT = torch.empty(max(wsbT, 1), dtype=torch.uint8, device=dev)

        def one(s, i, T=T, xT=xT, yT=yT, wsT=wsT, wsbT=wsbT):
            q = sets[i % 5]
            fm.fmlp_mlp_gelu(q["x"] if T == 1 else xT, q["W1"], q["b1"], q["W2"], q["b2"], yT,
                             T, w.D, w.H, w.Dout, fm.FMLP_GELU_ERF, wsT, wsbT, s)

        def twenty(s, one=one):
            for i in range(20):
                one(s, i)
        for _ in range(3):
            twenty(stream)
        ms_graph = graph_time(torch, dev, twenty, 20) / 20
        gbs = wbytes / (ms_graph * 1e-3) / 1e9
        entry = {"us": round(ms_graph * 1e3, 2), "weight_GBps": round(gbs, 1),
                 "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                 "plan": fm.fmlp_mlp_gelu_plan(T, w.D, w.H, w.Dout),
                 "timing": "CUDA graph of 20 consecutive forwards over 5 rotating weight sets "
                           "(336 MB > 2x L2), replayed 20 times"}
        # raw stream launches (no graph) too
        ms_stream = events_time(lambda: twenty(stream), 10) / 20
        entry["us_stream_launched"] = round(ms_stream * 1e3, 2)
        entry["kernels"] = fm.fmlp_describe_plan("mlp", T, w.D, w.H, w.Dout)
        if "one few-token tcgen05 launch" in entry["kernels"]:
            # the same forwards as two few-token launches, which the plan does not choose here
            fm.fmlp_test_fewtoken_block(-1)
            try:
                entry["us_two_launches"] = round(graph_time(torch, dev, twenty, 20) / 20 * 1e3, 2)
            finally:
                fm.fmlp_test_fewtoken_block(0)
        # oracle agreement of the last forward (weight set 4)
        one(stream, 4)
        torch.cuda.synchronize(dev)
        hs = host_sets[4]
        xin = hs["x"] if T == 1 else xall[:T]
        entry["oracle"] = error_stats(np, host(yT), oracle.mlp_gelu(
            xin, hs["W1"], hs["b1"], hs["W2"], hs["b2"], gelu_mode=oracle.GELU_ERF),
            f"all {T} rows")
        out[f"mlp_4096_t{T}"] = entry
        if T == 1:
            # the same forward as the one-kernel decode (both layers in one launch, a grid
            # barrier between them), which the plans do not choose: measured beside the GEMVs
            fm.fmlp_test_prefer_decode(1)
            try:
                for _ in range(3):
                    twenty(stream)
                ms_g = graph_time(torch, dev, twenty, 20) / 20
                ms_s = events_time(lambda: twenty(stream), 10) / 20
                one(stream, 4)
                torch.cuda.synchronize(dev)
                yk = host(yT)
            finally:
                fm.fmlp_test_prefer_decode(0)
            gk = wbytes / (ms_g * 1e-3) / 1e9
            out["mlp_4096_t1_one_kernel_decode"] = {
                "us": round(ms_g * 1e3, 2), "us_stream_launched": round(ms_s * 1e3, 2),
                "weight_GBps": round(gk, 1), "frac_hbm": round(gk / pk["hbm_gbs"], 4),
                "plan": fm.FMLP_PLAN_DECODE, "selected_by_default": False,
                "timing": entry["timing"],
                "oracle": error_stats(np, yk, oracle.mlp_gelu(
                    host_sets[4]["x"], host_sets[4]["W1"], host_sets[4]["b1"],
                    host_sets[4]["W2"], host_sets[4]["b2"], gelu_mode=oracle.GELU_ERF),
                    "the token")}
    sets.clear()
    host_sets.clear()

    # one-token decode of the GeGLU blocks: GPT-2-small-shaped (rotating 5 weight sets) and
    # 70B-class (1.41 GB of weights, far beyond L2)
    for name, reps in (("geglu_8192x768x3072", 5), ("geglu_8192x8192x28672", 1)):
        w = synth.WORKLOADS[name]
        hsets = [w.generate(names=["Wg", "Wu", "Wd"], replica=r) for r in range(reps)]
        dsets = [{k: up(v) for k, v in h.items()} for h in hsets]
        x1h = rne_normal_rows(np, synth, 1, w.D)
        x1 = up(x1h)
        y1 = torch.empty((1, w.D), dtype=torch.bfloat16, device=dev)
        wsb = fm.fmlp_geglu_workspace_size(1, w.D, w.H)
        ws1 = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)

        def twenty(s, dsets=dsets, x1=x1, y1=y1, ws1=ws1, wsb=wsb, w=w):
            for i in range(20):
                q = dsets[i % len(dsets)]
                fm.fmlp_geglu(x1, q["Wg"], q["Wu"], q["Wd"], y1, 1, w.D, w.H, ws1, wsb, s)
        for _ in range(2):
            twenty(stream)
        ms_graph = graph_time(torch, dev, twenty, 10) / 20
        ms_stream = events_time(lambda: twenty(stream), 5) / 20
        wb = 3 * w.D * w.H * 2
        gbs = wb / (ms_graph * 1e-3) / 1e9
        q = dsets[-1]
        fm.fmlp_geglu(x1, q["Wg"], q["Wu"], q["Wd"], y1, 1, w.D, w.H, ws1, wsb, stream)
        torch.cuda.synchronize(dev)
        h = hsets[-1]
        out[name.replace("geglu_8192x", "geglu_decode_t1_")] = {
            "us": round(ms_graph * 1e3, 2), "us_stream_launched": round(ms_stream * 1e3, 2),
            "weight_GBps": round(gbs, 1),
            "frac_hbm": round(gbs / pk["hbm_gbs"], 4), "plan": fm.fmlp_geglu_plan(1, w.D, w.H),
            "timing": f"CUDA graph of 20 consecutive one-token forwards over {reps} weight "
                      "set(s), replayed 10 times",
            "oracle": error_stats(np, host(y1), oracle.geglu(x1h, h["Wg"], h["Wu"], h["Wd"]),
                                  "the token")}
        del dsets, hsets

    # small fully fused GeGLU block and the single Linear: launch-latency bound, against the
    # launch -> complete floor of an empty kernel on the same box
    def empty_kernel(st):
        with torch.cuda.stream(st):
            torch.cuda._sleep(0)
    for _ in range(10):
        empty_kernel(stream)
    floor_stream = events_time(lambda: empty_kernel(stream), 200)
    floor_graph = graph_time(torch, dev, lambda st: [empty_kernel(st) for _ in range(20)], 20) / 20
    out["empty_kernel_floor"] = {"us": round(floor_graph * 1e3, 2),
                                 "us_stream_launched": round(floor_stream * 1e3, 2),
                                 "what": "a zero-length spin kernel (torch.cuda._sleep(0)), the "
                                         "launch -> complete floor of one kernel"}
    for name in ("geglu_1024x32x64", "linear_1024x32x64"):
        w = synth.WORKLOADS[name]
        t = w.generate()
        d = {k: up(v) for k, v in t.items()}
        if w.op == "geglu":
            y = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
            wsb = fm.fmlp_geglu_workspace_size(w.T, w.D, w.H)
            ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)

            def fn(st, d=d, y=y, ws=ws, wsb=wsb, w=w):
                fm.fmlp_geglu(d["x"], d["Wg"], d["Wu"], d["Wd"], y, w.T, w.D, w.H, ws, wsb, st)
            plan = fm.fmlp_geglu_plan(w.T, w.D, w.H)

            def ref(nth, t=t):
                return oracle.geglu(t["x"], t["Wg"], t["Wu"], t["Wd"], nthreads=nth)
        else:
            y = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)

            def fn(st, d=d, y=y, w=w):
                fm.fmlp_linear_bias(d["x"], d["W"], d["b"], y, w.T, w.D, w.H, st)
            plan = fm.fmlp_linear_plan(w.T, w.D, w.H)

            def ref(nth, t=t):
                return oracle.linear(t["x"], t["W"], t["b"], nthreads=nth)
        for _ in range(10):
            fn(stream)
        ms_stream = events_time(lambda: fn(stream), 200)
        ms_graph = graph_time(torch, dev, lambda st: [fn(st) for _ in range(20)], 20) / 20
        fn(stream)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        expect = ref(1)
        cpu1 = time.perf_counter() - t0
        out[name] = {"us": round(ms_graph * 1e3, 2), "us_stream_launched": round(ms_stream * 1e3, 2),
                     "plan": plan, "bound": "launch latency",
                     "x_empty_kernel_floor": round(ms_graph / floor_graph, 2),
                     "timing": "CUDA graph of 20 back-to-back calls, replayed 20 times",
                     "oracle_1_thread_us": round(cpu1 * 1e6, 1),
                     "oracle": error_stats(np, host(y), expect, "all rows")}
    return out


def rne_normal_rows(np, synth, T, D):
    """T x D bf16 bits ~ N(0, 1) for the token rows of the few-token lines (seed 7000)."""
    a = np.empty((T, D), dtype=np.uint16)
    synth.fill_bf16(a, a.size, 7000 + T, "normal")
    return a


def graph_time(torch, dev, fn, replays):
    """ms per replay of a CUDA graph that captures fn(stream)."""
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        fn(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    g.replay()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        a.record(s)
        for _ in range(replays):
            g.replay()
        b.record(s)
    b.synchronize()
    return a.elapsed_time(b) / replays


# ------------------------------------------------------------------------- CPU oracle

def cpu_baseline(t, w, rows_req: int):
    """The oracle on a bounded sample of the headline workload's token rows."""
    import numpy as np

    import oracle
    nthreads = oracle.threads()
    rows_n = rows_req or 24 * nthreads   # about 10 s on 16 cores
    rows = np.arange(rows_n, dtype=np.int64)
    t0 = time.perf_counter()
    ref = oracle.geglu(t["x"], t["Wg"], t["Wu"], t["Wd"], rows=rows, nthreads=nthreads)
    dt = time.perf_counter() - t0
    flops = w.flops() * rows_n / w.T
    return ({"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s",
             "cores": min(nthreads, rows_n), "kind": "oracle",
             "sample": f"{rows_n} of {w.T} token rows of {w.name} (full H), fp64 C oracle, "
                       f"{dt:.2f} s; flops scaled to the rows computed"}, ref)


# ------------------------------------------------------------------------- reference arm

def run_reference(args, dist: Dist):
    """The oracle (the plain fp64 CPU implementation) as the reference arm: each step is a
    bounded sample of the headline workload's rows."""
    if dist.rank != 0:
        return None
    import numpy as np

    import oracle
    import synth
    w = synth.WORKLOADS[HEADLINE]
    t = w.generate()
    nthreads = oracle.threads()
    rows_n = max(2, min(16, nthreads))
    for i in range(args.warmup):
        oracle.geglu(t["x"], t["Wg"], t["Wu"], t["Wd"], rows=np.arange(1, dtype=np.int64),
                     nthreads=1)
    t0 = time.perf_counter()
    for s in range(args.steps):
        rows = (np.arange(rows_n, dtype=np.int64) + s * rows_n) % w.T
        oracle.geglu(t["x"], t["Wg"], t["Wu"], t["Wd"], rows=rows, nthreads=nthreads)
    dt = (time.perf_counter() - t0) / args.steps
    flops = w.flops() * rows_n / w.T
    value = flops / dt / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{HEADLINE} (oracle on {rows_n} token rows per step)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                         "cores": min(nthreads, rows_n), "kind": "oracle",
                         "sample": f"{rows_n} of {w.T} token rows per step, full H"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_profile_case(args):
    """Launch one entry point a few times on device-random inputs (for ncu captures)."""
    import numpy as np
    import torch

    import feed_forward_gemm_gb300 as fm
    T, D, H = (int(v) for v in args.shape.split(","))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fm.load()
    g = torch.Generator(device=dev)
    g.manual_seed(0)

    def rnd(*shape, scale=1.0):
        return (torch.randn(shape, generator=g, device=dev) * scale).to(torch.bfloat16)

    x = rnd(T, D)
    W1, W2, W3 = rnd(H, D, scale=D ** -0.5), rnd(H, D, scale=D ** -0.5), rnd(D, H, scale=H ** -0.5)
    b1, b2 = rnd(H, scale=0.1), rnd(D, scale=0.1)
    mid = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    k = args.profile_kernel
    if k == "moe":
        # 8 experts with the benchmark's uneven shares of the T rows
        share = np.array([16, 12, 10, 8, 6, 5, 4, 3], dtype=np.float64)
        cnt = np.floor(share / share.sum() * T).astype(np.int64)
        cnt[0] += T - cnt.sum()
        moe_off = torch.tensor(np.concatenate([[0], np.cumsum(cnt)]), dtype=torch.int32,
                               device=dev)
        moe_g, moe_u = rnd(8, H, D, scale=D ** -0.5), rnd(8, H, D, scale=D ** -0.5)
        moe_d = rnd(8, D, H, scale=H ** -0.5)
    fm.fmlp_set_tile_policy({"auto": fm.FMLP_TILES_AUTO, "single": fm.FMLP_TILES_SINGLE,
                             "pair": fm.FMLP_TILES_PAIR}[args.tiles])
    for _ in range(args.launches):
        if k == "gate_up":
            fm.fmlp_geglu_gate_up(x, W1, W2, mid, T, D, H)
        elif k == "down":
            fm.fmlp_linear_bias(mid, W3, None, y, T, H, D)
        elif k == "geglu":
            fm.fmlp_geglu(x, W1, W2, W3, y, T, D, H, mid, mid.numel() * 2)
        elif k == "mlp_up":
            fm.fmlp_linear_bias_gelu(x, W1, b1, mid, T, D, H, fm.FMLP_GELU_ERF)
        elif k in ("mlp", "mlp_decode"):
            # mlp_decode: blocks of 1..4 tokens as the one-kernel decode (plan switch)
            fm.fmlp_test_prefer_decode(1 if k == "mlp_decode" else 0)
            fm.fmlp_mlp_gelu(x, W1, b1, W3, b2, y, T, D, H, D, fm.FMLP_GELU_ERF, mid,
                             mid.numel() * 2)
            fm.fmlp_test_prefer_decode(0)
        elif k == "linear":
            fm.fmlp_linear_bias(x, W1, b1, mid, T, D, H)
        elif k == "moe":
            fm.fmlp_moe_geglu(x, moe_off, moe_g, moe_u, moe_d, y, T, D, H, 8, mid,
                              mid.numel() * 2)
    torch.cuda.synchronize()
    st = fm.fmlp_device_status()
    if st != fm.FMLP_OK:
        raise SystemExit(f"device status {st}: {fm.fmlp_last_error()}")
    print(f"profile case {k} {T}x{D}x{H} tiles={args.tiles}: {args.launches} launches ok")


def main():
    args = parse()
    if args.profile_kernel:
        run_profile_case(args)
        return
    dist = Dist(args.gpus)
    if args.impl == "reference":
        out = run_reference(args, dist)
    else:
        out = run_ours(args, dist)
    if out is not None and dist.rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
