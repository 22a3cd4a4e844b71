"""Benchmark of the fused GEMM/conv chains on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: the FFN-like b2b GEMM, bf16, A[262144,256] . W0[256,256] (+b0,
Hardswish) . W1[256,128] (+b1, Hardswish) -- the largest point of that chain's M sweep
(4096 .. 262144 rows), the largest single-GPU configuration of the chain.  One step = one
fused launch over one batch.  Prints ONE JSON line (rank 0).

  value        whole-job TFLOP/s (MMA FLOPs 2*M*(K0*N0 + N0*N1) per step), inputs resident
               in HBM; the K timed steps rotate through input/output sets whose total size
               exceeds twice the L2, so every step streams its A from HBM.
  roofline     the fused kernel against the resource that bounds it: the slower of its
               FLOPs at the measured tensor peak and its algorithmic bytes (A + W0 + b0 +
               W1 + b1 + out) at the measured HBM copy rate.  HBM-bound: achieved GB/s of
               algorithmic bytes over the average launch time; tensor-bound: TFLOP/s.
  pct_of_roofline  100 * max(FLOPs / tensor peak, bytes / HBM peak) / measured time.
  sweep        the FFN-like chain over its M sweep: per M, microseconds per launch,
               TFLOP/s, percent of roofline and the unfused path's microseconds.
  unfused      the same chain as two launches (GEMM0 + epilogue -> HBM -> GEMM1), its
               time and algorithmic bytes (the intermediate written and read back).
  e2e          the same metric through the public API from pinned host buffers: every step
               uploads its activations and downloads its result (weights resident), the
               upload of step i+1, compute of step i and download of step i-1 overlapping.
  cpu_baseline the CPU oracle (single thread) on a bounded sample of rows.
  workloads    every workload (the headline too), fused and unfused, measured the same way.

--impl reference times the CPU oracle instead (the method's plain unfused definition),
on a per-step sample of the same workload sized so the whole run takes about a minute.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import platform
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gemm_conv_chains_gb300 import workloads as wl  # noqa: E402

METRIC = "fused-chain TFLOPS and % of roofline; HBM bytes vs unfused 2-kernel path"
UNIT = "TFLOP/s"
HEADLINE = wl.GEMM_FFN_LARGE


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def kernel_source_sha():
    """Hash of the kernel and launch-planner sources, comments and blank lines left out, so
    that a comment edit keeps the counters taken on the same code valid."""
    h = hashlib.sha256()
    for name in ("chain_kernel.cuh", "chain_cta2_kernel.cuh", "ptx.cuh", "kernel_params.h",
                 "kernel_units.cuh", "kernels_cta2_units.cuh", "api.cu"):
        with open(os.path.join(ROOT, "gemm_conv_chains_gb300", "csrc", name)) as f:
            for line in f.read().splitlines():
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def load_traffic(workload_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha") != kernel_source_sha():
        return None
    entry = d.get("workloads", {}).get(workload_name)
    return None if entry is None else entry.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for (t, line) in self.lines:
            if any(a - 0.05 <= t <= b + 0.05 for a, b in self.windows):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[6 + i]
                          and "Not" not in r[6 + i]})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------------------------
# workload runners: each returns (step(i) callable, flops, floor_bytes, unfused step,
# unfused_bytes, bytes of one input/output set)
# ------------------------------------------------------------------------------------
def make_sets(nsets, make_one):
    return [make_one(i) for i in range(nsets)]


def l2_bytes(dev):
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20))


def rotation_sets(set_bytes, dev):
    return max(2, math.ceil(2 * l2_bytes(dev) / set_bytes) + 1)


def gemm_runner(w: wl.GemmChain, dev):
    from gemm_conv_chains_gb300 import ops
    t = wl.gemm_inputs(w, seed=0)
    W0, b0, W1, b1 = (t[k].to(dev) for k in ("W0", "b0", "W1", "b1"))
    set_bytes = 2 * w.M * (w.K0 + w.N1)
    n = rotation_sets(set_bytes, dev)
    A0 = t["A"].to(dev)
    sets = []
    for i in range(n):
        A = A0 if i == 0 else A0.roll(i, dims=0).contiguous()
        sets.append((A, torch.empty((w.M, w.N1), dtype=A0.dtype, device=dev),
                     torch.empty((w.M, w.N0), dtype=A0.dtype, device=dev)))

    def fused(i):
        A, D, _ = sets[i % n]
        ops.b2b_gemm(A, W0, b0, W1, b1, w.act0, w.act1, out=D)

    def unfused(i):
        A, D, H = sets[i % n]
        ops.gemm_bias_act(A, W0, b0, w.act0, out=H)
        ops.gemm_bias_act(H, W1, b1, w.act1, out=D)

    # the library's single operators stop at N = 256: a wider GEMM0 has no unfused leg
    return fused, (unfused if w.N0 <= 256 else None), n, set_bytes


def gemm3_runner(w: wl.GemmChain3, dev):
    from gemm_conv_chains_gb300 import ops
    t = wl.gemm3_inputs(w, seed=0)
    W = [(t[f"W{i}"].to(dev), t[f"b{i}"].to(dev)) for i in range(3)]
    acts = (w.act0, w.act1, w.act2)
    set_bytes = 2 * w.M * (w.K0 + w.N2)
    n = rotation_sets(set_bytes, dev)
    A0 = t["A"].to(dev)
    sets = []
    for i in range(n):
        A = A0 if i == 0 else A0.roll(i, dims=0).contiguous()
        sets.append((A, torch.empty((w.M, w.N2), dtype=A0.dtype, device=dev),
                     torch.empty((w.M, w.N0), dtype=A0.dtype, device=dev),
                     torch.empty((w.M, w.N1), dtype=A0.dtype, device=dev)))

    def fused(i):
        A, D, _, _ = sets[i % n]
        ops.b2b_gemm3(A, W[0][0], W[0][1], W[1][0], W[1][1], W[2][0], W[2][1], *acts, out=D)

    def unfused(i):
        A, D, H0, H1 = sets[i % n]
        ops.gemm_bias_act(A, W[0][0], W[0][1], acts[0], out=H0)
        ops.gemm_bias_act(H0, W[1][0], W[1][1], acts[1], out=H1)
        ops.gemm_bias_act(H1, W[2][0], W[2][1], acts[2], out=D)

    return fused, unfused, n, set_bytes


def conv_runner(w: wl.ConvChain, dev):
    from gemm_conv_chains_gb300 import ops
    t = wl.conv_inputs(w, seed=0)
    W0, b0, W1, b1 = (t[k].to(dev) for k in ("W0", "b0", "W1", "b1"))
    set_bytes = 2 * (w.N * w.H * w.W * w.C + w.M * w.C1)
    n = rotation_sets(set_bytes, dev)
    x0 = t["x"].to(dev)
    sets = []
    for i in range(n):
        x = x0 if i == 0 else x0.roll(i, dims=0).contiguous()
        sets.append((x, torch.empty((w.N, w.Ho, w.Wo, w.C1), dtype=x0.dtype, device=dev),
                     torch.empty((w.N, w.Ho, w.Wo, w.C0), dtype=x0.dtype, device=dev)))
    W1_as_conv = W1.view(w.C1, 1, 1, w.C0)

    def fused(i):
        x, y, _ = sets[i % n]
        if w.stride == 1:
            ops.b2b_conv_nhwc(x, W0, b0, W1, b1, w.pad, w.act0, w.act1, out=y)
        else:
            ops.b2b_conv_nhwc_strided(x, W0, b0, W1, b1, w.pad, w.stride, w.act0, w.act1, out=y)

    def unfused(i):
        x, y, h = sets[i % n]
        if w.stride == 1:
            ops.conv_bias_act_nhwc(x, W0, b0, w.pad, w.act0, out=h)
        else:
            ops.conv_bias_act_nhwc_strided(x, W0, b0, w.pad, w.stride, w.act0, out=h)
        ops.conv_bias_act_nhwc(h, W1_as_conv, b1, 0, w.act1, out=y)

    return fused, unfused, n, set_bytes


def pool_runner(w: wl.ConvPool, dev):
    from gemm_conv_chains_gb300 import ops
    t = wl.pool_inputs(w, seed=0)
    Wt, b = t["Wt"].to(dev), t["b"].to(dev)
    set_bytes = 2 * (w.N * w.H * w.W * w.Cin + w.N * (w.H // 2) * (w.W // 2) * w.Cout)
    n = rotation_sets(set_bytes, dev)
    x0 = t["x"].to(dev)
    sets = []
    for i in range(n):
        x = x0 if i == 0 else x0.roll(i, dims=0).contiguous()
        sets.append((x, torch.empty((w.N, w.H // 2, w.W // 2, w.Cout), dtype=x0.dtype, device=dev),
                     torch.empty((w.N, w.H, w.W, w.Cout), dtype=x0.dtype, device=dev)))

    def fused(i):
        x, y, _ = sets[i % n]
        ops.conv_relu_maxpool(x, Wt, b, out=y)

    def unfused(i):
        x, y, c = sets[i % n]
        ops.conv_bias_act_nhwc(x, Wt, b, 1, "relu", out=c)
        ops.maxpool2x2_nhwc(c, out=y)

    return fused, unfused, n, set_bytes


def roofline_of(w, t_step, peaks):
    """The bound of workload `w` (the slower of FLOPs at the tensor peak and algorithmic
    bytes at the HBM peak) and what one step of `t_step` seconds achieves against it."""
    t_flop = w.flops / (peaks["bf16_tflops"] * 1e12)
    t_byte = w.floor_bytes / (peaks["hbm_gbs"] * 1e9)
    if t_flop > t_byte:
        achieved = w.flops / t_step / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4)}
    achieved = w.floor_bytes / t_step / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}


def shape_config(w):
    """The shape keys of a workload, for the printed config."""
    if isinstance(w, wl.GemmChain):
        return {"M": w.M, "K0": w.K0, "N0": w.N0, "N1": w.N1, "act0": w.act0, "act1": w.act1}
    if isinstance(w, wl.GemmChain3):
        return {"M": w.M, "K0": w.K0, "N0": w.N0, "N1": w.N1, "N2": w.N2,
                "acts": [w.act0, w.act1, w.act2]}
    if isinstance(w, wl.ConvChain):
        return {"N": w.N, "H": w.H, "W": w.W, "C": w.C, "C0": w.C0, "R": w.R, "S": w.S,
                "pad": w.pad, "stride": w.stride, "C1": w.C1, "act0": w.act0, "act1": w.act1}
    return {"N": w.N, "H": w.H, "W": w.W, "Cin": w.Cin, "Cout": w.Cout}


def runner_for(w, dev):
    if isinstance(w, wl.GemmChain):
        return gemm_runner(w, dev)
    if isinstance(w, wl.GemmChain3):
        return gemm3_runner(w, dev)
    if isinstance(w, wl.ConvChain):
        return conv_runner(w, dev)
    return pool_runner(w, dev)


def time_steps(step, steps, warmup, nsets, dev, graph_len=None):
    """Runs `warmup` untimed steps, then times exactly `steps` steps with CUDA events on
    the current stream.  Steps are captured in CUDA graphs of up to `graph_len` launches
    (a whole rotation of the input sets, repeated) and replayed; returns seconds."""
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if graph_len is None:
        graph_len = nsets * max(1, 96 // nsets)
    graphs = {}

    def graph_of(length):
        if length not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(length):
                    step(i)
            graphs[length] = g
        return graphs[length]

    full, rem = divmod(steps, graph_len)
    if full:
        graph_of(graph_len)
    if rem:
        graph_of(rem)
    # one untimed replay of each graph
    for g in graphs.values():
        g.replay()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(full):
        graphs[graph_len].replay()
    if rem:
        graphs[rem].replay()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


# ------------------------------------------------------------------------------------
# the oracle as CPU baseline
# ------------------------------------------------------------------------------------
def oracle_sample(w: wl.GemmChain, rows: int, seed: int = 0):
    t = wl.gemm_inputs(w.with_m(rows), seed=seed)
    return {k: wl.to_bits(v) for k, v in t.items()}


def time_oracle(w: wl.GemmChain, rows: int, reps: int = 1):
    import oracle
    b = oracle_sample(w, rows)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.b2b_gemm(w.dtype, b["A"], b["W0"], b["b0"], b["W1"], b["b1"], w.act0, w.act1)
    return time.perf_counter() - t0


def cpu_baseline(w: wl.GemmChain, target_s: float = 10.0):
    per_row_flops = w.flops / w.M
    calib_rows = 256
    t = time_oracle(w, calib_rows)
    rows = int(min(w.M, max(calib_rows, target_s / max(t, 1e-9) * calib_rows)))
    t = time_oracle(w, rows)
    return {"value": rows * per_row_flops / t / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{rows} of {w.M} rows of {w.name} (rows are independent), "
                      f"{t:.1f} s single-threaded C, double-precision sums",
            "host": platform.machine()}


# ------------------------------------------------------------------------------------
# end to end through the public API from host buffers
# ------------------------------------------------------------------------------------
def e2e_gemm(w: wl.GemmChain, dev, steps=60):
    """The headline metric through the public API from pinned host memory, as a serving
    loop runs it: every step uploads its activations A and downloads its result; the
    weights and biases are uploaded once, before the timed region (model parameters stay
    resident).  Steps are pipelined over three streams -- upload of step i+1, compute of
    step i, download of step i-1 -- with device and host buffers double-buffered and
    events ordering every reuse."""
    from gemm_conv_chains_gb300 import ops
    t = wl.gemm_inputs(w, seed=0)
    A_host = t["A"].pin_memory()
    W0, b0, W1, b1 = (t[k].to(dev) for k in ("W0", "b0", "W1", "b1"))
    A_dev = [torch.empty_like(A_host, device=dev) for _ in range(2)]
    out_dev = [torch.empty((w.M, w.N1), dtype=A_host.dtype, device=dev) for _ in range(2)]
    out_host = [torch.empty((w.M, w.N1), dtype=A_host.dtype).pin_memory() for _ in range(2)]
    h2d = A_host.numel() * A_host.element_size()
    d2h = out_host[0].numel() * out_host[0].element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_comp = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event()   # noqa: E731
    uploaded = [ev(), ev()]    # A_dev[b] holds this step's input
    consumed = [ev(), ev()]    # the kernel has finished with A_dev[b] and written out_dev[b]
    drained = [ev(), ev()]     # out_dev[b] has been copied to the host
    for b in range(2):
        consumed[b].record(s_comp)
        drained[b].record(s_comp)

    def step(i):
        b = i & 1
        s_in.wait_event(consumed[b])
        with torch.cuda.stream(s_in):
            A_dev[b].copy_(A_host, non_blocking=True)
        uploaded[b].record(s_in)
        s_comp.wait_event(uploaded[b])
        s_comp.wait_event(drained[b])
        ops.b2b_gemm(A_dev[b], W0, b0, W1, b1, w.act0, w.act1, out=out_dev[b])
        consumed[b].record(s_comp)
        s_out.wait_event(consumed[b])
        with torch.cuda.stream(s_out):
            out_host[b].copy_(out_dev[b], non_blocking=True)
        drained[b].record(s_out)

    for i in range(4):
        step(i)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_comp)
    s_in.wait_event(start)
    for i in range(steps):
        step(i)
    s_comp.wait_stream(s_in)
    s_comp.wait_stream(s_out)
    end.record(s_comp)
    end.synchronize()
    sec = start.elapsed_time(end) / 1e3 / steps
    torch.cuda.synchronize(dev)
    # the last result really came back
    ref = torch.empty_like(out_dev[0])
    ops.b2b_gemm(A_dev[0], W0, b0, W1, b1, w.act0, w.act1, out=ref)
    torch.cuda.synchronize(dev)
    assert torch.equal(out_host[(steps - 1) & 1].view(torch.int16), ref.cpu().view(torch.int16))
    return {"value": w.flops / sec / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": sec * 1e3, "steps": steps,
            "pipelined": "upload i+1 / compute i / download i-1 on three streams; weights resident"}


# ------------------------------------------------------------------------------------
# arms
# ------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(sec, pg, dev):
    """The slowest rank's time (the job finishes when its last replica does): an all-reduce
    MAX over the process group `pg` (torch.distributed), or `sec` itself without one."""
    if pg is None:
        return sec
    t = torch.tensor([float(sec)], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_step, steps, sec, world):
    """Whole-job TFLOP/s: every replica runs `steps` steps of the workload (weak scaling),
    all of them done when the slowest rank's `sec` seconds have passed."""
    return world * flops_per_step * steps / sec / 1e12


def workload_config(w, world):
    par = f"replicas{world}" if world > 1 else "single-gpu"
    if w is HEADLINE:
        desc = (f"{w.name}: b2b GEMM {w.dtype} A[{w.M},{w.K0}] W0[{w.K0},{w.N0}] "
                f"W1[{w.N0},{w.N1}], bias+{w.act0}/bias+{w.act1} (FFN-like chain, the largest "
                f"point of its M sweep)")
    else:
        desc = w.name
    return {"workload": desc, **shape_config(w), "dtype": w.dtype, "parallelism": par}


def headline_config(world):
    return workload_config(HEADLINE, world)


def print_trace(fused, cta: int, dev) -> None:
    """Prints the event timeline of CTA `cta` over one fused launch of the traced build of
    the kernel (after two launches of it that warm its code and data in the caches), one
    event per line: microseconds since the CTA's first event, event, epilogue group or
    buffer, tile."""
    from gemm_conv_chains_gb300 import ops
    fused(0)
    torch.cuda.synchronize(dev)
    try:
        for i in range(3):
            buf = torch.zeros(2 * (1 << 15), dtype=torch.int64, device=dev)
            ops.set_trace(buf, cta=cta)
            fused(0)
            torch.cuda.synchronize(dev)
    finally:
        ops.set_trace(None)
    for t, e, g, it in ops.read_trace(buf):
        print(f"{t / 1e3:9.3f} {e:18s} g{g} t{it}")
    st, _ = ops.get_device_error()
    if st != 0:
        raise SystemExit(f"device error {st}")


def run_ours(args):
    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    from gemm_conv_chains_gb300 import ops
    ops.lib()
    ops.get_device_error()
    peaks = load_peaks()
    w = wl.WORKLOADS[args.workload]
    if args.rows is not None:
        if not isinstance(w, wl.GemmChain):
            raise SystemExit("--rows applies to the GEMM-chain workloads only")
        w = w.with_m(args.rows)
    if args.batch is not None:
        if not isinstance(w, (wl.ConvChain, wl.ConvPool)):
            raise SystemExit("--batch applies to the conv workloads only")
        w = dataclasses.replace(w, N=args.batch, name=f"{w.name}_n{args.batch}")
    fused, unfused, nsets, set_bytes = runner_for(w, dev)
    if args.trace is not None:
        print_trace(fused, args.trace, dev)
        return
    clocks = ClockSampler(torch.cuda.current_device() if not os.environ.get("CUDA_VISIBLE_DEVICES")
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    clocks.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    sec = time_steps(fused, args.steps, args.warmup, nsets, dev)
    clocks.mark(t_wall0, time.time())
    sec = max_over_ranks(sec, pg, dev)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    st, info = ops.get_device_error()
    if st != 0:
        raise RuntimeError(f"device error word after the timed region: {st} {info}")
    unfused_steps = max(args.steps // 4, 8)
    sec_unfused = (time_steps(unfused, unfused_steps, args.warmup, nsets, dev) if unfused
                   else None)
    clocks.stop()

    ms = sec / args.steps * 1e3
    t_step = sec / args.steps
    tflops = w.flops / t_step / 1e12
    value = whole_job_value(w.flops, args.steps, sec, world)
    achieved_gbs = w.floor_bytes / t_step / 1e9
    t_roof = max(w.flops / (peaks["bf16_tflops"] * 1e12), w.floor_bytes / (peaks["hbm_gbs"] * 1e9))
    t_unf = sec_unfused / unfused_steps if sec_unfused else None
    traffic = load_traffic(w.name)
    roof = roofline_of(w, t_step, peaks)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; A ~ N(0,1) or U[-1,1], W ~ N(0, 1/K), b ~ U[-0.1, 0.1])",
        "config": {**workload_config(w, world),
                   "l2": f"{nsets} rotating input/output sets of {set_bytes / 2**20:.0f} MiB "
                         f"(> 2x L2) replayed in CUDA graphs"},
        "pct_of_roofline": round(100.0 * t_roof / t_step, 2),
        "roofline": {**roof, "traffic": traffic, "algorithmic_bytes_per_launch": w.floor_bytes,
                     "flops_per_launch": w.flops,
                     "kernel_source_sha": kernel_source_sha(),
                     "peak_source": peaks["source"],
                     "hbm": {"achieved_gbs": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"],
                             "frac": round(achieved_gbs / peaks["hbm_gbs"], 4)},
                     "tensor": {"achieved_tflops": round(tflops, 1), "peak": peaks["bf16_tflops"],
                                "frac": round(tflops / peaks["bf16_tflops"], 4)}},
        "unfused": ({"ms_per_step": round(t_unf * 1e3, 6),
                     "tflops": round(w.flops / t_unf / 1e12, 2),
                     "algorithmic_bytes": w.unfused_bytes,
                     "launches_per_step": 3 if isinstance(w, wl.GemmChain3) else 2,
                     "fused_speedup": round(t_unf / t_step, 3)} if t_unf else None),
        "gpu_launches": args.steps,
    }
    if rank == 0:
        if isinstance(w, wl.GemmChain):
            line["e2e"] = e2e_gemm(w, dev)
        if not args.skip_cpu and isinstance(w, wl.GemmChain):
            line["cpu_baseline"] = cpu_baseline(w, target_s=args.cpu_seconds)
        if not args.headline_only:
            line["sweep"] = ffn_sweep(dev, peaks, args.warmup)
            line["workloads"] = other_workloads(dev, peaks, max(args.steps // 8, 64), args.warmup)
        line["clocks"] = clocks.summary()
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def other_workloads(dev, peaks, steps, warmup):
    out = {}
    for w in wl.WORKLOADS.values():
        fused, unfused, nsets, _ = runner_for(w, dev)
        s_f = time_steps(fused, steps, warmup, nsets, dev) / steps
        s_u = time_steps(unfused, steps, warmup, nsets, dev) / steps if unfused else None
        t_roof = max(w.flops / (peaks["bf16_tflops"] * 1e12), w.floor_bytes / (peaks["hbm_gbs"] * 1e9))
        out[w.name] = {"us_per_step": round(s_f * 1e6, 3), "tflops": round(w.flops / s_f / 1e12, 1),
                       "pct_of_roofline": round(100 * t_roof / s_f, 1),
                       "hbm_gbs_algorithmic": round(w.floor_bytes / s_f / 1e9, 1),
                       "bound": roofline_of(w, s_f, peaks)["bound"], "dtype": w.dtype,
                       "config": shape_config(w),
                       "unfused_us_per_step": round(s_u * 1e6, 3) if s_u else None,
                       "fused_speedup": round(s_u / s_f, 3) if s_u else None,
                       "floor_bytes": w.floor_bytes, "unfused_bytes": w.unfused_bytes}
        del fused, unfused
        torch.cuda.empty_cache()
    from gemm_conv_chains_gb300 import ops
    st, info = ops.get_device_error()
    if st != 0:
        raise RuntimeError(f"device error word: {st} {info}")
    return out


def ffn_sweep(dev, peaks, warmup):
    """The FFN-like chain over its M sweep, fused and unfused, each point timed over about
    the same span of device time (inputs rotating through sets larger than twice L2)."""
    out = {}
    for M in wl.FFN_SWEEP_M:
        w = wl.GEMM_FFN.with_m(M)
        fused, unfused, nsets, _ = runner_for(w, dev)
        steps = max(32, min(1024, (1 << 22) // M))
        s_f = time_steps(fused, steps, warmup, nsets, dev) / steps
        s_u = time_steps(unfused, steps, warmup, nsets, dev) / steps
        t_roof = max(w.flops / (peaks["bf16_tflops"] * 1e12), w.floor_bytes / (peaks["hbm_gbs"] * 1e9))
        out[str(M)] = {"us_per_step": round(s_f * 1e6, 3), "tflops": round(w.flops / s_f / 1e12, 1),
                       "pct_of_roofline": round(100 * t_roof / s_f, 1),
                       "roofline": roofline_of(w, s_f, peaks), "steps": steps,
                       "unfused_us_per_step": round(s_u * 1e6, 3),
                       "fused_speedup": round(s_u / s_f, 3)}
        del fused, unfused
        torch.cuda.empty_cache()
    return out


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = HEADLINE
    per_row = w.flops / w.M
    t_cal = time_oracle(w, 128) / 128
    budget = 60.0
    rows = int(max(1, min(4096, budget / max(args.steps + args.warmup, 1) / max(t_cal, 1e-9))))
    import oracle
    b = oracle_sample(w, rows)
    for _ in range(args.warmup):
        oracle.b2b_gemm(w.dtype, b["A"], b["W0"], b["b0"], b["W1"], b["b1"], w.act0, w.act1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.b2b_gemm(w.dtype, b["A"], b["W0"], b["b0"], b["W1"], b["b1"], w.act0, w.act1)
    sec = time.perf_counter() - t0
    value = rows * per_row * args.steps / sec / 1e12
    sample = (f"{rows} of {w.M} rows of {w.name} per step (rows are independent), "
              f"single-threaded C oracle, double-precision sums")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": headline_config(world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the per-workload table")
    ap.add_argument("--skip-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", choices=sorted(wl.WORKLOADS), default=HEADLINE.name,
                    help="workload of the timed line (default: the FFN-like chain at its "
                         "largest M); the others are for profiling single kernels")
    ap.add_argument("--rows", type=int, default=None,
                    help="for profiling: run a GEMM-chain workload over this many rows "
                         "instead of its own M")
    ap.add_argument("--batch", type=int, default=None,
                    help="for profiling: run a conv workload over this many images instead "
                         "of its own N")
    ap.add_argument("--trace", type=int, default=None, metavar="CTA",
                    help="for profiling: print the event timeline of this CTA over one launch "
                         "of the workload instead of timing it")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
