#!/usr/bin/env python3
"""Throughput of the quantized decode GEMV on raw GGUF blocks.

Workload (one step): the dense-27B-like FFN shapes at M = 1 for Q4_0 and Q4_K -- gate/up
K=5120 N=17408 and down K=17408 N=5120 -- i.e. four GEMV calls per step, each quantizing its
activation row on the GPU and multiplying it against 50,135,040 bytes of raw blocks.  The
headline value is the effective weight bandwidth (weight bytes / time, decimal GB/s) over
the whole job; the roofline fraction is that bandwidth divided by the measured HBM copy
bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

  * our arm: 16 steps are captured as one CUDA graph and replayed to K steps between CUDA
    events on the launch stream; two copies of every matrix alternate, so the 200 MB a
    step reads never comes from L2 (129 MB);
  * e2e: the same K steps through the public Python API with host buffers: every step the
    four calls read their activation rows from page-locked host memory and write their
    results into it, the kernels addressing host memory directly over NVLink-C2C (no
    staging copy); the same steps with one staged copy each way are reported beside it;
  * reference arm: the plain CPU oracle (the checker of the CUDA path) on the host cores,
    each step a bounded sample of the same workload;
  * N > 1 (torchrun): replicas only -- every rank runs the whole workload on its own GPU;
    the value is the weight bytes of all ranks over the slowest rank's time;
  * --one FMT:NxK:M (e.g. Q4_K:17408x5120:1): three untimed GEMV calls of one shape on
    seeded synthetic input and nothing else -- the small case a profiler captures;
    --one-moe M does the same for the MoE FFN of M tokens, --one-prefill FMT:NxK:M for the
    prefill GEMM on the tensor cores (qg_prefill_gemm).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "effective weight GB/s per quant GEMV (fraction of HBM peak); MoE FFN tokens/s"
WORKLOAD_NAME = "Q4_0 + Q4_K GEMV, M=1, dense-27B FFN shapes (17408x5120 gate/up, 5120x17408 down)"
CONFIG_ID = 2  # seed id of this workload (synth.seed_for)
MATRICES = [(synth.Q4_0, 17408, 5120), (synth.Q4_0, 5120, 17408), (synth.Q4_K, 17408, 5120), (synth.Q4_K, 5120, 17408)]
M_TOKENS = 1
ONE_FUSED_K_MAX = 8192        # rows up to this length are quantized inside the one-token engine
ROTATE = 2                    # weight copies per matrix
STEPS_PER_GRAPH = 16          # steps captured in one CUDA graph
FALLBACK_HBM_GBS = 6800.0     # used only when no measured peak is available
# Integer roof of the batched decode: dp4a issues at 64 lanes per SM per clock (4 int8 MACs
# each) on 152 SMs at 2.07 GHz
DP4A_MAC_PER_S = 152 * 64 * 4 * 2.07e9
CLOCK_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


# ----------------------------------------------------------------------------- helpers
def weight_bytes_per_step() -> int:
    return sum(synth.matrix_bytes(f, n, k) for f, n, k in MATRICES)


def algorithmic_bytes_per_launch(fmt: int, N: int, K: int, M: int) -> int:
    """Weight bytes + fp32 activations read + fp32 results written by one GEMV call."""
    return synth.matrix_bytes(fmt, N, K) + 4 * M * K + 4 * M * N


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(ms: float, units: float, world: int):
    """Slowest rank's time and the units of all ranks (replicas: no data exchange)."""
    if world <= 1:
        return ms, units
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError, TypeError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor-core peak (TFLOP/s) measured on this machine: burst (a kernel timed
    alone) and sustained (inside a long loop); fp16 runs at the bf16 rate.  Fallback 1900."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError, TypeError):
        return 1900.0, 1700.0, "fallback"


def kernel_source_sha() -> str:
    csrc = os.path.join(ROOT, "gguf_block_quantized_quant_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def dram_traffic_per_launch():
    """DRAM bytes (read + write) of one engine launch from the committed ncu summary, or
    None when the kernel sources changed since that capture."""
    path = os.path.join(ROOT, "profiles", "engine1_q4k_17408x5120_m1.txt")
    try:
        with open(path) as f:
            kv = dict(line.split(":", 1) for line in f if ":" in line and not line.startswith("#"))
        kv = {k.strip(): v.strip() for k, v in kv.items()}
        if kv.get("source_sha") != kernel_source_sha():
            return None
        return int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while it runs."""

    def __init__(self, uuid: str | None, period_ms: int = 100):
        self.uuid, self.period_ms, self.proc, self.out = uuid, period_ms, None, ""

    def __enter__(self):
        q = "uuid,clocks.sm,clocks.max.sm,power.draw," + ",".join(f"clocks_event_reasons.{r}" for r in CLOCK_REASONS)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.period_ms)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    @staticmethod
    def _norm(u: str) -> str:
        u = u.strip().lower()
        return (u[4:] if u.startswith("gpu-") else u).replace("-", "")

    def summary(self):
        sm, smax, reasons = [], [], set()
        rows = [[x.strip() for x in line.split(",")] for line in self.out.splitlines()]
        rows = [f for f in rows if len(f) >= 4 + len(CLOCK_REASONS)]
        mine = [f for f in rows if self.uuid and self._norm(f[0]) == self._norm(self.uuid)]
        if not mine and len({f[0] for f in rows}) == 1:
            mine = rows  # one GPU visible: its samples are ours
        for f in mine:
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for r, v in zip(CLOCK_REASONS, f[4:]):
                if v.lower().startswith("active"):
                    reasons.add(r)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(rows_per_matrix: int, seed_salt: int = 0):
    """A bounded sample of the workload for the oracle: the first rows of every matrix."""
    out = []
    for i, (fmt, N, K) in enumerate(MATRICES):
        g = synth.rng(CONFIG_ID, 10 + i + seed_salt)
        r = min(rows_per_matrix, N)
        out.append((fmt, r, K, synth.weights(fmt, r, K, g), synth.activations(M_TOKENS, K, g)))
    return out


def time_oracle(sample, min_seconds: float):
    """Runs the oracle over the sample until min_seconds have passed; weight GB/s."""
    import oracle
    oracle.build()
    nbytes, t0, reps = 0, time.perf_counter(), 0
    while True:
        for fmt, r, K, W, x in sample:
            oracle.gemv(fmt, W, x, r, K)
            nbytes += synth.matrix_bytes(fmt, r, K)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            return nbytes / el / 1e9, oracle.get_threads(), reps, el


def cpu_baseline_block(seconds: float = 10.0):
    """The oracle on all host cores (the reported baseline) and, beside it, single-threaded."""
    import oracle
    rows = 256
    sample = oracle_sample(rows)
    gbs, cores, reps, el = time_oracle(sample, seconds)
    nthreads = oracle.get_threads()
    oracle.set_threads(1)
    try:
        gbs1, _, reps1, el1 = time_oracle(oracle_sample(32), max(2.0, seconds / 4))
    finally:
        oracle.set_threads(0 if nthreads == cores else nthreads)
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} rows of each of the 4 matrices ({sum(synth.matrix_bytes(f, r, k) for f, r, k, _, _ in sample)} "
                      f"weight bytes), repeated {reps}x in {el:.1f} s, fp64 oracle with OpenMP over rows",
            "single_thread": {"value": gbs1, "unit": "GB/s", "cores": 1,
                              "sample": f"first 32 rows of each matrix, repeated {reps1}x in {el1:.1f} s"}}


def run_reference(args, budget_s: float = 150.0):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    # rows per matrix per step: at most 64, fewer when K steps of 64 would exceed the budget
    rows = 64
    sample = oracle_sample(rows)
    t0 = time.perf_counter()
    for fmt, r, K, W, x in sample:
        oracle.gemv(fmt, W, x, r, K)
    t1 = time.perf_counter() - t0
    if t1 * (args.steps + args.warmup) > budget_s:
        rows = max(1, int(rows * budget_s / (t1 * (args.steps + args.warmup))))
        sample = oracle_sample(rows)
    for _ in range(args.warmup):
        for fmt, r, K, W, x in sample:
            oracle.gemv(fmt, W, x, r, K)
    step_bytes = sum(synth.matrix_bytes(f, r, k) for f, r, k, _, _ in sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for fmt, r, K, W, x in sample:
            oracle.gemv(fmt, W, x, r, K)
    el = time.perf_counter() - t0
    gbs = step_bytes * args.steps / el / 1e9
    desc = (f"first {rows} rows of each of the 4 matrices per step ({step_bytes} weight bytes), "
            f"fp64 oracle with OpenMP over rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; block codes/scales uniform, x ~ N(0,1))",
        "config": {"workload": WORKLOAD_NAME, "M": M_TOKENS, "sample_rows_per_matrix": rows},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": oracle.get_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def run_ours(args):
    import torch
    import gguf_block_quantized_quant_gb300 as qg

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "") or None

    # inputs: seeded on the host, uploaded once; ROTATE copies of every matrix
    mats = []
    for i, (fmt, N, K) in enumerate(MATRICES):
        g = synth.rng(CONFIG_ID, i)
        W = torch.from_numpy(synth.weights(fmt, N, K, g)).to(dev)
        x_host = torch.from_numpy(synth.activations(M_TOKENS, K, g)).pin_memory()
        copies = [W] + [W.clone() for _ in range(ROTATE - 1)]
        nws = qg.qg_workspace_size(qg.QG_OP_GEMV, fmt, M_TOKENS, N, K)
        mats.append(dict(fmt=fmt, N=N, K=K, W=copies, x_host=x_host, x=x_host.to(dev),
                         y=torch.empty((M_TOKENS, N), dtype=torch.float32, device=dev),
                         y_host=torch.empty((M_TOKENS, N), dtype=torch.float32).pin_memory(),
                         ws=torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)))
    step_weight_bytes = weight_bytes_per_step()
    # kernels per GEMV call at one token with x in device memory: the engine alone where it
    # quantizes the row itself (rows of up to 8192 elements), else the activation tile
    # preparation and the engine
    launches_per_step = sum(1 if K <= ONE_FUSED_K_MAX else 2 for _, _, K in MATRICES)

    s = torch.cuda.Stream(device=dev)

    def step(c):
        for m in mats:
            qg.qg_gemv(m["fmt"], m["W"][c], m["x"], m["N"], y=m["y"], ws=m["ws"], stream=s)

    # G steps per graph (weight copies alternate inside it), so consecutive calls overlap
    # (programmatic dependent launch) across the steps and not only within one; K steps are
    # G-step replays plus one graph for the remainder
    G = max(ROTATE, min(STEPS_PER_GRAPH, args.steps) // ROTATE * ROTATE)

    def capture(nsteps):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for i in range(nsteps):
                step(i % ROTATE)
        return gr

    with torch.cuda.stream(s):
        for i in range(max(args.warmup, 1)):
            step(i % ROTATE)
        s.synchronize()
        g_full = capture(G)
        rem = args.steps % G
        g_rem = capture(rem) if rem else None
        for i in range(max(1, args.warmup // G)):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()  # every graph of the timed region has run once
        s.synchronize()
    err = qg.qg_device_error()
    if err:
        raise SystemExit(f"bench.py: device error word {err:#x} after warm-up")

    # ---- timed region: K graph replays
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(uuid) as clk:
        with torch.cuda.stream(s):
            # untimed: back to steady clocks after the sampler's start-up pause
            g_full.replay()
            e0.record(s)
            for _ in range(args.steps // G):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            e1.record(s)
        torch.cuda.synchronize()
    barrier(world)
    ms_local = e0.elapsed_time(e1)
    ms, total_bytes = aggregate(ms_local, step_weight_bytes * args.steps, world)
    gbs = total_bytes / (ms * 1e-3) / 1e9
    # the same K steps timed again (spread of the measurement; value is the first region)
    rep_gbs = [gbs]
    for _ in range(args.repeats - 1):
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            r0.record(s)
            for _ in range(args.steps // G):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            r1.record(s)
        torch.cuda.synchronize()
        rms, rtb = aggregate(r0.elapsed_time(r1), step_weight_bytes * args.steps, world)
        rep_gbs.append(rtb / (rms * 1e-3) / 1e9)

    # ---- e2e: public API, host buffers, transfers inside the timed region.  Every step the
    # four calls take their activation rows from page-locked host memory and write their
    # results into page-locked host memory: the kernels read x and write y over the host
    # link (NVLink-C2C) themselves, so no staging copy is issued.  For comparison the same
    # steps are also timed with staged copies: one upload of the four inputs (packed in one
    # pinned buffer) and one read-back of the four results per step.
    xs_host = [m["x_host"].pin_memory() for m in mats]
    ys_host = [torch.empty(m["y_host"].shape, dtype=torch.float32, pin_memory=True) for m in mats]
    z0, z1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):  # untimed: the same calls once (host buffers seen, code paths warm)
        for i in range(max(args.warmup, 1)):
            c = i % ROTATE
            for m, xh, yh in zip(mats, xs_host, ys_host):
                qg.qg_gemv(m["fmt"], m["W"][c], xh, m["N"], y=yh, ws=m["ws"], stream=s)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        z0.record(s)
        for i in range(args.steps):
            c = i % ROTATE
            for m, xh, yh in zip(mats, xs_host, ys_host):
                qg.qg_gemv(m["fmt"], m["W"][c], xh, m["N"], y=yh, ws=m["ws"], stream=s)
        z1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    ms_e2e, tb_e2e = aggregate(z0.elapsed_time(z1), step_weight_bytes * args.steps, world)
    e2e_gbs = tb_e2e / (ms_e2e * 1e-3) / 1e9

    def packed(sizes):
        offs, o = [], 0
        for n in sizes:
            offs.append(o)
            o += -(-n // 64) * 64  # 256-byte aligned slices (fp32 elements)
        return offs, o
    xoffs, xtot = packed([m["x_host"].numel() for m in mats])
    yoffs, ytot = packed([m["y_host"].numel() for m in mats])
    x_all_h = torch.empty(xtot, dtype=torch.float32).pin_memory()
    y_all_h = torch.empty(ytot, dtype=torch.float32).pin_memory()
    x_all = torch.empty(xtot, dtype=torch.float32, device=dev)
    y_all = torch.empty(ytot, dtype=torch.float32, device=dev)
    for m, o in zip(mats, xoffs):
        x_all_h[o:o + m["x_host"].numel()] = m["x_host"].reshape(-1)
    xs_dev = [x_all[o:o + m["x_host"].numel()].view(m["x_host"].shape) for m, o in zip(mats, xoffs)]
    ys_dev = [y_all[o:o + m["y_host"].numel()].view(m["y_host"].shape) for m, o in zip(mats, yoffs)]
    h2d = sum(m["x_host"].numel() * 4 for m in mats)
    d2h = sum(m["y_host"].numel() * 4 for m in mats)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):  # untimed: the staged steps once
        x_all.copy_(x_all_h, non_blocking=True)
        for m, xd_, yd_ in zip(mats, xs_dev, ys_dev):
            qg.qg_gemv(m["fmt"], m["W"][0], xd_, m["N"], y=yd_, ws=m["ws"], stream=s)
        y_all_h.copy_(y_all, non_blocking=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        f0.record(s)
        for i in range(args.steps):
            c = i % ROTATE
            x_all.copy_(x_all_h, non_blocking=True)
            for m, xd_, yd_ in zip(mats, xs_dev, ys_dev):
                qg.qg_gemv(m["fmt"], m["W"][c], xd_, m["N"], y=yd_, ws=m["ws"], stream=s)
            y_all_h.copy_(y_all, non_blocking=True)
        f1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    ms_st, tb_st = aggregate(f0.elapsed_time(f1), step_weight_bytes * args.steps, world)
    staged_gbs = tb_st / (ms_st * 1e-3) / 1e9
    err = qg.qg_device_error()
    if err:
        raise SystemExit(f"bench.py: device error word {err:#x} after the timed region")

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel (the GEMV engine; each call also runs its small
    # activation preparation kernel, which the per-launch duration includes)
    peak, peak_kind = measured_peak()
    launch_ms = ms_local / (args.steps * len(MATRICES))
    algo = sum(algorithmic_bytes_per_launch(f, n, k, M_TOKENS) for f, n, k in MATRICES) / len(MATRICES)
    achieved = algo / (launch_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": dram_traffic_per_launch(), "peak_source": peak_kind,
                "kernel": "engine1_kernel (one-token GEMV) + activation tile preparation, per call",
                "algorithmic_bytes_per_launch": algo}

    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded; block codes/scales uniform, fp16 scales from U[1e-3,2e-3], x ~ N(0,1))",
        "config": {"workload": WORKLOAD_NAME, "M": M_TOKENS,
                   "matrices": [f"{synth.FORMAT_NAMES[f]} {n}x{k}" for f, n, k in MATRICES],
                   "weight_bytes_per_step": step_weight_bytes, "frac_of_hbm_peak": gbs / world / peak,
                   "l2": f"inputs larger than L2: {ROTATE} rotating copies of every matrix, "
                         f"{ROTATE * step_weight_bytes} weight bytes in rotation",
                   "timing": f"CUDA graphs of {G} steps (weight copies alternating inside), replayed to K steps "
                             "between CUDA events on the launch stream",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "value_gib_s": gbs / 2 ** 30 * 1e9,
                   "repeats": {"n": len(rep_gbs), "unit": "GB/s", "median": statistics.median(rep_gbs),
                               "min": min(rep_gbs), "max": max(rep_gbs),
                               "note": "the K timed steps repeated; value is the first repeat"}},
        "roofline": roofline,
        "cpu_baseline": None,
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "transfer": "the kernels read x from and write y to page-locked host memory (zero-copy over "
                            "NVLink-C2C), every step",
                "staged_copies_value": staged_gbs},
        "clocks": clk.summary(),
        "gpu_launches": launches_per_step * args.steps,
    }
    if world == 1:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_block(args.cpu_seconds)
        if not args.no_secondary:
            line["secondary"] = secondary(qg, torch, dev, s)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _eager_time_us(torch, s, fn, reps: int, warm: int = 3):
    """Mean µs of fn() launched from the host each time (no graph) on stream s."""
    with torch.cuda.stream(s):
        for _ in range(warm):
            fn()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            fn()
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def _graph_time_us(torch, s, fn, reps: int, warm: int = 3, per_graph: int = 8):
    """Mean µs of fn() from CUDA graphs of per_graph calls each (consecutive calls inside a
    graph overlap through programmatic dependent launch; a graph boundary does not)."""
    with torch.cuda.stream(s):
        for _ in range(warm):
            fn()
        s.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for _ in range(per_graph):
                fn()
        gr.replay()
        s.synchronize()
        n = max(1, reps // per_graph)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(n):
            gr.replay()
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (n * per_graph)


def secondary(qg, torch, dev, s):
    """The other workloads, for context: format sweep, Q8_0 1024^2, MoE FFN tokens/s, FFN
    sublayer.  Small matrices rotate through copies totalling > 4x L2 ("cold")."""
    out = {}
    l2 = 4 * torch.cuda.get_device_properties(dev).L2_cache_size
    for fmt, N, K in [(synth.Q8_0, 1024, 1024), (synth.Q5_K, 4096, 4096), (synth.Q6_K, 4096, 4096),
                      (synth.IQ4_XS, 4096, 4096), (synth.Q2_K, 4096, 4096), (synth.Q3_K, 4096, 4096),
                      (synth.Q4_1, 4096, 4096), (synth.Q5_0, 4096, 4096), (synth.Q5_1, 4096, 4096),
                      (synth.IQ4_NL, 4096, 4096)]:
        g = synth.rng(3 if fmt != synth.Q8_0 else 1, 0)
        nb = synth.matrix_bytes(fmt, N, K)
        R = max(2, -(-l2 // nb))
        base = torch.from_numpy(synth.weights(fmt, N, K, g)).to(dev)
        Ws = [base] + [base.clone() for _ in range(R - 1)]
        x = torch.from_numpy(synth.activations(1, K, g)).to(dev)
        y = torch.empty((1, N), dtype=torch.float32, device=dev)
        ws = torch.empty(max(qg.qg_workspace_size(qg.QG_OP_GEMV, fmt, 1, N, K), 16), dtype=torch.uint8, device=dev)

        def fn():
            for W in Ws:
                qg.qg_gemv(fmt, W, x, N, y=y, ws=ws, stream=s)
        us = _graph_time_us(torch, s, fn, 20) / R
        peak, _ = measured_peak()
        out[f"{synth.FORMAT_NAMES[fmt]} {N}x{K} M=1 cold"] = {"us": us, "GB/s": nb / us / 1e3,
                                                            "GiB/s": nb / us * 1e6 / 2 ** 30,
                                                            "frac_of_hbm": nb / us / 1e3 / peak}
        # warm: the same buffer every call (it stays in L2), for context beside the cold figure
        uw = _graph_time_us(torch, s, lambda: qg.qg_gemv(fmt, base, x, N, y=y, ws=ws, stream=s), 40)
        out[f"{synth.FORMAT_NAMES[fmt]} {N}x{K} M=1 warm"] = {"us": uw, "GB/s": nb / uw / 1e3}
        del Ws, base
    # MoE FFN: Q4_K experts, H=2048, E=256 routed (I=512) + 1 shared, top-8
    H, E, I, topk = 2048, 256, 512, 8
    g = synth.rng(4, 0)
    Wr = torch.from_numpy(synth.router_weights(E, H, g)).to(dev)
    fq = synth.Q4_K
    Wg = torch.from_numpy(synth.stacked_experts(fq, E, I, H, g)).to(dev)
    Wu = torch.from_numpy(synth.stacked_experts(fq, E, I, H, g)).to(dev)
    Wd = torch.from_numpy(synth.stacked_experts(fq, E, H, I, g)).to(dev)
    Wgs = torch.from_numpy(synth.weights(fq, I, H, g)).to(dev)
    Wus = torch.from_numpy(synth.weights(fq, I, H, g)).to(dev)
    Wds = torch.from_numpy(synth.weights(fq, H, I, g)).to(dev)
    for M in (1, 2, 4):
        x = torch.from_numpy(synth.activations(M, H, g)).to(dev)
        y = torch.empty((M, H), dtype=torch.float32, device=dev)
        ws = torch.empty(qg.qg_workspace_size(qg.QG_OP_MOE_FFN, fq, M, H, H, E, topk, I), dtype=torch.uint8,
                         device=dev)
        ids = torch.empty((M, topk), dtype=torch.int32, device=dev)
        call = lambda: qg.qg_moe_ffn(fq, x, Wr, topk, Wg, Wu, Wd, Wgs, Wus, Wds, I, y=y, topk_ids=ids, ws=ws, stream=s)  # noqa
        us = _graph_time_us(torch, s, call, 200)
        # the same chain launched from the host call by call: the launch gaps a graph removes
        ue = _eager_time_us(torch, s, call, 200)
        # algorithmic bytes: every distinct routed expert once, the shared expert, the router
        nb = (len(set(ids.cpu().numpy().ravel().tolist())) + 1) * 3 * synth.matrix_bytes(fq, I, H) + 4 * E * H
        peak, _ = measured_peak()
        out[f"MoE FFN Q4_K H=2048 E=256+1 I=512 top-8 M={M}"] = {"us": us, "tokens/s": M / (us * 1e-6),
                                                                  "us_eager": ue, "GB/s": nb / us / 1e3,
                                                                  "frac_of_hbm": nb / us / 1e3 / peak,
                                                                  "algorithmic_bytes": nb}
        # the same with s16 activations (two int8 planes per activation row)
        ws16 = torch.empty(qg.qg_workspace_size(qg.QG_OP_MOE_FFN_S16, fq, M, H, H, E, topk, I), dtype=torch.uint8,
                           device=dev)
        call16 = lambda: qg.qg_moe_ffn_s16(fq, x, Wr, topk, Wg, Wu, Wd, Wgs, Wus, Wds, I, y=y, ws=ws16, stream=s)  # noqa
        us16 = _graph_time_us(torch, s, call16, 200)
        out[f"MoE FFN s16 Q4_K H=2048 E=256+1 I=512 top-8 M={M}"] = {"us": us16, "tokens/s": M / (us16 * 1e-6)}
    del Wg, Wu, Wd
    # FFN sublayer: H=5120, I=17408 (150 / 219 MB of weights: larger than L2)
    H, I = 5120, 17408
    for fmt in (synth.Q4_K, synth.Q6_K):
        g = synth.rng(5, fmt)
        Wg = torch.from_numpy(synth.weights(fmt, I, H, g)).to(dev)
        Wu = torch.from_numpy(synth.weights(fmt, I, H, g)).to(dev)
        Wd = torch.from_numpy(synth.weights(fmt, H, I, g)).to(dev)
        nb = 2 * synth.matrix_bytes(fmt, I, H) + synth.matrix_bytes(fmt, H, I)
        for M in (1, 2, 4, 8, 16):
            x = torch.from_numpy(synth.activations(M, H, g)).to(dev)
            y = torch.empty((M, H), dtype=torch.float32, device=dev)
            ws = torch.empty(qg.qg_workspace_size(qg.QG_OP_FFN_SUBLAYER, fmt, M, H, H, 0, 0, I), dtype=torch.uint8,
                             device=dev)
            call = lambda: qg.qg_ffn_sublayer(fmt, Wg, Wu, Wd, x, I, y=y, ws=ws, stream=s)  # noqa: E731
            us = _graph_time_us(torch, s, call, 80)
            ue = _eager_time_us(torch, s, call, 40)
            peak, _ = measured_peak()
            hbm_us = nb / (peak * 1e3)
            alu_us = 3.0 * M * H * I / DP4A_MAC_PER_S * 1e6
            roof_us = max(hbm_us, alu_us)
            out[f"FFN sublayer {synth.FORMAT_NAMES[fmt]} H=5120 I=17408 M={M}"] = {
                "us": us, "GB/s": nb / us / 1e3, "us_eager": ue,
                "roof": {"bound": "hbm" if hbm_us >= alu_us else "alu", "hbm_us": hbm_us, "alu_us": alu_us,
                         "frac": roof_us / us}}
        del Wg, Wu, Wd
    out.update(prefill_secondary(qg, torch, dev, s))
    return out


PREFILL_M = 512
PREFILL_MATRICES = [(synth.Q4_K, 17408, 5120), (synth.Q4_K, 5120, 17408), (synth.Q4_0, 17408, 5120),
                    (synth.Q4_0, 5120, 17408)]


def prefill_secondary(qg, torch, dev, s):
    """Prefill GEMM on the tensor cores (qg_prefill_gemm), 512 tokens, dense-27B FFN shapes:
    TFLOP/s = 2 M N K / call time, against the measured dense bf16 peak (fp16 runs at the
    same rate), burst figure (each call is timed inside a short graph of calls)."""
    out = {}
    burst, _, kind = measured_tensor_peak()
    M = PREFILL_M
    for fmt, N, K in PREFILL_MATRICES:
        g = synth.rng(6, fmt * 7 + (N > K))
        W = torch.from_numpy(synth.weights(fmt, N, K, g)).to(dev)
        x = torch.from_numpy(synth.activations(M, K, g)).to(dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        ws = torch.empty(qg.qg_workspace_size(qg.QG_OP_PREFILL, fmt, M, N, K), dtype=torch.uint8, device=dev)
        call = lambda: qg.qg_prefill_gemm(fmt, W, x, N, y=y, ws=ws, stream=s)  # noqa: E731
        us = _graph_time_us(torch, s, call, 40, per_graph=4)
        tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
        out[f"prefill {synth.FORMAT_NAMES[fmt]} {N}x{K} M={M}"] = {
            "us": us, "TFLOP/s": tf, "frac_of_tensor_peak": tf / burst,
            "peak": {"value": burst, "unit": "TFLOP/s", "source": kind, "which": "dense bf16 burst"},
            "tokens/s": M / (us * 1e-6)}
        del W, x, y, ws
    return out


def run_one_prefill(spec: str):
    """Three qg_prefill_gemm calls of one shape (format name:NxK:M), for a profiler."""
    import torch

    import gguf_block_quantized_quant_gb300 as qg

    name, shape, m = spec.split(":")
    N, K = (int(v) for v in shape.lower().split("x"))
    fmt = synth.FORMATS[name]
    g = np.random.default_rng(synth.seed_for(6, fmt))
    W = torch.from_numpy(synth.weights(fmt, N, K, g)).cuda()
    x = torch.from_numpy(synth.activations(int(m), K, g)).cuda()
    for _ in range(3):
        y = qg.qg_prefill_gemm(fmt, W, x, N)
    torch.cuda.synchronize()
    if qg.qg_device_error():
        raise SystemExit("bench.py: device error word set by the prefill calls")
    print(json.dumps({"one_prefill": spec, "y_abs_sum": float(y.abs().sum())}))
    return 0


def run_one(spec: str):
    """Three qg_gemv calls of one shape (format name:NxK:M), for a profiler to capture."""
    import torch

    import gguf_block_quantized_quant_gb300 as qg

    name, shape, m = spec.split(":")
    N, K = (int(v) for v in shape.lower().split("x"))
    fmt = synth.FORMATS[name]
    g = np.random.default_rng(synth.seed_for(CONFIG_ID, fmt))
    W = torch.from_numpy(synth.weights(fmt, N, K, g)).cuda()
    x = torch.from_numpy(synth.activations(int(m), K, g)).cuda()
    for _ in range(3):
        y = qg.qg_gemv(fmt, W, x, N)
    torch.cuda.synchronize()
    print(json.dumps({"one": spec, "weight_bytes": int(W.numel()), "y_abs_sum": float(y.abs().sum())}))
    return 0


def run_one_moe(m: int):
    """Three qg_moe_ffn calls (Q4_K experts, H=2048, 256 routed + 1 shared, I=512, top-8) of
    m tokens, for a profiler to capture."""
    import torch

    import gguf_block_quantized_quant_gb300 as qg

    H, E, I, topk, fq = 2048, 256, 512, 8, synth.Q4_K
    g = synth.rng(4, 0)
    Wr = torch.from_numpy(synth.router_weights(E, H, g)).cuda()
    Wg = torch.from_numpy(synth.stacked_experts(fq, E, I, H, g)).cuda()
    Wu = torch.from_numpy(synth.stacked_experts(fq, E, I, H, g)).cuda()
    Wd = torch.from_numpy(synth.stacked_experts(fq, E, H, I, g)).cuda()
    sg = torch.from_numpy(synth.weights(fq, I, H, g)).cuda()
    su = torch.from_numpy(synth.weights(fq, I, H, g)).cuda()
    sd = torch.from_numpy(synth.weights(fq, H, I, g)).cuda()
    x = torch.from_numpy(synth.activations(m, H, g)).cuda()
    for _ in range(3):
        y = qg.qg_moe_ffn(fq, x, Wr, topk, Wg, Wu, Wd, sg, su, sd, I)
    torch.cuda.synchronize()
    print(json.dumps({"one_moe": m, "y_abs_sum": float(y.abs().sum())}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time budget of cpu_baseline")
    ap.add_argument("--repeats", type=int, default=5, help="timed regions of K steps (spread)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--one", metavar="FMT:NxK:M", help="three untimed GEMV calls of one shape, then exit")
    ap.add_argument("--one-moe", type=int, metavar="M", help="three untimed MoE FFN calls of M tokens, then exit")
    ap.add_argument("--one-prefill", metavar="FMT:NxK:M", help="three untimed prefill GEMM calls, then exit")
    ap.add_argument("--prefill-only", action="store_true", help="print the prefill secondary entries only")
    args = ap.parse_args(argv)
    if args.one:
        return run_one(args.one)
    if args.one_prefill:
        return run_one_prefill(args.one_prefill)
    if args.prefill_only:
        import torch

        import gguf_block_quantized_quant_gb300 as qg
        s = torch.cuda.Stream()
        print(json.dumps(prefill_secondary(qg, torch, torch.device("cuda", 0), s)), flush=True)
        return 0
    if args.one_moe:
        return run_one_moe(args.one_moe)
    if args.warmup < 3:
        raise SystemExit("bench.py: at least 3 warm-up steps")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
