"""Benchmark of the SVDQ W4A4 NVFP4 linear (and the AWQ W4A16 modulation GEMV)
on B300.

One step = one pass of the per-forward hot path of the SVDQ linear over one
batch: svdq_quantize_act (smoothing, rank-r down projection, e2m1/e4m3
quantization) then svdq_gemm_w4a4 (tcgen05 NVFP4 product + rank-r up
projection + bias), on the attention out-projection workload of a 1024x1024
diffusion transformer: M = 4096 tokens, K = N = 3072, rank 32, synthetic
outlier-heavy activations.  Weights are packed once, offline, by
svdq_pack_weights (not timed).  Inputs rotate over enough buffer sets that
every step reads from HBM, not L2.

The AWQ phase times the 57 stacked adaLN modulation GEMVs (K = 3072,
N = 6 x 3072, M in {1, 2, 4}) back to back; the MLP phase times the MLP's
first linear (M = 4096, K = 3072, N = 12288) with GELU fused into its epilogue
against the same GEMM without it; the QKV phase times the fused QKV projection
(M = 4608, K = 3072, N = 9216) with the per-head RMS normalization of Q and K
and the rotary embedding in its epilogue against the plain GEMM.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
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

import workloads  # noqa: E402

METRIC = "SVDQ W4A4 NVFP4 linear TFLOP/s & % FP4 tensor peak; AWQ W4A16 HBM GB/s"
_SAMPLE = {}  # device output rows kept for the quality figures
L2_BYTES = 126 * 1024 * 1024
FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense ratio of the tensor cores


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of the attn_out workload, each valid only while the kernel's
# sources hash to what was captured (the summaries are under profiles/).
MEASURED_TRAFFIC = {
    "svdq_gemm_w4a4": {
        "bytes": 12891648 + 23296,
        "sources": {"gemm_w4a4.cu": "b4d5668611bd8376b6807d366c6d05c029b11b32419fd8be6a03f349f4966da1",
                    "act_quant.cuh": "bea739112402fcfe84521d48b6e661028f64613e645ba281febb8147d55b1520",
                    "device_common.cuh": "aa6078eb6ec5f726d817e11391c6444f445b6172a148942c18c694f17a14beff"},
        "profile": "profiles/svdq_gemm_w4a4_attn_out_ncu.md"},
    "svdq_quantize_act": {
        "bytes": 25392128 + 0,
        "sources": {"quantize_act.cu": "d0998b9fff12f198db08792f7ce47d2c9cf9e804fa3f37fad0e7afd06ea2da2e",
                    "act_quant.cuh": "bea739112402fcfe84521d48b6e661028f64613e645ba281febb8147d55b1520",
                    "int4_quant.cuh": "a4a9954f799df30b652ac915d56273d1f9ef5b94d2ec3dbc03eaafcd92a4dc09",
                    "device_common.cuh": "aa6078eb6ec5f726d817e11391c6444f445b6172a148942c18c694f17a14beff"},
        "profile": "profiles/svdq_quantize_act_attn_out_ncu.md"},
    "svdq_quantize_act_int4": {
        "bytes": 25395328 + 0,
        "sources": {"quantize_act.cu": "d0998b9fff12f198db08792f7ce47d2c9cf9e804fa3f37fad0e7afd06ea2da2e",
                    "act_quant.cuh": "bea739112402fcfe84521d48b6e661028f64613e645ba281febb8147d55b1520",
                    "int4_quant.cuh": "a4a9954f799df30b652ac915d56273d1f9ef5b94d2ec3dbc03eaafcd92a4dc09",
                    "device_common.cuh": "aa6078eb6ec5f726d817e11391c6444f445b6172a148942c18c694f17a14beff"},
        "profile": "profiles/svdq_gemm_w4a4_int4_attn_out_ncu.md"},
    "svdq_gemm_w4a4_int4": {
        "bytes": 12188672 + 1280,
        "sources": {"gemm_int4.cu": "8d501f172976557d91ca4fba9f9e93abb8197acf27f688ada3365dd8c8d1c426",
                    "device_common.cuh": "aa6078eb6ec5f726d817e11391c6444f445b6172a148942c18c694f17a14beff"},
        "profile": "profiles/svdq_gemm_w4a4_int4_attn_out_ncu.md"},
    "awq_gemv_w4a16": {
        "bytes": 31934464 + 0,
        "sources": {"awq_gemv.cu": "cc0f366eeff3794b51fa8afa39adfe5516d626fb278178ce229587cf12f163d8",
                    "device_common.cuh": "aa6078eb6ec5f726d817e11391c6444f445b6172a148942c18c694f17a14beff"},
        "profile": "profiles/awq_gemv_w4a16_modulation_ncu.md"},
}


def measured_traffic(kernel: str):
    """Bytes per launch from the recorded capture, or None if the kernel's
    sources changed since."""
    import hashlib
    rec = MEASURED_TRAFFIC[kernel]
    csrc = os.path.join(ROOT, "bit_w4a4_diffusion_quantize_b300", "csrc")
    for name, digest in rec["sources"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return rec["bytes"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# --------------------------------------------------------------------------- dist
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons with
    nvidia-smi every 50 ms while the timed loop and its repeats run
    (read-only queries: no setting of the GPU is changed)."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        self.t0 = time.perf_counter()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        self.t1 = time.perf_counter()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, power, mx, reasons = [], [], None, set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(self.REASONS, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None,
                "window_s": round(self.t1 - self.t0, 3), "source": "nvidia-smi, 50 ms period"}


# --------------------------------------------------------------------------- CPU oracle timing
def time_oracle(case, sample_rows: int, steps: int):
    """The CPU oracle on `sample_rows` rows of the workload per step (its own
    packing is offline, not timed).  Returns (seconds per step, flop per step,
    threads)."""
    from oracle import svdq
    X = workloads.make_activations(case, M=sample_rows)
    W, b = workloads.make_weights(case)
    xm = svdq.calib_absmax(workloads.make_activations(case))
    packed = svdq.pack_weights(W, xm, case.rank)
    svdq.linear_forward(X, packed, b)  # warm-up
    ts = []
    for _ in range(steps):
        t0 = time.perf_counter()
        svdq.linear_forward(X, packed, b)
        ts.append(time.perf_counter() - t0)
    return statistics.median(ts), 2.0 * sample_rows * case.N * case.K, os.cpu_count()


def quality_sample(case, rows: int, y_dev_rows):
    """The quality invariant on the first `rows` rows of the workload: relative
    Frobenius error against float64 X W^T + b of the device's SVDQ output, of
    smoothing alone (no low-rank branch) and of plain W4A4 (neither), the
    latter two by the oracle with the same NVFP4 rules."""
    from oracle import svdq
    X_full = workloads.make_activations(case)
    X = X_full[:rows]
    W, b = workloads.make_weights(case)
    exact = X.astype(np.float64) @ W.T.astype(np.float64) + b
    nrm = np.linalg.norm(exact)
    smooth = svdq.linear_forward(X, svdq.pack_weights(W, svdq.calib_absmax(X_full), 0), b)["Y"]
    naive = svdq.naive_w4a4(X, W, b)
    e = {"svdq_device": float(np.linalg.norm(y_dev_rows - exact) / nrm),
         "smoothing_only": float(np.linalg.norm(smooth - exact) / nrm),
         "naive_w4a4": float(np.linalg.norm(naive - exact) / nrm)}
    return {"sample": f"first {rows} of {case.M} rows of the {case.name} workload",
            "rel_fro_err_vs_fp64": {k: round(v, 5) for k, v in e.items()},
            "svdq_below_naive": e["svdq_device"] < e["naive_w4a4"],
            "svdq_below_smoothing_only": e["svdq_device"] < e["smoothing_only"]}


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args, world, rank, local):
    import torch
    import bit_w4a4_diffusion_quantize_b300 as lib

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    case = workloads.CASES[args.workload]
    M, K, N, r = case.M, case.K, case.N, case.rank

    # ---- inputs and offline packing (not timed)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    Xbits = workloads.bf16_bits_of(X)
    xm = lib.svdq_calib_absmax(Xbits)
    t0 = time.perf_counter()
    packed = lib.svdq_pack_weights(W, xm, r)
    pack_s = time.perf_counter() - t0

    def dbits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    set_bytes = (M * K * 2 + M * K // 2 + lib.scale_bytes(M, K) + M * r * 2 + M * N * 2 +
                 N * K // 2 + lib.scale_bytes(N, K) + r * (N + K) * 2 + N * 2 + K * 4)
    nsets = max(2, math.ceil(3 * L2_BYTES / set_bytes))
    sets = []
    for _ in range(nsets):
        s = {
            "X": dbits(Xbits).view(torch.bfloat16).view(M, K),
            "inv": torch.from_numpy(packed["inv_lambda"]).to(dev),
            "L1s": dbits(packed["L1s"]).view(torch.bfloat16),
            "L2s": dbits(packed["L2s"]).view(torch.bfloat16),
            "wc": torch.from_numpy(packed["w_codes"]).to(dev),
            "ws": torch.from_numpy(packed["w_scales"]).to(dev),
            "bias": dbits(workloads.bf16_bits_of(b)).view(torch.bfloat16),
            "ac": torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
            "as": torch.empty(lib.scale_bytes(M, K), dtype=torch.uint8, device=dev),
            "lora": torch.empty((M, r), dtype=torch.bfloat16, device=dev),
            "Y": torch.empty((M, N), dtype=torch.bfloat16, device=dev),
        }
        sets.append(s)
    sT = packed["w_tensor_scale"]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def quantize(i, st):
        s = sets[i % nsets]
        lib.svdq_quantize_act(s["X"], s["inv"], s["L1s"], r, s["ac"], s["as"], s["lora"],
                              dev_status=status, stream=st)

    def gemm(i, st):
        s = sets[i % nsets]
        lib.svdq_gemm_w4a4(s["ac"], s["as"], s["wc"], s["ws"], sT, s["lora"], s["L2s"],
                           s["bias"], M, N, K, r, Y=s["Y"], dev_status=status, stream=st)

    def step(i, st):
        quantize(i, st)
        gemm(i, st)

    # The timed loops are CUDA graphs of the library's own launches (what a
    # serving loop replays); the host's launch cost stays out of the kernel
    # numbers and is part of `e2e` below.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream(dev)
            for i in range(args.steps):
                fn(i, cs)
        return g

    def timed(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3

    def repeated(g, reps):
        """`reps` timed replays of a graph of exactly `steps` launches, each
        bracketed by barrier + synchronize; seconds per replay."""
        ts = []
        for _ in range(reps):
            barrier(world)
            torch.cuda.synchronize()
            ts.append(timed(g))
        return ts

    for i in range(args.warmup):            # eager warm-up: module load, every set written
        step(i, stream)
    torch.cuda.synchronize()
    g_step, g_q, g_g = capture(step), capture(quantize), capture(gemm)
    with ClockSampler(local) as clk:
        for g in (g_step, g_q, g_g):          # untimed replays (clocks up, graphs resident)
            g.replay()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        # the timed region: `reps` replays of exactly `steps` steps each
        ts_step = repeated(g_step, args.reps)
        wall = time.perf_counter() - wall0
        barrier(world)
        ts_q = repeated(g_q, args.reps)
        ts_g = repeated(g_g, args.reps)
        t_total = statistics.median(ts_step)
        t_q = statistics.median(ts_q) / args.steps
        t_g = statistics.median(ts_g) / args.steps
        # keep the same load running so the clock record spans >= clock_window s
        t_end = time.perf_counter() + max(0.0, args.clock_window - (time.perf_counter() - wall0))
        while time.perf_counter() < t_end:
            g_step.replay()
            torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status set during the timed region")
    # device output rows for the quality figures (every set holds the same X)
    _SAMPLE["y_rows"] = sets[0]["Y"][:args.oracle_rows].view(torch.int16).cpu().numpy().view(
        np.uint16)
    t_total = max_over_ranks(t_total, world, dev)
    flop = 2.0 * M * N * K
    value = world * args.steps * flop / t_total / 1e12

    # ---- end to end: host (pinned) X in, host Y out, through the layer API
    layer = lib.SVDQLinear(packed | {"N": N, "K": K, "rank": r}, workloads.bf16_bits_of(b), dev)
    Xh = torch.from_numpy(Xbits.view(np.int16)).view(torch.bfloat16).pin_memory()
    Yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    Xd = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    Yd = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    bufs = (sets[0]["ac"], sets[0]["as"], sets[0]["lora"])

    def e2e_step():
        Xd.copy_(Xh, non_blocking=True)
        layer.forward(Xd, out=Yd, act_buffers=bufs, stream=stream)
        Yh.copy_(Yd, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world, dev)
    e2e = {"value": world * args.steps * flop / t_e2e / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2,
           "ms_per_step": t_e2e / args.steps * 1e3}
    # the host link on its own: the step's two copies timed alone (pinned
    # memory, this stream), and the share of a step they account for
    link = host_link(Xh, Xd, Yd, Yh, stream, reps=max(3, min(args.steps, 20)))
    e2e["host_link"] = link
    e2e["copies_share_of_step"] = round(
        (link["h2d_ms"] + link["d2h_ms"]) / e2e["ms_per_step"], 3)
    try:
        e2e_pipe = e2e_pipelined(args, layer, Xbits, M, K, N, dev, stream, bufs, world, flop)
    except Exception as exc:  # reported in the line; the serial e2e above stands alone
        try:
            torch.cuda.synchronize()
        except Exception:
            pass
        e2e_pipe = {"error": f"{type(exc).__name__}: {exc}"}
    if "error" not in e2e_pipe:
        # with the two directions on their own streams, the longer copy bounds a step
        e2e_pipe["copies_bound_ms_per_step"] = max(link["h2d_ms"], link["d2h_ms"])

    # ---- AWQ W4A16: the stacked modulation GEMVs
    awq = None
    if args.awq_blocks > 0:
        awq = run_awq(args, lib, dev, stream, world)

    # the tensor cores' own NVFP4 rate on this device, at the GEMM's shape:
    # back-to-back CTA-pair M256 N256 K64 block-scaled MMAs on every SM pair
    # (no memory traffic)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ctas = 2 * (sms // 2)
    iters = 8192
    for _ in range(2):
        lib.bench_mma_rate(3, 256, iters, ctas, dev_status=status, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    lib.bench_mma_rate(3, 256, iters, ctas, dev_status=status, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    mma_tflops = 2.0 * 128 * 256 * 64 * iters * ctas / (e0.elapsed_time(e1) * 1e-3) / 1e12

    pk = peaks()
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    g_avg = t_g
    q_avg = t_q
    gemm_tflops = flop / g_avg / 1e12
    q_bytes = M * K * 2 + M * K // 2 + M * K // 16 + M * r * 2
    g_bytes = (M * K // 2 + M * K // 16 + N * K // 2 + N * K // 16 + M * r * 2 + r * N * 2 +
               N * 2 + M * N * 2)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_total / args.steps * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4",
        "data": "synthetic (seeded; DiT attention out-projection shapes and outlier statistics)",
        "config": {"workload": f"{case.name}: SVDQ W4A4 linear M={M} K={K} N={N} rank={r}",
                   "M": M, "K": K, "N": N, "rank": r,
                   "l2": f"inputs rotate over {nsets} buffer sets ({nsets * set_bytes / 2**20:.0f}"
                         " MiB > 3x L2)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {
            "bound": "tensor", "kernel": "svdq_gemm_w4a4",
            "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
            "frac": round(gemm_tflops / fp4_peak, 4),
            "peak_source": f"{pk['source']} bf16 {pk['bf16_tflops']} TFLOP/s x {FP4_OVER_BF16:g} "
                           "(nominal fp4/bf16 dense ratio)",
            "traffic": measured_traffic("svdq_gemm_w4a4"),
            "traffic_note": "ncu dram read+write of one launch (Y is written back from L2 "
                            "after the kernel, so it is not in the count)",
            "algorithmic_bytes": g_bytes,
            "achieved_hbm_gbs": round(g_bytes / g_avg / 1e9, 1),
            "measured_mma_tflops": round(mma_tflops, 1),
            "frac_of_measured_mma": round(gemm_tflops / mma_tflops, 4),
        },
        "kernels": {
            "svdq_quantize_act": {"us": round(q_avg * 1e6, 2), "bound": "hbm",
                                  "achieved_gbs": round(q_bytes / q_avg / 1e9, 1),
                                  "peak_gbs": pk["hbm_gbs"],
                                  "frac": round(q_bytes / q_avg / 1e9 / pk["hbm_gbs"], 4),
                                  "algorithmic_bytes": q_bytes,
                                  "traffic": measured_traffic("svdq_quantize_act")},
            "svdq_gemm_w4a4": {"us": round(g_avg * 1e6, 2), "tflops": round(gemm_tflops, 1)},
        },
        "e2e": {k: (round(v, 3) if isinstance(v, float) else v) for k, v in e2e.items()},
        "e2e_pipelined": {k: (round(v, 3) if isinstance(v, float) else v)
                          for k, v in e2e_pipe.items()},
        "gpu_launches": 2 * args.steps * args.reps,
        "timing": f"median of {args.reps} replays of a CUDA graph of the {args.steps} steps "
                  "(CUDA events around each replay, barrier + synchronize on both sides); "
                  "per-kernel times the same way from graphs of that kernel alone",
        "spread": {"replays": args.reps,
                   "step_us": _spread([t / args.steps for t in ts_step]),
                   "svdq_quantize_act_us": _spread([t / args.steps for t in ts_q]),
                   "svdq_gemm_w4a4_us": _spread([t / args.steps for t in ts_g])},
        "clocks": clk.summary(),
        "pack_seconds": round(pack_s, 2),
        "wall_s_timed": round(wall, 4),
    }
    if awq is not None:
        line["awq"] = awq
        line["gpu_launches"] += awq["launches"]
    if not args.no_mlp_gelu:
        mlp = run_mlp_gelu(args, lib, dev, stream, world)
        line["mlp_fc1_gelu"] = mlp
        line["gpu_launches"] += mlp["launches"]
    if not args.no_qkv_epilogue:
        qk = run_qkv_epilogue(args, lib, dev, stream, world)
        line["qkv_norm_rope"] = qk
        line["gpu_launches"] += qk["launches"]
    if not args.no_int4:
        i4 = run_int4(args, lib, dev, stream, world)
        line["int4"] = i4
        line["gpu_launches"] += i4["launches"]
    return line


def _spread(ts):
    """min / 10th percentile / median / 90th percentile / max, microseconds."""
    q = np.percentile(np.asarray(ts) * 1e6, [0, 10, 50, 90, 100])
    return {k: round(float(v), 3) for k, v in zip(("min", "p10", "median", "p90", "max"), q)}


def _time_graph(args, launch, fn, stream, dev, world):
    """Per-launch seconds of `args.steps` launches of fn captured in a CUDA
    graph (eager warm-up first), max over ranks."""
    import torch
    for i in range(args.warmup):
        launch(fn, i, stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream(dev)
        for i in range(args.steps):
            launch(fn, i, cs)
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(1, min(args.reps, 20))):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3 / args.steps)
    return max_over_ranks(statistics.median(ts), world, dev)


def run_qkv_epilogue(args, lib, dev, stream, world):
    """The fused QKV projection (M = 4608 tokens: 512 text + 4096 image,
    K = 3072, N = 9216 = 3 x 24 heads x 128, rank 32) with the per-head RMS
    normalization of Q and K and the rotary embedding in the GEMM epilogue
    (svdq_gemm_w4a4_qkv), against the plain GEMM on the same operands.
    Unfused, normalization and rotation would read and write the Q and K
    columns once more each (2 x 2 x M x 2N/3 x 2 bytes)."""
    import torch
    case = workloads.CASES["qkv"]
    M, K, N, r = case.M, case.K, case.N, case.rank
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    Xbits = workloads.bf16_bits_of(X)
    packed = lib.svdq_pack_weights(W, lib.svdq_calib_absmax(Xbits), r)
    nq, nk = workloads.make_qk_norm_weights()
    cos, sin = workloads.make_rope_tables(workloads.rope_positions())

    def dbits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sets = []
    for _ in range(3):        # three weight + output sets (> 3 x L2 in all), rotated
        s = {"wc": torch.from_numpy(packed["w_codes"]).to(dev),
             "ws": torch.from_numpy(packed["w_scales"]).to(dev),
             "L2s": dbits(packed["L2s"]), "bias": dbits(workloads.bf16_bits_of(b)),
             "Y": torch.empty((M, N), dtype=torch.bfloat16, device=dev)}
        s["ac"], s["as"], s["lora"] = lib.svdq_quantize_act(
            dbits(Xbits).view(M, K), torch.from_numpy(packed["inv_lambda"]).to(dev),
            dbits(packed["L1s"]), r, dev_status=status, stream=stream)
        sets.append(s)
    nq_d, nk_d = dbits(workloads.bf16_bits_of(nq)), dbits(workloads.bf16_bits_of(nk))
    cos_d, sin_d = torch.from_numpy(cos).to(dev), torch.from_numpy(sin).to(dev)

    def plain(s, st):
        lib.svdq_gemm_w4a4(s["ac"], s["as"], s["wc"], s["ws"], packed["w_tensor_scale"],
                           s["lora"], s["L2s"], s["bias"], M, N, K, r, s["Y"],
                           dev_status=status, stream=st)

    def fused(s, st):
        lib.svdq_gemm_w4a4_qkv(s["ac"], s["as"], s["wc"], s["ws"], packed["w_tensor_scale"],
                               s["lora"], s["L2s"], s["bias"], nq_d, nk_d, cos_d, sin_d, M, N,
                               K, r, QKV=s["Y"], dev_status=status, stream=st)

    def launch(fn, i, st):
        fn(sets[i % len(sets)], st)

    res = {"workload": f"qkv: SVDQ W4A4 linear + Q/K RMS norm + rotary M={M} K={K} N={N} "
                       f"rank={r}", "launches": 2 * args.steps}
    for name, fn in (("fused", fused), ("plain", plain)):
        t = _time_graph(args, launch, fn, stream, dev, world)
        res[f"us_{name}"] = round(t * 1e6, 2)
        res[f"tflops_{name}"] = round(world * 2.0 * M * N * K / t / 1e12, 1)
    if int(status.item()) != 0:
        raise RuntimeError("device status set during the QKV epilogue phase")
    res["epilogue_cost"] = round(res["us_fused"] / res["us_plain"] - 1.0, 4)
    res["separate_pass_bytes_avoided"] = 2 * 2 * M * (2 * N // 3) * 2
    return res


def run_int4(args, lib, dev, stream, world):
    """The INT4 variant at the attention out-projection shape (M = 4096,
    K = N = 3072, rank 32): svdq_quantize_act_int4 and svdq_gemm_w4a4_int4,
    each alone and as the layer's step, weights from svdq_pack_weights_int4
    (three input, weight and output sets rotated, > L2 in all).  The GEMM runs
    on tcgen05 f16 MMAs: its denominator is the measured bf16 tensor rate (the
    f16 rate of the same instruction); the quantizer's is the HBM copy rate."""
    import torch
    case = workloads.CASES["attn_out"]
    M, K, N, r = case.M, case.K, case.N, case.rank
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    Xbits = workloads.bf16_bits_of(X)
    t0 = time.perf_counter()
    packed = lib.svdq_pack_weights_int4(W, lib.svdq_calib_absmax(Xbits), r)
    pack_s = time.perf_counter() - t0

    def dbits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    inv = torch.from_numpy(packed["inv_lambda"]).to(dev)
    L1s = dbits(packed["L1s"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sets = []
    for _ in range(3):
        sets.append({
            "X": dbits(Xbits).view(M, K), "wc": torch.from_numpy(packed["w_codes"]).to(dev),
            "ws": dbits(packed["w_scales"]), "L2": dbits(packed["L2"]),
            "bias": dbits(workloads.bf16_bits_of(b)),
            "ac": torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
            "as": torch.empty((M, K // 64), dtype=torch.bfloat16, device=dev),
            "lora": torch.empty((M, r), dtype=torch.bfloat16, device=dev),
            "Y": torch.empty((M, N), dtype=torch.bfloat16, device=dev)})

    def quant(s, st):
        lib.svdq_quantize_act_int4(s["X"], inv, L1s, r, s["ac"], s["as"], s["lora"],
                                   dev_status=status, stream=st)

    def gemm(s, st):
        lib.svdq_gemm_w4a4_int4(s["ac"], s["as"], s["wc"], s["ws"], s["lora"], s["L2"],
                                s["bias"], M, N, K, r, s["Y"], dev_status=status, stream=st)

    def step(s, st):
        quant(s, st)
        gemm(s, st)

    def launch(fn, i, st):
        fn(sets[i % len(sets)], st)

    t_step = _time_graph(args, launch, step, stream, dev, world)
    t_q = _time_graph(args, launch, quant, stream, dev, world)
    t_g = _time_graph(args, launch, gemm, stream, dev, world)
    if int(status.item()) != 0:
        raise RuntimeError("device status set during the INT4 phase")
    flop = 2.0 * M * N * K
    q_bytes = M * K * 2 + M * K // 2 + M * (K // 64) * 2 + M * r * 2
    gemm_tflops = world * flop / t_g / 1e12
    pk = peaks()
    hbm = pk["hbm_gbs"]
    return {
        "workload": f"attn_out, INT4 variant: M={M} K={K} N={N} rank={r}, group 64, bf16 "
                    f"scales", "launches": 4 * args.steps,
        "pack_seconds": round(pack_s, 2),
        "us_step": round(t_step * 1e6, 2), "tflops_step": round(world * flop / t_step / 1e12, 1),
        "us_quantize_act_int4": round(t_q * 1e6, 2),
        "quantize_act_int4_gbs": round(q_bytes / t_q / 1e9, 1),
        "quantize_act_int4_frac_hbm": round(q_bytes / t_q / 1e9 / hbm, 4),
        "quantize_act_int4_traffic": measured_traffic("svdq_quantize_act_int4"),
        "us_gemm_int4": round(t_g * 1e6, 2), "tflops_gemm_int4": round(gemm_tflops, 1),
        "gemm_int4_traffic": measured_traffic("svdq_gemm_w4a4_int4"),
        "gemm_int4_peak_tflops": pk["bf16_tflops"],
        "gemm_int4_frac": round(gemm_tflops / pk["bf16_tflops"], 4),
        "gemm_int4_peak_source": f"{pk['source']} bf16 (tcgen05 f16 and bf16 MMAs run at one rate)",
    }


def run_mlp_gelu(args, lib, dev, stream, world):
    """The MLP's first linear (fc1: M = 4096, K = 3072, N = 12288, rank 32)
    with GELU fused into the GEMM epilogue (svdq_gemm_w4a4_gelu), against the
    plain GEMM on the same quantized operands.  A separate GELU pass would
    read and write the M x N bf16 output once more."""
    import torch
    case = workloads.CASES["fc1"]
    M, K, N, r = case.M, case.K, case.N, case.rank
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    Xbits = workloads.bf16_bits_of(X)
    packed = lib.svdq_pack_weights(W, lib.svdq_calib_absmax(Xbits), r)

    def dbits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sets = []
    for _ in range(3):        # three weight + output sets (> 3 x L2 in all), rotated
        s = {"wc": torch.from_numpy(packed["w_codes"]).to(dev),
             "ws": torch.from_numpy(packed["w_scales"]).to(dev),
             "L2s": dbits(packed["L2s"]), "bias": dbits(workloads.bf16_bits_of(b)),
             "Y": torch.empty((M, N), dtype=torch.bfloat16, device=dev)}
        s["ac"], s["as"], s["lora"] = lib.svdq_quantize_act(
            dbits(Xbits).view(M, K), torch.from_numpy(packed["inv_lambda"]).to(dev),
            dbits(packed["L1s"]), r, dev_status=status, stream=stream)
        sets.append(s)

    def launch(fn, i, st):
        s = sets[i % len(sets)]
        fn(s["ac"], s["as"], s["wc"], s["ws"], packed["w_tensor_scale"], s["lora"], s["L2s"],
           s["bias"], M, N, K, r, s["Y"], dev_status=status, stream=st)

    res = {"workload": f"fc1: SVDQ W4A4 linear + GELU (tanh) M={M} K={K} N={N} rank={r}",
           "launches": 0}
    for name, fn in (("gelu", lib.svdq_gemm_w4a4_gelu), ("plain", lib.svdq_gemm_w4a4)):
        t = _time_graph(args, launch, fn, stream, dev, world)
        res[f"us_{name}"] = round(t * 1e6, 2)
        res[f"tflops_{name}"] = round(world * 2.0 * M * N * K / t / 1e12, 1)
        res["launches"] += args.steps
    if int(status.item()) != 0:
        raise RuntimeError("device status set during the fc1 GELU phase")
    res["gelu_epilogue_cost"] = round(res["us_gelu"] / res["us_plain"] - 1.0, 4)
    res["separate_gelu_bytes_avoided"] = 2 * M * N * 2

    # fc2's activation side (K2 = N, rank 32) fused as well
    # (svdq_gemm_w4a4_gelu_quant, H not written), against fc1 + GELU followed by
    # svdq_quantize_act on H.  fc2's smoothing and down-projection factor are
    # synthetic here (inv_lambda2 = 2^u, u ~ U(-3, 3); L1s2 ~ N(0, 0.05^2) in
    # bf16): the kernels' work does not depend on their values.
    r2 = workloads.CASES["fc2"].rank
    rng = np.random.default_rng(77)
    inv2 = torch.from_numpy(np.exp2(rng.uniform(-3.0, 3.0, N)).astype(np.float32)).to(dev)
    l1s2 = dbits(workloads.bf16_bits_of(
        workloads.to_bf16_values(rng.standard_normal((r2, N)) * 0.05)))
    for s in sets:
        s["a2c"] = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
        s["a2s"] = torch.empty(lib.scale_bytes(M, N), dtype=torch.uint8, device=dev)
        s["l2"] = torch.empty((M, r2), dtype=torch.bfloat16, device=dev)
        s["scr"] = torch.empty(lib.gelu_quant_scratch_bytes(M, N, r2), dtype=torch.uint8,
                               device=dev)

    def fused_quant(s, st):
        lib.svdq_gemm_w4a4_gelu_quant(s["ac"], s["as"], s["wc"], s["ws"],
                                      packed["w_tensor_scale"], s["lora"], s["L2s"], s["bias"],
                                      inv2, l1s2, r2, M, N, K, r, a2_codes=s["a2c"],
                                      a2_scales=s["a2s"], lora_act2=s["l2"], scratch=s["scr"],
                                      dev_status=status, stream=st)

    def gelu_then_quant(s, st):
        lib.svdq_gemm_w4a4_gelu(s["ac"], s["as"], s["wc"], s["ws"], packed["w_tensor_scale"],
                                s["lora"], s["L2s"], s["bias"], M, N, K, r, s["Y"],
                                dev_status=status, stream=st)
        lib.svdq_quantize_act(s["Y"], inv2, l1s2, r2, s["a2c"], s["a2s"], s["l2"],
                              dev_status=status, stream=st)

    def launch2(fn, i, st):
        fn(sets[i % len(sets)], st)

    for name, fn in (("gelu_quant", fused_quant), ("gelu_then_quantize_act", gelu_then_quant)):
        t = _time_graph(args, launch2, fn, stream, dev, world)
        res[f"us_{name}"] = round(t * 1e6, 2)
        res["launches"] += 2 * args.steps
    if int(status.item()) != 0:
        raise RuntimeError("device status set during the fc1 GELU + quantization phase")
    res["gelu_quant_workload"] = (f"fc1 + GELU + fc2 activation quantization and down "
                                  f"projection (K2={N}, rank2={r2})")
    res["gelu_quant_saving"] = round(1.0 - res["us_gelu_quant"] /
                                     res["us_gelu_then_quantize_act"], 4)
    return res


def host_link(Xh, Xd, Yd, Yh, stream, reps):
    """GB/s of the host-to-device copy of X and the device-to-host copy of Y
    (pinned host buffers), each timed alone with CUDA events on `stream`."""
    import torch
    out = {}
    for name, dst, src in (("h2d", Xd, Xh), ("d2h", Yh, Yd)):
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                dst.copy_(src, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        nbytes = src.numel() * src.element_size()
        out[f"{name}_ms"] = round(ms, 4)
        out[f"{name}_gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    return out


def e2e_pipelined(args, layer, Xbits, M, K, N, dev, stream, bufs, world, flop):
    """The end-to-end step of `e2e` as a serving loop runs it: two X and Y
    buffer pairs and two copy streams, so that step i's host-to-device copy
    overlaps step i-1's compute and its device-to-host read step i+1's.  Every
    step still moves its own input and result inside the timed region; events
    order each buffer's reuse after the copy or compute that last used it."""
    import torch
    nb = 2
    Xh = [torch.from_numpy(Xbits.view(np.int16)).view(torch.bfloat16).pin_memory()
          for _ in range(nb)]
    Yh = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    Xd = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in range(nb)]
    Yd = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(nb)]
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    x_ready = [torch.cuda.Event() for _ in range(nb)]  # Xd[b] holds this step's input
    computed = [torch.cuda.Event() for _ in range(nb)]  # done reading Xd[b], Yd[b] written
    y_read = [torch.cuda.Event() for _ in range(nb)]    # Yd[b] copied out
    used = [False] * nb

    def run(n):
        for i in range(n):
            b = i % nb
            if used[b]:
                h2d.wait_event(computed[b])
            with torch.cuda.stream(h2d):
                Xd[b].copy_(Xh[b], non_blocking=True)
            x_ready[b].record(h2d)
            stream.wait_event(x_ready[b])
            if used[b]:
                stream.wait_event(y_read[b])
            layer.forward(Xd[b], out=Yd[b], act_buffers=bufs, stream=stream)
            computed[b].record(stream)
            d2h.wait_event(computed[b])
            with torch.cuda.stream(d2h):
                Yh[b].copy_(Yd[b], non_blocking=True)
            y_read[b].record(d2h)
            used[b] = True

    run(args.warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d)
    run(args.steps)
    e1.record(d2h)
    torch.cuda.synchronize()
    t = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world, dev)
    return {"value": world * args.steps * flop / t / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2,
            "ms_per_step": t / args.steps * 1e3, "buffers": nb}


def run_awq(args, lib, dev, stream, world):
    import torch
    pk = peaks()
    blocks = []
    for blk in range(args.awq_blocks):
        W, b = workloads.make_awq_weights(blk)
        q, s, z = lib.awq_pack_weights(W)
        blocks.append((torch.from_numpy(q).to(dev),
                       torch.from_numpy(s.view(np.int16)).to(dev).view(torch.float16),
                       torch.from_numpy(z.view(np.int16)).to(dev).view(torch.float16),
                       torch.from_numpy(workloads.bf16_bits_of(b).view(np.int16)).to(dev).view(
                           torch.bfloat16)))
    N, K = workloads.AWQ_N, workloads.AWQ_K
    res = {"metric": "AWQ W4A16 HBM GB/s", "blocks": args.awq_blocks, "K": K, "N": N,
           "by_M": {}, "launches": 0}
    for M in (1, 2, 4):
        X = torch.from_numpy(workloads.bf16_bits_of(workloads.make_awq_activations(M)).view(
            np.int16)).to(dev).view(torch.bfloat16)
        Y = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in blocks]
        for i, (q, s, z, b) in enumerate(blocks):   # eager warm-up
            lib.awq_gemv_w4a16(X, q, s, z, b, Y=Y[i], stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()                  # the stack of block GEMVs, one graph
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream(dev)
            for i, (q, s, z, b) in enumerate(blocks):
                lib.awq_gemv_w4a16(X, q, s, z, b, Y=Y[i], stream=cs)
        g.replay()
        torch.cuda.synchronize()
        reps = max(1, args.steps // 4)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e-3 / reps
        t = max_over_ranks(t, world, dev)
        nbytes = len(blocks) * (N * K // 2 + 4 * N * (K // 64) + M * K * 2 + M * N * 2 + N * 2)
        gbs = nbytes / t / 1e9
        res["by_M"][str(M)] = {"us_per_stack": round(t * 1e6, 1), "gbs": round(world * gbs, 1),
                               "frac": round(gbs / pk["hbm_gbs"], 4)}
        res["launches"] += reps * len(blocks)
    res["roofline"] = {"bound": "hbm", "kernel": "awq_gemv_w4a16",
                       "achieved": res["by_M"]["1"]["gbs"] / world, "peak": pk["hbm_gbs"],
                       "unit": "GB/s", "frac": res["by_M"]["1"]["frac"],
                       "traffic": measured_traffic("awq_gemv_w4a16"),
                       "algorithmic_bytes_per_launch":
                           N * K // 2 + 4 * N * (K // 64) + K * 2 + N * 2 + N * 2}
    return res


# --------------------------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    case = workloads.CASES[args.workload]
    rows = args.oracle_rows
    t, flop, cores = time_oracle(case, rows, args.steps)
    value = flop / t / 1e12
    sample = (f"{rows} of {case.M} rows of the {case.name} workload per step "
              f"(K={case.K}, N={case.N}, rank {case.rank}); oracle packing not timed")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{case.name}: SVDQ W4A4 linear M={case.M} K={case.K} "
                               f"N={case.N} rank={case.rank}", "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--reps", type=int, default=50,
                    help="timed replays of the K-step graph (the median is reported)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="attn_out", choices=sorted(workloads.CASES))
    ap.add_argument("--awq-blocks", type=int, default=workloads.AWQ_BLOCKS)
    ap.add_argument("--oracle-rows", type=int, default=512)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-mlp-gelu", action="store_true",
                    help="skip the fc1 + fused GELU phase")
    ap.add_argument("--no-qkv-epilogue", action="store_true",
                    help="skip the QKV + normalization + rotary phase")
    ap.add_argument("--no-int4", action="store_true", help="skip the INT4 variant's phase")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of repeated steps (untimed) over which clocks are sampled")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, world, rank)), flush=True)
        return 0

    line = run_gpu(args, world, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            case = workloads.CASES[args.workload]
            t, flop, cores = time_oracle(case, args.oracle_rows, 3)
            line["cpu_baseline"] = {
                "value": round(flop / t / 1e12, 5), "unit": "TFLOP/s", "cores": cores,
                "kind": "oracle",
                "sample": f"{args.oracle_rows} of {case.M} rows per step, median of 3 "
                          "(oracle packing not timed)"}
            if "y_rows" in _SAMPLE:
                y = (_SAMPLE["y_rows"].astype(np.uint32) << 16).view(np.float32).astype(
                    np.float64)
                line["quality"] = quality_sample(case, args.oracle_rows, y)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
