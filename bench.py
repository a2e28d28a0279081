#!/usr/bin/env python
"""Benchmark of the FMPQ W4Ax hot path on GB300.

A step is one pass of the hot path over one batch: the fused activation quantizer
(gather-permute, per-block scales, INT4/INT8 codes) followed by the W4Ax GEMM with its FP32
epilogue, on the LLaMA-70B down-projection shape (M=4096 tokens, K=28672, N=8192; synthetic
Laplace activations with 10% outlier channels, 27 of 224 blocks INT8). The INT4 weights are
packed once beforehand (offline preparation; timed separately and reported, not in the step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --sweep      # the other workloads: one JSON line each (not the step metric)

Prints one JSON line. `value` is effective TOPS (2*M*N*K per step, INT4 and INT8 blocks
counted alike) summed over ranks with the max per-rank step time; `e2e` is the same metric
with the host->device copy of X and the device->host copy of Y inside every step.
`--impl reference` times the CPU oracle (test infrastructure, never tuned) on bounded
samples of the same workload.
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

WORKLOAD = "llama70b_down"
METRIC = "W4Ax GEMM effective TOPS (% INT8 TC peak) at M=4096; quantizer HBM GB/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "gemm_traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many untimed steps and exit (for profilers)")
    ap.add_argument("--sweep-only", default="",
                    help="with --sweep: run only the named workload (e.g. decode_m16)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the quantizer and GEMM on the LLaMA-7B QKV, decode (M=1..128) and "
                         "load-balance (INT8 fraction 0-50%%) workloads, and the calibration "
                         "statistics kernel, one JSON line each")
    return ap.parse_args()


# ------------------------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: the whole job takes as long as its slowest rank. One all-reduce
    of a scalar (NCCL on the GPU in the benchmark, gloo on the CPU in the tests); the data path
    itself has no collective (each rank runs its own batch against replicated weights)."""
    if world == 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_tops(world: int, ops_per_rank: float, ms: float) -> float:
    """Whole-job throughput (weak scaling): every rank does ops_per_rank in ms."""
    return world * ops_per_rank / (ms * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fmpq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            sms.append(sm)
            maxs.append(mx)
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms)}


# Sources each recorded kernel is compiled from: a recorded figure stays valid while these are
# unchanged (an edit to another kernel's file does not touch this kernel's code).
KERNEL_SOURCES = {
    "w4ax_gemm": ("fmpq_gemm.cu", "fmpq_device.cuh", "fmpq_internal.h"),
    "fmpq_quantize": ("fmpq_quantize.cu", "fmpq_device.cuh", "fmpq_internal.h"),
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_quantized_gemm_fmpq_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def quant_algorithmic_bytes(M: int, K: int, n8: int) -> int:
    """Algorithmic HBM bytes of one quantizer pass: the fp16 input (2MK), the codes at their
    nominal widths (INT4 blocks half a byte per code, INT8 blocks one byte) and one fp16 scale
    per token and block."""
    nb = K // 128
    k8 = 128 * n8
    return 2 * M * K + M * ((K - k8) // 2 + k8) + 2 * M * nb


# ------------------------------------------------------------------------------- CPU oracle

def oracle_sample_rate(w, target_s: float, rows: int = 8, cols: int = 4096, max_rounds: int = 2000):
    """Time the oracle (quantizer on `rows` tokens + per-block partials and fp64 epilogue for
    rows x cols outputs, weights pre-quantized) repeatedly until `target_s` seconds of CPU
    work; return effective TOPS and a description."""
    import oracle
    Wq, sw = oracle.quantize_weights(w.W[:cols], w.perm)
    done_ops, elapsed, rounds, r0 = 0.0, 0.0, 0, 0
    while elapsed < target_s and rounds < max_rounds:
        Xs = w.X[r0:r0 + rows]
        t0 = time.perf_counter()
        _, sx, Aq = oracle.quantize_activations(Xs, w.perm, w.mask)
        ms, ns = np.meshgrid(np.arange(rows, dtype=np.int32), np.arange(cols, dtype=np.int32), indexing="ij")
        oracle.gemm_sample(Aq, Wq, sx, sw, ms.ravel(), ns.ravel())
        elapsed += time.perf_counter() - t0
        done_ops += 2.0 * rows * cols * w.K
        rounds += 1
        r0 = (r0 + rows) % (w.M - rows)
    sample = (f"{rounds} rounds x ({rows} tokens quantized + {rows}x{cols} outputs over K={w.K}) "
              f"of the {w.M}x{w.K}x{w.N} workload, weights pre-quantized")
    return done_ops / elapsed / 1e12, elapsed, sample, oracle.num_threads()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from bit_quantized_gemm_fmpq_gb300 import workloads as wl
    import oracle
    oracle.build()
    w = wl.llama70b_down()
    per_step = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_rate(w, per_step / 4, max_rounds=1)
    vals, total = [], 0.0
    sample = ""
    cores = oracle.num_threads()
    for _ in range(args.steps):
        v, el, sample, cores = oracle_sample_rate(w, per_step, max_rounds=64)
        vals.append(v)
        total += el
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8/int64 (fp64 epilogue)",
        "data": "synthetic", "config": {"workload": WORKLOAD, "M": w.M, "K": w.K, "N": w.N, "n8_blocks": int(w.mask.sum()),
                                        "sample": "bounded sample per step"},
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)



# ------------------------------------------------------------------------------- sweep

def run_sweep(args):
    """Quantizer and GEMM alone on the other workloads of the method's evaluation shapes, each
    against its own roofline: the GEMM is tensor-bound at large M (2MNK over the fp8 peak) and
    HBM-bound in decode (packed A + scales + packed W + Y over the measured copy bandwidth).
    Inputs larger than L2 are not guaranteed here, so L2 is flushed before every timed launch;
    decode is also timed as a CUDA graph of back-to-back launches over weight copies that
    together exceed L2 (the serving case: no flush, no launch gaps)."""
    import torch
    from bit_quantized_gemm_fmpq_gb300 import build as fbuild
    fbuild.build()
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    from bit_quantized_gemm_fmpq_gb300 import workloads as wl
    fmpq.load_library()
    torch.cuda.set_device(0)
    peaks = measured_peaks()
    fp8_peak = peaks["bf16_tflops"] * 2.0
    hbm = peaks["hbm_gbs"]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    iters = max(10, min(args.steps, 100))

    def timed(fn):
        for _ in range(5):
            fn()
            flush.zero_()
        torch.cuda.synchronize()
        ts = []
        for _ in range(iters):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ts)

    configs = [("llama7b_qkv", lambda: wl.llama7b_qkv())]
    configs += [(f"decode_m{m}", (lambda m=m: wl.decode(m))) for m in (1, 8, 16, 32, 64, 128)]
    configs += [(f"load_balance_{int(f * 100)}pct", (lambda f=f: wl.load_balance(f))) for f in (0.0, 0.10, 0.25, 0.50)]
    if args.sweep_only:
        names = [c[0] for c in configs] + ["rmsnorm_quantize_llama70b_down", "swiglu_quantize_llama70b_down",
                                           "outlier_split_llama70b_down",
                                           "quik_asym_llama70b_down", "qoq_w4a8_llama70b_down",
                                           "calibrate_llama70b_down"]
        if args.sweep_only not in names:
            raise SystemExit(f"unknown workload {args.sweep_only}; one of {names}")
        configs = [c for c in configs if c[0] == args.sweep_only]
    sampler = ClockSampler(0)
    for name, make in configs:
        w = make()
        M, K, N = w.M, w.K, w.N
        layout = fmpq.Layout(K, w.perm, w.mask)
        X = torch.from_numpy(w.X).cuda()
        Wd = torch.from_numpy(w.W).cuda()
        Wp, sw = fmpq.w4_pack_weights(layout, Wd)
        del Wd
        A = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device="cuda")
        sx = torch.empty((layout.nb, M), dtype=torch.float16, device="cuda")
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        ws = layout.workspace(M, N)
        sampler.start()
        q_ms = timed(lambda: fmpq.fmpq_quantize(layout, X, A, sx))
        g_ms = timed(lambda: fmpq.w4ax_gemm(layout, A, sx, Wp, sw, M, N, Y, workspace=ws))
        graph_ms = quant_graph_ms = step_graph_ms = step_graph_one_call_ms = None
        if M <= 128:
            copies = [Wp] + [Wp.clone() for _ in range(4)]   # 5 x packed W > L2
            reps = 20

            def graph_time(body):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for r in range(reps):
                        body(r)
                for _ in range(3):
                    g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(5):
                    g.replay()
                e1.record()
                torch.cuda.synchronize()
                return e0.elapsed_time(e1) / (5 * reps)

            def gemm(r):
                fmpq.w4ax_gemm(layout, A, sx, copies[r % len(copies)], sw, M, N, Y, workspace=ws)

            graph_ms = graph_time(gemm)
            quant_graph_ms = graph_time(lambda r: fmpq.fmpq_quantize(layout, X, A, sx))
            # the decode step: quantize the token(s), then the GEMM
            step_graph_ms = graph_time(lambda r: (fmpq.fmpq_quantize(layout, X, A, sx), gemm(r)))
            # the same step as one call: the GEMM's prologue and weight stream overlap the quantizer
            step_graph_one_call_ms = graph_time(lambda r: fmpq.fmpq_quantize_gemm(
                layout, X, copies[r % len(copies)], sw, N, A_packed=A, a_scales=sx, Y=Y, workspace=ws))
            del copies
        clocks = sampler.stop()
        if fmpq.fmpq_device_status(layout) != 0:
            raise RuntimeError(f"device status after {name}")
        flops = 2.0 * M * N * K
        k8 = 128 * int(w.mask.sum())
        a_alg = M * ((K - k8) // 2 + k8)   # codes at their nominal widths
        gbytes = a_alg + 2 * layout.nb * M + layout.packed_w_bytes(N) + 2 * layout.nb * N + 2 * M * N
        qbytes = quant_algorithmic_bytes(M, K, int(w.mask.sum()))
        t_tensor = flops / (fp8_peak * 1e12) * 1e3
        t_hbm = gbytes / (hbm * 1e9) * 1e3
        bound = "tensor" if t_tensor >= t_hbm else "hbm"
        line = {
            "sweep": name, "M": M, "K": K, "N": N, "n8_blocks": int(w.mask.sum()), "bound": bound,
            "gemm_ms": g_ms, "gemm_tflops_effective": flops / (g_ms * 1e-3) / 1e12,
            "gemm_gbs": gbytes / (g_ms * 1e-3) / 1e9,
            "gemm_frac": max(t_tensor, t_hbm) / g_ms,
            "gemm_frac_of": "fp8 peak (measured bf16 burst x 2)" if bound == "tensor" else "measured HBM copy bandwidth",
            "gemm_graph_ms": graph_ms,
            "gemm_graph_frac": (max(t_tensor, t_hbm) / graph_ms) if graph_ms else None,
            "quant_ms": q_ms, "quant_gbs": qbytes / (q_ms * 1e-3) / 1e9,
            "quant_frac_hbm": qbytes / (q_ms * 1e-3) / 1e9 / hbm,
            "quant_graph_ms": quant_graph_ms, "step_graph_ms": step_graph_ms,
            "step_graph_one_call_ms": step_graph_one_call_ms,
            "l2": "flushed before every timed launch (graphs: back-to-back launches, 5 rotating weight "
                  "copies, no flush)",
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
        del X, A, sx, Y, Wp, sw, ws, layout
        torch.cuda.empty_cache()
    if not args.sweep_only or args.sweep_only == "rmsnorm_quantize_llama70b_down":
        # the quantizer fused with the preceding RMSNorm, on the 4096 x 28672 activations
        w = wl.llama70b_down()
        layout = fmpq.Layout(w.K, w.perm, w.mask)
        X = torch.from_numpy(w.X).cuda()
        gperm = torch.from_numpy(np.ascontiguousarray(
            np.random.default_rng(5).uniform(0.5, 1.5, w.K).astype(np.float16)[w.perm])).cuda()
        A = torch.empty(layout.packed_a_bytes(w.M), dtype=torch.uint8, device="cuda")
        sx = torch.empty((layout.nb, w.M), dtype=torch.float16, device="cuda")
        sampler.start()
        ms_plain = timed(lambda: fmpq.fmpq_quantize(layout, X, A, sx))
        ms = timed(lambda: fmpq.fmpq_rmsnorm_quantize(layout, X, gperm, 1e-5, A, sx))
        clocks = sampler.stop()
        nbytes = quant_algorithmic_bytes(w.M, w.K, int(w.mask.sum())) + 2 * w.K
        print(json.dumps({"sweep": "rmsnorm_quantize_llama70b_down", "M": w.M, "K": w.K, "bound": "hbm",
                          "kernel": "quantize_kernel<true>", "ms": ms, "quantize_only_ms": ms_plain,
                          "gbs": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
                          "l2": "flushed before every timed launch", "clocks": clocks}), flush=True)
        del layout
    if not args.sweep_only or args.sweep_only == "swiglu_quantize_llama70b_down":
        # the quantizer fused with SwiGLU on the LLaMA-70B down projection's 4096 x 28672 activations
        w = wl.llama70b_down()
        layout = fmpq.Layout(w.K, w.perm, w.mask)
        rng = np.random.default_rng(8)
        G = torch.from_numpy((rng.standard_normal((w.M, w.K)) * 2.0).astype(np.float16)).cuda()
        U = torch.from_numpy(w.X).cuda()
        A = torch.empty(layout.packed_a_bytes(w.M), dtype=torch.uint8, device="cuda")
        sx = torch.empty((layout.nb, w.M), dtype=torch.float16, device="cuda")
        sampler.start()
        ms = timed(lambda: fmpq.fmpq_swiglu_quantize(layout, G, U, A, sx))
        clocks = sampler.stop()
        nbytes = quant_algorithmic_bytes(w.M, w.K, int(w.mask.sum())) + 2 * w.M * w.K   # G and U read
        print(json.dumps({"sweep": "swiglu_quantize_llama70b_down", "M": w.M, "K": w.K, "bound": "hbm",
                          "kernel": "swiglu_quantize_kernel", "ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
                          "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
                          "l2": "flushed before every timed launch", "clocks": clocks}), flush=True)
        del layout, G, U, A, sx
        torch.cuda.empty_cache()
    if not args.sweep_only or args.sweep_only == "outlier_split_llama70b_down":
        # outlier split: 256 outlier channels in FP16 (tensor-core kernel), the other 28416 through the INT4 path
        w = wl.llama70b_down()
        n_out = 256
        rng = np.random.default_rng(6)
        out_cols = np.sort(rng.choice(w.K, size=n_out, replace=False)).astype(np.int32)
        base = np.setdiff1d(np.arange(w.K), out_cols).astype(np.int32)
        Kb = base.size
        layout = fmpq.select_layout(Kb, w.K, base, np.zeros(Kb // 128, dtype=np.uint8))
        X = torch.from_numpy(w.X).cuda()
        Wd = torch.from_numpy(w.W).cuda()
        Wp, sw = fmpq.w4_pack_weights(layout, Wd)
        W_out = Wd[:, torch.from_numpy(out_cols).long().cuda()].contiguous()
        del Wd
        cols = torch.from_numpy(out_cols).cuda()
        A = torch.empty(layout.packed_a_bytes(w.M), dtype=torch.uint8, device="cuda")
        sx = torch.empty((layout.nb, w.M), dtype=torch.float16, device="cuda")
        Y = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
        X_out = torch.empty((w.M, n_out), dtype=torch.float16, device="cuda")
        ws = layout.workspace(w.M, w.N)
        fmpq.fmpq_quantize(layout, X, A, sx)
        sampler.start()
        ms_q = timed(lambda: fmpq.fmpq_quantize(layout, X, A, sx))
        ms_qs = timed(lambda: fmpq.fmpq_quantize_split(layout, X, cols, A_packed=A, a_scales=sx, X_out=X_out))
        ms_base = timed(lambda: fmpq.w4ax_gemm(layout, A, sx, Wp, sw, w.M, w.N, Y, workspace=ws))
        ms_out = timed(lambda: fmpq.fmpq_outlier_gemm_fp16(layout, X, cols, W_out, Y, X_out))
        ms_prod = timed(lambda: fmpq.fmpq_outlier_product_fp16(layout, X_out, W_out, Y))

        def fused_step():
            # the QUIK forward pass with the split in the quantizer's pass over X
            fmpq.fmpq_quantize_split(layout, X, cols, A_packed=A, a_scales=sx, X_out=X_out)
            fmpq.w4ax_gemm(layout, A, sx, Wp, sw, w.M, w.N, Y, workspace=ws)
            fmpq.fmpq_outlier_product_fp16(layout, X_out, W_out, Y)
        ms_step = timed(fused_step)
        clocks = sampler.stop()
        print(json.dumps({"sweep": "outlier_split_llama70b_down", "M": w.M, "K_base": Kb, "n_out": n_out, "N": w.N,
                          "quantize_ms": ms_q, "quantize_split_ms": ms_qs,
                          "int4_path_ms": ms_base, "fp16_outlier_path_ms": ms_out, "fp16_product_ms": ms_prod,
                          "fused_step_ms": ms_step,
                          "fused_step_tops": 2.0 * w.M * w.N * w.K / (ms_step * 1e-3) / 1e12,
                          "int4_path_tflops_effective": 2.0 * w.M * w.N * Kb / (ms_base * 1e-3) / 1e12,
                          "fp16_outlier_path_tflops": 2.0 * w.M * w.N * n_out / (ms_out * 1e-3) / 1e12,
                          "l2": "flushed before every timed launch", "clocks": clocks}), flush=True)
        del layout, Wp, sw, W_out, X, A, sx, Y, X_out, ws
        torch.cuda.empty_cache()
    if not args.sweep_only or args.sweep_only == "quik_asym_llama70b_down":
        # QUIK asymmetric activations (every block 4-bit, zero point per token and block)
        w = wl.llama70b_down()
        layout = fmpq.Layout(w.K, w.perm, np.zeros(w.K // 128, dtype=np.uint8))
        X = torch.from_numpy(w.X).cuda()
        Wd = torch.from_numpy(w.W).cuda()
        Wp, sw = fmpq.w4_pack_weights(layout, Wd)
        del Wd
        wsum = fmpq.w4_weight_sums(layout, Wp, sw, w.N)
        A = torch.empty(layout.packed_a_bytes(w.M), dtype=torch.uint8, device="cuda")
        sx = torch.empty((layout.nb, w.M), dtype=torch.float16, device="cuda")
        z = torch.empty((layout.nb, w.M), dtype=torch.float16, device="cuda")
        Y = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
        ws = layout.workspace(w.M, w.N, variant=True)
        sampler.start()
        q_ms = timed(lambda: fmpq.fmpq_quantize_asym(layout, X, A, sx, z))
        g_ms = timed(lambda: fmpq.w4ax_gemm_asym(layout, A, sx, z, Wp, sw, wsum, w.M, w.N, Y, workspace=ws))
        clocks = sampler.stop()
        flops = 2.0 * w.M * w.N * w.K
        qbytes = 2 * w.M * w.K + layout.packed_a_bytes(w.M) + 4 * layout.nb * w.M
        print(json.dumps({"sweep": "quik_asym_llama70b_down", "M": w.M, "K": w.K, "N": w.N, "n8_blocks": 0,
                          "gemm_ms": g_ms, "gemm_tflops_effective": flops / (g_ms * 1e-3) / 1e12,
                          "gemm_frac_fp8_peak": flops / (g_ms * 1e-3) / 1e12 / fp8_peak,
                          "quant_ms": q_ms, "quant_gbs": qbytes / (q_ms * 1e-3) / 1e9,
                          "quant_frac_hbm": qbytes / (q_ms * 1e-3) / 1e9 / hbm,
                          "l2": "flushed before every timed launch", "clocks": clocks}), flush=True)
        del layout, Wp, sw, wsum, X, A, sx, z, Y, ws
        torch.cuda.empty_cache()
    if not args.sweep_only or args.sweep_only == "qoq_w4a8_llama70b_down":
        # QoQ: per-token INT8 activations (two code planes per block), progressive UINT4 weights
        w = wl.llama70b_down()
        layout = fmpq.Layout(w.K, w.perm, np.ones(w.K // 128, dtype=np.uint8))
        X = torch.from_numpy(w.X).cuda()
        Wd = torch.from_numpy(w.W).cuda()
        Wp, s1, s2, z2 = fmpq.qoq_pack_weights(layout, Wd)
        del Wd
        A = torch.empty(layout.packed_a_bytes(w.M), dtype=torch.uint8, device="cuda")
        sx = torch.empty(w.M, dtype=torch.float16, device="cuda")
        sums = torch.empty((layout.nb, w.M), dtype=torch.int32, device="cuda")
        Y = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
        ws = layout.workspace(w.M, w.N, variant=True)
        sampler.start()
        q_ms = timed(lambda: fmpq.qoq_quantize(layout, X, A, sx, sums))
        g_ms = timed(lambda: fmpq.qoq_gemm(layout, A, sx, sums, Wp, s1, s2, z2, w.M, w.N, Y, workspace=ws))
        clocks = sampler.stop()
        flops = 2.0 * w.M * w.N * w.K
        qbytes = 2 * w.M * w.K + layout.packed_a_bytes(w.M) + 2 * w.M + 4 * layout.nb * w.M
        print(json.dumps({"sweep": "qoq_w4a8_llama70b_down", "M": w.M, "K": w.K, "N": w.N,
                          "gemm_ms": g_ms, "gemm_tflops_effective": flops / (g_ms * 1e-3) / 1e12,
                          "gemm_frac_fp8_peak_of_mma_work": 2 * flops / (g_ms * 1e-3) / 1e12 / fp8_peak,
                          "quant_ms": q_ms, "quant_gbs": qbytes / (q_ms * 1e-3) / 1e9,
                          "quant_frac_hbm": qbytes / (q_ms * 1e-3) / 1e9 / hbm,
                          "l2": "flushed before every timed launch", "clocks": clocks}), flush=True)
        del layout, Wp, s1, s2, z2, X, A, sx, sums, Y, ws
        torch.cuda.empty_cache()
    if not args.sweep_only or args.sweep_only == "calibrate_llama70b_down":
        # offline calibration: per-channel absmax over the 4096 x 28672 activations (HBM-bound)
        w = wl.llama70b_down()
        X = torch.from_numpy(w.X).cuda()
        out = torch.empty(w.K, dtype=torch.int32, device="cuda")
        sampler.start()
        ms = timed(lambda: fmpq.fmpq_channel_absmax(X, out))
        clocks = sampler.stop()
        nbytes = 2 * w.M * w.K + 4 * w.K
        print(json.dumps({"sweep": "calibrate_llama70b_down", "M": w.M, "K": w.K, "bound": "hbm",
                          "kernel": "channel_absmax_kernel", "ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
                          "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
                          "l2": "flushed before every timed launch", "clocks": clocks}), flush=True)

# ------------------------------------------------------------------------------- our arm

def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    world, rank, local = dist_env()
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    from bit_quantized_gemm_fmpq_gb300 import build as fbuild
    if rank == 0:
        fbuild.build()
    if world > 1:
        torch.distributed.barrier()
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    from bit_quantized_gemm_fmpq_gb300 import workloads as wl
    fmpq.load_library()

    w = wl.llama70b_down()
    M, K, N = w.M, w.K, w.N
    layout = fmpq.Layout(K, w.perm, w.mask)
    stream = torch.cuda.current_stream()
    X = torch.from_numpy(w.X).cuda()
    Wd = torch.from_numpy(w.W).cuda()
    # offline weight preparation (timed once, not part of the step)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fmpq.w4_pack_weights(layout, Wd)  # warm
    Wp = torch.empty(layout.packed_w_bytes(N), dtype=torch.uint8, device="cuda")
    sw = torch.empty((layout.nb, N), dtype=torch.float16, device="cuda")
    e0.record()
    fmpq.w4_pack_weights(layout, Wd, Wp, sw)
    e1.record()
    torch.cuda.synchronize()
    pack_ms = e0.elapsed_time(e1)
    del Wd
    A = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device="cuda")
    sx = torch.empty((layout.nb, M), dtype=torch.float16, device="cuda")
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = layout.workspace(M, N)
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")

    def step():
        fmpq.fmpq_quantize(layout, X, A, sx, stream=stream)
        fmpq.w4ax_gemm(layout, A, sx, Wp, sw, M, N, Y, workspace=ws, stream=stream)

    if args.profile_steps:
        for _ in range(args.profile_steps):
            step()
        torch.cuda.synchronize()
        return

    for _ in range(max(3, args.warmup)):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record(stream)
        fmpq.fmpq_quantize(layout, X, A, sx, stream=stream)
        ev[i][1].record(stream)
        fmpq.w4ax_gemm(layout, A, sx, Wp, sw, M, N, Y, workspace=ws, stream=stream)
        ev[i][2].record(stream)
        flush.zero_()  # L2 flush between steps (outside the timed events)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    q_ms = [e[0].elapsed_time(e[1]) for e in ev]
    g_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_ms = max_over_ranks(sum(q + g for q, g in zip(q_ms, g_ms)) / args.steps, world, "cuda")
    status = fmpq.fmpq_device_status(layout)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    flops = 2.0 * M * N * K
    value = aggregate_tops(world, flops, step_ms)
    gemm_ms = statistics.mean(g_ms)
    quant_ms = statistics.mean(q_ms)
    peaks = measured_peaks()
    fp8_peak = peaks["bf16_tflops"] * 2.0   # nominal dense fp8/bf16 ratio (4.5 / 2.25)
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    # algorithmic bytes of the quantizer: read X (2MK), write the codes at their nominal widths
    # (half a byte per INT4 code, one per INT8 code) and the fp16 scales
    quant_bytes = quant_algorithmic_bytes(M, K, int(w.mask.sum()))
    quant_moved = 2 * M * K + layout.packed_a_bytes(M) + 2 * layout.nb * M   # what the kernel writes
    quant_gbs = quant_bytes / (quant_ms * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers: every step copies its input from
    # pinned host memory and its result back. The steps run as a serving pipeline would: the
    # input of step k + 1 is copied (on its own stream) while step k computes, and the result
    # of step k is read back while step k + 1 computes (two device buffers for each). One timed
    # region over all steps; no L2 flush inside it (X and the packed weights exceed L2).
    e2e = None
    if not args.no_e2e:
        Xh = torch.from_numpy(w.X).pin_memory()
        Yhs = [torch.empty((M, N), dtype=torch.float16).pin_memory() for _ in range(2)]
        Xs = [X, torch.empty_like(X)]
        Ys = [Y, torch.empty_like(Y)]
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        n_e2e = max(3, min(args.steps, 50))

        def step_on(Xk, Yk):
            fmpq.fmpq_quantize_gemm(layout, Xk, Wp, sw, N, A_packed=A, a_scales=sx, Y=Yk, workspace=ws,
                                    stream=stream)

        def pipeline(n):
            ev = lambda: torch.cuda.Event(enable_timing=False)
            h2d_ev, comp_ev, d2h_ev = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            h2d.wait_event(t0)
            with torch.cuda.stream(h2d):
                Xs[0].copy_(Xh, non_blocking=True)
            h2d_ev[0].record(h2d)
            for k in range(n):
                stream.wait_event(h2d_ev[k])
                if k >= 2:
                    stream.wait_event(d2h_ev[k - 2])        # result buffer k % 2 has been read back
                step_on(Xs[k % 2], Ys[k % 2])
                comp_ev[k].record(stream)
                if k + 1 < n:
                    if k >= 1:
                        h2d.wait_event(comp_ev[k - 1])      # input buffer (k + 1) % 2 is free
                    with torch.cuda.stream(h2d):
                        Xs[(k + 1) % 2].copy_(Xh, non_blocking=True)
                    h2d_ev[k + 1].record(h2d)
                d2h.wait_event(comp_ev[k])
                with torch.cuda.stream(d2h):
                    Yhs[k % 2].copy_(Ys[k % 2], non_blocking=True)
                d2h_ev[k].record(d2h)
            stream.wait_event(d2h_ev[n - 1])
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / n

        pipeline(3)   # warm-up
        e2e_ms = max_over_ranks(pipeline(n_e2e), world, "cuda")
        e2e = {"value": aggregate_tops(world, flops, e2e_ms), "unit": "TOPS",
               "h2d_bytes_per_step": int(Xh.numel() * 2), "d2h_bytes_per_step": int(Yhs[0].numel() * 2),
               "ms_per_step": e2e_ms,
               "pipeline": "each step's input copy and result read-back overlap the neighbouring steps' "
                           "compute (two device buffers each, copy streams); one timed region over the steps"}

    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, el, sample, cores = oracle_sample_rate(w, target_s=10.0)
        cpu = {"value": v, "unit": "TOPS", "cores": cores, "kind": "oracle", "sample": sample, "seconds": el}

    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4/int8 codes on e4m3 tensor cores, fp32 epilogue",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "n8_blocks": int(w.mask.sum()), "nb": layout.nb,
                   "step": "fmpq_quantize + w4ax_gemm", "l2": "flushed between steps (2x L2 write, untimed)",
                   "parallelism": f"replicated weights, one {M}-token batch per GPU"},
        "gemm": {"ms": gemm_ms, "tflops_effective": gemm_tflops, "frac_fp8_peak": gemm_tflops / fp8_peak},
        "quantizer": {"ms": quant_ms, "gbs": quant_gbs, "frac_hbm": quant_gbs / peaks["hbm_gbs"],
                      "bytes": quant_bytes, "bytes_basis": "2MK + M(K4/2 + K8) + 2M*nb (algorithmic)",
                      "bytes_moved": quant_moved, "traffic": recorded_traffic("fmpq_quantize")},
        "offline_pack_ms": pack_ms,
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": gemm_tflops / fp8_peak, "traffic": recorded_traffic("w4ax_gemm"),
                     "kernel": "w4ax_gemm_kernel",
                     "peak_source": f"{peaks['source']} bf16 burst x 2 (nominal fp8/bf16 dense ratio)"},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
