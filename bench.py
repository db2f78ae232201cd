"""Benchmark of the BaKron solve (bakron_quantize) on one m x n layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c3] [--impl ours|reference]

One step = one bakron_quantize call over the whole layer (every anti-
diagonal, every propagation), inputs resident in HBM; the factor preparation
is timed once and reported separately, as the paper's Table 3 excludes it.
Default workload: c3, the 4096 x 4096 attention-projection shape with an
AR(1) output factor and a 4-bit alphabet (see workloads/configs.py).

Multi-GPU: one layer per GPU, no communication (independent replicas):
`value` = N * m * n / max over ranks of the timed time.  L2 is flushed
(a 512 MiB write) before every timed step, outside the step's events.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload: the first R rows of the layer (their codes do
not depend on later rows), so the unit stays weights/s.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "BaKron solve time & weights quantized/s per m×n layer; % of tensor roofline"
UNIT = "weights/s"
SM_COUNT = 152
FP32_LANES_PER_SM = 128
# One double-float multiply-add (2 algorithmic flops) costs 5 fp32 pipe
# instructions (offset accumulator, df.cuh).
DF_INSTR_PER_MAC = 5


def alu_peak_tflops(sm_max_mhz: float) -> float:
    """Algorithmic TFLOP/s of the fp32 pipes running double-float MACs."""
    lane_ops = SM_COUNT * FP32_LANES_PER_SM * sm_max_mhz * 1e6
    return 2.0 * lane_ops / DF_INSTR_PER_MAC / 1e12


# Kernel classes on the tensor cores, with the bf16 multiply-adds their exact
# digit split performs per algorithmic multiply-add (5 factor digits x 6
# source digits, the 20 pairs of levels 0..5).  "sweep" is the persistent
# solve (--method persistent), one kernel that runs the whole solve (the band
# sweep on the fp32 pipes and every product on the tensor cores): its entry
# is the solve's own rate against the tensor roofline of the precision mode,
# i.e. the measured bf16 peak divided by the 20 digit pairs.
TENSOR_CLASSES = {"chunk_push": 20, "sweep": 20}
# Kernel launches of one solve on the persistent sweep: input check, offset,
# two factor exponent and two factor digit kernels, three task-queue
# kernels, the sweep.
SWEEP_LAUNCHES = 10
BF16_FALLBACK_TFLOPS = 1900.0  # used only without a measured peak


def roofline_for(kernel: str, alg_flops: float, ms: float, peaks: dict) -> dict:
    """Roofline entry of one kernel class from its algorithmic flops (2 per
    multiply-add of the products L_B E L_A^T it computes) and its summed
    event time.  Tensor-core classes: bf16 tensor flops (digit pairs x
    algorithmic flops) against the measured bf16 burst peak (the profile pass
    times each kernel alone); the other classes: double-float flops against
    the fp32-pipe peak derived from the unit counts and the maximum clock."""
    sec = ms * 1e-3
    alg = alg_flops / sec / 1e12 if sec > 0 else 0.0
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    if kernel in TENSOR_CLASSES:
        pairs = TENSOR_CLASSES[kernel]
        measured = "bf16_tflops" in peaks
        peak = float(peaks["bf16_tflops"]) if measured else BF16_FALLBACK_TFLOPS
        achieved = pairs * alg
        return {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "alg_tflops_fp64_equiv": alg,
                "peak_basis": ("measured" if measured else "fallback") + " bf16 dense burst peak; achieved = "
                              f"{pairs} bf16 digit-pair multiply-adds per algorithmic multiply-add"}
    peak = alu_peak_tflops(sm_max)
    return {"bound": "alu", "kernel": kernel, "achieved": alg, "peak": peak, "unit": "TFLOP/s", "frac": alg / peak,
            "peak_basis": f"{SM_COUNT} SMs x {FP32_LANES_PER_SM} fp32 lanes x {sm_max:.0f} MHz / "
                          f"{DF_INSTR_PER_MAC} instr per double-float MAC x 2 flops"}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def aggregate_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world <= 1:
        return
    import torch.distributed as dist

    if device is not None and device.type == "cuda":
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows)}


def load_workload(key: str):
    """A named workload (c1 .. c5), or "rand:MxN": an M x N layer with
    damped Gaussian Gram factors, W ~ N(0, 0.02^2) and 4-bit per-row scales
    (the shape of a layer without a named workload)."""
    from workloads import make_config, random_problem

    if key.startswith("rand:"):
        m, n = (int(x) for x in key[5:].lower().split("x"))
        return random_problem(m, n, bits=4, seed=m + 7 * n, w_std=0.02)
    return make_config(key)


def workload_config(p, world: int) -> dict:
    alpha = "Z" if p.bits == 0 else "{%d..%d}" % (-(1 << (p.bits - 1)), (1 << (p.bits - 1)) - 1)
    return {"workload": p.name, "m": p.m, "n": p.n, "bits": p.bits, "alphabet": alpha,
            "scales": "per-row absmax" if p.scales is not None else "none",
            "global_batch": world, "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": "flushed by a 512 MiB write before every timed step", "inputs": p.digest()}


def oracle_sample(p, rows: int, LA64, LB64):
    """The oracle on the first `rows` rows (codes of a row depend only on rows
    above it).  Returns (weights solved, seconds, layer-equivalent weights):
    the sample costs r n (r + n) multiply-adds where the layer costs
    m n (m + n), so a sample of r rows stands for r n (r + n) / (m + n)
    weights of the whole layer at the same rate of work."""
    import oracle as O

    r = min(rows, p.m)
    s = None if p.scales is None else p.scales[:r]
    t0 = time.perf_counter()
    O.bakron(p.W[:r], LA=LA64, LB=LB64[:r, :r], scales=s, bits=p.bits)
    return r * p.n, time.perf_counter() - t0, r * p.n * (r + p.n) / (p.m + p.n)


def sample_text(p, rows: int, secs: float, raw_rate: float) -> str:
    r = min(rows, p.m)
    return (f"first {r} of {p.m} rows x {p.n} columns per solve ({secs:.1f} s, fp64 numpy, Alg. 5 recursion); "
            f"the value is scaled to whole-layer work: the sample costs r n (r + n) = "
            f"{r * p.n * (r + p.n):.3g} multiply-adds against m n (m + n) = {p.m * p.n * (p.m + p.n):.3g} for "
            f"the layer, so {raw_rate:.4g} sampled weights/s stand for {raw_rate * (r + p.n) / (p.m + p.n):.4g} "
            f"layer weights/s")


def cpu_cores() -> int:
    return len(os.sched_getaffinity(0))


def run_reference(args, rank, world):
    """The fp64 oracle on the host cores, on a bounded sample per step."""
    if rank != 0:
        return None
    import oracle as O

    p = load_workload(args.config)
    LA64, LB64 = O.factors_of(p.A, p.B)
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(p, rows, LA64, LB64)
    times, units, equiv = [], 0, 0.0
    for _ in range(args.steps):
        u, t, eq = oracle_sample(p, rows, LA64, LB64)
        times.append(t)
        units, equiv = u, eq
    tot = sum(times)
    value = equiv * args.steps / tot
    sample = sample_text(p, rows, tot / args.steps, units * args.steps / tot)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": workload_config(p, 1), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


KERNEL_SOURCES = ("kronecker_hessian_gptq_gb300/csrc/quantize.cu", "kronecker_hessian_gptq_gb300/csrc/df.cuh",
                  "kronecker_hessian_gptq_gb300/csrc/tc.cuh")


def kernel_source_digest() -> str:
    """sha256 over the code of the sources the solve kernels are compiled
    from: comments removed and whitespace collapsed, so that an edit of a
    comment does not void a traffic measurement of unchanged code."""
    import hashlib
    import re

    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(rel.encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` (dram__bytes_read.sum +
    dram__bytes_write.sum, averaged over the captured launches), from the data
    record profiles/<kernel>_<workload>_dram.json that accompanies the ncu
    summary of the same name.  None when there is no such record or the
    kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_dram.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_digest():
        return None
    b = rec.get("traffic_bytes_per_launch")
    return int(b) if b is not None else None


# fp32 operations of one candidate evaluation in the scale search (counted
# from csrc/scales.cu: quotient and tie test 8, clamp 2, power-of-two scaling
# 2, exact error 15, its square 4, double-float accumulation 20).
SCALE_OPS_PER_EVAL = 51


def run_scales(args, p, W, LA, LB, s, ws, out, flush, world, dev):
    """The base quantizer's side kernels on the layer: the App. D scale search
    (grid `--scale-grid` shrink factors, alphabet {-2^(b-1) .. 2^(b-1)-1}) and
    the packing of the layer's codes to b bits; one step = both kernels."""
    import torch

    import kronecker_hessian_gptq_gb300 as bk

    m, n, bits = p.m, p.n, p.bits
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    V = bk.quantize(W, LA, LB, s, bits, ws=ws, out=out)[0]
    S = torch.empty(m, dtype=torch.float32, device=dev)
    P = torch.empty((m, (n * bits + 7) // 8), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        bk.row_scales(W, lo, hi, args.scale_grid, out=S)
        bk.pack_codes(V, bits, out=P)
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    sampler = ClockSampler(dev.index)
    sampler.start()
    barrier(world, dev)
    marks = [[ev(), ev(), ev()] for _ in range(args.steps)]
    for a, b, c in marks:
        flush.zero_()
        a.record()
        bk.row_scales(W, lo, hi, args.scale_grid, out=S)
        b.record()
        bk.pack_codes(V, bits, out=P)
        c.record()
    torch.cuda.synchronize()
    barrier(world, dev)
    clocks = sampler.stop()
    scale_ms = sum(a.elapsed_time(b) for a, b, _ in marks) / args.steps
    pack_ms = sum(b.elapsed_time(c) for _, b, c in marks) / args.steps
    total_ms = aggregate_max(sum(a.elapsed_time(c) for a, _, c in marks), world, dev)
    peaks = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    alu_peak = SM_COUNT * FP32_LANES_PER_SM * sm_max * 1e6 / 1e12  # T fp32 lane operations / s
    achieved = m * n * args.scale_grid * SCALE_OPS_PER_EVAL / (scale_ms * 1e-3) / 1e12
    pack_bytes = 4 * m * n + m * ((n * bits + 7) // 8)
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    cfg = workload_config(p, world)
    cfg["method"] = f"scale search ({args.scale_grid} shrink factors) + {bits}-bit packing"
    return {
        "metric": "scale search + code packing, weights/s per m x n layer", "unit": UNIT,
        "value": world * m * n * args.steps / (total_ms * 1e-3), "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 decisions, f32x2 error sums; int32 -> packed bits", "data": "synthetic",
        "config": cfg, "clocks": clocks, "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "alu", "kernel": "row_scales", "achieved": achieved, "peak": alu_peak,
                     "unit": "T fp32 ops/s", "frac": achieved / alu_peak, "traffic": None,
                     "peak_basis": f"{SM_COUNT} SMs x {FP32_LANES_PER_SM} fp32 lanes x {sm_max:.0f} MHz; "
                                   f"{SCALE_OPS_PER_EVAL} ops per candidate evaluation"},
        "kernels": {"row_scales": {"ms": scale_ms},
                    "pack_codes": {"ms": pack_ms, "bound": "hbm", "bytes": pack_bytes,
                                   "achieved_gbs": pack_bytes / (pack_ms * 1e-3) / 1e9, "peak_gbs": hbm,
                                   "frac": pack_bytes / (pack_ms * 1e-3) / 1e9 / hbm}},
        "e2e": None,
    }


def run_gram(args, world, dev):
    """Kronecker-factor accumulation (Sec. 4.2): the K-FAC Gram E[a a^T] and
    the one-step Shampoo Gram E[|b|^2 a a^T] of the 4096-feature input side
    from 65536 bf16 samples, on the tensor cores."""
    import numpy as np
    import torch

    import kronecker_hessian_gptq_gb300 as bk
    from workloads.activations import make_sample_config

    s = make_sample_config(args.config if args.config.startswith("g") else "g3")
    d, N = s.n, s.N
    Xh = torch.from_numpy(s.a_bits.view(np.int16)).view(torch.bfloat16)
    X = Xh.to(dev)
    w = bk.sq_norms(torch.from_numpy(s.b_bits.view(np.int16)).view(torch.bfloat16).to(dev))
    G = torch.empty((d, d), dtype=torch.float32, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        marks = [(ev(), ev()) for _ in range(args.steps)]
        for a, b in marks:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in marks) / args.steps

    sampler = ClockSampler(dev.index)
    sampler.start()
    barrier(world, dev)
    kfac_ms = timed(lambda: bk.gram(X, out=G))
    shampoo_ms = timed(lambda: bk.gram(X, w, out=G))
    barrier(world, dev)
    clocks = sampler.stop()
    kfac_ms = aggregate_max(kfac_ms * args.steps, world, dev) / args.steps
    # End to end: pinned host samples in, the factor out.
    Xp = Xh.pin_memory()
    Gh = torch.empty((d, d), dtype=torch.float32, pin_memory=True)
    t_e2e = []
    for _ in range(max(1, args.steps // 2)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        Xd = Xp.to(dev, non_blocking=True)
        bk.gram(Xd, out=G)
        Gh.copy_(G, non_blocking=True)
        torch.cuda.synchronize()
        t_e2e.append(time.perf_counter() - t0)
    e2e_s = aggregate_max(min(t_e2e), world, dev)
    flops = float(d) * (d + 1) * N  # d(d+1)/2 distinct entries, 2N flops each
    peaks = measured_peaks()
    peak = float(peaks["bf16_tflops"]) if "bf16_tflops" in peaks else BF16_FALLBACK_TFLOPS
    achieved = flops / (kfac_ms * 1e-3) / 1e12
    return {
        "metric": "Kronecker-factor accumulation (K-FAC Gram) TFLOP/s", "unit": "TFLOP/s",
        "value": world * achieved, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": kfac_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 samples, fp32 accumulation", "data": "synthetic",
        "config": {"workload": f"{s.name}: {d} features x {N} samples, Student-t (nu = 4)", "d": d, "N": N,
                   "l2": f"inputs ({d * N * 2 / 2**20:.0f} MiB) larger than L2"},
        "shampoo_ms": shampoo_ms, "shampoo_tflops": flops / (shampoo_ms * 1e-3) / 1e12,
        "clocks": clocks, "gpu_launches": 2 * args.steps,  # per K-FAC call: the packing pass and the products
        "roofline": {"bound": "tensor", "kernel": "gram_kernel", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_basis": ("measured" if "bf16_tflops" in peaks else "fallback")
                                   + " bf16 dense burst peak; algorithmic flops d (d + 1) N"},
        "e2e": {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": d * N * 2,
                "d2h_bytes_per_step": d * d * 4},
    }


# The pages' own BaKron times for the same layer shapes ("BaKron: Efficient
# Quantization with Kronecker-Factored Hessians", Sec. 6, Table 3: one RTX
# PRO 6000, float32; their inputs' Hessians and alphabet are not stated):
# context beside the measured line, not a target and not vs_baseline.
PAGES_TABLE3_BAKRON_S = {(1024, 1024): 0.025, (2048, 2048): 0.074, (4096, 4096): 0.288, (8192, 8192): 1.839,
                         (8192, 2048): 0.335, (2048, 8192): 0.322, (14336, 4096): 1.600, (4096, 14336): 1.717}


def pages_same_shape(m: int, n: int, ms_per_step: float):
    """The pages' BaKron time for an m x n layer, if Table 3 lists that shape."""
    t = PAGES_TABLE3_BAKRON_S.get((m, n))
    if t is None:
        return None
    return {"seconds": t, "hardware": "RTX PRO 6000, float32 (Table 3)", "ratio_pages_over_this": t / (ms_per_step * 1e-3)}


def antidiag_macs(m: int, n: int) -> int:
    """Multiply-adds of Algorithm 3 with triangular factors: entry (p, q)
    receives one per earlier entry (i, j) with i <= p, j <= q."""
    return (m * (m + 1) // 2) * (n * (n + 1) // 2) - m * n


def run_antidiag(args, p, W, LA, LB, s, ws, out, flush, world, dev):
    """BaKron-antidiagonal (Algorithm 3) on the layer, and the BaKron solve
    on the same inputs: the pages' speedup column (Table 3) on this GPU."""
    import torch

    import kronecker_hessian_gptq_gb300 as bk

    m, n = p.m, p.n
    ws_ad = torch.empty(bk.load_library().bakron_antidiag_workspace_size(m, n), dtype=torch.uint8, device=dev)
    out_ad = (torch.empty((m, n), dtype=torch.int32, device=dev), torch.empty((m, n), dtype=torch.float32, device=dev),
              torch.zeros(1, dtype=torch.int32, device=dev))
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def timed(fn, steps):
        marks = [(ev(), ev()) for _ in range(steps)]
        for a, b in marks:
            flush.zero_()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in marks)

    solve_ad = lambda: bk.antidiag(W, LA, LB, s, p.bits, ws=ws_ad, out=out_ad)  # noqa: E731
    solve_bk = lambda: bk.quantize(W, LA, LB, s, p.bits, ws=ws, out=out)  # noqa: E731
    for _ in range(args.warmup):
        solve_ad()
        solve_bk()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    sampler.start()
    barrier(world, dev)
    ad_ms = aggregate_max(timed(solve_ad, args.steps), world, dev)
    barrier(world, dev)
    clocks = sampler.stop()
    bk_ms = aggregate_max(timed(solve_bk, args.steps), world, dev)
    if out_ad[2].item() != 0 or out[2].item() != 0:
        raise RuntimeError(f"device status {out_ad[2].item()} / {out[2].item()}")
    same = float((out_ad[0] == out[0]).float().mean().item())
    peaks = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    alg = 2.0 * antidiag_macs(m, n) / (ad_ms / args.steps * 1e-3) / 1e12
    peak = alu_peak_tflops(sm_max)
    cfg = workload_config(p, world)
    cfg["method"] = "BaKron-antidiagonal (Algorithm 3), double-float"
    return {
        "metric": "BaKron-antidiagonal solve time & weights quantized/s per m x n layer", "unit": UNIT,
        "value": world * m * n * args.steps / (ad_ms * 1e-3), "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ad_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32x2 double-float", "data": "synthetic", "config": cfg, "clocks": clocks,
        "gpu_launches": (m + n + 1) * args.steps,
        "bakron_ms_per_step": bk_ms / args.steps, "speedup_bakron_over_antidiag": ad_ms / bk_ms,
        "codes_identical_fraction": same,
        "roofline": {"bound": "alu", "kernel": "ad_step", "achieved": alg, "peak": peak, "unit": "TFLOP/s",
                     "frac": alg / peak, "traffic": None, "alg_macs": antidiag_macs(m, n),
                     "peak_basis": f"{SM_COUNT} SMs x {FP32_LANES_PER_SM} fp32 lanes x {sm_max:.0f} MHz / "
                                   f"{DF_INSTR_PER_MAC} instr per double-float MAC x 2 flops"},
        "e2e": None,
    }


def run_ours(args, rank, local_rank, world):
    import ctypes

    import numpy as np
    import torch

    import kronecker_hessian_gptq_gb300 as bk
    from kronecker_hessian_gptq_gb300 import _lib

    lib = bk.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if args.method == "gram":
        return run_gram(args, world, dev)
    p = load_workload(args.config)
    m, n = p.m, p.n
    A, B, W = (torch.from_numpy(x).to(dev) for x in (p.A, p.B, p.W))
    s = None if p.scales is None else torch.from_numpy(p.scales).to(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    torch.cuda.synchronize()
    prep_times = []
    for _ in range(6):  # the first call includes the process's first launches of the factor kernels
        e0, e1 = ev(), ev()
        e0.record()
        LA, LB, info = bk.prepare(A, B)
        e1.record()
        torch.cuda.synchronize()
        prep_times.append(e0.elapsed_time(e1))
    cold_prep_ms, prep_ms = prep_times[0], statistics.median(prep_times[1:])
    if info.abs().sum().item() != 0:
        raise RuntimeError(f"factor preparation reported a non-positive pivot: {info.tolist()}")

    ws = torch.empty(bk.quantize_workspace_size(m, n), dtype=torch.uint8, device=dev)
    out = (torch.empty((m, n), dtype=torch.int32, device=dev), torch.empty((m, n), dtype=torch.float32, device=dev),
           torch.zeros(1, dtype=torch.int32, device=dev))
    flush = torch.empty((512 << 20) // 4, dtype=torch.float32, device=dev)
    if args.method == "scales":
        return run_scales(args, p, W, LA, LB, s, ws, out, flush, world, dev)
    if args.method == "antidiag":
        return run_antidiag(args, p, W, LA, LB, s, ws, out, flush, world, dev)
    if args.method == "gptq":  # row-wise GPTQ: the one-sided case B = I of the same solve
        solve = lambda: bk.gptq(W, LA, s, p.bits, ws=ws, out=out)  # noqa: E731
    elif args.method == "persistent":  # the same solve as one persistent cooperative kernel
        solve = lambda: bk.quantize_persistent(W, LA, LB, s, p.bits, ws=ws, out=out)  # noqa: E731
    else:
        solve = lambda: bk.quantize(W, LA, LB, s, p.bits, ws=ws, out=out)  # noqa: E731
    for _ in range(args.warmup):
        solve()
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    sampler.start()
    barrier(world, dev)
    torch.cuda.synchronize()
    starts, ends = [ev() for _ in range(args.steps)], [ev() for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        starts[k].record()
        solve()
        ends[k].record()
    torch.cuda.synchronize()
    barrier(world, dev)
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    if out[2].item() != 0:
        raise RuntimeError(f"device status {out[2].item()}")
    total_ms = aggregate_max(sum(step_ms), world, dev)
    if args.method == "gptq":
        cfg = workload_config(p, world)
        cfg["method"] = "gptq (B = I)"
        return {
            "metric": "row-wise GPTQ solve time & weights quantized/s per m x n layer", "unit": UNIT,
            "value": world * m * n * args.steps / (total_ms * 1e-3), "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32x2 double-float", "data": "synthetic", "config": cfg,
            "prep_ms": prep_ms, "cold_prep_ms": cold_prep_ms, "clocks": clocks, "roofline": None, "e2e": None,
            "gpu_launches": None,
        }

    if args.method == "persistent":
        cfg = workload_config(p, world)
        cfg["method"] = "persistent sweep (bakron_quantize_persistent)"
        step_s = total_ms / args.steps * 1e-3
        f_alg = float(m) * n * (m + n)
        # the whole solve against the tensor roofline of the precision mode
        # (20 bf16 digit-pair multiply-adds per algorithmic multiply-add)
        roof = roofline_for("sweep", f_alg, step_s * 1e3, measured_peaks())
        roof["traffic"] = None
        return {
            "metric": "persistent BaKron solve time & weights quantized/s per m x n layer", "unit": UNIT,
            "value": world * m * n * args.steps / (total_ms * 1e-3), "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32x2 double-float; bf16 digit products on tensor cores",
            "data": "synthetic", "config": cfg, "solve_alg_tflops": f_alg / step_s / 1e12,
            "us_per_antidiagonal_step": total_ms / args.steps * 1e3 / (m + n - 1), "prep_ms": prep_ms,
            "cold_prep_ms": cold_prep_ms, "clocks": clocks, "roofline": roof, "e2e": None,
            "gpu_launches": SWEEP_LAUNCHES * args.steps,
        }

    # Per-kernel timing pass (events around every launch), after the timed region.
    ncls = len(_lib.KERNEL_CLASSES)
    kms = (ctypes.c_double * ncls)()
    kl = (ctypes.c_int64 * ncls)()
    kf = (ctypes.c_double * ncls)()
    for _ in range(2):
        flush.zero_()
        st = lib.bakron_quantize_profile(W.data_ptr(), LA.data_ptr(), LB.data_ptr(), None if s is None else s.data_ptr(),
                                         p.bits, m, n, out[0].data_ptr(), out[1].data_ptr(), ws.data_ptr(), ws.numel(),
                                         out[2].data_ptr(), torch.cuda.current_stream().cuda_stream, kms, kl, kf)
        _lib.check(st, "bakron_quantize_profile")
    kernels = {name: {"ms": kms[c], "launches": kl[c], "alg_tflops": (kf[c] / (kms[c] * 1e-3) / 1e12) if kms[c] else 0}
               for c, name in enumerate(_lib.KERNEL_CLASSES)}
    dom = max(range(ncls), key=lambda c: kms[c])
    # launch-per-step schedule: the set-up class (one timed span) is the input
    # check, the offset, the two factors' block exponents and, from 2^22 weights
    # on, their packed digits; then every tile solve, mid push and chunk product
    setup_launches = 4 + (2 if m * n >= (1 << 22) else 0)
    launches_per_step = setup_launches * kl[0] + sum(kl[c] for c in range(1, ncls))

    # End to end through the host entry point: pinned host inputs in, codes out.
    Wh = torch.from_numpy(p.W).pin_memory()
    LAh, LBh = LA.cpu().pin_memory(), LB.cpu().pin_memory()
    sh = None if p.scales is None else torch.from_numpy(p.scales).pin_memory()
    hout = (torch.empty((m, n), dtype=torch.int32, pin_memory=True),
            torch.empty((m, n), dtype=torch.float32, pin_memory=True))
    dws = torch.empty(lib.bakron_quantize_host_workspace_size(m, n), dtype=torch.uint8, device=dev)
    bk.quantize_host(Wh, LAh, LBh, sh, p.bits, dev_ws=dws, out=hout)
    barrier(world, dev)
    e2e = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        bk.quantize_host(Wh, LAh, LBh, sh, p.bits, dev_ws=dws, out=hout)
        e2e.append(time.perf_counter() - t0)
    e2e_s = aggregate_max(sum(e2e), world, dev)
    if not np.array_equal(hout[0].numpy(), out[0].cpu().numpy()):
        raise RuntimeError("host entry point disagrees with the device entry point")

    peaks = measured_peaks()
    roof = roofline_for(_lib.KERNEL_CLASSES[dom], kf[dom], kms[dom], peaks)
    roof["traffic"] = profiled_traffic(_lib.KERNEL_CLASSES[dom], p.name.split("_")[0])
    f_alg = float(m) * n * (m + n)
    res = {
        "metric": METRIC, "value": world * m * n * args.steps / (total_ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32x2 double-float; bf16 digit products on tensor cores", "data": "synthetic",
        "config": workload_config(p, world),
        "solve_alg_tflops": f_alg / (total_ms / args.steps * 1e-3) / 1e12,
        # the solve is a chain of m + n - 1 anti-diagonal steps; on small layers the chain sets the time
        "us_per_antidiagonal_step": total_ms / args.steps * 1e3 / (m + n - 1),
        "pages_same_shape": pages_same_shape(m, n, total_ms / args.steps),
        "prep_ms": prep_ms,  # median of 5 warm bakron_prepare calls
        "cold_prep_ms": cold_prep_ms,  # the first call of the process
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clocks,
        "e2e": {"value": world * m * n * args.steps / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": 4 * (m * n + n * n + m * m + (m if p.scales is not None else 0)),
                "d2h_bytes_per_step": 8 * m * n + 4},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle as O

        LA64, LB64 = O.factors_of(p.A, p.B)
        units, secs, equiv = oracle_sample(p, args.cpu_rows, LA64, LB64)
        res["cpu_baseline"] = {"value": equiv / secs, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                               "sample": sample_text(p, args.cpu_rows, secs, units / secs)}
    return res


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="c3", help="c1 .. c5, or rand:MxN for a random layer of that shape")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=2048)
    ap.add_argument("--ref-rows", type=int, default=512)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scale-grid", type=int, default=100, help="shrink factors of --method scales")
    ap.add_argument("--method", default="bakron", choices=["bakron", "persistent", "gptq", "scales", "antidiag", "gram"],
                    help="bakron (default, the headline); persistent: the same solve as one persistent "
                         "cooperative kernel; gptq: row-wise GPTQ, the case B = I; scales: the "
                         "scale search and code packing kernels; antidiag: Algorithm 3 beside BaKron "
                         "(give --config c2 for a short run); gram: Kronecker-factor accumulation")
    args = ap.parse_args(argv)
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist

        if args.impl == "reference":
            if rank != 0:
                return 0
            world = 1
        else:
            import torch

            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    res = run_reference(args, rank, world) if args.impl == "reference" else run_ours(args, rank, local_rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
