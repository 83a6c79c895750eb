#!/usr/bin/env python
"""Per-layer GEMM benchmark of the quantized linear-layer hot path on GB300.

Workload: one CodonFM-5B-shaped transformer layer (hidden 4096, intermediate
16384, micro-batch 31 x sequence 512 = 15872 tokens): four linears x Fprop /
Dgrad / Wgrad = 12 GEMMs, 19.17 TFLOP ("How to Optimize Transformer-Based
Models for Low-Precision Training", sections "モデル設定とトレーニング入力" and
"autocast モードの使用と事前量子化の比較").  Inputs are synthetic and seeded
(X ~ N(0,1), W ~ N(0,0.02^2), dY ~ N(0,1e-3^2), bf16); no dataset, no weights.

One timed step runs, for each recipe (bf16, fp8_delayed, fp8_current, mxfp8,
nvfp4), the layer in autocast mode (both operands quantized before every GEMM)
and then in pre-quantized mode (the 12 GEMMs alone on the operands the
autocast pass produced).  The headline ``value`` is the FP8 CurrentScaling
autocast time per layer; every recipe and mode is in ``per_recipe``.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the layer (the path
has no exchange step on one node's replicas), the timed region is bracketed by
a barrier and the maximum over ranks is reported.
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

METRIC = "ms and TFLOP/s per layer GEMMs (autocast & pre-quantized), % of tensor/HBM peak"
# The pages' per-layer numbers (B300 SXM6 AC, autocast unless noted): context, not targets.
PAGES_MS = {("fp8_delayed", "autocast"): 7.80, ("fp8_current", "autocast"): 9.15, ("mxfp8", "autocast"): 8.98,
            ("fp8_current", "prequant"): 6.81}
HEADLINE = ("fp8_current", "autocast")
RECIPE_DTYPE = {"bf16": "bf16", "fp8_delayed": "fp8", "fp8_current": "fp8", "mxfp8": "fp8", "nvfp4": "fp4"}
PEAK_RATIO = {"bf16": 1.0, "fp8": 2.0, "fp4": 6.0}   # nominal dense ratios to bf16 (2.25 / 4.5 / 13.5 PF)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--recipes", default="bf16,fp8_delayed,fp8_current,mxfp8,nvfp4")
    p.add_argument("--tokens", type=int, default=31 * 512)
    p.add_argument("--hidden", type=int, default=4096)
    p.add_argument("--ffn", type=int, default=16384)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=0,
                   help="steps of the end-to-end run (0: as many as --steps, at least 5)")
    p.add_argument("--schedule-layers", type=int, default=24,
                   help="layers of the DelayedScaling schedule measured eager and as CUDA graphs (0: skip)")
    p.add_argument("--schedule-steps", type=int, default=4)
    p.add_argument("--case", default="", help="time one kernel case instead of the layer (see KERNEL_CASES)")
    p.add_argument("--shape", type=int, nargs="+", default=None, help="rows cols (quantizers) or M N K (GEMMs)")
    p.add_argument("--iters", type=int, default=50, help="--case: timed repetitions (median reported)")
    p.add_argument("--case-warmup", type=int, default=None, help="--case: untimed launches first (10; 1 when --iters 1)")
    p.add_argument("--no-flush", action="store_true", help="--case: do not evict L2 between repetitions")
    p.add_argument("--layer-shapes", action="store_true", help="--case (GEMMs): time all 12 GEMM shapes of the layer")
    return p.parse_args()


# ---- distributed plumbing (replicas) -------------------------------------------------------------

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def reduce_max(value: float, ws: int) -> float:
    """Maximum of a host float over ranks (identity for a single process)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- clocks -----------------------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        self.gpu_index = gpu_index

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu_index)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---- measured peaks ------------------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---- DRAM traffic of the dominant kernel (from a committed ncu summary) ---------------------------

def fp8_gemm_traffic():
    """DRAM bytes per FP8 GEMM launch (mean over the layer's 12 shapes) from the committed ncu
    figures (``profiles/gemm_fp8_dram_traffic_codonfm_layer.json``), else None.

    The figures record the sha256 prefix of the GEMM source they were measured on; a changed
    kernel reports no traffic until it is measured again."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "gemm_fp8_dram_traffic_codonfm_layer.json")
    csrc = os.path.join(ROOT, "nvfp4_precision_transformer_gb300", "csrc")
    try:
        d = json.load(open(prof))
        h = hashlib.sha256()
        for name in ("gemm.cu", "common.cuh"):
            h.update(open(os.path.join(csrc, name), "rb").read())
        if d.get("kernel_source_sha256_prefix") != h.hexdigest()[:16]:
            return None, d.get("algorithmic_bytes_per_launch"), "GEMM source changed since the ncu capture"
        return int(d["traffic_bytes_per_launch"]), int(d["algorithmic_bytes_per_launch"]), d.get("how")
    except (OSError, KeyError, ValueError):
        return None, None, "no ncu traffic figures committed"


# ---- CPU oracle baseline ---------------------------------------------------------------------------
#
# The oracle (numpy, as it stands) on the host cores.  Its quantizers are row-independent
# once the tensor's amax / scale is known, so rows are split over a pool of worker processes
# (started with "spawn": the parent has already used the GPU); the fp64 GEMMs run in the
# parent on the BLAS threads.  Both arms time the same sample: the attention-output linear
# (4096 -> 4096) at SAMPLE_TOKENS tokens under FP8 CurrentScaling autocast (amax, row and col
# copies of X, W and dY; Fprop, Dgrad and Wgrad in fp64).  The per-layer figure is
# extrapolated from it per quantized element and per GEMM flop, and labelled so.

SAMPLE_TOKENS = 1024
_POOL = None


def _pool_init():
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"


def oracle_pool():
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        _POOL = mp.get_context("spawn").Pool(cpu_threads(), initializer=_pool_init)
    return _POOL


def close_pool():
    global _POOL
    if _POOL is not None:
        _POOL.terminate()
        _POOL.join()
        _POOL = None


def _oracle_job(job):
    """One row slab of one oracle quantizer (runs in a pool worker); returns a small checksum."""
    from oracle import quantize as Q
    kind, arr = job[0], job[1]
    if kind == "amax":
        return float(Q.amax(arr))
    if kind == "rht_amax":
        return float(Q.amax(Q.rht16(arr, job[2])))
    if kind == "fp8":
        return int(Q.fp8_cast(arr, job[2], job[3])[:1].sum())
    if kind == "mx":
        return int(Q.mxfp8_quantize(arr)[1][:1].sum())
    if kind == "nv":
        z = Q.rht16(arr, job[3]) if job[3] is not None else arr
        return int(Q.nvfp4_quantize(z, job[2])[1][:1].sum())
    raise ValueError(kind)


def _pmap(kind, arr, *extra):
    """Run one oracle quantizer over ``arr`` [R, C] in row slabs on the pool."""
    import numpy as np
    n = max(1, min(arr.shape[0] // 16, 2 * cpu_threads()))
    bounds = np.linspace(0, arr.shape[0] // 16, n + 1).astype(int) * 16   # whole 16-row groups
    jobs = [(kind, np.ascontiguousarray(arr[a:b]), *extra) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    return oracle_pool().map(_oracle_job, jobs)


def oracle_linear_sample(hidden: int, layer_flops: float, layer_elems: float):
    """FP8 CurrentScaling autocast of the attention-output linear at SAMPLE_TOKENS tokens by the
    oracle.  Returns (ms per layer extrapolated, measured sample seconds, description)."""
    import numpy as np
    from oracle import gemm as OG, quantize as Q, recipes as Rc
    from oracle.formats import bf16_bits_to_f32
    from synthetic import gaussian, bf16_bits
    T = SAMPLE_TOKENS
    x = bf16_bits_to_f32(bf16_bits(gaussian((T, hidden), 1.0, 901)))
    w = bf16_bits_to_f32(bf16_bits(gaussian((hidden, hidden), 0.02, 902)))
    dy = bf16_bits_to_f32(bf16_bits(gaussian((T, hidden), 1e-3, 903)))
    oracle_pool()
    t0 = time.perf_counter()
    deq = {}
    for name, t, fmt in (("x", x, "e4m3"), ("w", w, "e4m3"), ("dy", dy, "e5m2")):
        amax = np.float32(max(_pmap("amax", t)))
        s, si = Rc.current_scale(amax, fmt)
        _pmap("fp8", t, s, fmt)                                   # row copy
        _pmap("fp8", np.ascontiguousarray(t.T), s, fmt)           # col copy
        deq[name] = (s, si, fmt)
    t1 = time.perf_counter()
    # the GEMMs consume the dequantized copies (the casts are repeated here for the operands,
    # outside the timed quantizer region)
    op = {k: Q.fp8_dequant(Q.fp8_cast(v, deq[k][0], deq[k][2]), deq[k][1], deq[k][2])
          for k, v in (("x", x), ("w", w), ("dy", dy))}
    t2 = time.perf_counter()
    OG.gemm(op["x"], op["w"])                 # Fprop  Y  = X W^T
    OG.gemm(op["dy"], op["w"].T)              # Dgrad  dX = dY W
    OG.gemm(op["dy"].T, op["x"].T)            # Wgrad  dW = dY^T X
    t3 = time.perf_counter()
    elems = 2.0 * (x.size + w.size + dy.size)
    flops = 3 * 2.0 * T * hidden * hidden
    ms = 1e3 * ((t1 - t0) / elems * layer_elems + (t3 - t2) / flops * layer_flops)
    desc = (f"oracle FP8-current autocast of the attn-out linear at {T} tokens (X {T}x{hidden}, W {hidden}x{hidden}, "
            f"dY {T}x{hidden}: amax + row + col copies on {cpu_threads()} pool processes, Fprop/Dgrad/Wgrad fp64 on the "
            f"BLAS threads); per-layer value EXTRAPOLATED per quantized element ({layer_elems:.3g}/layer) and per "
            f"GEMM flop ({layer_flops:.3g}/layer)")
    return ms, (t1 - t0) + (t3 - t2), desc, {"quantize_s": round(t1 - t0, 3), "gemm_s": round(t3 - t2, 3),
                                             "gemm_gflops": round(flops / (t3 - t2) / 1e9, 2)}


def oracle_full_quantizers(tokens: int, hidden: int):
    """The oracle's quantizers on one full CodonFM activation X [tokens, hidden] (bf16 N(0,1)):
    FP8 CurrentScaling (amax, row + col), MXFP8 (row + col), NVFP4 (amax + rotated amax, RN
    row, RHT col).  Wall ms on the pool and the algorithmic GB/s the GPU kernels are held to."""
    import numpy as np
    from oracle import quantize as Q, recipes as Rc
    from oracle.formats import bf16_bits_to_f32
    from synthetic import gaussian, bf16_bits, rht_sign_mask
    x = bf16_bits_to_f32(bf16_bits(gaussian((tokens, hidden), 1.0, 904)))
    xt = np.ascontiguousarray(x.T)
    n = x.size
    signs = rht_sign_mask(7)
    oracle_pool()
    out = {}

    def timed(name, fn, bytes_):
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        out[name] = {"ms": round(1e3 * dt, 1), "gbs": round(bytes_ / dt / 1e9, 4)}

    def fp8():
        s, _ = Rc.current_scale(np.float32(max(_pmap("amax", x))), "e4m3")
        _pmap("fp8", x, s, "e4m3")
        _pmap("fp8", xt, s, "e4m3")

    def mx():
        _pmap("mx", x)
        _pmap("mx", xt)

    def nv():
        a = np.float32(max(_pmap("amax", x)))
        ar = np.float32(max(_pmap("rht_amax", xt, signs)))
        _pmap("nv", x, a, None)
        _pmap("nv", xt, ar, signs)

    timed("fp8_current_row_col", fp8, 6 * n)
    timed("mxfp8_row_col", mx, 2 * n + 2 * (n + n / 32))
    timed("nvfp4_row_rn_col_rht", nv, 2 * n + 2 * n + 2 * (n / 2 + n / 16))
    out["tensor"] = f"X [{tokens}, {hidden}] bf16"
    return out


def cpu_threads():
    return os.cpu_count() or 1


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads") or 0) for i in threadpool_info()) or None
    except Exception:
        return os.environ.get("OPENBLAS_NUM_THREADS") or "library default (all cores)"


# ---- reference arm -------------------------------------------------------------------------------

def run_reference(args, ws, rank):
    if rank != 0:
        return
    from nvfp4_precision_transformer_gb300.shapes import LayerConfig, layer_flops, linears
    cfg = LayerConfig(hidden=args.hidden, intermediate=args.ffn, micro_batch=1, seq_len=args.tokens)
    lf = float(layer_flops(cfg))
    elems = 2.0 * sum(cfg.tokens * ki + no * ki + cfg.tokens * no for _, ki, no in linears(cfg))
    est, secs = [], []
    desc, parts = "", {}
    for i in range(args.warmup + args.steps):
        ms, s, desc, parts = oracle_linear_sample(args.hidden, lf, elems)
        if i >= args.warmup:
            est.append(ms)
            secs.append(s)
    v = statistics.median(est)
    sample_ms = 1e3 * statistics.median(secs)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "ms/layer", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sample_ms, 1),
            "step": f"one oracle sample (measured): {desc}", "value_is": "extrapolated from the measured sample",
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args),
            "cpu_baseline": {"value": round(v, 1), "unit": "ms/layer", "cores": cpu_threads(),
                             "blas_threads": blas_threads(), "kind": "oracle", "sample": desc,
                             "sample_seconds": round(sample_ms / 1e3, 3), "extrapolated": True, **parts},
            "e2e": {"value": round(v, 1), "unit": "ms/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(args):
    return {"workload": f"CodonFM-5B layer GEMMs: M={args.tokens} tokens, hidden {args.hidden}, ffn {args.ffn}, "
                        f"12 shapes (QKV/attn-out/MLP-up/MLP-down x Fprop/Dgrad/Wgrad); headline FP8 "
                        f"CurrentScaling HYBRID (E4M3 X/W, E5M2 dY), autocast",
            "tokens": args.tokens, "hidden": args.hidden, "ffn": args.ffn, "recipe": "fp8_current",
            "l2": "inputs larger than L2 (X, W, dY of the layer: ~2.5 GB bf16 per step)",
            "parallelism": "replicas"}


# ---- our arm ---------------------------------------------------------------------------------------

KERNEL_CASES = ("amax", "amax_rht", "amax_rht_only", "fp8_row", "fp8_col", "fp8_both", "fp8_col_dbias", "mxfp8_row",
                "mxfp8_col", "mxfp8_both", "nvfp4_rn_row",
                "nvfp4_rht_col", "nvfp4_sr_row", "nvfp4_sr_rht_col", "nvfp4_2d_both", "nvfp4_2d_row", "nvfp4_2d_col",
                "layernorm_fp8",
                "gemm_bf16", "gemm_fp8", "gemm_mxfp8", "gemm_nvfp4",
                "cublaslt_bf16", "cublaslt_fp8", "cublaslt_mxfp8", "cublaslt_nvfp4")


def run_case(args):
    """One kernel on one shape: ``--case-warmup`` untimed launches, then ``--iters`` launches each
    timed alone with CUDA events, L2 evicted between them by reading a 2x-L2 buffer outside the
    timed events (reading, not writing, so that no dirty lines are written back during the next
    launch), median reported: the per-kernel measurements (and, with ``--iters 1``, the command
    the ncu summaries are taken with)."""
    import torch
    import nvfp4_precision_transformer_gb300 as te
    from synthetic import gaussian, rht_sign_mask
    assert args.case in KERNEL_CASES, f"--case one of {KERNEL_CASES}"
    dev = torch.device("cuda", 0)
    u8 = dict(dtype=torch.uint8, device=dev)
    f1 = lambda v=0.0: torch.full((1,), v, device=dev)
    signs = rht_sign_mask(7)
    if args.case.startswith("cublaslt"):
        # context only: the same operand bytes through torch's cuBLASLt path (torch._scaled_mm /
        # torch.matmul), never on the library's path
        M, N, K = args.shape or (15872, 4096, 16384)
        if args.case == "cublaslt_bf16":
            A, B = gaussian((M, K), 1.0, 1, device=dev), gaussian((N, K), 1.0, 2, device=dev)
            fn = lambda: torch.matmul(A, B.t())
        else:
            one = torch.ones((), device=dev)
            if args.case == "cublaslt_fp8":
                A = torch.randint(0, 120, (M, K), **u8).view(torch.float8_e4m3fn)
                B = torch.randint(0, 120, (N, K), **u8).view(torch.float8_e4m3fn)
                sa, sb = one, one
            elif args.case == "cublaslt_mxfp8":
                A = torch.randint(0, 120, (M, K), **u8).view(torch.float8_e4m3fn)
                B = torch.randint(0, 120, (N, K), **u8).view(torch.float8_e4m3fn)
                sa = torch.full((te.te_scale_bytes(te.E8M0, M, K),), 127, **u8).view(torch.float8_e8m0fnu)
                sb = torch.full((te.te_scale_bytes(te.E8M0, N, K),), 127, **u8).view(torch.float8_e8m0fnu)
            else:
                A = torch.randint(0, 256, (M, K // 2), **u8).view(torch.float4_e2m1fn_x2)
                B = torch.randint(0, 256, (N, K // 2), **u8).view(torch.float4_e2m1fn_x2)
                sa = torch.full((te.te_scale_bytes(te.UE4M3, M, K),), 0x38, **u8).view(torch.float8_e4m3fn)
                sb = torch.full((te.te_scale_bytes(te.UE4M3, N, K),), 0x38, **u8).view(torch.float8_e4m3fn)
            fn = lambda: torch._scaled_mm(A, B.t(), sa, sb, out_dtype=torch.bfloat16)
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    elif args.case.startswith("gemm"):
        M, N, K = args.shape or (15872, 4096, 16384)
        D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        if args.case == "gemm_bf16":
            A, B = gaussian((M, K), 1.0, 1, device=dev), gaussian((N, K), 1.0, 2, device=dev)
            fn = lambda: te.te_gemm_bf16(A, B, D)
        elif args.case == "gemm_fp8":
            A, B = torch.randint(0, 120, (M, K), **u8), torch.randint(0, 120, (N, K), **u8)
            one = f1(1.0)
            fn = lambda: te.te_gemm_fp8(A, te.E4M3, B, te.E4M3, one, one, D)
        elif args.case == "gemm_mxfp8":
            A, B = torch.randint(0, 120, (M, K), **u8), torch.randint(0, 120, (N, K), **u8)
            sA = torch.full((te.te_scale_bytes(te.E8M0, M, K),), 127, **u8)
            sB = torch.full((te.te_scale_bytes(te.E8M0, N, K),), 127, **u8)
            fn = lambda: te.te_gemm_mxfp8(A, sA, B, sB, D)
        else:
            A, B = torch.randint(0, 256, (M, K // 2), **u8), torch.randint(0, 256, (N, K // 2), **u8)
            sA = torch.full((te.te_scale_bytes(te.UE4M3, M, K),), 0x38, **u8)
            sB = torch.full((te.te_scale_bytes(te.UE4M3, N, K),), 0x38, **u8)
            one = f1(1.0)
            fn = lambda: te.te_gemm_nvfp4(A, sA, one, B, sB, one, D)
        work, unit = 2.0 * M * N * K, "TFLOP/s"
    else:
        R, C = args.shape or (15872, 16384)
        x = gaussian((R, C), 1e-3, 3, device=dev)
        amax, amax_r, sinv = f1(), f1(), f1()
        te.te_amax_reduce(x, amax, amax_r, signs)
        n = R * C
        qr, qc = torch.empty(R, C, **u8), torch.empty(C, R, **u8)
        nr, nc = torch.empty(R, C // 2, **u8), torch.empty(C, R // 2, **u8)
        snr = torch.empty(te.te_scale_bytes(te.UE4M3, R, C), **u8)
        snc = torch.empty(te.te_scale_bytes(te.UE4M3, C, R), **u8)
        smr = torch.empty(te.te_scale_bytes(te.E8M0, R, C), **u8)
        smc = torch.empty(te.te_scale_bytes(te.E8M0, C, R), **u8)
        gr, gc = f1(), f1()
        scale = f1(2.0 ** 14)
        RHT, SR, D2 = te.NVFP4_RHT_COL, te.NVFP4_SR, te.NVFP4_2D
        nv = lambda flags, row, col: te.te_quantize_nvfp4(
            x, flags, signs, 7, 3, amax, amax_r, *((nr, snr, gr) if row else (None, None, None)),
            *((nc, snc, gc) if col else (None, None, None)))
        cases = {
            "amax": (lambda: te.te_amax_reduce(x, amax), 2 * n),
            "amax_rht": (lambda: te.te_amax_reduce(x, amax, amax_r, signs), 2 * n),
            "amax_rht_only": (lambda: te.te_amax_reduce(x, None, amax_r, signs), 2 * n),
            "fp8_row": (lambda: te.te_quantize_fp8(x, te.E4M3, scale, 0, qr, None, amax, sinv), 3 * n),
            "fp8_both": (lambda: te.te_quantize_fp8(x, te.E4M3, scale, 0, qr, qc, amax, sinv), 4 * n),
            "fp8_col": (lambda: te.te_quantize_fp8(x, te.E4M3, scale, 0, None, qc, amax, sinv), 3 * n),
            "mxfp8_row": (lambda: te.te_quantize_mxfp8(x, qr, smr), 2 * n + n + n // 32),
            "mxfp8_col": (lambda: te.te_quantize_mxfp8(x, None, None, qc, smc), 2 * n + n + n // 32),
            "mxfp8_both": (lambda: te.te_quantize_mxfp8(x, qr, smr, qc, smc), 2 * n + 2 * (n + n // 32)),
            "nvfp4_rn_row": (lambda: nv(0, True, False), 2 * n + n // 2 + n // 16),
            "nvfp4_rht_col": (lambda: nv(RHT, False, True), 2 * n + n // 2 + n // 16),
            "nvfp4_sr_row": (lambda: nv(SR, True, False), 2 * n + n // 2 + n // 16),
            "nvfp4_sr_rht_col": (lambda: nv(SR | RHT, False, True), 2 * n + n // 2 + n // 16),
            "nvfp4_2d_both": (lambda: nv(D2, True, True), 2 * n + n + n // 8),
            # the one-copy 16 x 16 launches autocast runs on W (Fprop row copy, Dgrad col copy)
            "nvfp4_2d_row": (lambda: nv(D2, True, False), 2 * n + n // 2 + n // 16),
            "nvfp4_2d_col": (lambda: nv(D2, False, True), 2 * n + n // 2 + n // 16),
        }
        if args.case == "fp8_col_dbias":
            db = torch.empty(C, device=dev)
            wsp = torch.empty(te.te_dbias_workspace_bytes(R, C) // 4, device=dev)
            cases["fp8_col_dbias"] = (lambda: te.te_quantize_fp8_dbias(x, te.E5M2, db, wsp, scale=scale, q_col=qc,
                                                                      amax_out=amax, scale_inv_out=sinv), 3 * n)
        if args.case == "layernorm_fp8":
            g, b = torch.ones(C, device=dev), torch.zeros(C, device=dev)
            cases["layernorm_fp8"] = (lambda: te.te_layernorm_fp8(x, g, b, 1e-5, te.E4M3, scale, qr), 3 * n)
        fn, work = cases[args.case]
        unit = "GB/s"
    warm = args.case_warmup if args.case_warmup is not None else (1 if args.iters == 1 else 10)
    for _ in range(max(warm, 1)):
        fn()
    torch.cuda.synchronize()
    flush = None if args.no_flush else torch.zeros(68 << 20, dtype=torch.float32, device=dev)
    if flush is not None:
        flush.sum()
        torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.iters)]
    for e0, e1 in evs:
        if flush is not None:
            flush.sum()        # reads 272 MB > 2 x the 129 MB L2: nothing of the last launch stays cached
        e0.record()
        torch.cuda.nvtx.range_push("timed")     # ncu captures select the timed launches by this range
        fn()
        torch.cuda.nvtx.range_pop()
        e1.record()
    torch.cuda.synchronize()
    assert te.te_get_last_error() == 0
    times = sorted(e0.elapsed_time(e1) for e0, e1 in evs)
    if args.case.startswith("cublaslt"):
        te_launches = "library (cuBLASLt via torch), context only"
    else:
        te_launches = "libte_gb300"
    ms = times[len(times) // 2]
    rate = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"case": args.case, "impl": te_launches, "gemm": getattr(args, "label", None),
                      "shape": list(args.shape) if args.shape else None,
                      "ms": round(ms, 4),
                      "rate": round(rate, 1), "unit": unit,
                      "work": "flops" if unit == "TFLOP/s" else "algorithmic bytes",
                      "timing": {"reps": args.iters, "warmup": max(warm, 1), "stat": "median",
                                 "min_ms": round(times[0], 4), "max_ms": round(times[-1], 4),
                                 "l2": "evicted between reps" if flush is not None else "not evicted"}}), flush=True)


PER_GEMM_FIELDS = ["recipe", "mode", "linear", "pass", "M", "N", "K", "ms", "tflops", "frac_of_peak"]


def per_gemm_table(per_g, pk):
    """One row per (recipe, mode, linear, pass): mean CUDA-event ms of that GEMM launch over the
    timed steps, its TFLOP/s and the fraction of the recipe's tensor peak (measured bf16
    sustained x the nominal dtype ratio).  Rows as lists under ``fields``."""
    rows = []
    for (r, m, lname, p, M, N, K), ts in per_g.items():
        ms = statistics.mean(ts)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        peak = pk["bf16_tflops_sustained"] * PEAK_RATIO[RECIPE_DTYPE[r]]
        rows.append([r, m, lname, p, M, N, K, round(ms, 4), round(tf, 1), round(tf / peak, 4)])
    return {"fields": PER_GEMM_FIELDS, "rows": rows,
            "timing": "CUDA events around each GEMM launch inside the timed steps (quantizers excluded), mean"}


def roofline_by_kind(agg, pk):
    """Tensor roofline of each GEMM kind over its pre-quantized layer GEMMs in the step (BF16: its
    autocast run, which has no quantizers): achieved TFLOP/s from the per-GEMM CUDA events against
    the measured sustained bf16 peak times the nominal dtype ratio."""
    out = {}
    for (r, m), d in agg.items():
        if m != ("autocast" if r == "bf16" else "prequant") or d["gemm_ms"] <= 0:
            continue
        tf = d["gemm_flops"] / (d["gemm_ms"] * 1e-3) / 1e12
        peak = pk["bf16_tflops_sustained"] * PEAK_RATIO[RECIPE_DTYPE[r]]
        out[r] = {"bound": "tensor", "achieved": round(tf, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                  "frac": round(tf / peak, 4)}
    return out


def nvfp4_over_bf16(per):
    """The pages' NVFP4-over-BF16 speed-ups: autocast (quantizers included) and kernel-only
    (pre-quantized NVFP4 GEMMs against the BF16 GEMMs)."""
    b = per.get("bf16/autocast")
    na, npq = per.get("nvfp4/autocast"), per.get("nvfp4/prequant")
    if not b or not na or not npq:
        return None
    return {"autocast": round(b["ms_per_layer"] / na["ms_per_layer"], 3),
            "prequant_kernel_only": round(b["gemm_ms_per_layer"] / npq["gemm_ms_per_layer"], 3),
            "pages_b300": {"autocast": 1.98, "prequant_kernel_only": 3.48}}


def main():
    args = parse()
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        try:
            run_reference(args, ws, rank)
        finally:
            close_pool()
        return
    if args.case:
        if args.layer_shapes:
            # every GEMM shape of the layer, one JSON line each (GEMM cases only)
            from nvfp4_precision_transformer_gb300.shapes import LayerConfig, layer_gemms
            cfg = LayerConfig(hidden=args.hidden, intermediate=args.ffn, micro_batch=1, seq_len=args.tokens)
            for g in layer_gemms(cfg):
                args.shape = [g.M, g.N, g.K]
                args.label = f"{g.linear}/{g.pass_}"
                run_case(args)
        else:
            run_case(args)
        return

    import torch
    import nvfp4_precision_transformer_gb300 as te
    from nvfp4_precision_transformer_gb300.linear import Layer
    from nvfp4_precision_transformer_gb300.shapes import LayerConfig, layer_flops, linears
    from synthetic import gaussian, rht_sign_mask, seed_for

    assert torch.cuda.is_available(), "bench.py needs a GPU"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    recipes = [r for r in args.recipes.split(",") if r]
    cfg = LayerConfig(hidden=args.hidden, intermediate=args.ffn, micro_batch=1, seq_len=args.tokens)
    lf = float(layer_flops(cfg))

    tensors = []
    for i, (_, k_in, n_out) in enumerate(linears(cfg)):
        x = gaussian((cfg.tokens, k_in), 1.0, seed_for(2, i, 0) + 97 * rank, device=dev)
        w = gaussian((n_out, k_in), 0.02, seed_for(2, i, 1), device=dev)
        dy = gaussian((cfg.tokens, n_out), 1e-3, seed_for(2, i, 2) + 97 * rank, device=dev)
        b = gaussian((n_out,), 0.02, seed_for(2, i, 3), dtype=torch.float32, device=dev)
        tensors.append((x, w, dy, b))
    layer = Layer(tensors, recipes, history_len=16, rht_signs=rht_sign_mask(7), sr_seed=1234, device=dev)

    modes = []
    for r in recipes:
        modes.append((r, "autocast"))
        if r != "bf16":
            modes.append((r, "prequant"))

    def one_step(rec):
        for r, m in modes:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            gemms = []

            def on_gemm(lin, p, phase, _g=gemms):
                ev = torch.cuda.Event(enable_timing=True)
                ev.record()
                if phase == 0:
                    _g.append([lin.gemm_shape(p), ev, None, (lin.name, p)])
                else:
                    _g[-1][2] = ev
            e0.record()
            layer.run(r, autocast=(m == "autocast"), on_gemm=on_gemm if rec is not None else None)
            e1.record()
            if rec is not None:
                rec.append((r, m, e0, e1, gemms))
        layer.step_idx += 1

    for _ in range(args.warmup):
        one_step(None)
    torch.cuda.synchronize()
    barrier(ws)

    records = []
    launches0 = te.te_launch_count()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier(ws)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record()
        for _ in range(args.steps):
            one_step(records)
        t_end.record()
        torch.cuda.synchronize()
        barrier(ws)
    launches = te.te_launch_count() - launches0
    assert te.te_get_last_error() == 0, "device error during the timed region"
    total_ms = reduce_max(t_start.elapsed_time(t_end), ws)
    clocks = clk.summary()

    # per recipe / mode aggregation, and per GEMM (recipe, mode, linear, pass)
    pk = peaks()
    agg = {}
    per_g = {}
    for r, m, e0, e1, gemms in records:
        d = agg.setdefault((r, m), {"seg": [], "gemm_ms": 0.0, "gemm_flops": 0.0})
        d["seg"].append(e0.elapsed_time(e1))
        for (M, N, K), g0, g1, (lname, p) in gemms:
            t = g0.elapsed_time(g1)
            d["gemm_ms"] += t
            d["gemm_flops"] += 2.0 * M * N * K
            per_g.setdefault((r, m, lname, p, M, N, K), []).append(t)
    per = {}
    for (r, m), d in agg.items():
        ms = statistics.mean(d["seg"])
        peak = pk["bf16_tflops_sustained"] * PEAK_RATIO[RECIPE_DTYPE[r]]
        gemm_tflops = d["gemm_flops"] / (d["gemm_ms"] * 1e-3) / 1e12
        per[f"{r}/{m}"] = {"ms_per_layer": round(ms, 4), "tflops": round(lf / (ms * 1e-3) / 1e12, 1),
                           "frac_of_peak": round(lf / (ms * 1e-3) / 1e12 / peak, 4),
                           "gemm_ms_per_layer": round(d["gemm_ms"] / args.steps, 4),
                           "gemm_tflops": round(gemm_tflops, 1), "gemm_frac_of_peak": round(gemm_tflops / peak, 4),
                           "peak_tflops": round(peak, 1),
                           "pages_ms_b300": PAGES_MS.get((r, m))}
    per_gemm = per_gemm_table(per_g, pk)
    ratios = nvfp4_over_bf16(per)
    head = per.get(f"{HEADLINE[0]}/{HEADLINE[1]}") or next(iter(per.values()))
    head_ms = reduce_max(head["ms_per_layer"], ws)     # per replica: the slowest rank's ms per layer
    # dominant kernel of the headline: the FP8 GEMM
    hd = agg.get(HEADLINE) or next(iter(agg.values()))
    fp8_peak = pk["bf16_tflops_sustained"] * PEAK_RATIO["fp8"]
    achieved = hd["gemm_flops"] / (hd["gemm_ms"] * 1e-3) / 1e12
    traffic, alg_bytes, traffic_note = fp8_gemm_traffic()
    roofline = {"kernel": "gemm_kernel<FP8> (tcgen05 kind::f8f6f4)", "bound": "tensor", "achieved": round(achieved, 1),
                "peak": round(fp8_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                "traffic": traffic, "algorithmic_bytes": alg_bytes, "traffic_note": traffic_note,
                "flops_per_launch": round(hd["gemm_flops"] / (12 * args.steps)),
                "peak_note": f"{pk['source']} bf16 sustained {pk['bf16_tflops_sustained']} x 2 (nominal FP8/BF16 ratio)",
                "launches_per_layer": 12}
    line = {"metric": METRIC, "value": round(head_ms, 4), "unit": "ms/layer", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": round(head_ms / PAGES_MS[HEADLINE], 4), "dtype": "fp8",
            "data": "synthetic", "config": workload_config(args), "per_recipe": per, "per_gemm": per_gemm,
            "nvfp4_over_bf16": ratios, "roofline": roofline, "roofline_by_kind": roofline_by_kind(agg, pk),
            "gpu_launches": int(launches), "clocks": clocks,
            "aggregate": {"layers_per_s": round(ws * 1e3 / head_ms, 3), "replicas": ws,
                          "note": "value is ms per layer of one replica (max over ranks); replicas run in parallel"}}

    # end to end through the C ABI from pinned host buffers (headline recipe)
    if not args.no_e2e and HEADLINE[0] in recipes:
        line["e2e"] = run_e2e(layer, args, ws)
    if args.schedule_layers > 0:
        del layer, tensors
        torch.cuda.empty_cache()
        line["schedule"] = run_schedule(args, cfg, dev, rank, ws)
    if rank == 0 and not args.no_cpu:
        elems = 2.0 * sum(cfg.tokens * ki + no * ki + cfg.tokens * no for _, ki, no in linears(cfg))
        ms, secs, desc, parts = oracle_linear_sample(args.hidden, lf, elems)
        line["cpu_baseline"] = {"value": round(ms, 1), "unit": "ms/layer", "cores": cpu_threads(),
                                "blas_threads": blas_threads(), "kind": "oracle", "sample": desc,
                                "sample_seconds": round(secs, 3), "extrapolated": True, **parts,
                                "full_tensor_quantizers": oracle_full_quantizers(cfg.tokens, args.hidden)}
    close_pool()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_schedule(args, cfg, dev, rank, ws):
    """The 24-layer step under FP8 DelayedScaling (each tensor quantized once per step into
    both copies, batched scale updates; X Student-t(3) with 0.1 % outliers x100, distinct
    W per layer), timed eager and replayed as CUDA graphs (one per history slot)."""
    import torch
    from nvfp4_precision_transformer_gb300.linear import ScheduleGraphs, ScheduleStep
    from nvfp4_precision_transformer_gb300.shapes import linears
    from synthetic import gaussian, seed_for, student_t_outliers
    import nvfp4_precision_transformer_gb300 as te
    layers = []
    for l in range(args.schedule_layers):
        lin = []
        for i, (_, k_in, n_out) in enumerate(linears(cfg)):
            s = seed_for(5, 100 * l + i, 0) + 97 * rank
            lin.append((student_t_outliers((cfg.tokens, k_in), s, device=dev),
                        gaussian((n_out, k_in), 0.02, s + 1, device=dev),
                        gaussian((cfg.tokens, n_out), 1e-3, s + 2, device=dev),
                        gaussian((n_out,), 0.02, s + 3, dtype=torch.float32, device=dev)))
        layers.append(lin)
    sched = ScheduleStep(layers, history_len=16, device=dev)
    flops = sched.gemm_flops()

    def timed(run, first):
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0 = te.te_launch_count()
        e0.record()
        for t in range(first, first + args.schedule_steps):
            run(t)
        e1.record()
        torch.cuda.synchronize()
        return reduce_max(e0.elapsed_time(e1), ws) / args.schedule_steps, te.te_launch_count() - n0

    for t in range(2):
        sched.run(t)
    eager_ms, eager_launches = timed(sched.run, 2)
    graphs = ScheduleGraphs(sched)
    graphs.run(2 + args.schedule_steps)
    graph_ms, _ = timed(graphs.run, 3 + args.schedule_steps)
    del graphs
    # the same step with the long amax history (NeMo's fp8_amax_history_len 1024): eager, the
    # per-slot graphs would be 1024 captures
    long_h = ScheduleStep(layers, history_len=1024, device=dev)
    for t in range(2):
        long_h.run(t)
    long_ms, _ = timed(long_h.run, 2)
    del long_h
    # the BF16 GEMM path on the same tensors, alongside
    bf = ScheduleStep(layers, device=dev, recipe="bf16")
    bf.run(0)
    bf_ms, _ = timed(bf.run, 1)
    del bf
    assert te.te_get_last_error() == 0, "device error in the schedule"
    L = args.schedule_layers
    out = {"layers": L, "recipe": "fp8_delayed (each tensor quantized once per step, both copies)",
           "history_len": 16, "steps": args.schedule_steps,
           "eager_ms_per_step": round(eager_ms, 3), "graph_ms_per_step": round(graph_ms, 3),
           "eager_ms_per_layer": round(eager_ms / L, 4),
           "graph_ms_per_layer": round(graph_ms / L, 4),
           "gemm_tflops_graph": round(flops / (graph_ms * 1e-3) / 1e12, 1),
           "launches_per_step": int(eager_launches // args.schedule_steps),
           "history_len_1024": {"eager_ms_per_step": round(long_ms, 3), "eager_ms_per_layer": round(long_ms / L, 4)},
           "bf16": {"eager_ms_per_step": round(bf_ms, 3), "eager_ms_per_layer": round(bf_ms / L, 4),
                    "gemm_tflops": round(flops / (bf_ms * 1e-3) / 1e12, 1),
                    "fp8_delayed_speedup_graph": round(bf_ms / graph_ms, 3)}}
    del sched, layers
    torch.cuda.empty_cache()
    return out


def e2e_steps(args) -> int:
    """Steps of the end-to-end run: ``--e2e-steps`` when given, else as many as the device-timed
    region (at least 5). The copies of consecutive steps overlap as in a training loop, so the
    pipeline's fill (the first inputs alone on the link) and drain (the last outputs alone) are
    spread over the same K steps as the bench line's other figures."""
    return args.e2e_steps if args.e2e_steps > 0 else max(5, args.steps)


def run_e2e(layer, args, ws):
    """The headline recipe end to end: every step copies the layer's inputs from pinned host
    memory, runs it, and copies its outputs back (``HostStreamedLayer``: each linear's input
    and output copies overlap its neighbours' compute)."""
    import torch
    from nvfp4_precision_transformer_gb300.linear import HostStreamedLayer
    lins = layer.linears
    host_in = [(l.x.cpu().pin_memory(), l.w.cpu().pin_memory(), l.dy.cpu().pin_memory(),
                l.bias.cpu().pin_memory()) for l in lins]
    host_out = [(torch.empty_like(l.y, device="cpu").pin_memory(), torch.empty_like(l.dx, device="cpu").pin_memory(),
                 torch.empty_like(l.dw, device="cpu").pin_memory()) for l in lins]
    h2d = sum(t.numel() * t.element_size() for tup in host_in for t in tup)
    d2h = sum(t.numel() * t.element_size() for tup in host_out for t in tup)
    hs = HostStreamedLayer(layer, host_in, host_out)
    link = host_link(host_in, host_out, lins)
    for _ in range(2):
        hs.step(HEADLINE[0])
    torch.cuda.synchronize()
    barrier(ws)
    main_s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main_s)
    for s in hs.streams():
        s.wait_event(e0)
    steps = e2e_steps(args)
    for _ in range(steps):
        hs.step(HEADLINE[0])
    for s in hs.streams():
        main_s.wait_stream(s)
    e1.record(main_s)
    torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1), ws) / steps      # per replica (max over ranks)
    link["bound_ms_per_layer"] = round(1e3 * max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                                                 (h2d + d2h) / (link["both_gbs"] * 1e9)), 3)
    return {"value": round(ms, 4), "unit": "ms/layer", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "recipe": HEADLINE[0], "steps": steps,
            "overlap": "per-linear input / output copies on their own streams overlap the compute",
            "host_link": link}


def host_link(host_in, host_out, lins):
    """This box's pinned host <-> device bandwidth, measured before the end-to-end run: the largest
    input copied in, the largest output copied out, then both at once on two streams (the
    end-to-end figure cannot beat the layer's bytes at these rates)."""
    import torch
    src = max((t for tup in host_in for t in tup), key=lambda t: t.numel() * t.element_size())
    out_dev = max((t for l in lins for t in (l.y, l.dx, l.dw)), key=lambda t: t.numel() * t.element_size())
    dst_dev = torch.empty_like(src, device=out_dev.device)
    dst_host = torch.empty_like(out_dev, device="cpu").pin_memory()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn, reps=3):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) * 1e-3
            best = t if best is None else min(best, t)
        return best

    bi, bo = src.numel() * src.element_size(), out_dev.numel() * out_dev.element_size()
    t_in = timed(lambda: dst_dev.copy_(src, non_blocking=True))
    t_out = timed(lambda: dst_host.copy_(out_dev, non_blocking=True))

    def both():
        cur = torch.cuda.current_stream()
        s1.wait_stream(cur)
        s2.wait_stream(cur)
        with torch.cuda.stream(s1):
            dst_dev.copy_(src, non_blocking=True)
        with torch.cuda.stream(s2):
            dst_host.copy_(out_dev, non_blocking=True)
        cur.wait_stream(s1)
        cur.wait_stream(s2)
    t_both = timed(both)
    del dst_dev, dst_host
    return {"h2d_gbs": round(bi / t_in / 1e9, 1), "d2h_gbs": round(bo / t_out / 1e9, 1),
            "both_gbs": round((bi + bo) / t_both / 1e9, 1)}


if __name__ == "__main__":
    main()
