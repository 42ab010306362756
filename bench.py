#!/usr/bin/env python
"""Benchmark of the QLoRA linear hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama33b|llama7b]

Workload (one step, the default): the LLaMA-33B-shaped stack, 60 layers x 7
QLoRA linears (q/k/v/o 6656x6656, gate/up 17920x6656, down 6656x17920) with
NF4 + double-quant weights (16.6 GB, all resident) and a rank-64 LoRA adapter
(alpha 16) on every linear, M = 2048 tokens: the forward of all 420 linears
in order, then the backward of all 420 in reverse order, through the
library's C ABI.  Every linear has its own seeded synthetic X and dY (bf16,
N(0, 1)); weights are N(0, 0.015^2) bf16 drawn on the device and quantized
once before timing, as in QLoRA finetuning where the frozen 4-bit weights are
stored once.  `--workload llama7b` times the 7 LLaMA-7B linears at M = 4096
instead (also reported as a sub-result of the default run).

The metric is algorithmic TFLOP/s: 4MNK + 6Mr(N+K) per linear per step.
One JSON line is printed by rank 0.  Extra keys: `roofline` of the dominant
kernel (the tensor-core dequant GEMM, timed inside the timed steps by its own
first-CTA-start / last-CTA-end %globaltimer stamps), `cpu_baseline` (the CPU
oracle on a bounded sample), `e2e` (the same metric with host buffers and
host<->device copies inside the timed region), `clocks`, `gpu_launches`, and
sub-results for the LLaMA-7B linears, the decode GEMV and the quantizer.

With N > 1 ranks (torchrun) the run is data parallel: every rank holds the
same weights and processes its own 2048 tokens (weak scaling), and after
each linear's backward the adapter gradients dA, dB are summed over the
ranks (an NCCL all-reduce on a side stream).

`--impl reference` times the CPU oracle (the plain fp64 restatement of the
method, the only reference this subject has) on the same config with a
bounded sample per step.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "QLoRA linear fwd+bwd TFLOP/s and decode GB/s, % of B300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["llama33b", "llama7b"], default="llama33b",
                   help="the timed step: the 60x7 LLaMA-33B stack (default) or the 7 LLaMA-7B linears")
    p.add_argument("--layers", type=int, default=60, help="layers of the 33B stack (profiling runs only)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-extras", action="store_true", help="skip the decode and quantizer sub-results")
    p.add_argument("--linears", default="", help="comma-separated subset of the 7 linears (profiling runs)")
    p.add_argument("--only", choices=["all", "decode", "quantize", "single", "fp8"], default="all",
                   help="run only one sub-benchmark (profiling runs)")
    p.add_argument("--decode-m", default="1,4,16", help="decode token counts")
    p.add_argument("--decode-shapes", default="0,1,2", help="indices of the LLaMA-13B decode shapes")
    p.add_argument("--decode-calls", type=int, default=240)
    return p.parse_args()


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def ncu_traffic(kernel, src_files):
    """DRAM bytes per launch of `kernel` from the ncu capture recorded in
    profiles/ncu_traffic.json, if it was taken on the current kernel source
    (sha256 over `src_files`), else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    h = hashlib.sha256()
    for f in src_files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid):
        self.samples = []
        self.proc = None
        self.uuid = gpu_uuid

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for t, s in self.samples if t0 - 0.06 <= t <= t1 + 0.06]
        if not rows and self.samples:
            rows = [min(self.samples, key=lambda ts: abs(ts[0] - t1))[1]]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample_setup(workload="llama33b", M_sample=512):
    """The workload's first linear (q_proj: 6656x6656 for the 33B stack,
    4096x4096 for the 7B linears) quantized by the oracle, with M_sample tokens."""
    from bit_nf4_quantized_38_b300.workloads import bf16_bits, case_inputs, case_weight, llama33b_stack, \
        llama7b_linears
    from oracle import nf4
    case = (llama7b_linears() if workload == "llama7b" else llama33b_stack(layers=1)).cases[0]
    W = case_weight(case)
    X, A, B, dY = case_inputs(case, M=M_sample)
    qt = nf4.quantize(bf16_bits(W))
    return dict(case=case, qt=qt, X=bf16_bits(X), A=bf16_bits(A), B=bf16_bits(B), dY=bf16_bits(dY),
                M=M_sample, workload=workload)


def oracle_sample_step(s):
    """One oracle step on the sample: dequantize, forward, backward (fp64 numpy)."""
    from oracle import linear, nf4
    Wh = nf4.dequantize(s["qt"])
    linear.lora_forward(s["X"], Wh, s["A"], s["B"], s["case"].scale)
    linear.lora_backward(s["dY"], s["X"], Wh, s["A"], s["B"], s["case"].scale)


def oracle_sample_flops(s):
    c = s["case"]
    return 4 * s["M"] * c.N * c.K + 6 * s["M"] * c.r * (c.N + c.K)


def oracle_sample_text(s):
    c = s["case"]
    return (f"{c.name} {c.N}x{c.K} linear of the workload, {s['M']} tokens, r={c.r}: NF4+DQ dequantize + fwd + "
            f"bwd in fp64 numpy")


def cpu_oracle_details(s, workload_flops_step):
    """Bounded samples of the other workloads, timed once each on the host's
    cores with the same oracle: the single 1024 x 1024 linear in full; the
    training sample on one BLAS thread; 512 rows of the 5120 x 5120 decode
    layer (dequantize + forward, M = 1); 512 rows of an 8192-wide LLaMA-65B
    weight (quantize, then dequantize).  Rates use the algorithmic bytes or
    flops of the sample itself; the time of a whole step of the workload at
    the sample's rate is given as an extrapolation."""
    from bit_nf4_quantized_38_b300.workloads import (bf16_bits, case_inputs, case_weight, llama13b_decode,
                                                     single_linear_1024, student_t4_bf16)
    from oracle import linear, nf4
    out = {"host_cores": cpu_cores(), "blas_threads": blas_threads()}
    # the single linear (quantize + dequantize + fwd + bwd), in full
    c = single_linear_1024().cases[0]
    W = bf16_bits(case_weight(c))
    X, A, B, dY = (bf16_bits(t) for t in case_inputs(c))
    t0 = time.perf_counter()
    Wh = nf4.dequantize(nf4.quantize(W))
    linear.lora_forward(X, Wh, A, B, c.scale)
    linear.lora_backward(dY, X, Wh, A, B, c.scale)
    out["single_linear_1024_us"] = (time.perf_counter() - t0) * 1e6
    # the training sample on one thread: a child process started with the
    # BLAS thread counts set to 1 (they are fixed when numpy loads)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys, time, json; sys.path.insert(0, %r); import bench; s = bench.oracle_sample_setup(%r); "
            "t0 = time.perf_counter(); bench.oracle_sample_step(s); dt = time.perf_counter() - t0; "
            "print(json.dumps(bench.oracle_sample_flops(s) / dt / 1e12))"
            % (os.path.dirname(os.path.abspath(__file__)), s["workload"]))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        out["training_sample_1thread_tflops"] = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # the all-core figures above and below stand on their own
        out["training_sample_1thread_tflops"] = None
        out["one_thread_error"] = f"{type(e).__name__}: {e}"[:200]
    # decode: 512 of the 5120 rows of the 13B 5120 x 5120 layer, M = 1
    c = llama13b_decode(M=1).cases[0]
    rows = 512
    W = bf16_bits(case_weight(c))[:rows]
    X, A, B, _ = (bf16_bits(t) for t in case_inputs(c))
    qt = nf4.quantize(W)
    t0 = time.perf_counter()
    linear.lora_forward(X, nf4.dequantize(qt), A, B[:, :rows], c.scale)
    dt = time.perf_counter() - t0
    n_b = rows * c.K // 64
    byts = rows * c.K // 2 + n_b + 4 * ((n_b + 255) // 256) + 2 * c.r * (c.K + rows) + 2 * (c.K + rows)
    out["llama13b_decode_sample_gbs"] = byts / dt / 1e9
    # quantize / dequantize: 512 rows of an 8192-wide Student-t(4) weight
    W = bf16_bits(student_t4_bf16((512, 8192), 0.015, 300, "cpu"))
    n = W.size
    t0 = time.perf_counter()
    qt = nf4.quantize(W)
    t1 = time.perf_counter()
    nf4.dequantize(qt)
    t2 = time.perf_counter()
    byts = n * (2 + 0.5 + 1 / 64 + 4 / (64 * 256))
    out["llama65b_quantize_sample_gbs"] = byts / (t1 - t0) / 1e9
    out["llama65b_dequantize_sample_gbs"] = byts / (t2 - t1) / 1e9
    out["samples"] = ("single linear 1024x1024 M=16 r=8 in full; the training sample on 1 BLAS thread; "
                      "512 of 5120 rows of the 13B 5120x5120 decode layer (M=1, dequantize + fwd); "
                      "512 x 8192 Student-t(4) weight (quantize, dequantize)")
    return out


def cpu_baseline(workload, workload_flops_step, repeats=3):
    s = oracle_sample_setup(workload)
    oracle_sample_step(s)  # warm
    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle_sample_step(s)
    dt = (time.perf_counter() - t0) / repeats
    rate = oracle_sample_flops(s) / dt / 1e12
    return {"value": rate, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{oracle_sample_text(s)}, mean of {repeats} runs ({dt:.2f} s each)",
            "extrapolated_s_per_step": workload_flops_step / (rate * 1e12),
            "extrapolation": "one step of the whole workload at the sample's rate (extrapolated, not run)",
            "details": cpu_oracle_details(s, workload_flops_step)}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else cpu_cores()
    except Exception:
        return cpu_cores()


# ----------------------------------------------------------------------------- ranks (N > 1: replicas)

def rank_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks_of(x, world, device):
    """The largest of the ranks' values of x (each rank passes its own)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_rank_step, ms_per_step):
    """Whole-job rate: every rank does the same step (weak scaling), timed by the slowest."""
    return world * flops_per_rank_step / (ms_per_step / 1e3) / 1e12


def workload_of(name, layers=60):
    from bit_nf4_quantized_38_b300.workloads import llama33b_stack, llama7b_linears
    return llama7b_linears() if name == "llama7b" else llama33b_stack(layers=layers)


def step_flops(wl):
    return sum(4 * c.M * c.N * c.K + 6 * c.M * c.r * (c.N + c.K) for c in wl.cases)


def config_of(wl, world):
    c0 = wl.cases[0]
    shapes = []
    for c in wl.cases:
        name = c.name.split(".")[-1]
        if (name, c.N, c.K) not in shapes:
            shapes.append((name, c.N, c.K))
    return {"workload": wl.name, "layers": wl.layers, "linears_per_layer": [f"{n} {N}x{K}" for n, N, K in shapes],
            "M": c0.M, "r": c0.r, "alpha": c0.alpha, "quant": "NF4 block 64 + double quant block 256",
            "step": f"fwd of {len(wl.cases)} linears in order, then bwd in reverse",
            "l2": "inputs larger than L2 (each linear has its own weight and activations; one step touches "
                  f"{'~80' if wl.layers > 1 else '~0.7'} GB)",
            "parallelism": f"data parallel x{world} (own tokens per rank, dA/dB all-reduced)" if world > 1
            else "single GPU"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = oracle_sample_setup(args.workload)
    for _ in range(args.warmup):
        oracle_sample_step(s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(s)
    dt = (time.perf_counter() - t0) / args.steps
    v = oracle_sample_flops(s) / dt / 1e12
    wl = workload_of(args.workload, args.layers)
    cfg = config_of(wl, 1)
    cfg["sample_per_step"] = oracle_sample_text(s)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": "per step: " + oracle_sample_text(s)},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ----------------------------------------------------------------------------- sub-benchmarks

def clone_nf4(ql, q):
    import torch
    t = ql.NF4Tensor(q.rows, q.cols, q.packed.clone(), blocksize=q.blocksize, dq_blocksize=q.dq_blocksize,
                     quant_type=q.quant_type, dq_type=q.dq_type)
    for f in ("absmax", "absmax_code", "dq_step", "dq_mean"):
        v = getattr(q, f)
        setattr(t, f, None if v is None else v.clone())
    return t


def bench_decode(ql, dev, hbm_gbs, calls=240, Ms=(1, 4, 16), shapes=(0, 1, 2)):
    """LLaMA-13B decode shapes, M in {1, 4, 16}, r = 64: a CUDA graph of `calls`
    forward calls cycling over weight copies that together exceed 3x L2."""
    import torch
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight, llama13b_decode
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = []
    for M in Ms:
        for c in [llama13b_decode(M=M).cases[i] for i in shapes]:
            W = case_weight(c, device=dev)
            q0 = ql.nf4_quantize(W)
            del W
            copies = max(2, math.ceil(3 * l2 / q0.nbytes()))
            qs = [q0] + [clone_nf4(ql, q0) for _ in range(copies - 1)]
            X, A, B, _ = (t.to(dev) for t in case_inputs(c))
            Y = torch.empty(M, c.N, dtype=torch.bfloat16, device=dev)
            XA = torch.empty(M, c.r, dtype=torch.bfloat16, device=dev)
            ws = torch.empty(ql.workspace_size(ql.OP_LINEAR_FWD, M, c.N, c.K, c.r), dtype=torch.uint8, device=dev)
            for q in qs:
                ql.qlora_linear_fwd(X, q, A, B, c.scale, Y=Y, XA=XA, ws=ws)
            torch.cuda.synchronize()
            n = copies * max(1, calls // copies)
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for i in range(n):
                        ql.qlora_linear_fwd(X, qs[i % copies], A, B, c.scale, Y=Y, XA=XA, ws=ws)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 5
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (reps * n)
            n_b = c.N * c.K // 64
            alg = c.N * c.K // 2 + n_b + 4 * ((n_b + 255) // 256) + 4 + 2 * c.r * (c.K + c.N) + 2 * M * (c.K + c.N)
            gbs = alg / (us * 1e-6) / 1e9
            out.append({"shape": f"{c.N}x{c.K}", "M": M, "us_per_call": us, "bytes": alg, "GB/s": gbs,
                        "frac_hbm": gbs / hbm_gbs, "weight_copies": copies})
            del qs, q0
            torch.cuda.empty_cache()
    return out


def bench_single_linear(ql, dev, iters=200):
    """The small 1024 x 1024 linear (16 tokens, r = 8): latency of quantize,
    forward and backward, each timed over `iters` back-to-back calls from the
    host (launch overhead included; a latency case, no roofline claim)."""
    import torch
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight, single_linear_1024
    c = single_linear_1024().cases[0]
    W = case_weight(c).to(dev)
    X, A, B, dY = (t.to(dev) for t in case_inputs(c))
    q = ql.nf4_quantize(W)
    Y, XA = ql.qlora_linear_fwd(X, q, A, B, c.scale)
    dX, dA, dB = ql.qlora_linear_bwd(dY, X, XA, q, A, B, c.scale)
    wsq = torch.empty(ql.workspace_size(ql.OP_QUANTIZE, 0, c.N, c.K, 0), dtype=torch.uint8, device=dev)
    wsf = torch.empty(ql.workspace_size(ql.OP_LINEAR_FWD, c.M, c.N, c.K, c.r), dtype=torch.uint8, device=dev)
    wsb = torch.empty(ql.workspace_size(ql.OP_LINEAR_BWD, c.M, c.N, c.K, c.r), dtype=torch.uint8, device=dev)
    calls = {
        "quantize": lambda: ql.nf4_quantize(W, out=q, ws=wsq),
        "fwd": lambda: ql.qlora_linear_fwd(X, q, A, B, c.scale, Y=Y, XA=XA, ws=wsf),
        "bwd": lambda: ql.qlora_linear_bwd(dY, X, XA, q, A, B, c.scale, dX=dX, dA=dA, dB=dB, ws=wsb),
    }
    out = {"workload": "single linear 1024x1024, M=16, r=8, alpha=16", "iters": iters}
    for name, fn in calls.items():
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            fn()
        e1.record()
        torch.cuda.synchronize()
        out[f"us_{name}"] = e0.elapsed_time(e1) * 1e3 / iters
    out["us_total"] = out["us_quantize"] + out["us_fwd"] + out["us_bwd"]
    ql.device_status()
    return out


def bench_quantize(ql, dev, hbm_gbs, reps=5):
    """NF4 + double quant of the 7 weights of one LLaMA-65B layer (Student-t(4)
    values with std 0.015, drawn on the device), and the dequantize round trip."""
    import torch
    from bit_nf4_quantized_38_b300.workloads import case_weight, llama65b_layer_quant
    cases = llama65b_layer_quant().cases
    Ws = [case_weight(c, device=dev) for c in cases]
    qs = [ql.nf4_quantize(W) for W in Ws]
    outs = [torch.empty_like(W) for W in Ws]
    wss = [torch.empty(ql.workspace_size(ql.OP_QUANTIZE, 0, c.N, c.K, 0), dtype=torch.uint8, device=dev)
           for c in cases]
    params = sum(c.N * c.K for c in cases)
    n_b = sum(c.N * c.K // 64 for c in cases)
    n_2 = sum((c.N * c.K // 64 + 255) // 256 for c in cases)
    alg = 2 * params + params // 2 + n_b + 4 * n_2 + 4 * len(cases)
    res = {}
    for name, fn in (("quantize", lambda i: ql.nf4_quantize(Ws[i], out=qs[i], ws=wss[i])),
                     ("dequantize", lambda i: ql.nf4_dequantize(qs[i], out=outs[i]))):
        for i in range(len(cases)):
            fn(i)
        torch.cuda.synchronize()
        # the 7 calls of a layer as one CUDA graph, so host call overhead is not timed
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(len(cases)):
                    fn(i)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        gbs = alg / (us * 1e-6) / 1e9
        res[name] = {"us_per_layer": us, "bytes": alg, "GB/s": gbs, "frac_hbm": gbs / hbm_gbs,
                     "timing": "CUDA graph of the 7 calls, replayed; inputs larger than L2"}
    res["params"] = params
    res["workload"] = "llama65b_layer_7_weights_student_t4"
    del Ws, qs, outs
    torch.cuda.empty_cache()
    return res


def run_only(args):
    """One sub-benchmark alone, printed as a JSON line (for profiling)."""
    import torch
    from bit_nf4_quantized_38_b300 import qlora as ql
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, _ = load_peaks()
    if args.only == "decode":
        res = bench_decode(ql, dev, peaks["hbm_gbs"], args.decode_calls,
                           tuple(int(m) for m in args.decode_m.split(",")),
                           tuple(int(i) for i in args.decode_shapes.split(",")))
    elif args.only == "single":
        res = bench_single_linear(ql, dev)
    elif args.only == "fp8":
        res = bench_forward_fp8(ql, dev, peaks)
    else:
        res = bench_quantize(ql, dev, peaks["hbm_gbs"])
    print(json.dumps({"only": args.only, "results": res}), flush=True)


def bench_forward_fp8(ql, dev, peaks, steps=20, warmup=5, rounds=3):
    """The LLaMA-7B linears (M = 4096 tokens, r = 64): the bf16 and the E4M3
    forward, and the bf16 and the E4M3 backward (dX main product on E4M3),
    each timed over `steps` passes of the 7 calls with CUDA events; flops
    counted as 2 M N K + 2 M r (N + K) per linear forward and
    2 M N K + 4 M r (N + K) per linear backward for both.  The two variants
    alternate over `rounds` rounds (the order flipped each round, so that a
    drifting clock under the power cap favours neither) and each reports its
    median."""
    import torch
    wl = workload_of("llama7b")
    layers = build_layers(ql, dev, wl)
    ws_bytes = max(max(ql.workspace_size(op, c.M, c.N, c.K, c.r)
                       for op in (ql.OP_LINEAR_FWD, ql.OP_LINEAR_FWD_FP8, ql.OP_LINEAR_BWD, ql.OP_LINEAR_BWD_FP8))
                   for c in wl.cases)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fwd_flops = sum(2.0 * c.M * c.N * c.K + 2.0 * c.M * c.r * (c.N + c.K) for c in wl.cases)
    bwd_flops = sum(2.0 * c.M * c.N * c.K + 4.0 * c.M * c.r * (c.N + c.K) for c in wl.cases)
    out = {"workload": wl.name + " forward and backward", "flops_per_pass": fwd_flops,
           "bwd_flops_per_pass": bwd_flops}

    def fwd(fn):
        def one_pass():
            for L in layers:
                c = L["case"]
                fn(L["X"], L["q"], L["A"], L["B"], c.scale, Y=L["Y"], XA=L["XA"], ws=ws)
        return one_pass

    def bwd(fn):
        def one_pass():
            for L in layers:
                c = L["case"]
                fn(L["dY"], L["X"], L["XA"], L["q"], L["A"], L["B"], c.scale, dX=L["dX"], dA=L["dA"], dB=L["dB"],
                   ws=ws)
        return one_pass

    def timed(one_pass, flops):
        for _ in range(warmup):
            one_pass()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            one_pass()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        return {"ms_per_pass": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12}

    def alternate(name_a, pass_a, name_b, pass_b, flops):
        ms = {name_a: [], name_b: []}
        for rd in range(rounds):
            order = ((name_a, pass_a), (name_b, pass_b)) if rd % 2 == 0 else ((name_b, pass_b), (name_a, pass_a))
            for name, one_pass in order:
                ms[name].append(timed(one_pass, flops)["ms_per_pass"])
        for name in (name_a, name_b):
            med = sorted(ms[name])[len(ms[name]) // 2]
            out[name] = {"ms_per_pass": med, "TFLOP/s": flops / (med * 1e-3) / 1e12, "rounds_ms": ms[name]}

    alternate("bf16", fwd(ql.qlora_linear_fwd), "e4m3", fwd(ql.qlora_linear_fwd_fp8), fwd_flops)
    out["speedup_e4m3_over_bf16"] = out["bf16"]["ms_per_pass"] / out["e4m3"]["ms_per_pass"]
    alternate("bwd_bf16", bwd(ql.qlora_linear_bwd), "bwd_e4m3", bwd(ql.qlora_linear_bwd_fp8), bwd_flops)
    out["bwd_speedup_e4m3_over_bf16"] = out["bwd_bf16"]["ms_per_pass"] / out["bwd_e4m3"]["ms_per_pass"]
    out["peak_e4m3_tflops"] = 2.0 * peaks["bf16_tflops"]
    out["peak_note"] = "E4M3 dense peak taken as 2x the measured bf16 burst peak (nominal ratio)"
    del layers
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- GPU arm

def build_layers(ql, dev, wl):
    """Quantized weights and seeded inputs / outputs of every linear, on the device."""
    import torch
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight
    layers = []
    for c in wl.cases:
        W = case_weight(c, device=dev)
        q = ql.nf4_quantize(W)
        del W
        X, A, B, dY = case_inputs(c, device=dev)
        layers.append(dict(case=c, q=q, X=X, A=A, B=B, dY=dY,
                           Y=torch.empty(c.M, c.N, dtype=torch.bfloat16, device=dev),
                           XA=torch.empty(c.M, c.r, dtype=torch.bfloat16, device=dev),
                           dX=torch.empty(c.M, c.K, dtype=torch.bfloat16, device=dev),
                           dA=torch.empty(c.K, c.r, dtype=torch.float32, device=dev),
                           dB=torch.empty(c.r, c.N, dtype=torch.float32, device=dev)))
    torch.cuda.synchronize()
    return layers


def run_workload(ql, dev, wl, args, world, sampler=None, e2e=True):
    """Time args.steps steps of the workload (after args.warmup untimed ones).
    Returns the result dict (value, ms_per_step, roofline, launches, e2e)."""
    import torch
    import torch.distributed as dist
    layers = build_layers(ql, dev, wl)
    ws_bytes = max(max(ql.workspace_size(ql.OP_LINEAR_FWD, c.M, c.N, c.K, c.r),
                       ql.workspace_size(ql.OP_LINEAR_BWD, c.M, c.N, c.K, c.r)) for c in wl.cases)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    comm = torch.cuda.Stream() if world > 1 else None
    for L in layers:
        L["ev_bwd"], L["ev_red"] = torch.cuda.Event(), torch.cuda.Event()
        L["ev_red"].record(stream)

    def bwd(L):
        if comm is not None:
            stream.wait_event(L["ev_red"])  # the previous step's all-reduce of dA, dB is done
        ql.qlora_linear_bwd(L["dY"], L["X"], L["XA"], L["q"], L["A"], L["B"], L["case"].scale,
                            dX=L["dX"], dA=L["dA"], dB=L["dB"], ws=ws)
        if comm is not None:  # data parallel: the adapter gradients summed over the ranks
            L["ev_bwd"].record(stream)
            comm.wait_event(L["ev_bwd"])
            with torch.cuda.stream(comm):
                dist.all_reduce(L["dA"])
                dist.all_reduce(L["dB"])
            L["ev_red"].record(comm)

    def step():
        for L in layers:
            ql.qlora_linear_fwd(L["X"], L["q"], L["A"], L["B"], L["case"].scale, Y=L["Y"], XA=L["XA"], ws=ws)
        for L in reversed(layers):
            bwd(L)

    flops = step_flops(wl)
    for _ in range(args.warmup):
        step()
    if comm is not None:
        stream.wait_stream(comm)
    torch.cuda.synchronize()

    n_gemm = 2 * len(layers) * args.steps
    spans = torch.empty(2 * n_gemm, dtype=torch.int64, device=dev)
    ql.spans_start(spans)
    torch.cuda.synchronize()
    rank_barrier(world)
    n_launch0 = ql.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    if comm is not None:
        stream.wait_stream(comm)  # the last all-reduces belong to the timed region
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    rank_barrier(world)
    launches = ql.launch_count() - n_launch0
    n_rec, gemm_flops = ql.spans_stop()
    ql.device_status()
    sp = spans.view(-1, 2)[:n_rec].cpu()
    busy_ms = union_ms(sp.tolist())
    sum_ms = float((sp[:, 1] - sp[:, 0]).sum()) / 1e6
    ms_total = max_over_ranks_of(ev0.elapsed_time(ev1), world, dev)
    ms_step = ms_total / args.steps
    res = {"value": job_tflops(world, flops, ms_step), "ms_per_step": ms_step, "ms_total": ms_total,
           "flops_per_step": flops, "gpu_launches": launches, "t_wall": (t_wall0, t_wall1),
           "gemm": {"launches": n_rec, "flops": gemm_flops, "busy_ms": busy_ms, "sum_ms": sum_ms}}

    # ---- end to end through the public API with host buffers
    if e2e:
        res["e2e"] = run_e2e(ql, dev, layers, ws, stream, args, world, flops)
    del layers, ws
    torch.cuda.empty_cache()
    return res


def union_ms(pairs):
    """Length in ms of the union of [start, end) nanosecond intervals
    (consecutive GEMMs overlap: one's main loop runs in the other's last wave)."""
    total, cur0, cur1 = 0, None, None
    for a, b in sorted(pairs):
        if cur1 is None or a > cur1:
            if cur1 is not None:
                total += cur1 - cur0
            cur0, cur1 = a, b
        else:
            cur1 = max(cur1, b)
    if cur1 is not None:
        total += cur1 - cur0
    return total / 1e6


def run_e2e(ql, dev, layers, ws, stream, args, world, flops):
    """The same step with every linear's X and dY copied from pinned host
    memory on a copy stream running ahead of the compute, and dA, dB read back
    on a second copy stream after each backward.  The host holds the inputs of
    up to 8 layers (each distinct and seeded); layer l copies from host set
    l mod 8.  Y and dX stay on the device."""
    import torch
    per_layer = 7 if len(layers) % 7 == 0 else len(layers)
    n_sets = min(8, len(layers) // per_layer)
    host = []
    for i in range(n_sets * per_layer):
        L = layers[i]
        host.append(dict(X=torch.empty(L["X"].shape, dtype=torch.bfloat16).pin_memory(),
                         dY=torch.empty(L["dY"].shape, dtype=torch.bfloat16).pin_memory(),
                         dA=torch.empty(L["dA"].shape, dtype=torch.float32).pin_memory(),
                         dB=torch.empty(L["dB"].shape, dtype=torch.float32).pin_memory()))
        host[-1]["X"].copy_(L["X"])
        host[-1]["dY"].copy_(L["dY"])
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    for i, L in enumerate(layers):
        L["h"] = host[i % len(host)]
        L["ev_x"], L["ev_dy"] = torch.cuda.Event(), torch.cuda.Event()
        L["ev_b"], L["ev_d2h"] = torch.cuda.Event(), torch.cuda.Event()
        L["ev_b"].record(stream)
        L["ev_d2h"].record(stream)

    def step_e2e():
        for L in layers:
            h2d_stream.wait_event(L["ev_b"])  # the previous step's backward is done with X
            with torch.cuda.stream(h2d_stream):
                L["X"].copy_(L["h"]["X"], non_blocking=True)
            L["ev_x"].record(h2d_stream)
        for L in reversed(layers):
            with torch.cuda.stream(h2d_stream):
                L["dY"].copy_(L["h"]["dY"], non_blocking=True)
            L["ev_dy"].record(h2d_stream)
        for L in layers:
            stream.wait_event(L["ev_x"])
            ql.qlora_linear_fwd(L["X"], L["q"], L["A"], L["B"], L["case"].scale, Y=L["Y"], XA=L["XA"], ws=ws)
        for L in reversed(layers):
            stream.wait_event(L["ev_dy"])
            stream.wait_event(L["ev_d2h"])  # the previous step's read-back of dA, dB is done
            ql.qlora_linear_bwd(L["dY"], L["X"], L["XA"], L["q"], L["A"], L["B"], L["case"].scale,
                                dX=L["dX"], dA=L["dA"], dB=L["dB"], ws=ws)
            L["ev_b"].record(stream)
            d2h_stream.wait_event(L["ev_b"])
            with torch.cuda.stream(d2h_stream):
                L["h"]["dA"].copy_(L["dA"], non_blocking=True)
                L["h"]["dB"].copy_(L["dB"], non_blocking=True)
            L["ev_d2h"].record(d2h_stream)

    steps = args.steps if len(layers) <= 7 else min(args.steps, 5)
    for _ in range(2):
        step_e2e()
    torch.cuda.synchronize()
    rank_barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_stream.wait_event(e0)
    d2h_stream.wait_event(e0)
    for _ in range(steps):
        step_e2e()
    stream.wait_stream(d2h_stream)  # the last read-backs belong to the timed region
    stream.wait_stream(h2d_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    rank_barrier(world)
    e_ms = max_over_ranks_of(e0.elapsed_time(e1), world, dev) / steps
    h2d = sum(2 * L["case"].M * (L["case"].K + L["case"].N) for L in layers)
    d2h = sum(4 * L["case"].r * (L["case"].K + L["case"].N) for L in layers)
    return {"value": job_tflops(world, flops, e_ms), "unit": "TFLOP/s", "ms_per_step": e_ms, "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": f"per step: X and dY of all {len(layers)} linears copied from pinned host memory "
                    f"({len(host)} distinct linears' inputs held on the host, reused in turn) on a copy stream "
                    "running ahead of the compute, dA and dB read back on a second copy stream; Y and dX stay "
                    "on the device"}


def roofline_of(res, peaks, peak_src, wl):
    """The tensor-core GEMM inside the timed steps: algorithmic flops of its
    launches over the sum of their in-step durations (first CTA past its
    dependency wait to last CTA done, %globaltimer)."""
    g = res["gemm"]
    achieved = g["flops"] / (g["busy_ms"] / 1e3) / 1e12 if g["busy_ms"] > 0 else 0.0
    long_region = res["ms_total"] >= 1000.0
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    traffic = ncu_traffic("k_nf4_gemm_pair " + wl.name, ["bit_nf4_quantized_38_b300/csrc/tc_gemm.cu",
                                                         "bit_nf4_quantized_38_b300/csrc/convert.cuh"])
    return {"kernel": "k_nf4_gemm_pair (tcgen05 fused NF4-dequant GEMM, fwd Y and bwd dX)",
            "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": traffic,
            "peak_source": f"{peak_src} bf16 dense, "
                           f"{'sustained (timed region of seconds)' if long_region else 'burst'}",
            "frac_of_burst": achieved / peaks["bf16_tflops"],
            "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
            "launches_timed": g["launches"], "kernel_ms_per_step": g["busy_ms"] / res["ms_total"] * res["ms_per_step"],
            "share_of_step": g["busy_ms"] / res["ms_total"] if res["ms_total"] else None,
            "sum_of_launch_ms_per_step": g["sum_ms"] / res["ms_total"] * res["ms_per_step"],
            "timing": "per launch: earliest CTA start to latest CTA end (%globaltimer stamps the kernel "
                      "records in the timed steps themselves); achieved = the launches' algorithmic flops over "
                      "the union of their intervals (consecutive GEMMs overlap)"}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist

    if args.only != "all":
        return run_only(args)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from bit_nf4_quantized_38_b300 import qlora as ql

    peaks, peak_src = load_peaks()
    wl = workload_of(args.workload, args.layers)
    uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.2)
    res = run_workload(ql, dev, wl, args, world, e2e=not args.no_e2e)
    time.sleep(0.1)
    clocks = sampler.summary(*res["t_wall"])

    out = {
        "metric": METRIC, "value": res["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(wl, world),
        "roofline": roofline_of(res, peaks, peak_src, wl),
        "gpu_launches": res["gpu_launches"],
        "clocks": clocks,
    }
    if "e2e" in res:
        out["e2e"] = res["e2e"]
    if not args.no_extras and world == 1:
        if args.workload != "llama7b":
            wl7 = workload_of("llama7b")
            r7 = run_workload(ql, dev, wl7, argparse.Namespace(steps=max(args.steps, 20), warmup=args.warmup),
                              1, e2e=False)
            out["llama7b"] = {"workload": wl7.name, "value": r7["value"], "unit": "TFLOP/s",
                              "ms_per_step": r7["ms_per_step"], "steps": max(args.steps, 20),
                              "roofline": roofline_of(r7, peaks, peak_src, wl7),
                              "clocks": sampler.summary(*r7["t_wall"])}
        out["decode"] = {"workload": "llama13b decode shapes, M in {1,4,16}, r=64, fwd, CUDA graph over "
                                     "weight copies > 3x L2",
                         "peak_hbm_gbs": peaks["hbm_gbs"],
                         "results": bench_decode(ql, dev, peaks["hbm_gbs"], args.decode_calls,
                                                 tuple(int(m) for m in args.decode_m.split(",")),
                                                 tuple(int(i) for i in args.decode_shapes.split(",")))}
        out["prefill"] = {"workload": "llama13b shapes, M in {32,48,64,128} tokens (32: one 32-token pass "
                                      "of the weight-streaming kernel; 48-128: the few-token tensor-core "
                                      "kernel), r=64, fwd, CUDA graph over weight copies > 3x L2",
                          "peak_hbm_gbs": peaks["hbm_gbs"],
                          "results": bench_decode(ql, dev, peaks["hbm_gbs"], 120, (32, 48, 64, 128), (0, 1, 2))}
        out["quantize"] = bench_quantize(ql, dev, peaks["hbm_gbs"])
        out["single_linear"] = bench_single_linear(ql, dev)
        out["forward_e4m3"] = bench_forward_fp8(ql, dev, peaks)
    sampler.stop()
    if rank == 0 and world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(args.workload, step_flops(wl))
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
