#!/usr/bin/env python
"""Benchmark of the QLoRA linear hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (one step): the 7 LLaMA-7B linears (q/k/v/o 4096x4096, gate/up
11008x4096, down 4096x11008) with NF4 + double-quant weights and a rank-64
LoRA adapter (alpha 16) on all 7, M = 4 x 1024 = 4096 tokens: the forward of
all 7 in order, then the backward of all 7 in reverse order, through the
library's C ABI.  Inputs are seeded synthetic bf16 data shaped like the
pages' LLaMA workloads (weights N(0, 0.02^2) with 0.1% outliers x20,
activations N(0, 1)); the weights are quantized once before timing, as in
QLoRA finetuning where the frozen 4-bit weights are stored once.

The metric is algorithmic TFLOP/s: 4MNK + 6Mr(N+K) per linear per step.
One JSON line is printed by rank 0.  Extra keys: `roofline` of the dominant
kernel (the tensor-core dequant GEMM), `cpu_baseline` (the CPU oracle on a
bounded sample), `e2e` (the same metric with host buffers and host<->device
copies inside the timed region), `clocks`, `gpu_launches`, and sub-results
for the decode GEMV and the quantizer.

`--impl reference` times the CPU oracle (the plain fp64 restatement of the
method, the only reference this subject has) on the same config with a
bounded sample per step.
"""
import argparse
import hashlib
import json
import math
import os
import re
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
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-extras", action="store_true", help="skip the decode and quantizer sub-results")
    p.add_argument("--linears", default="", help="comma-separated subset of the 7 linears (profiling runs)")
    p.add_argument("--only", choices=["all", "decode", "quantize", "single"], default="all",
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


def profile_traffic(name, src_files):
    """Per-launch DRAM bytes recorded in profiles/<name>.md for the current kernel source, else None."""
    path = os.path.join(ROOT, "profiles", name + ".md")
    try:
        text = open(path).read()
    except OSError:
        return None
    h = hashlib.sha256()
    for f in src_files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    m_src = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_src or not m_tr or m_src.group(1) != h.hexdigest():
        return None
    return float(m_tr.group(1))


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


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample_setup(M_sample=512):
    """The first LLaMA-7B linear (q_proj 4096x4096) quantized by the oracle, with M_sample tokens."""
    from bit_nf4_quantized_38_b300.workloads import bf16_bits, case_inputs, case_weight, llama7b_linears
    from oracle import nf4
    case = llama7b_linears().cases[0]
    W = case_weight(case)
    X, A, B, dY = case_inputs(case, M=M_sample)
    qt = nf4.quantize(bf16_bits(W))
    return dict(case=case, qt=qt, X=bf16_bits(X), A=bf16_bits(A), B=bf16_bits(B), dY=bf16_bits(dY),
                M=M_sample)


def oracle_sample_step(s):
    """One oracle step on the sample: dequantize, forward, backward (fp64 numpy)."""
    from oracle import linear, nf4
    Wh = nf4.dequantize(s["qt"])
    linear.lora_forward(s["X"], Wh, s["A"], s["B"], s["case"].scale)
    linear.lora_backward(s["dY"], s["X"], Wh, s["A"], s["B"], s["case"].scale)


def oracle_sample_flops(s):
    c = s["case"]
    return 4 * s["M"] * c.N * c.K + 6 * s["M"] * c.r * (c.N + c.K)


def cpu_oracle_details(s):
    """Bounded samples of the other workloads, timed once each on the host's
    cores with the same oracle: the single 1024 x 1024 linear in full; the
    q_proj sample on one BLAS thread; 512 rows of the 5120 x 5120 decode layer
    (dequantize + forward, M = 1); 512 rows of an 8192-wide LLaMA-65B weight
    (quantize, then dequantize).  Rates use the algorithmic bytes or flops of
    the sample itself."""
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
    # the q_proj training sample on one thread: a child process started with
    # the BLAS thread counts set to 1 (they are fixed when numpy loads)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import sys, time, json; sys.path.insert(0, %r); import bench; s = bench.oracle_sample_setup(); "
            "t0 = time.perf_counter(); bench.oracle_sample_step(s); dt = time.perf_counter() - t0; "
            "print(json.dumps(bench.oracle_sample_flops(s) / dt / 1e12))" % os.path.dirname(os.path.abspath(__file__)))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        out["llama7b_q_proj_sample_1thread_tflops"] = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # the all-core figures above and below stand on their own
        out["llama7b_q_proj_sample_1thread_tflops"] = None
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
    out["samples"] = ("single linear 1024x1024 M=16 r=8 in full; q_proj 512-token sample on 1 BLAS thread; "
                      "512 of 5120 rows of the 13B 5120x5120 decode layer (M=1, dequantize + fwd); "
                      "512 x 8192 Student-t(4) weight (quantize, dequantize)")
    return out


def cpu_baseline(repeats=3):
    s = oracle_sample_setup()
    oracle_sample_step(s)  # warm
    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle_sample_step(s)
    dt = (time.perf_counter() - t0) / repeats
    return {"value": oracle_sample_flops(s) / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"q_proj 4096x4096 linear, {s['M']} tokens, r=64: NF4+DQ dequantize + fwd + bwd in "
                      f"fp64 numpy, mean of {repeats} runs ({dt:.2f} s each)",
            "details": cpu_oracle_details(s)}


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


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = oracle_sample_setup()
    for _ in range(args.warmup):
        oracle_sample_step(s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(s)
    dt = (time.perf_counter() - t0) / args.steps
    v = oracle_sample_flops(s) / dt / 1e12
    from bit_nf4_quantized_38_b300.workloads import llama7b_linears
    wl = llama7b_linears()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "linears": [c.name for c in wl.cases], "M": 4096, "r": 64,
                   "alpha": 16, "sample_per_step": "q_proj linear, 512 tokens"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": "per step: q_proj 4096x4096 linear, 512 tokens, r=64: NF4+DQ dequantize "
                                   "+ fwd + bwd in fp64 numpy"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ----------------------------------------------------------------------------- sub-benchmarks

def clone_nf4(ql, q):
    import torch
    t = ql.NF4Tensor(q.rows, q.cols, q.packed.clone(), blocksize=q.blocksize, dq_blocksize=q.dq_blocksize)
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
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            for i in range(len(cases)):
                fn(i)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        gbs = alg / (us * 1e-6) / 1e9
        res[name] = {"us_per_layer": us, "bytes": alg, "GB/s": gbs, "frac_hbm": gbs / hbm_gbs}
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
    else:
        res = bench_quantize(ql, dev, peaks["hbm_gbs"])
    print(json.dumps({"only": args.only, "results": res}), flush=True)


# ----------------------------------------------------------------------------- GPU arm

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
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight, llama7b_linears

    wl = llama7b_linears()
    if args.linears:
        keep = set(args.linears.split(","))
        wl.cases = [c for c in wl.cases if c.name in keep]
        wl.name += "_subset_" + "+".join(c.name for c in wl.cases)
    layers = []
    for c in wl.cases:
        W = case_weight(c).to(dev)
        q = ql.nf4_quantize(W)
        del W
        X, A, B, dY = case_inputs(c)
        L = dict(case=c, q=q, X=X.to(dev), A=A.to(dev), B=B.to(dev), dY=dY.to(dev),
                 Y=torch.empty(c.M, c.N, dtype=torch.bfloat16, device=dev),
                 XA=torch.empty(c.M, c.r, dtype=torch.bfloat16, device=dev),
                 dX=torch.empty(c.M, c.K, dtype=torch.bfloat16, device=dev),
                 dA=torch.empty(c.K, c.r, dtype=torch.float32, device=dev),
                 dB=torch.empty(c.r, c.N, dtype=torch.float32, device=dev))
        if not args.no_e2e:
            L["X_h"] = X.pin_memory()
            L["dY_h"] = dY.pin_memory()
            L["dA_h"] = torch.empty(c.K, c.r, dtype=torch.float32).pin_memory()
            L["dB_h"] = torch.empty(c.r, c.N, dtype=torch.float32).pin_memory()
        layers.append(L)
    ws_bytes = max(max(ql.workspace_size(ql.OP_LINEAR_FWD, c.M, c.N, c.K, c.r),
                       ql.workspace_size(ql.OP_LINEAR_BWD, c.M, c.N, c.K, c.r)) for c in wl.cases)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def step():
        for L in layers:
            ql.qlora_linear_fwd(L["X"], L["q"], L["A"], L["B"], L["case"].scale, Y=L["Y"], XA=L["XA"], ws=ws)
        for L in reversed(layers):
            ql.qlora_linear_bwd(L["dY"], L["X"], L["XA"], L["q"], L["A"], L["B"], L["case"].scale,
                                dX=L["dX"], dA=L["dA"], dB=L["dB"], ws=ws)

    # End to end: the inputs of every linear come from pinned host memory and
    # dA, dB go back to it, as a training loop would do it: host-to-device
    # copies on their own stream run ahead of the compute (each waits until
    # the previous step's backward has finished with that linear's buffers),
    # the device-to-host copies on a third stream follow each backward.
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    for L in layers:
        L["ev_x"], L["ev_dy"] = torch.cuda.Event(), torch.cuda.Event()
        L["ev_bwd"], L["ev_d2h"] = torch.cuda.Event(), torch.cuda.Event()
        L["ev_bwd"].record(stream)
        L["ev_d2h"].record(stream)

    def step_e2e():
        for L in layers:
            h2d_stream.wait_event(L["ev_bwd"])
            with torch.cuda.stream(h2d_stream):
                L["X"].copy_(L["X_h"], non_blocking=True)
            L["ev_x"].record(h2d_stream)
        for L in reversed(layers):
            with torch.cuda.stream(h2d_stream):
                L["dY"].copy_(L["dY_h"], non_blocking=True)
            L["ev_dy"].record(h2d_stream)
        for L in layers:
            stream.wait_event(L["ev_x"])
            ql.qlora_linear_fwd(L["X"], L["q"], L["A"], L["B"], L["case"].scale, Y=L["Y"], XA=L["XA"], ws=ws)
        for L in reversed(layers):
            stream.wait_event(L["ev_dy"])
            stream.wait_event(L["ev_d2h"])  # the previous step's read-back of dA, dB is done
            ql.qlora_linear_bwd(L["dY"], L["X"], L["XA"], L["q"], L["A"], L["B"], L["case"].scale,
                                dX=L["dX"], dA=L["dA"], dB=L["dB"], ws=ws)
            L["ev_bwd"].record(stream)
            d2h_stream.wait_event(L["ev_bwd"])
            with torch.cuda.stream(d2h_stream):
                L["dA_h"].copy_(L["dA"], non_blocking=True)
                L["dB_h"].copy_(L["dB"], non_blocking=True)
            L["ev_d2h"].record(d2h_stream)

    flops_step = sum(4 * c.M * c.N * c.K + 6 * c.M * c.r * (c.N + c.K) for c in wl.cases)

    def barrier():
        rank_barrier(world)

    def max_over_ranks(x):
        return max_over_ranks_of(x, world, dev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.2)

    barrier()
    torch.cuda.synchronize()
    n_launch0 = ql.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    launches = ql.launch_count() - n_launch0
    # The GEMM launch durations for the roofline come from a second pass of the
    # same steps with a CUDA event pair around every GEMM launch (events between
    # kernels would stop the programmatic overlap the timed pass above uses).
    ql.timing_start(14 * args.steps)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    gemm_ms, gemm_launches, gemm_flops = ql.timing_stop()
    ql.device_status()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1))
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    ms_step = ms_total / args.steps
    value = job_tflops(world, flops_step, ms_step)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        for _ in range(2):
            step_e2e()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        d2h_stream.wait_event(e0)
        for _ in range(args.steps):
            step_e2e()
        stream.wait_stream(d2h_stream)  # the last read-backs belong to the timed region
        stream.wait_stream(h2d_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e_ms = max_over_ranks(e0.elapsed_time(e1)) / args.steps
        h2d = sum(2 * c.M * (c.K + c.N) for c in wl.cases)
        d2h = sum(4 * c.r * (c.K + c.N) for c in wl.cases)
        e2e = {"value": job_tflops(world, flops_step, e_ms), "unit": "TFLOP/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "per step: X and dY of all 7 linears copied from pinned host memory on a copy "
                       "stream running ahead of the compute, dA and dB read back on a second copy "
                       "stream; Y and dX stay on the device"}

    peaks, peak_src = load_peaks()
    achieved = gemm_flops / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else 0.0
    traffic = profile_traffic("nf4_gemm_llama7b", ["bit_nf4_quantized_38_b300/csrc/tc_gemm.cu"])
    roofline = {"kernel": "k_nf4_gemm (tcgen05 fused NF4-dequant GEMM, fwd Y and bwd dX)",
                "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                "peak_source": f"{peak_src} bf16 dense (burst)",
                "frac_of_sustained": achieved / peaks.get("bf16_tflops_sustained", 1400.0),
                "launches_timed": gemm_launches, "kernel_ms_per_step": gemm_ms / args.steps,
                "timing": "CUDA event pair around each GEMM launch, in a second pass of the same steps",
                "share_of_step": gemm_ms / ms_total if ms_total else None}

    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "linears": [f"{c.name} {c.N}x{c.K}" for c in wl.cases], "M": 4096,
                   "r": 64, "alpha": 16, "quant": "NF4 block 64 + double quant block 256",
                   "step": "fwd of 7 linears in order, then bwd in reverse",
                   "l2": "inputs larger than L2 (each step touches ~0.7 GB of weights, activations "
                         "and gradients)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if e2e:
        out["e2e"] = e2e
    if not args.no_extras and world == 1:
        del layers, ws
        torch.cuda.empty_cache()
        out["decode"] = {"workload": "llama13b decode shapes, M in {1,4,16}, r=64, fwd, CUDA graph over "
                                     "weight copies > 3x L2",
                         "peak_hbm_gbs": peaks["hbm_gbs"],
                         "results": bench_decode(ql, dev, peaks["hbm_gbs"], args.decode_calls,
                                                 tuple(int(m) for m in args.decode_m.split(",")),
                                                 tuple(int(i) for i in args.decode_shapes.split(",")))}
        out["quantize"] = bench_quantize(ql, dev, peaks["hbm_gbs"])
        out["single_linear"] = bench_single_linear(ql, dev)
    if rank == 0 and world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
