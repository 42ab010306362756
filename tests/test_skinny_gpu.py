"""GPU parity of the few-token forward (32 < M <= 128 tokens: the transposed
tensor-core product split over all SMs, csrc/skinny.cu; and 17-32 tokens, run
by the decode path in one 32-token pass) against the fp64 oracle.

Same tolerance as the other GEMM results (relative Frobenius <= 5e-3,
|err| <= 1e-2 (|ref| + rms(ref)) per element, fp32 accumulation on the same
dequantized weights).  The in-kernel dequantization is pinned bit-exactly
with one-hot tokens: with B = 0 every output is one product of 1.0 and a
dequantized weight, so the sum over the CTAs' shares is exact."""
import numpy as np
import pytest
import torch

from oracle import linear, nf4
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_38_b300 import qlora
    return qlora


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def make(N, K, M, r, seed):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed)
    X = normal_bf16((M, K), 1.0, seed + 1)
    A = normal_bf16((K, r), 1.0 / np.sqrt(r), seed + 2)
    B = normal_bf16((r, N), 0.01, seed + 3)
    return W, X, A, B, 16.0 / r


SHAPES = [
    # N, K, M, r, dq, quant type
    (1032, 576, 33, 128, 256, 0),   # ragged N tile, two LoRA steps, Mp = 64
    (5120, 1024, 128, 64, 256, 0),  # full 128-token tile
    (328, 320, 100, 16, 256, 0),    # ragged N, Mp = 128 with 28 padding tokens
    (4096, 4096, 40, 64, 256, 0),   # LLaMA-7B attention shape, 40 tokens
    (256, 64, 128, 8, 256, 0),      # one main K-step per tile
    (776, 1088, 64, 32, 0, 0),      # double quantization off
    (520, 1088, 48, 16, 256, 1),    # FP4 code table, Mp = 64
    (136, 4160, 34, 64, 256, 0),    # two tiles, long reduction: many CTAs share each tile
    (1032, 576, 17, 128, 256, 0),   # 17 tokens: the decode path's 32-token pass, 15 empty columns
    (776, 1088, 32, 32, 0, 0),      # 32 tokens (decode path), double quantization off
]


@pytest.mark.parametrize("N,K,M,r,dq,qt", SHAPES)
def test_forward_within_tolerance(ql, N, K, M, r, dq, qt):
    W, X, A, B, s = make(N, K, M, r, seed=N + 3 * K + M)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), dq_blocksize=dq, quant_type=qt)
    Y, XA = ql.qlora_linear_fwd(X.to(dev), q, A.to(dev), B.to(dev), s)
    torch.cuda.synchronize()
    ql.device_status()
    ref = nf4.quantize(bits(W), dq_blocksize=dq, quant_type=qt)
    Yr, XAr = linear.lora_forward(bits(X), nf4.dequantize(ref), bits(A), bits(B), s)
    tag = f"{N}x{K} M={M} r={r} dq={dq} qt={qt}"
    assert_close(f"Y few-token {tag}", f64(Y), Yr)
    assert_close(f"XA few-token {tag}", f64(XA), XAr)


@pytest.mark.parametrize("N,K,M", [(1032, 576, 128), (296, 320, 100), (136, 4160, 33)])
def test_in_kernel_dequant_is_bit_exact(ql, N, K, M):
    """One-hot tokens in batches of M (the last one ragged), B = 0:
    Y[m, n] = W_hat[n, k_m] bit for bit, equal to the oracle's W_hat."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed=21)
    Wh = nf4.dequantize(nf4.quantize(bits(W)))
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev))
    r = 16
    A = torch.randn(K, r).to(torch.bfloat16).to(dev)
    Bz = torch.zeros(r, N, dtype=torch.bfloat16, device=dev)
    for k0 in range(0, K, M):
        # every batch stays above 32 tokens (M <= 32 takes the decode path)
        ks = np.arange(min(k0, K - 33), min(K, k0 + M))
        X = torch.zeros(len(ks), K, dtype=torch.bfloat16)
        X[torch.arange(len(ks)), torch.from_numpy(ks)] = 1.0
        Y, _ = ql.qlora_linear_fwd(X.to(dev), q, A, Bz, 2.0)
        torch.cuda.synchronize()
        assert np.array_equal(bits(Y), Wh.T[ks]), f"tokens {k0}..{ks[-1]}"


@pytest.mark.parametrize("idx,M", [(0, 128), (1, 128), (2, 128), (1, 48), (1, 32)])
def test_llama13b_full_size(ql, idx, M):
    """LLaMA-13B shapes (5120^2, 13824x5120, 5120x13824), r = 64, checked in
    full against the oracle (M = 32: the decode path)."""
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight, llama13b_decode
    case = llama13b_decode(M=M).cases[idx]
    W = case_weight(case)
    X, A, B, _ = case_inputs(case)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev))
    Y, XA = ql.qlora_linear_fwd(X.to(dev), q, A.to(dev), B.to(dev), case.scale)
    torch.cuda.synchronize()
    ql.device_status()
    Wh = nf4.dequantize(nf4.quantize(bits(W)))
    Yr, XAr = linear.lora_forward(bits(X), Wh, bits(A), bits(B), case.scale)
    tag = f"llama13b {case.N}x{case.K} M={M}"
    assert_close(f"Y {tag}", f64(Y), Yr)
    assert_close(f"XA {tag}", f64(XA), XAr)


def test_deterministic_and_back_to_back(ql):
    """The fixed-order sum of the shares makes repeated calls bit-identical,
    and calls issued back to back on one stream (where the GEMM may start
    before the previous call has finished) equal calls separated by a
    synchronisation."""
    dev = torch.device("cuda")
    cases = [make(1032, 576, 64, 32, seed=40 + i) for i in range(3)]
    qs = [ql.nf4_quantize(W.to(dev)) for W, *_ in cases]
    ins = [(X.to(dev), A.to(dev), B.to(dev), s) for _, X, A, B, s in cases]
    ws = torch.empty(ql.workspace_size(ql.OP_LINEAR_FWD, 64, 1032, 576, 32), dtype=torch.uint8, device=dev)
    sync = []
    for q, (X, A, B, s) in zip(qs, ins):
        Y, _ = ql.qlora_linear_fwd(X, q, A, B, s, ws=ws)
        torch.cuda.synchronize()
        sync.append(Y.clone())
    outs = [torch.empty_like(y) for y in sync]
    for _ in range(3):
        for q, (X, A, B, s), Y in zip(qs, ins, outs):
            ql.qlora_linear_fwd(X, q, A, B, s, Y=Y, ws=ws)
    torch.cuda.synchronize()
    ql.device_status()
    for a, b in zip(sync, outs):
        assert torch.equal(a, b)
