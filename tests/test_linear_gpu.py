"""GPU parity of the QLoRA linear forward and backward against the fp64 oracle.

Tolerance (fp32 accumulation vs fp64 on the same dequantized weights):
relative Frobenius error <= 5e-3 and |err| <= 1e-2 (|ref| + rms(ref)) per
element.  The in-GEMM dequantization is checked bit-exactly with one-hot
inputs."""
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


def make_case(N, K, M, r, seed, alpha=16.0, dq=256, B_zero=False):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed)
    X = normal_bf16((M, K), 1.0, seed + 1)
    A = normal_bf16((K, r), 1.0 / np.sqrt(r), seed + 2)
    B = torch.zeros((r, N), dtype=torch.bfloat16) if B_zero else normal_bf16((r, N), 0.01, seed + 3)
    dY = normal_bf16((M, N), 1.0, seed + 4)
    return W, X, A, B, dY, alpha / r


def run_gpu(ql, W, X, A, B, dY, s, dq=256, xa_from_fwd=True):
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), dq_blocksize=dq)
    Xd, Ad, Bd, dYd = X.to(dev), A.to(dev), B.to(dev), dY.to(dev)
    Y, XA = ql.qlora_linear_fwd(Xd, q, Ad, Bd, s)
    dX, dA, dB = ql.qlora_linear_bwd(dYd, Xd, XA if xa_from_fwd else None, q, Ad, Bd, s)
    torch.cuda.synchronize()
    ql.device_status()
    return q, Y, XA, dX, dA, dB


def oracle_all(W, X, A, B, dY, s, dq=256):
    ref = nf4.quantize(bits(W), dq_blocksize=dq)
    Wh = nf4.dequantize(ref)
    Y, XA = linear.lora_forward(bits(X), Wh, bits(A), bits(B), s)
    dX, dA, dB, _ = linear.lora_backward(bits(dY), bits(X), Wh, bits(A), bits(B), s)
    return Y, XA, dX, dA, dB


SHAPES = [
    # N, K, M, r
    (1024, 1024, 16, 8),    # the single 1024x1024 linear, 16 tokens
    (1024, 1024, 256, 64),  # two M tiles, four N tiles
    (328, 320, 200, 16),    # ragged in every dimension
    (512, 4160, 130, 32),   # long reduction, M just over one tile
    (264, 192, 129, 128),   # rank 128: two LoRA K-steps
    (328, 320, 600, 16),    # CTA-pair tiles, ragged
    (1032, 576, 1100, 32),  # CTA-pair tiles, partial pair in N and M
    (520, 448, 300, 8),     # rank 8 on the tensor-core forward path
    (264, 640, 17, 64),     # 17 tokens: the decode path's 32-token pass (forward)
    (264, 640, 33, 64),     # one token past the decode limit: the few-token kernel
]


@pytest.mark.parametrize("N,K,M,r", SHAPES)
def test_forward_backward_within_tolerance(ql, N, K, M, r):
    W, X, A, B, dY, s = make_case(N, K, M, r, seed=N + K + M + r)
    _, Y, XA, dX, dA, dB = run_gpu(ql, W, X, A, B, dY, s)
    Yr, XAr, dXr, dAr, dBr = oracle_all(W, X, A, B, dY, s)
    tag = f"{N}x{K} M={M} r={r}"
    assert_close(f"Y {tag}", f64(Y), Yr)
    assert_close(f"XA {tag}", f64(XA), XAr)
    assert_close(f"dX {tag}", f64(dX), dXr)
    assert_close(f"dA {tag}", f64(dA), dAr)
    assert_close(f"dB {tag}", f64(dB), dBr)


def test_double_quant_off(ql):
    W, X, A, B, dY, s = make_case(512, 512, 64, 16, seed=5)
    _, Y, XA, dX, dA, dB = run_gpu(ql, W, X, A, B, dY, s, dq=0)
    Yr, _, dXr, dAr, dBr = oracle_all(W, X, A, B, dY, s, dq=0)
    assert_close("Y dq off", f64(Y), Yr)
    assert_close("dX dq off", f64(dX), dXr)
    assert_close("dA dq off", f64(dA), dAr)
    assert_close("dB dq off", f64(dB), dBr)


@pytest.mark.parametrize("N,K", [(512, 384), (296, 320)])
def test_in_gemm_dequant_is_bit_exact(ql, N, K):
    """With B = 0 and one-hot tokens, Y[m, n] = W_hat[n, k_m] exactly (one
    fp32 product by 1.0, rounded to bf16 once); with one-hot dY,
    dX[m, k] = W_hat[n_m, k] exactly.  Both must equal the oracle's W_hat."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed=7)
    ref = nf4.quantize(bits(W))
    Wh = nf4.dequantize(ref)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev))
    r = 8
    A = torch.randn(K, r).to(torch.bfloat16).to(dev)
    Bz = torch.zeros(r, N, dtype=torch.bfloat16, device=dev)
    ks = np.arange(K)
    X = torch.zeros(K, K, dtype=torch.bfloat16)
    X[torch.arange(K), torch.from_numpy(ks)] = 1.0
    Y, _ = ql.qlora_linear_fwd(X.to(dev), q, A, Bz, 2.0)
    torch.cuda.synchronize()
    assert np.array_equal(bits(Y), Wh.T[ks])
    dY = torch.zeros(N, N, dtype=torch.bfloat16)
    dY[torch.arange(N), torch.arange(N)] = 1.0
    X2 = torch.zeros(N, K, dtype=torch.bfloat16, device=dev)
    dX, dA, dB = ql.qlora_linear_bwd(dY.to(dev), X2, None, q, A, Bz, 2.0)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dX), Wh)
    assert torch.count_nonzero(dA) == 0


def test_recomputed_xa_matches_forward_xa_bitwise(ql):
    W, X, A, B, dY, s = make_case(768, 640, 192, 64, seed=9)
    _, _, _, dX1, dA1, dB1 = run_gpu(ql, W, X, A, B, dY, s, xa_from_fwd=True)
    _, _, _, dX2, dA2, dB2 = run_gpu(ql, W, X, A, B, dY, s, xa_from_fwd=False)
    assert torch.equal(dX1, dX2) and torch.equal(dA1, dA2) and torch.equal(dB1, dB2)


def test_results_are_deterministic(ql):
    W, X, A, B, dY, s = make_case(1024, 1024, 300, 64, seed=10)
    a = run_gpu(ql, W, X, A, B, dY, s)
    b = run_gpu(ql, W, X, A, B, dY, s)
    for x, y in zip(a[1:], b[1:]):
        assert torch.equal(x, y)


def test_zero_B_gives_zero_dA(ql):
    W, X, A, B, dY, s = make_case(256, 256, 64, 8, seed=11, B_zero=True)
    _, Y, XA, dX, dA, dB = run_gpu(ql, W, X, A, B, dY, s)
    assert torch.count_nonzero(dA) == 0
    Yr, _, dXr, _, dBr = oracle_all(W, X, A, B, dY, s)
    assert_close("Y B=0", f64(Y), Yr)
    assert_close("dB B=0", f64(dB), dBr)


@pytest.mark.parametrize("idx", [0, 4, 6])
def test_llama7b_linear_full_size_sampled(ql, idx):
    """LLaMA-7B linears at M = 4096 tokens, r = 64: Y and dX checked on 64
    sampled rows, XA, dA and dB in full."""
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight, llama7b_linears
    case = llama7b_linears().cases[idx]
    W = case_weight(case)
    X, A, B, dY = case_inputs(case)
    s = case.scale
    _, Y, XA, dX, dA, dB = run_gpu(ql, W, X, A, B, dY, s)
    ref = nf4.quantize(bits(W))
    Wh = nf4.dequantize(ref)
    rows = np.sort(np.random.default_rng(idx).choice(case.M, 64, replace=False))
    Yr, _ = linear.lora_forward(bits(X)[rows], Wh, bits(A), bits(B), s)
    tag = f"llama7b {case.name}"
    assert_close(f"Y rows {tag}", f64(Y)[rows], Yr)
    dXr, _, _, _ = linear.lora_backward(bits(dY)[rows], bits(X)[rows], Wh, bits(A), bits(B), s)
    assert_close(f"dX rows {tag}", f64(dX)[rows], dXr)
    dAr, dBr, XAr = linear.lora_adapter_grads(bits(dY), bits(X), bits(A), bits(B), s)
    assert_close(f"XA {tag}", f64(XA), XAr)
    assert_close(f"dA {tag}", f64(dA), dAr)
    assert_close(f"dB {tag}", f64(dB), dBr)


def test_chained_calls_read_the_previous_calls_output(ql):
    """Layer 2 reads layer 1's Y, and layer 1's backward reads layer 2's dX, on
    one stream with one workspace: the kernels of a call may start alongside
    the previous call only when their inputs are disjoint from its writes, so
    these calls must see the finished values.  Each layer is checked on its
    own at the path's tolerance: the oracle's layer 2 takes the GPU's own bf16
    Y1 (the activation handed over), and layer 1's backward the GPU's own bf16
    dY1.  A read of unfinished data would miss by orders of magnitude."""
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    M, K, H, N, r, s = 512, 384, 640, 448, 16, 2.0
    dev = torch.device("cuda")
    W1 = normal_with_outliers_bf16((H, K), 0.02, 0.001, 20.0, 71)
    W2 = normal_with_outliers_bf16((N, H), 0.02, 0.001, 20.0, 72)
    X = normal_bf16((M, K), 1.0, 73)
    A1, B1 = normal_bf16((K, r), 0.25, 74), normal_bf16((r, H), 0.01, 75)
    A2, B2 = normal_bf16((H, r), 0.25, 76), normal_bf16((r, N), 0.01, 77)
    dY2 = normal_bf16((M, N), 1.0, 78)
    q1, q2 = ql.nf4_quantize(W1.to(dev)), ql.nf4_quantize(W2.to(dev))
    ws = torch.empty(max(ql.workspace_size(ql.OP_LINEAR_FWD, M, 640, 640, r),
                         ql.workspace_size(ql.OP_LINEAR_BWD, M, 640, 640, r)), dtype=torch.uint8, device=dev)
    Xd, A1d, B1d, A2d, B2d, dY2d = (t.to(dev) for t in (X, A1, B1, A2, B2, dY2))
    for _ in range(3):  # repeated, so later rounds follow a training call on the stream
        Y1, XA1 = ql.qlora_linear_fwd(Xd, q1, A1d, B1d, s, ws=ws)
        Y2, XA2 = ql.qlora_linear_fwd(Y1, q2, A2d, B2d, s, ws=ws)
        dY1, dA2, dB2 = ql.qlora_linear_bwd(dY2d, Y1, XA2, q2, A2d, B2d, s, ws=ws)
        dX, dA1, dB1 = ql.qlora_linear_bwd(dY1, Xd, XA1, q1, A1d, B1d, s, ws=ws)
    torch.cuda.synchronize()
    ql.device_status()

    Wh1 = nf4.dequantize(nf4.quantize(bits(W1)))
    Wh2 = nf4.dequantize(nf4.quantize(bits(W2)))
    H1 = bits(Y1)    # the activation handed to layer 2, as the GPU produced it
    G1 = bits(dY1)   # the gradient handed back to layer 1
    Y1r, _ = linear.lora_forward(bits(X), Wh1, bits(A1), bits(B1), s)
    Y2r, _ = linear.lora_forward(H1, Wh2, bits(A2), bits(B2), s)
    assert_close("Y1", f64(Y1), Y1r)
    assert_close("Y2", f64(Y2), Y2r)
    dY1r, dA2r, dB2r, _ = linear.lora_backward(bits(dY2), H1, Wh2, bits(A2), bits(B2), s)
    assert_close("dX of layer 2", f64(dY1), dY1r)
    assert_close("dA of layer 2", f64(dA2), dA2r)
    assert_close("dB of layer 2", f64(dB2), dB2r)
    dXr, dA1r, dB1r, _ = linear.lora_backward(G1, bits(X), Wh1, bits(A1), bits(B1), s)
    assert_close("dX of layer 1", f64(dX), dXr)
    assert_close("dA of layer 1", f64(dA1), dA1r)
    assert_close("dB of layer 1", f64(dB1), dB1r)


def test_back_to_back_independent_calls_equal_synchronised_calls(ql):
    """Independent linears issued back to back on one stream overlap: a GEMM
    whose inputs the previous call does not write starts its main loop in the
    previous GEMM's last wave and waits only before its LoRA steps.  Results
    must equal the same calls made one at a time with a synchronisation in
    between, bit for bit, over repeated rounds on one workspace."""
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    dev = torch.device("cuda")
    shapes = [(1032, 576, 1100, 64), (4096, 1024, 2048, 16), (520, 4160, 600, 32), (2048, 2048, 1500, 64),
              (1032, 576, 300, 128)]
    layers = []
    for i, (N, K, M, r) in enumerate(shapes):
        q = ql.nf4_quantize(normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, 90 + i).to(dev))
        X, A = normal_bf16((M, K), 1.0, 100 + i).to(dev), normal_bf16((K, r), 0.125, 110 + i).to(dev)
        B, dY = normal_bf16((r, N), 0.01, 120 + i).to(dev), normal_bf16((M, N), 1.0, 130 + i).to(dev)
        layers.append((q, X, A, B, dY, 16.0 / r))
    ws = torch.empty(max(max(ql.workspace_size(ql.OP_LINEAR_FWD, M, N, K, r),
                             ql.workspace_size(ql.OP_LINEAR_BWD, M, N, K, r)) for N, K, M, r in shapes),
                     dtype=torch.uint8, device=dev)

    def run(sync):
        outs = []
        for q, X, A, B, dY, s in layers:
            Y, XA = ql.qlora_linear_fwd(X, q, A, B, s, ws=ws)
            outs.append([Y, XA])
            if sync:
                torch.cuda.synchronize()
        for (q, X, A, B, dY, s), o in zip(reversed(layers), reversed(outs)):
            o.extend(ql.qlora_linear_bwd(dY, X, o[1], q, A, B, s, ws=ws))
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        ql.device_status()
        return outs

    ref = run(True)
    for _ in range(3):
        got = run(False)
        for a, b in zip(ref, got):
            for x, y in zip(a, b):
                assert torch.equal(x, y)


@pytest.mark.parametrize("N,K,M,r", [(1032, 576, 1100, 32), (264, 640, 17, 64), (520, 1088, 9, 16)])
def test_fp4_weights_forward_backward(ql, N, K, M, r):
    """The same layer with FP4-coded weights (tensor-core path and, for
    M <= 32, the decode path): within tolerance of the oracle on the FP4
    dequantized weight."""
    W, X, A, B, dY, s = make_case(N, K, M, r, seed=N + M + 3)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), quant_type=ql.QL_FP4)
    Xd, Ad, Bd, dYd = X.to(dev), A.to(dev), B.to(dev), dY.to(dev)
    Y, XA = ql.qlora_linear_fwd(Xd, q, Ad, Bd, s)
    dX, dA, dB = ql.qlora_linear_bwd(dYd, Xd, XA, q, Ad, Bd, s)
    torch.cuda.synchronize()
    ql.device_status()
    Wh = nf4.dequantize(nf4.quantize(bits(W), quant_type=nf4.QT_FP4))
    Yr, _ = linear.lora_forward(bits(X), Wh, bits(A), bits(B), s)
    dXr, dAr, dBr, _ = linear.lora_backward(bits(dY), bits(X), Wh, bits(A), bits(B), s)
    tag = f"fp4 {N}x{K} M={M} r={r}"
    assert_close(f"Y {tag}", f64(Y), Yr)
    assert_close(f"dX {tag}", f64(dX), dXr)
    assert_close(f"dA {tag}", f64(dA), dAr)
    assert_close(f"dB {tag}", f64(dB), dBr)


@pytest.mark.parametrize("N,K,M,r", [(1032, 576, 1100, 32), (520, 1088, 300, 16), (264, 640, 33, 64),
                                     (520, 1088, 9, 16)])
def test_e4m3_second_level_forward_backward(ql, N, K, M, r):
    """Weights double-quantized with E4M3 second-level codes through every
    forward path (CTA-pair and single-CTA tensor-core GEMMs, the few-token
    kernel, the decode path) and the backward, against the oracle on the same
    dequantized weights."""
    W, X, A, B, dY, s = make_case(N, K, M, r, seed=N + K + M + r + 5)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), dq_type=ql.QL_DQ_E4M3)
    Xd, Ad, Bd, dYd = X.to(dev), A.to(dev), B.to(dev), dY.to(dev)
    Y, XA = ql.qlora_linear_fwd(Xd, q, Ad, Bd, s)
    dX, dA, dB = ql.qlora_linear_bwd(dYd, Xd, XA, q, Ad, Bd, s)
    torch.cuda.synchronize()
    ql.device_status()
    Wh = nf4.dequantize(nf4.quantize(bits(W), dq_type=nf4.DQ_E4M3))
    tag = f"e4m3 dq {N}x{K} M={M} r={r}"
    if M > 16:  # the decode path computes with bf16(q) * m_hat (see test_decode_gpu)
        Yr, _ = linear.lora_forward(bits(X), Wh, bits(A), bits(B), s)
        assert_close(f"Y {tag}", f64(Y), Yr)
    dXr, dAr, dBr, _ = linear.lora_backward(bits(dY), bits(X), Wh, bits(A), bits(B), s)
    assert_close(f"dX {tag}", f64(dX), dXr)
    assert_close(f"dA {tag}", f64(dA), dAr)
    assert_close(f"dB {tag}", f64(dB), dBr)


def test_e4m3_second_level_in_gemm_dequant_is_bit_exact(ql):
    """One-hot tokens through the CTA-pair GEMM and the few-token kernel with
    E4M3 second-level codes: Y[m, n] = W_hat[n, k_m] bit for bit."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    N, K = 296, 320
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed=17)
    Wh = nf4.dequantize(nf4.quantize(bits(W), dq_type=nf4.DQ_E4M3))
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), dq_type=ql.QL_DQ_E4M3)
    A = torch.randn(K, 8).to(torch.bfloat16).to(dev)
    Bz = torch.zeros(8, N, dtype=torch.bfloat16, device=dev)
    for k0, k1 in ((0, K), (0, 100), (100, 217)):  # all tokens at once; few-token batches
        ks = np.arange(k0, k1)
        X = torch.zeros(len(ks), K, dtype=torch.bfloat16)
        X[torch.arange(len(ks)), torch.from_numpy(ks)] = 1.0
        Y, _ = ql.qlora_linear_fwd(X.to(dev), q, A, Bz, 2.0)
        torch.cuda.synchronize()
        assert np.array_equal(bits(Y), Wh.T[ks])
