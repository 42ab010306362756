"""GPU parity of the E4M3 forward and backward (qlora_linear_fwd_fp8,
qlora_linear_bwd_fp8) against the oracle's E4M3 forward and dX
(oracle/fp8.py): same quantized operands, fp32 accumulation on the GPU vs
fp64 -- the usual GEMM tolerance (relative Frobenius <= 5e-3, |err| <=
1e-2 (|ref| + rms(ref)) per element).  One-hot tokens (forward) and one-hot
gradient rows (dX, through the MN-major E4M3 operand) pin the weight
conversion, the row codes and the epilogue factor bit for bit."""
import numpy as np
import pytest
import torch

from oracle import fp8, linear, nf4
from oracle.bf16 import f32_to_bf16_bits
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


@pytest.mark.parametrize("N,K,M,r,dq,dqt", [
    (520, 1088, 200, 16, 256, 0),    # one accumulator per CTA (M <= 256)
    (1032, 576, 1100, 32, 256, 0),   # two accumulators, ragged in N and M
    (264, 640, 17, 64, 256, 0),      # few tokens, mostly padding
    (1024, 1024, 300, 128, 256, 1),  # rank 128; E4M3 second-level codes
    (776, 1088, 513, 8, 0, 0),       # double quantization off
    (520, 576, 1, 16, 256, 0),       # one token in a 256-row tile
])
def test_forward_matches_the_e4m3_oracle(ql, N, K, M, r, dq, dqt):
    W, X, A, B, s = make(N, K, M, r, seed=N + K + M + r)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), dq_blocksize=dq, dq_type=dqt)
    Y, XA = ql.qlora_linear_fwd_fp8(X.to(dev), q, A.to(dev), B.to(dev), s)
    torch.cuda.synchronize()
    ql.device_status()
    qt = nf4.quantize(bits(W), dq_blocksize=dq, dq_type=dqt)
    Yr, _ = fp8.lora_forward_e4m3(bits(X), qt, bits(A), bits(B), s)
    tag = f"{N}x{K} M={M} r={r} dq={dq} dqt={dqt}"
    assert_close(f"Y e4m3 {tag}", f64(Y), Yr)
    # XA_out is the same bf16 XA the bf16 forward hands to the backward
    _, XA16 = ql.qlora_linear_fwd(X.to(dev), q, A.to(dev), B.to(dev), s)
    torch.cuda.synchronize()
    assert torch.equal(XA, XA16)
    # and the E4M3 forward stays near the bf16 one (3 mantissa bits per operand)
    Y16, _ = linear.lora_forward(bits(X), nf4.dequantize(qt), bits(A), bits(B), s)
    assert np.linalg.norm(f64(Y) - Y16) / np.linalg.norm(Y16) < 0.06


def test_one_hot_tokens_are_bit_exact(ql):
    """X row m one-hot (1.0) at k_m, B = 0: the row exponent is 8, the row
    code 256, so Y[m, n] = bf16(Wq[n, k_m] 2^-E) exactly -- the weight's E4M3
    codes, read back bit for bit."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    N, K = 296, 320
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed=23)
    qt = nf4.quantize(bits(W))
    E, wq = fp8.weight_e4m3(qt)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev))
    A = torch.randn(K, 8).to(torch.bfloat16).to(dev)
    Bz = torch.zeros(8, N, dtype=torch.bfloat16, device=dev)
    ks = np.arange(K)
    X = torch.zeros(K, K, dtype=torch.bfloat16)
    X[torch.arange(K), torch.from_numpy(ks)] = 1.0
    Y, _ = ql.qlora_linear_fwd_fp8(X.to(dev), q, A, Bz, 2.0)
    torch.cuda.synchronize()
    Em, xq = fp8.rows_e4m3(bits(X))
    assert np.all(Em == 8) and np.all(xq[np.arange(K), ks] == 256.0)
    expect = f32_to_bf16_bits(np.ldexp(wq.T[ks], -E).astype(np.float32))
    assert np.array_equal(bits(Y), expect)


def test_llama7b_q_proj_full_size_sampled(ql):
    """LLaMA-7B q_proj (4096 x 4096) at 4096 tokens, r = 64: 64 sampled rows
    against the oracle (the weight's E4M3 codes in full)."""
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight, llama7b_linears
    case = llama7b_linears().cases[0]
    W = case_weight(case)
    X, A, B, _ = case_inputs(case)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev))
    Y, _ = ql.qlora_linear_fwd_fp8(X.to(dev), q, A.to(dev), B.to(dev), case.scale)
    torch.cuda.synchronize()
    ql.device_status()
    rows = np.sort(np.random.default_rng(7).choice(case.M, 64, replace=False))
    qt = nf4.quantize(bits(W))
    Yr, _ = fp8.lora_forward_e4m3(bits(X)[rows], qt, bits(A), bits(B), case.scale)
    assert_close("Y e4m3 llama7b q_proj rows", f64(Y)[rows], Yr)


# ------------------------------------------------------------------ backward (dX on E4M3)

@pytest.mark.parametrize("N,K,M,r,dq,dqt,saved_xa", [
    (528, 1088, 200, 16, 256, 0, True),    # one accumulator per CTA; ragged last reduction step (N % 128 = 16)
    (1040, 576, 1100, 32, 256, 0, False),  # two accumulators, ragged M and output columns; XA recomputed
    (272, 640, 17, 64, 256, 0, True),      # few tokens
    (1024, 1024, 300, 128, 256, 1, True),  # rank 128; E4M3 second-level codes
    (784, 1088, 513, 8, 0, 0, False),      # double quantization off
    (528, 576, 3, 16, 256, 0, False),      # three tokens in a 256-row tile
])
def test_backward_matches_the_e4m3_oracle(ql, N, K, M, r, dq, dqt, saved_xa):
    W, X, A, B, s = make(N, K, M, r, seed=N + 2 * K + M + r)
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    dY = normal_bf16((M, N), 1.0, N + M)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), dq_blocksize=dq, dq_type=dqt)
    Xd, Ad, Bd, dYd = X.to(dev), A.to(dev), B.to(dev), dY.to(dev)
    XA = ql.qlora_linear_fwd(Xd, q, Ad, Bd, s)[1] if saved_xa else None
    dX, dA, dB = ql.qlora_linear_bwd_fp8(dYd, Xd, XA, q, Ad, Bd, s)
    torch.cuda.synchronize()
    ql.device_status()
    qt = nf4.quantize(bits(W), dq_blocksize=dq, dq_type=dqt)
    dXr, _ = fp8.lora_backward_e4m3(bits(dY), qt, bits(A), bits(B), s)
    dAr, dBr, _ = linear.lora_adapter_grads(bits(dY), bits(X), bits(A), bits(B), s)
    tag = f"{N}x{K} M={M} r={r} dq={dq} dqt={dqt} xa={saved_xa}"
    assert_close(f"dX e4m3 {tag}", f64(dX), dXr)
    assert_close(f"dA e4m3 bwd {tag}", dA.double().cpu().numpy(), dAr)
    assert_close(f"dB e4m3 bwd {tag}", dB.double().cpu().numpy(), dBr)
    # and dX stays near the bf16 backward's (3 mantissa bits per operand)
    dX16 = linear.lora_backward(bits(dY), bits(X), nf4.dequantize(qt), bits(A), bits(B), s)[0]
    assert np.linalg.norm(f64(dX) - dX16) / np.linalg.norm(dX16) < 0.06


def test_backward_one_hot_gradients_are_bit_exact(ql):
    """dY row m one-hot (1.0) at n_m, B = 0 (so G = 0): the row exponent is 8
    and the code 256, so dX[m, k] = bf16(Wq[n_m, k] 2^-E) exactly -- the
    weight's E4M3 codes read back through the MN-major operand, bit for bit."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    N, K = 272, 576
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed=29)
    qt = nf4.quantize(bits(W))
    E, wq = fp8.weight_e4m3(qt)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev))
    X = torch.randn(N, K).to(torch.bfloat16).to(dev)
    A = torch.randn(K, 16).to(torch.bfloat16).to(dev)
    Bz = torch.zeros(16, N, dtype=torch.bfloat16, device=dev)
    ns = np.arange(N)
    dY = torch.zeros(N, N, dtype=torch.bfloat16)
    dY[torch.arange(N), torch.from_numpy(ns)] = 1.0
    dX, _, _ = ql.qlora_linear_bwd_fp8(dY.to(dev), X, None, q, A, Bz, 2.0)
    torch.cuda.synchronize()
    expect = f32_to_bf16_bits(np.ldexp(wq[ns], -E).astype(np.float32))
    assert np.array_equal(bits(dX), expect)


def test_backward_llama7b_q_proj_full_size_sampled(ql):
    """LLaMA-7B q_proj (4096 x 4096) at 4096 tokens, r = 64: 64 sampled rows
    of dX against the oracle."""
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight, llama7b_linears
    case = llama7b_linears().cases[0]
    W = case_weight(case)
    X, A, B, dY = case_inputs(case)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev))
    dX, _, _ = ql.qlora_linear_bwd_fp8(dY.to(dev), X.to(dev), None, q, A.to(dev), B.to(dev), case.scale)
    torch.cuda.synchronize()
    ql.device_status()
    rows = np.sort(np.random.default_rng(8).choice(case.M, 64, replace=False))
    qt = nf4.quantize(bits(W))
    dXr, _ = fp8.lora_backward_e4m3(bits(dY)[rows], qt, bits(A), bits(B), case.scale)
    assert_close("dX e4m3 llama7b q_proj rows", f64(dX)[rows], dXr)


def test_back_to_back_calls_equal_synchronised_calls(ql):
    """E4M3 forwards issued back to back on one stream with one workspace
    (the operand and LoRA kernels of a call may run alongside the previous
    call's GEMM) give bit-identical results to calls separated by a
    synchronisation; so does a chain where a call's X is the previous call's
    Y (which must wait for it), and a bf16 forward in between."""
    dev = torch.device("cuda")
    shapes = [(1024, 1024, 512, 32), (1024, 1024, 512, 32), (2048, 1024, 512, 16)]
    cases = [make(N, K, M, r, seed=60 + i) for i, (N, K, M, r) in enumerate(shapes)]
    qs = [ql.nf4_quantize(W.to(dev)) for W, *_ in cases]
    ins = [(X.to(dev), A.to(dev), B.to(dev), s) for _, X, A, B, s in cases]
    ws = torch.empty(max(ql.workspace_size(op, 512, 2048, 1024, 32) for op in (ql.OP_LINEAR_FWD_FP8, ql.OP_LINEAR_FWD)),
                     dtype=torch.uint8, device=dev)
    ref = []
    for q, (X, A, B, s) in zip(qs, ins):
        Y, XA = ql.qlora_linear_fwd_fp8(X, q, A, B, s, ws=ws)
        torch.cuda.synchronize()
        ref.append((Y.clone(), XA.clone()))
    outs = [(torch.empty_like(y), torch.empty_like(xa)) for y, xa in ref]
    for _ in range(3):
        for q, (X, A, B, s), (Y, XA) in zip(qs, ins, outs):
            ql.qlora_linear_fwd_fp8(X, q, A, B, s, Y=Y, XA=XA, ws=ws)
        # a bf16 forward on the same workspace between the E4M3 calls
        ql.qlora_linear_fwd(ins[0][0], qs[0], ins[0][1], ins[0][2], ins[0][3], ws=ws)
    torch.cuda.synchronize()
    ql.device_status()
    for (a, xa), (b, xb) in zip(ref, outs):
        assert torch.equal(a, b) and torch.equal(xa, xb)
    # chain: layer 2's input is layer 1's output (1024 -> 1024 -> 2048)
    X0, A0, B0, s0 = ins[0]
    A1, B1, s1 = ins[1][1], ins[1][2], ins[1][3]
    Y1s, _ = ql.qlora_linear_fwd_fp8(X0, qs[0], A0, B0, s0, ws=ws)
    torch.cuda.synchronize()
    Y2s, _ = ql.qlora_linear_fwd_fp8(Y1s, qs[1], A1, B1, s1, ws=ws)
    torch.cuda.synchronize()
    Y1, _ = ql.qlora_linear_fwd_fp8(X0, qs[0], A0, B0, s0, ws=ws)
    Y2, _ = ql.qlora_linear_fwd_fp8(Y1, qs[1], A1, B1, s1, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(Y2, Y2s)


def test_back_to_back_backward_calls_equal_synchronised_calls(ql):
    """E4M3 backward calls issued back to back on one stream and workspace,
    interleaved with E4M3 forwards (saved XA and recomputed XA), give
    bit-identical dX, dA, dB to calls separated by a synchronisation."""
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    dev = torch.device("cuda")
    shapes = [(1024, 1024, 512, 32), (2048, 1024, 512, 16), (1024, 2048, 512, 64)]
    cases = [make(N, K, M, r, seed=80 + i) for i, (N, K, M, r) in enumerate(shapes)]
    qs = [ql.nf4_quantize(W.to(dev)) for W, *_ in cases]
    ins = [(X.to(dev), A.to(dev), B.to(dev), normal_bf16((M, N), 1.0, 90 + i).to(dev), s)
           for i, ((_, X, A, B, s), (N, K, M, r)) in enumerate(zip(cases, shapes))]
    ws = torch.empty(max(ql.workspace_size(op, 512, 2048, 2048, 64)
                         for op in (ql.OP_LINEAR_FWD_FP8, ql.OP_LINEAR_BWD_FP8)), dtype=torch.uint8, device=dev)
    xas = [ql.qlora_linear_fwd_fp8(X, q, A, B, s)[1] for q, (X, A, B, dY, s) in zip(qs, ins)]
    torch.cuda.synchronize()
    ref = []
    for i, (q, (X, A, B, dY, s)) in enumerate(zip(qs, ins)):
        out = ql.qlora_linear_bwd_fp8(dY, X, xas[i] if i % 2 == 0 else None, q, A, B, s, ws=ws)
        torch.cuda.synchronize()
        ref.append(tuple(t.clone() for t in out))
    outs = [tuple(torch.empty_like(t) for t in r) for r in ref]
    Y = [torch.empty(X.shape[0], q.rows, dtype=torch.bfloat16, device=dev) for q, (X, *_) in zip(qs, ins)]
    for _ in range(3):
        for i, (q, (X, A, B, dY, s)) in enumerate(zip(qs, ins)):
            ql.qlora_linear_fwd_fp8(X, q, A, B, s, Y=Y[i], ws=ws)
            dX, dA, dB = outs[i]
            ql.qlora_linear_bwd_fp8(dY, X, xas[i] if i % 2 == 0 else None, q, A, B, s, dX=dX, dA=dA, dB=dB, ws=ws)
    torch.cuda.synchronize()
    ql.device_status()
    for r, o in zip(ref, outs):
        for a, b in zip(r, o):
            assert torch.equal(a, b)


def test_fp4_weights_forward_and_backward(ql):
    """The E4M3 forward and backward on FP4-coded weights (the comparison code
    table): the weight's E4M3 values come from the FP4 levels."""
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    N, K, M, r = 528, 640, 300, 16
    W, X, A, B, s = make(N, K, M, r, seed=101)
    dY = normal_bf16((M, N), 1.0, 102)
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), quant_type=ql.QL_FP4)
    Xd, Ad, Bd, dYd = X.to(dev), A.to(dev), B.to(dev), dY.to(dev)
    Y, XA = ql.qlora_linear_fwd_fp8(Xd, q, Ad, Bd, s)
    dX, dA, dB = ql.qlora_linear_bwd_fp8(dYd, Xd, XA, q, Ad, Bd, s)
    torch.cuda.synchronize()
    ql.device_status()
    qt = nf4.quantize(bits(W), quant_type=nf4.QT_FP4)
    Yr, _ = fp8.lora_forward_e4m3(bits(X), qt, bits(A), bits(B), s)
    dXr, _ = fp8.lora_backward_e4m3(bits(dY), qt, bits(A), bits(B), s)
    dAr, dBr, _ = linear.lora_adapter_grads(bits(dY), bits(X), bits(A), bits(B), s)
    assert_close("Y e4m3 fp4 weights", f64(Y), Yr)
    assert_close("dX e4m3 fp4 weights", f64(dX), dXr)
    assert_close("dA e4m3 fp4 weights", dA.double().cpu().numpy(), dAr)
    assert_close("dB e4m3 fp4 weights", dB.double().cpu().numpy(), dBr)
