"""GPU parity of the decode-sized forward (M <= 32 tokens) against the fp64
oracle.  The decode path forms every weight as the dequantized value
w_hat = bf16(fl32(q[c] * m_hat)) (pinned bit for bit by one-hot tokens below)
and accumulates in fp32, so its outputs differ from the oracle's only by the
order of the fp32 sums and the bf16 rounding of Y; the bar is the path's
tolerance (relative Frobenius error <= 5e-3, |err| <= 1e-2 (|ref| + rms(ref)))."""
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


def run(ql, W, X, A, B, s, dq=256):
    dev = torch.device("cuda")
    q = ql.nf4_quantize(W.to(dev), dq_blocksize=dq)
    Y, XA = ql.qlora_linear_fwd(X.to(dev), q, A.to(dev), B.to(dev), s)
    torch.cuda.synchronize()
    ql.device_status()
    return q, Y, XA


def reference(W, X, A, B, s, dq=256):
    Wh = nf4.dequantize(nf4.quantize(bits(W), dq_blocksize=dq))
    return linear.lora_forward(bits(X), Wh, bits(A), bits(B), s)


@pytest.mark.parametrize("N,K,M,r", [
    (1024, 1024, 1, 8), (1032, 576, 3, 8), (1032, 576, 9, 128), (520, 4160, 16, 32), (64, 64, 16, 16),
    (4096, 128, 7, 64), (256, 8192, 12, 64), (1536, 2048, 2, 16), (776, 1088, 5, 64), (512, 768, 8, 8),
    # K long enough that each XA CTA stages its slice of A in several chunks
    (256, 19968, 3, 64), (256, 20032, 1, 64), (512, 10240, 16, 128), (512, 40960, 4, 64),
    # 17-32 tokens: four 8-token tiles per pass, ragged last tile
    (1032, 576, 17, 128), (520, 4160, 32, 32), (776, 1088, 25, 64), (4096, 128, 24, 64),
    (256, 20032, 32, 64), (64, 64, 31, 16), (1536, 2048, 20, 8),
])
def test_decode_ragged_shapes(ql, N, K, M, r):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    seed = N + K + M
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed)
    X = normal_bf16((M, K), 1.0, seed + 1)
    A = normal_bf16((K, r), 1.0 / np.sqrt(r), seed + 2)
    B = normal_bf16((r, N), 0.01, seed + 3)
    s = 16.0 / r
    _, Y, XA = run(ql, W, X, A, B, s)
    Yr, XAr = reference(W, X, A, B, s)
    assert_close(f"decode Y {N}x{K} M={M} r={r}", Y.float().cpu().numpy(), Yr)
    assert_close(f"decode XA {N}x{K} M={M} r={r}", XA.float().cpu().numpy(), XAr)


def test_decode_double_quant_off(ql):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    W = normal_bf16((512, 1024), 0.02, 1)
    X = normal_bf16((4, 1024), 1.0, 2)
    A = normal_bf16((1024, 16), 0.25, 3)
    B = normal_bf16((16, 512), 0.01, 4)
    _, Y, _ = run(ql, W, X, A, B, 1.0, dq=0)
    Yr, _ = reference(W, X, A, B, 1.0, dq=0)
    assert_close("decode Y dq off", Y.float().cpu().numpy(), Yr)


@pytest.mark.parametrize("M", [1, 4, 16, 32])
@pytest.mark.parametrize("idx", [0, 1, 2])
def test_decode_llama13b_full_size(ql, idx, M):
    """LLaMA-13B shapes (5120x5120, 13824x5120, 5120x13824), r = 64: every output checked."""
    from bit_nf4_quantized_38_b300.workloads import case_inputs, case_weight, llama13b_decode
    case = llama13b_decode(M=M).cases[idx]
    W = case_weight(case)
    X, A, B, _ = case_inputs(case)
    _, Y, XA = run(ql, W, X, A, B, case.scale)
    Yr, XAr = reference(W, X, A, B, case.scale)
    assert_close(f"decode Y llama13b {case.N}x{case.K} M={M}", Y.float().cpu().numpy(), Yr)
    assert_close(f"decode XA llama13b {case.N}x{case.K} M={M}", XA.float().cpu().numpy(), XAr)


def test_decode_is_deterministic_and_repeatable(ql):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    dev = torch.device("cuda")
    W = normal_bf16((5120, 5120), 0.02, 5).to(dev)
    q = ql.nf4_quantize(W)
    X = normal_bf16((16, 5120), 1.0, 6).to(dev)
    A = normal_bf16((5120, 64), 0.125, 7).to(dev)
    B = normal_bf16((64, 5120), 0.01, 8).to(dev)
    outs = [ql.qlora_linear_fwd(X, q, A, B, 0.25)[0] for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_decode_chained_calls_and_any_workspace_contents(ql):
    """Layer chains on one stream: the second call reads the first call's Y (it
    must wait for it) while its weight may stream early.  Results must equal
    the same calls made one at a time with a synchronisation in between, on a
    workspace filled with arbitrary bytes (every workspace word a call reads
    was written by that call first, so no initialisation is needed)."""
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    dev = torch.device("cuda")
    K0, N1, N2, r = 1024, 2048, 1024, 16
    q1 = ql.nf4_quantize(normal_bf16((N1, K0), 0.02, 11).to(dev))
    q2 = ql.nf4_quantize(normal_bf16((N2, N1), 0.02, 12).to(dev))
    X = normal_bf16((4, K0), 1.0, 13).to(dev)
    A1, B1 = normal_bf16((K0, r), 0.25, 14).to(dev), normal_bf16((r, N1), 0.01, 15).to(dev)
    A2, B2 = normal_bf16((N1, r), 0.25, 16).to(dev), normal_bf16((r, N2), 0.01, 17).to(dev)
    nbytes = max(ql.workspace_size(ql.OP_LINEAR_FWD, 4, N1, K0, r), ql.workspace_size(ql.OP_LINEAR_FWD, 4, N2, N1, r))
    g = torch.Generator(device="cpu").manual_seed(5)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).to(dev)
    # one at a time
    Y1s, _ = ql.qlora_linear_fwd(X, q1, A1, B1, 1.0)
    torch.cuda.synchronize()
    Y2s, _ = ql.qlora_linear_fwd(Y1s.clone(), q2, A2, B2, 1.0)
    torch.cuda.synchronize()
    for _ in range(3):
        Y1, _ = ql.qlora_linear_fwd(X, q1, A1, B1, 1.0, ws=ws)
        Y2, _ = ql.qlora_linear_fwd(Y1, q2, A2, B2, 1.0, ws=ws)
        Y3, _ = ql.qlora_linear_fwd(X, q1, A1, B1, 1.0, ws=ws)  # reads nothing the previous call wrote
        torch.cuda.synchronize()
        ql.device_status()
        assert torch.equal(Y1, Y1s) and torch.equal(Y2, Y2s) and torch.equal(Y3, Y1s)


def test_decode_graph_replays_reuse_the_workspace(ql):
    """A captured sequence of decode calls on one workspace (the same
    workspace halves every replay) gives the eager results on every replay."""
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    dev = torch.device("cuda")
    shapes = [(1024, 1024, 1), (3072, 1024, 16), (1024, 3072, 9)]
    calls = []
    for i, (N, K, M) in enumerate(shapes):
        q = ql.nf4_quantize(normal_bf16((N, K), 0.02, 30 + i).to(dev))
        X = normal_bf16((M, K), 1.0, 40 + i).to(dev)
        A, B = normal_bf16((K, 64), 0.125, 50 + i).to(dev), normal_bf16((64, N), 0.01, 60 + i).to(dev)
        calls.append((X, q, A, B))
    nbytes = max(ql.workspace_size(ql.OP_LINEAR_FWD, M, N, K, 64) for N, K, M in shapes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    eager = []
    for X, q, A, B in calls:
        Y, XA = ql.qlora_linear_fwd(X, q, A, B, 0.25, ws=ws)
        eager.append((Y.clone(), XA.clone()))
    outs = [(torch.empty_like(Y), torch.empty_like(XA)) for Y, XA in eager]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for (X, q, A, B), (Y, XA) in zip(calls, outs):
                ql.qlora_linear_fwd(X, q, A, B, 0.25, Y=Y, XA=XA, ws=ws)
    for _ in range(4):
        for Y, XA in outs:
            Y.fill_(0)
            XA.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        ql.device_status()
        for (Y, XA), (Ye, XAe) in zip(outs, eager):
            assert torch.equal(Y, Ye) and torch.equal(XA, XAe)


@pytest.mark.parametrize("dq", [256, 0])
@pytest.mark.parametrize("M", [32, 16, 1])
def test_decode_weight_values_one_hot(ql, M, dq):
    """The decode path's per-weight value, read out bit for bit: with B = 0 and
    one-hot token rows, Y[m, n] is the weight of (n, k_m) that the path used,
    which must be the oracle's dequantized w_hat = bf16(fl32(q[c] * m_hat))."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    dev = torch.device("cuda")
    N, K, r = 264, 512, 8
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, 81 + dq)
    Wh = nf4.dequantize(nf4.quantize(bits(W), dq_blocksize=dq))
    q = ql.nf4_quantize(W.to(dev), dq_blocksize=dq)
    A = torch.randn(K, r, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).to(dev)
    Bz = torch.zeros(r, N, dtype=torch.bfloat16, device=dev)
    ks = np.arange(K) if M > 1 else np.array([0, 1, 63, 64, 200, 255, 256, 511])
    got = np.empty((ks.size, N), dtype=np.uint16)
    for i0 in range(0, ks.size, M):
        sel = ks[i0:i0 + M]
        X = torch.zeros(M, K, dtype=torch.bfloat16)
        X[torch.arange(sel.size), torch.from_numpy(sel)] = 1.0
        Y, _ = ql.qlora_linear_fwd(X.to(dev), q, A, Bz, 2.0)
        got[i0:i0 + sel.size] = bits(Y)[:sel.size]
    torch.cuda.synchronize()
    ql.device_status()
    assert np.array_equal(got, Wh.T[ks])
