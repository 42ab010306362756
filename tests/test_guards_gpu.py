"""Guard bytes around every output and workspace: no kernel writes outside
the buffers it is given.

Each buffer is carved out of a larger allocation with 4 KB on either side
filled with a fixed pattern; after quantize, dequantize, the forward (both
the tensor-core and the decode path) and the backward on ragged shapes (N,
M and K not multiples of the tiles, ranks 8 and 128), every guard byte must
still hold the pattern.  The outputs themselves are checked by the parity
tests; here only what lies around them is.  The E4M3 forward and backward
get the same check."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_38_b300 import qlora
    return qlora


class Guarded:
    """Buffers with guard regions; view() hands out the inside as a tensor."""

    def __init__(self, dev):
        self.dev = dev
        self.bufs = []

    def view(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        full = torch.full((GUARD + ((n + 255) // 256) * 256 + GUARD,), PATTERN, dtype=torch.uint8,
                          device=self.dev)
        self.bufs.append((full, n))
        return full[GUARD:GUARD + n].view(dtype).view(shape)

    def fill(self, t, value):
        t.view(torch.uint8).fill_(value)

    def check(self):
        torch.cuda.synchronize()
        for i, (full, n) in enumerate(self.bufs):
            lo = full[:GUARD]
            hi = full[GUARD + n:]
            assert bool((lo == PATTERN).all()), f"buffer {i}: guard before it overwritten"
            assert bool((hi == PATTERN).all()), f"buffer {i}: guard after it overwritten"


def guarded_nf4(ql, g, rows, cols, dq):
    n_b = rows * cols // 64
    q = ql.NF4Tensor(rows, cols, g.view((rows * cols // 2,), torch.uint8), dq_blocksize=dq)
    if dq:
        q.absmax_code = g.view((n_b,), torch.int8)
        q.dq_step = g.view(((n_b + 255) // 256,), torch.float32)
        q.dq_mean = g.view((1,), torch.float32)
    else:
        q.absmax = g.view((n_b,), torch.float32)
    return q


@pytest.mark.parametrize("N,K,M,r,dq", [
    (328, 320, 200, 16, 256),   # ragged tensor-core tiles
    (1032, 576, 1100, 128, 256),  # CTA-pair tiles, partial pair, rank 128
    (264, 640, 17, 8, 0),       # 17 tokens: the decode path's 32-token pass, DQ off
    (264, 640, 40, 8, 0),       # few-token forward past the decode limit, DQ off
    (1032, 576, 100, 128, 256), # few-token forward: ragged tile, shared tiles, rank 128
    (520, 4160, 16, 32, 256),   # decode path, long K
    (776, 1088, 5, 8, 256),     # decode path, ragged N
])
def test_no_write_outside_buffers(ql, N, K, M, r, dq):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    dev = torch.device("cuda")
    g = Guarded(dev)
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, N + K).to(dev)
    q = guarded_nf4(ql, g, N, K, dq)
    wsq = g.view((ql.workspace_size(ql.OP_QUANTIZE, 0, N, K, 0),), torch.uint8)
    ql.nf4_quantize(W, dq_blocksize=dq, out=q, ws=wsq)
    Wd = g.view((N, K), torch.bfloat16)
    ql.nf4_dequantize(q, out=Wd)
    X = normal_bf16((M, K), 1.0, 1).to(dev)
    A = normal_bf16((K, r), 0.25, 2).to(dev)
    B = normal_bf16((r, N), 0.01, 3).to(dev)
    dY = normal_bf16((M, N), 1.0, 4).to(dev)
    Y = g.view((M, N), torch.bfloat16)
    XA = g.view((M, r), torch.bfloat16)
    wsf = g.view((ql.workspace_size(ql.OP_LINEAR_FWD, M, N, K, r),), torch.uint8)
    ql.qlora_linear_fwd(X, q, A, B, 0.5, Y=Y, XA=XA, ws=wsf)
    dX = g.view((M, K), torch.bfloat16)
    dA = g.view((K, r), torch.float32)
    dB = g.view((r, N), torch.float32)
    wsb = g.view((ql.workspace_size(ql.OP_LINEAR_BWD, M, N, K, r),), torch.uint8)
    for xa in (XA, None):  # saved XA, and the recompute into the workspace
        ql.qlora_linear_bwd(dY, X, xa, q, A, B, 0.5, dX=dX, dA=dA, dB=dB, ws=wsb)
    ql.device_status()
    g.check()
    # the outputs were written (not left at the pattern)
    assert not bool((Y.view(torch.uint8) == PATTERN).all())
    assert not bool((dX.view(torch.uint8) == PATTERN).all())


@pytest.mark.parametrize("N,K,M,r", [
    (336, 320, 200, 16),    # one accumulator, ragged output tiles and reduction steps
    (1040, 576, 1100, 128), # two accumulators, partial pair tile, rank 128
    (272, 640, 17, 8),      # few tokens
])
def test_e4m3_calls_write_no_byte_outside_their_buffers(ql, N, K, M, r):
    """The E4M3 forward and backward: the operand kernel's codes and row
    exponents in the workspace, the MN-major dX path and both epilogues."""
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    dev = torch.device("cuda")
    g = Guarded(dev)
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, N + K + 1).to(dev)
    q = guarded_nf4(ql, g, N, K, 256)
    wsq = g.view((ql.workspace_size(ql.OP_QUANTIZE, 0, N, K, 0),), torch.uint8)
    ql.nf4_quantize(W, out=q, ws=wsq)
    X = normal_bf16((M, K), 1.0, 5).to(dev)
    A = normal_bf16((K, r), 0.25, 6).to(dev)
    B = normal_bf16((r, N), 0.01, 7).to(dev)
    dY = normal_bf16((M, N), 1.0, 8).to(dev)
    Y = g.view((M, N), torch.bfloat16)
    XA = g.view((M, r), torch.bfloat16)
    wsf = g.view((ql.workspace_size(ql.OP_LINEAR_FWD_FP8, M, N, K, r),), torch.uint8)
    ql.qlora_linear_fwd_fp8(X, q, A, B, 0.5, Y=Y, XA=XA, ws=wsf)
    dX = g.view((M, K), torch.bfloat16)
    dA = g.view((K, r), torch.float32)
    dB = g.view((r, N), torch.float32)
    wsb = g.view((ql.workspace_size(ql.OP_LINEAR_BWD_FP8, M, N, K, r),), torch.uint8)
    for xa in (XA, None):
        ql.qlora_linear_bwd_fp8(dY, X, xa, q, A, B, 0.5, dX=dX, dA=dA, dB=dB, ws=wsb)
    ql.device_status()
    g.check()
    assert not bool((Y.view(torch.uint8) == PATTERN).all())
    assert not bool((dX.view(torch.uint8) == PATTERN).all())
