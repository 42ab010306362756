"""The data-parallel split on one GPU: ranks emulated one after the other
(each rank's calls complete before the next starts; no kernel waits on
another), with the all-reduce done on the host.

* Row-sharded quantization (nf4_quantize_shard_begin / _end) with the shards'
  fp64 absmax sums added: codes, second-level codes, steps and mean equal the
  unsharded quantization bit for bit (and the oracle's).
* Token-sliced backward: dX rows, and dA and dB summed over the slices, are
  within the path's tolerance of the oracle."""
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


@pytest.mark.parametrize("rows,cols,world,dq", [(264, 1152, 3, 256), (4096, 4096, 8, 256), (300, 640, 2, 0)])
def test_row_sharded_quantize_equals_unsharded(ql, rows, cols, world, dq):
    from bit_nf4_quantized_38_b300 import dp
    from bit_nf4_quantized_38_b300.workloads import student_t4_bf16
    dev = torch.device("cuda")
    W = student_t4_bf16((rows, cols), 0.015, rows + cols).to(dev)
    full = ql.nf4_quantize(W, dq_blocksize=dq)
    shards = [dp.quant_row_shard(rows, cols, world, k) for k in range(world)]
    parts = []
    for r0, r1 in shards:
        if r1 > r0:
            parts.append(ql.nf4_quantize_shard_begin(W[r0:r1].contiguous(), dq_blocksize=dq))
    total_sum = sum(float(p[2].item()) for p in parts)  # the all-reduce, on the host
    for q, ws, partial in parts:
        partial.fill_(total_sum)
        ql.nf4_quantize_shard_end(q, ws, rows * cols // 64)
    torch.cuda.synchronize()
    ql.device_status()
    cat = lambda f: torch.cat([getattr(p[0], f) for p in parts])
    assert torch.equal(cat("packed"), full.packed)
    if dq:
        assert torch.equal(cat("absmax_code"), full.absmax_code)
        assert torch.equal(cat("dq_step").view(torch.int32), full.dq_step.view(torch.int32))
        for p in parts:
            assert torch.equal(p[0].dq_mean.view(torch.int32), full.dq_mean.view(torch.int32))
    else:
        assert torch.equal(cat("absmax").view(torch.int32), full.absmax.view(torch.int32))
    ref = nf4.quantize(bits(W), dq_blocksize=dq)
    assert np.array_equal(full.packed.cpu().numpy(), ref["packed"])
    if dq:
        assert np.array_equal(full.absmax_code.cpu().numpy(), ref["code"])


def test_shard_end_rejects_a_total_below_the_shard(ql):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    W = normal_bf16((64, 256), 0.02, 3).to("cuda")
    q, ws, _ = ql.nf4_quantize_shard_begin(W)
    with pytest.raises(ql.QLError) as e:
        ql.nf4_quantize_shard_end(q, ws, 10)
    assert e.value.code == ql.QL_ERR_INVALID


@pytest.mark.parametrize("M,world", [(4096, 2), (1100, 3)])
def test_token_sliced_backward_sums_to_the_full_batch(ql, M, world):
    from bit_nf4_quantized_38_b300 import dp
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    dev = torch.device("cuda")
    N, K, r, s = 1032, 576, 64, 0.25
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, 21)
    X, A = normal_bf16((M, K), 1.0, 22), normal_bf16((K, r), 0.125, 23)
    B, dY = normal_bf16((r, N), 0.01, 24), normal_bf16((M, N), 1.0, 25)
    q = ql.nf4_quantize(W.to(dev))
    Xd, Ad, Bd, dYd = (t.to(dev) for t in (X, A, B, dY))
    dX_full, _, _ = ql.qlora_linear_bwd(dYd, Xd, None, q, Ad, Bd, s)
    dA = torch.zeros(K, r, device=dev)
    dB = torch.zeros(r, N, device=dev)
    dX = torch.empty_like(dX_full)
    for k in range(world):
        m0, m1 = dp.token_slice(M, world, k)
        _, XA = ql.qlora_linear_fwd(Xd[m0:m1], q, Ad, Bd, s)
        dXk, dAk, dBk = ql.qlora_linear_bwd(dYd[m0:m1], Xd[m0:m1], XA, q, Ad, Bd, s)
        dX[m0:m1] = dXk
        dA += dAk  # the all-reduce
        dB += dBk
    torch.cuda.synchronize()
    ql.device_status()
    # dX of a token depends on that token only (the LoRA term's split of the
    # reduction over N may differ with the slice size, so not bit for bit)
    Wh = nf4.dequantize(nf4.quantize(bits(W)))
    rows = np.sort(np.random.default_rng(M).choice(M, 48, replace=False))
    dXr, _, _, _ = linear.lora_backward(bits(dY)[rows], bits(X)[rows], Wh, bits(A), bits(B), s)
    assert_close(f"dp dX rows M={M} world={world}", dX.float().cpu().numpy()[rows], dXr)
    assert_close(f"dX rows full batch M={M}", dX_full.float().cpu().numpy()[rows], dXr)
    dAr, dBr, _ = linear.lora_adapter_grads(bits(dY), bits(X), bits(A), bits(B), s)
    assert_close(f"dp dA M={M} world={world}", dA.cpu().numpy(), dAr)
    assert_close(f"dp dB M={M} world={world}", dB.cpu().numpy(), dBr)
