"""LoRA merge (qlora_merge): W' = bf16(w_hat + s (A B)^T) against the fp64
oracle's merged weight (LoRA tutorial: W' = W + W_A W_B gives the same
output with no extra cost at inference).

* B = 0: W' is the dequantized weight bit for bit.
* Random adapters: within the path's tolerance of the fp64 merge, and every
  element within one bf16 step of the fp64 value rounded to bf16 plus the
  fp32 accumulation error of w_hat + s acc.
* Requantizing W' (nf4_quantize) gives the oracle's codes of the GPU's W'.
(That the merged weight reproduces the layer's output, X W'^T = Y, is the
oracle's own pin, in fp64; a bf16 W' carries one more rounding per weight.)"""
import numpy as np
import pytest
import torch

from oracle import linear, nf4
from oracle.bf16 import f64_to_bf16_bits_via_f32
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


def _case(N, K, r, seed, dq=256):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    W = normal_with_outliers_bf16((N, K), 0.02, 0.001, 20.0, seed)
    A = normal_bf16((K, r), 1.0 / np.sqrt(r), seed + 1)
    B = normal_bf16((r, N), 0.01, seed + 2)
    return W, A, B


@pytest.mark.parametrize("dq", [256, 0])
def test_merge_with_zero_B_is_the_dequantized_weight(ql, dq):
    W, A, _ = _case(264, 640, 16, 3, dq)
    q = ql.nf4_quantize(W.cuda(), dq_blocksize=dq)
    Bz = torch.zeros(16, 264, dtype=torch.bfloat16, device="cuda")
    Wm = ql.qlora_merge(q, A.cuda(), Bz, 2.0)
    torch.cuda.synchronize()
    assert np.array_equal(bits(Wm), nf4.dequantize(nf4.quantize(bits(W), dq_blocksize=dq)))


@pytest.mark.parametrize("N,K,r,dq", [(1024, 1024, 8, 256), (264, 640, 128, 256), (4096, 4096, 64, 256),
                                      (1032, 576, 32, 0), (72, 192, 16, 256)])
def test_merge_matches_oracle_and_requantizes(ql, N, K, r, dq):
    W, A, B = _case(N, K, r, N + K + r, dq)
    s = 16.0 / r
    q = ql.nf4_quantize(W.cuda(), dq_blocksize=dq)
    Wm = ql.qlora_merge(q, A.cuda(), B.cuda(), s)
    q2 = ql.nf4_quantize(Wm, dq_blocksize=dq)
    torch.cuda.synchronize()
    ql.device_status()
    Wh = nf4.dequantize(nf4.quantize(bits(W), dq_blocksize=dq))
    ref = linear.merged_weight(Wh, bits(A), bits(B), s)
    got = bits(Wm)
    assert_close(f"merge {N}x{K} r={r}", linear.as_f64(got), ref)
    # one bf16 step from the correctly rounded value at most
    # one bf16 rounding of the result, plus the fp32 accumulation error of
    # w_hat + s sum_j A B (bounded relative to the summands' magnitudes; it
    # matters where they nearly cancel)
    rbf = linear.as_f64(f64_to_bf16_bits_via_f32(ref))
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(rbf), 2.0 ** -126))) - 7)
    mag = np.abs(linear.as_f64(Wh)) + s * (np.abs(linear.as_f64(bits(A))) @ np.abs(linear.as_f64(bits(B)))).T
    ratio = np.abs(linear.as_f64(got) - rbf) / (step + 2.0 ** -18 * mag)
    i = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert ratio[i] <= 1.0, (f"worst {ratio[i]:.3f} at {i}: got {linear.as_f64(got)[i]!r} ref {ref[i]!r} "
                             f"w_hat {linear.as_f64(Wh)[i]!r}")
    # requantized merged weight = the oracle's quantization of the GPU's W'
    ref2 = nf4.quantize(got, dq_blocksize=dq)
    assert np.array_equal(q2.packed.cpu().numpy(), ref2["packed"])
    if dq:
        assert np.array_equal(q2.absmax_code.cpu().numpy(), ref2["code"])


def test_merge_fp4_weight(ql):
    W, A, B = _case(520, 1088, 64, 77)
    q = ql.nf4_quantize(W.cuda(), quant_type=ql.QL_FP4)
    Wm = ql.qlora_merge(q, A.cuda(), B.cuda(), 0.25)
    torch.cuda.synchronize()
    Wh = nf4.dequantize(nf4.quantize(bits(W), quant_type=nf4.QT_FP4))
    assert_close("merge fp4", linear.as_f64(bits(Wm)), linear.merged_weight(Wh, bits(A), bits(B), 0.25))


def test_merge_e4m3_second_level_weight(ql):
    W, A, B = _case(520, 1088, 64, 78)
    q = ql.nf4_quantize(W.cuda(), dq_type=ql.QL_DQ_E4M3)
    Wm = ql.qlora_merge(q, A.cuda(), B.cuda(), 0.25)
    torch.cuda.synchronize()
    Wh = nf4.dequantize(nf4.quantize(bits(W), dq_type=nf4.DQ_E4M3))
    assert_close("merge e4m3 dq", linear.as_f64(bits(Wm)), linear.merged_weight(Wh, bits(A), bits(B), 0.25))
