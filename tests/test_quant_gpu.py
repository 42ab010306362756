"""GPU parity of NF4 quantization, double quantization and dequantization
against the CPU oracle: bit-exact codes, constants and bf16 weights."""
import numpy as np
import pytest
import torch

from oracle import nf4
from oracle.bf16 import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_38_b300 import qlora
    return qlora


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _gpu_quant(ql, W, dq=256):
    q = ql.nf4_quantize(W, dq_blocksize=dq)
    torch.cuda.synchronize()
    ql.device_status()
    return q


def _compare_quant(q, ref, rows=None):
    """Compare the GPU tensor q with the oracle dict ref (optionally some rows)."""
    R, C = ref["rows"], ref["cols"]
    pk = q.packed.cpu().numpy().reshape(R, C // 2)
    rpk = ref["packed"].reshape(R, C // 2)
    if rows is None:
        assert np.array_equal(pk, rpk)
    else:
        assert np.array_equal(pk[rows], rpk[rows])
    if ref["dq_blocksize"]:
        assert ref["mean_exact"]
        assert q.dq_mean.cpu().numpy()[0].view(np.uint32) == np.float32(ref["mean"]).view(np.uint32)
        assert np.array_equal(q.dq_step.cpu().numpy().view(np.uint32), ref["step"].view(np.uint32))
        assert np.array_equal(q.absmax_code.cpu().numpy(), ref["code"])
    else:
        assert np.array_equal(q.absmax.cpu().numpy().view(np.uint32), ref["absmax"].view(np.uint32))


CASES = [
    # rows, cols, dq, description
    (1024, 1024, 256, "single 1024x1024 linear"),
    (3, 64, 256, "one partial second-level group"),
    (7, 320, 256, "ragged: 35 blocks"),
    (37, 4160, 256, "ragged: 2405 blocks, partial last group"),
    (129, 1088, 0, "double quant off"),
]


@pytest.mark.parametrize("rows,cols,dq,desc", CASES)
def test_quantize_and_dequantize_bit_exact(ql, rows, cols, dq, desc):
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    W = normal_with_outliers_bf16((rows, cols), 0.02, 0.001, 20.0, seed=rows * 7 + cols)
    wb = _bits(W)
    ref = nf4.quantize(wb, dq_blocksize=dq)
    q = _gpu_quant(ql, W.cuda(), dq)
    _compare_quant(q, ref)
    Wd = ql.nf4_dequantize(q)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(Wd), nf4.dequantize(ref))


def test_every_bf16_value_and_zero_blocks(ql):
    """All finite bf16 patterns against several block absmax values (both the
    division-free and the IEEE-division ranges), plus all-zero and -0 blocks."""
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (b.astype(np.uint32) << 16).view(np.float32)
    finite = np.isfinite(vals)
    blocks = []
    for m in (1.0, 0.02, 3.0, 1e-4, 2.0 ** -70, 1e30):
        mb = f32_to_bf16_bits(np.float32(m))[0]
        mval = (np.uint32(mb) << np.uint32(16)).view(np.float32)
        keep = b[finite & (np.abs(vals) <= mval)]
        n = -(-keep.size // 63) * 63
        blk = np.zeros(n, np.uint16)
        blk[:keep.size] = keep
        blk = blk.reshape(-1, 63)
        # first element of every block is m itself, so every block's absmax is m
        blocks.append(np.concatenate([np.full((blk.shape[0], 1), mb, np.uint16), blk], axis=1))
    data = np.concatenate([x.reshape(-1) for x in blocks])
    extra = np.zeros(64 * 4, np.uint16)
    extra[64:128] = 0x8000  # a block of -0
    data = np.concatenate([data, extra])
    cols = 4096
    data = np.concatenate([data, np.zeros((-data.size) % cols, np.uint16)]).reshape(-1, cols)
    W = torch.from_numpy(data.view(np.int16)).view(torch.bfloat16).cuda()
    for dq in (0, 256):
        ref = nf4.quantize(data, dq_blocksize=dq)
        q = _gpu_quant(ql, W, dq)
        # codes do not depend on double quant; its constants are not compared
        # here because this tensor's absmax values span ~100 binades
        assert np.array_equal(q.packed.cpu().numpy(), ref["packed"])
        if not dq:
            assert np.array_equal(q.absmax.cpu().numpy().view(np.uint32), ref["absmax"].view(np.uint32))
            assert np.array_equal(_bits(ql.nf4_dequantize(q)), nf4.dequantize(ref))


def test_quantize_is_deterministic(ql):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16
    W = normal_bf16((2048, 4096), 0.02, seed=11).cuda()
    q1 = _gpu_quant(ql, W)
    q2 = _gpu_quant(ql, W)
    for a, b in ((q1.packed, q2.packed), (q1.absmax_code, q2.absmax_code), (q1.dq_step, q2.dq_step),
                 (q1.dq_mean, q2.dq_mean)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("idx", [0, 4, 6])
def test_llama65b_layer_weights_full_size(ql, idx):
    """One LLaMA-65B-layer weight at full size (Student-t values): every code,
    constant and the mean bit-exact; dequantized rows sampled."""
    from bit_nf4_quantized_38_b300.workloads import case_weight, llama65b_layer_quant
    case = llama65b_layer_quant().cases[idx]
    W = case_weight(case)
    wb = _bits(W)
    ref = nf4.quantize(wb, dq_blocksize=256)
    q = _gpu_quant(ql, W.cuda())
    _compare_quant(q, ref)
    rng = np.random.default_rng(idx)
    rows = np.sort(rng.choice(case.N, 64, replace=False))
    Wd = ql.nf4_dequantize(q)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(Wd)[rows], nf4.dequantize(ref, rows=rows))


@pytest.mark.parametrize("offset_elems", [0, 8])
def test_weight_only_16_byte_aligned(ql, offset_elems):
    """The quantizer reads whole 32-byte sectors when W is 32-byte aligned and
    16-byte pieces otherwise (the interface asks only for 16): both give the
    oracle's codes bit for bit."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    rows, cols = 520, 1088
    W = normal_with_outliers_bf16((rows, cols), 0.02, 0.001, 20.0, seed=61)
    buf = torch.empty(rows * cols + 64, dtype=torch.bfloat16, device="cuda")
    Wd = buf[offset_elems:offset_elems + rows * cols].view(rows, cols)
    Wd.copy_(W.cuda())
    assert (Wd.data_ptr() % 32 == 0) == (offset_elems == 0)
    ref = nf4.quantize(_bits(W), dq_blocksize=256)
    _compare_quant(_gpu_quant(ql, Wd, 256), ref)


@pytest.mark.parametrize("rows,cols,dq", [(1024, 1024, 256), (37, 4160, 256), (129, 1088, 0)])
def test_fp4_quantize_and_dequantize_bit_exact(ql, rows, cols, dq):
    """The FP4 comparison table behind the same interface (quant_type = FP4):
    codes, constants and dequantized weights equal the oracle's bit for bit."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    W = normal_with_outliers_bf16((rows, cols), 0.02, 0.001, 20.0, seed=rows + cols + 5)
    ref = nf4.quantize(_bits(W), dq_blocksize=dq, quant_type=nf4.QT_FP4)
    q = ql.nf4_quantize(W.cuda(), dq_blocksize=dq, quant_type=ql.QL_FP4)
    torch.cuda.synchronize()
    ql.device_status()
    _compare_quant(q, ref)
    assert np.array_equal(_bits(ql.nf4_dequantize(q)), nf4.dequantize(ref))
    # the same weight under NF4 codes differently
    assert not np.array_equal(ref["packed"], nf4.quantize(_bits(W), dq_blocksize=dq)["packed"])


def test_fp4_every_bf16_value(ql):
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (b.astype(np.uint32) << 16).view(np.float32)
    keep = b[np.isfinite(vals) & (np.abs(vals) <= 1.0)]
    mb = f32_to_bf16_bits(np.float32(1.0))[0]
    n = -(-keep.size // 63) * 63
    blk = np.zeros(n, np.uint16)
    blk[:keep.size] = keep
    blk = np.concatenate([np.full((n // 63, 1), mb, np.uint16), blk.reshape(-1, 63)], axis=1).reshape(-1)
    cols = 1024
    data = np.concatenate([blk, np.zeros((-blk.size) % cols, np.uint16)]).reshape(-1, cols)
    W = torch.from_numpy(data.view(np.int16)).view(torch.bfloat16).cuda()
    ref = nf4.quantize(data, dq_blocksize=0, quant_type=nf4.QT_FP4)
    q = ql.nf4_quantize(W, dq_blocksize=0, quant_type=ql.QL_FP4)
    torch.cuda.synchronize()
    assert np.array_equal(q.packed.cpu().numpy(), ref["packed"])
    assert np.array_equal(_bits(ql.nf4_dequantize(q)), nf4.dequantize(ref))


@pytest.mark.parametrize("rows,cols,pinned,dq", [(4096, 4096, True, 256), (1000, 11008, True, 256),
                                                 (37, 4160, False, 256), (3000, 2048, False, 0)])
def test_quantize_on_load_equals_device_quantize(ql, rows, cols, pinned, dq):
    """nf4_quantize_host streams a host weight through two staging chunks
    (copies on their own stream overlapping the coding): the result equals
    quantizing the same weight already on the device, bit for bit, and the
    oracle's codes."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    W = normal_with_outliers_bf16((rows, cols), 0.02, 0.001, 20.0, seed=rows + cols)
    Wh = W.pin_memory() if pinned else W.clone()
    dev = torch.device("cuda")
    copy = torch.cuda.Stream()
    got = ql.nf4_quantize_host(Wh, dev, dq_blocksize=dq, copy_stream=copy)
    want = ql.nf4_quantize(W.to(dev), dq_blocksize=dq)
    torch.cuda.synchronize()
    ql.device_status()
    for f in ("packed", "absmax", "absmax_code", "dq_step", "dq_mean"):
        a, b = getattr(got, f), getattr(want, f)
        assert (a is None) == (b is None), f
        if a is not None:
            assert torch.equal(a, b), f
    if rows * cols <= 4096 * 4096:
        _compare_quant(got, nf4.quantize(_bits(W), dq_blocksize=dq))


@pytest.mark.parametrize("rows,cols", [(1024, 1024), (37, 4160), (3, 64), (8192, 2752)])
def test_e4m3_second_level_bit_exact(ql, rows, cols):
    """Double quantization with E4M3 second-level codes: packed codes, the
    E4M3 bytes, steps and mean bit-exact against the oracle, and the
    dequantized weight too (ragged groups, and a LLaMA-65B-sized slab)."""
    from bit_nf4_quantized_38_b300.workloads import normal_with_outliers_bf16
    W = normal_with_outliers_bf16((rows, cols), 0.015, 0.001, 20.0, seed=rows + 3 * cols)
    ref = nf4.quantize(_bits(W), dq_blocksize=256, dq_type=nf4.DQ_E4M3)
    q = ql.nf4_quantize(W.cuda(), dq_type=ql.QL_DQ_E4M3)
    torch.cuda.synchronize()
    ql.device_status()
    _compare_quant(q, ref)
    assert not np.any((q.absmax_code.cpu().numpy().view(np.uint8) & 0x7F) == 0x7F)  # no NaN bytes
    Wd = ql.nf4_dequantize(q)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(Wd), nf4.dequantize(ref))
