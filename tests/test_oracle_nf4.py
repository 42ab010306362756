"""Pins for the NF4 / double-quant oracle against closed forms, brute force,
library routines and the figures the pages print (CPU only)."""
import json
import math
import os
import statistics
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nf4
from oracle.bf16 import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


def _torch_bf16_bits(x_f32):
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------- bf16

def test_bf16_rounding_matches_torch_on_ties_and_random():
    rng = np.random.default_rng(0)
    # every low-half pattern class around ties, on many exponents and both signs
    hi = rng.integers(0, 0x7F00, size=4096, dtype=np.uint32)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    u = ((hi[:, None] << 16) | lows[None, :]).reshape(-1)
    u = np.concatenate([u, u | 0x80000000])
    x = u.view(np.float32)
    x = np.concatenate([x, rng.standard_normal(100_000).astype(np.float32),
                        np.array([0.0, -0.0, 1e-40, -1e-40], dtype=np.float32)])
    assert np.array_equal(f32_to_bf16_bits(x), _torch_bf16_bits(x))


def test_bf16_widening_is_exact():
    b = np.arange(0, 0x7F80, 7, dtype=np.uint16)
    f = bf16_bits_to_f32(b)
    assert np.array_equal(f32_to_bf16_bits(f), b)


# --------------------------------------------------------------------------- codebook

def test_codebook_invariants():
    q = nf4.nf4_levels()
    assert q.dtype == np.float32 and q.shape == (16,)
    assert np.all(np.diff(q.astype(np.float64)) > 0)
    assert q[0] == -1.0 and q[15] == 1.0 and q[nf4.ZERO_CODE] == 0.0
    assert (q > 0).sum() == 8 and (q < 0).sum() == 7


def _phi(x):
    """Standard normal CDF from the closed form 0.5 * erfc(-x / sqrt 2)."""
    return 0.5 * math.erfc(-x / math.sqrt(2.0))


def test_codebook_levels_are_normalised_normal_quantiles():
    """Each positive level times z(DELTA) is the standard-normal quantile at its
    probability, and each negative level likewise (checked through the CDF)."""
    q = nf4.nf4_levels_f64()
    pos_p, neg_p = nf4.nf4_probabilities()
    z_max = statistics.NormalDist().inv_cdf(nf4.DELTA)
    assert abs(_phi(z_max) - nf4.DELTA) < 1e-14
    pos = q[q > 0][::-1]   # descending: DELTA first
    neg = -q[q < 0]        # |levels|, descending
    assert len(pos) == 8 and len(neg) == 7
    for lv, p in zip(pos, pos_p):
        assert abs(_phi(lv * z_max) - p) < 1e-13
    for lv, p in zip(neg, neg_p):
        assert abs(_phi(lv * z_max) - p) < 1e-13
    # probabilities equally spaced from DELTA towards 1/2 (9 and 8 points, 1/2 dropped)
    assert np.allclose(np.diff(pos_p), -(nf4.DELTA - 0.5) / 8, rtol=0, atol=1e-15)
    assert np.allclose(np.diff(neg_p), -(nf4.DELTA - 0.5) / 7, rtol=0, atol=1e-15)


def test_quantile_routine_matches_independent_implementation():
    nd = statistics.NormalDist()
    for p in np.concatenate(nf4.nf4_probabilities()):
        assert abs(float(nf4.normal_quantile(p)) - nd.inv_cdf(float(p))) < 1e-12


# --------------------------------------------------------------------------- coding

def _brute_code(x_f32):
    q = nf4.nf4_levels().astype(np.float64)
    d = np.abs(np.asarray(x_f32, dtype=np.float32).astype(np.float64)[..., None] - q)
    return np.argmin(d, axis=-1)  # first minimum: ties to the lower index


def test_nearest_code_equals_brute_force_argmin_dense_sweep():
    rng = np.random.default_rng(1)
    t = nf4.nf4_midpoints()
    xs = [rng.uniform(-1, 1, 200_000).astype(np.float32)]
    # neighbourhood of every midpoint, several fp32 steps each side
    for tj in t:
        c = np.float32(tj)
        v = [c]
        up, dn = c, c
        for _ in range(8):
            up = np.nextafter(up, np.float32(2)); dn = np.nextafter(dn, np.float32(-2))
            v += [up, dn]
        xs.append(np.array(v, dtype=np.float32))
    # strided walk over every fp32 bit pattern in [-1, 1]
    pos = np.arange(0, 0x3F800001, 997, dtype=np.uint32).view(np.float32)
    xs += [pos, -pos, nf4.nf4_levels()]
    x = np.concatenate(xs)
    assert np.array_equal(nf4.nearest_code(x), _brute_code(x))


def test_midpoint_ties_go_to_lower_index():
    q = nf4.nf4_levels().astype(np.float64)
    t = nf4.nf4_midpoints()
    for j, tj in enumerate(t):
        if float(np.float32(tj)) == tj:  # an exactly representable midpoint is a tie
            assert nf4.nearest_code(np.float32(tj)) == j
    # equivalent definition check: counting thresholds below x
    assert np.all((q[:-1] < t) & (t < q[1:]))


@pytest.mark.parametrize("m", [1.0, 0.02, 3.0, 0.0001, 3.3e38])
def test_all_bf16_weights_code_to_nearest_level(m):
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    w = bf16_bits_to_f32(b)
    m32 = np.float32(bf16_bits_to_f32(f32_to_bf16_bits(np.float32(m)))[0])
    keep = np.isfinite(w) & (np.abs(w) <= m32)
    w = w[keep]
    W = np.zeros((1, 64 * ((w.size + 63) // 64)), dtype=np.float32)
    W[0, :w.size] = w
    W = W.reshape(-1, 64)
    W[:, 0] = m32  # each block's absmax is m: put m in every block
    absmax = nf4.block_absmax(W)
    assert np.all(absmax == m32)
    codes = nf4.nf4_codes(W, absmax)
    x = (W / m32).astype(np.float32)
    assert np.array_equal(codes, _brute_code(x))


def test_block_coding_matches_per_element_loop():
    rng = np.random.default_rng(2)
    W = (rng.standard_normal((3, 192)) * 0.02).astype(np.float32)
    W = bf16_bits_to_f32(f32_to_bf16_bits(W))
    W[1, 64:128] = 0.0  # an all-zero block
    q = nf4.nf4_levels().astype(np.float64)
    absmax = nf4.block_absmax(W)
    codes = nf4.nf4_codes(W, absmax)
    for i in range(3):
        for k in range(192):
            blk = W[i, (k // 64) * 64:(k // 64 + 1) * 64]
            m = float(np.max(np.abs(blk)))
            assert absmax[i, k // 64] == m
            if m == 0:
                want = 7
            else:
                x = float(np.float32(W[i, k]) / np.float32(m))
                d = [abs(x - float(v)) for v in q]
                want = d.index(min(d))
            assert codes[i, k] == want


def test_nibble_order_and_roundtrip():
    assert list(nf4.pack_nibbles(np.array([1, 2, 3, 4, 15, 0]))) == [0x12, 0x34, 0xF0]
    rng = np.random.default_rng(3)
    c = rng.integers(0, 16, 4096).astype(np.uint8)
    assert np.array_equal(nf4.unpack_nibbles(nf4.pack_nibbles(c)), c)


# --------------------------------------------------------------------------- round trip bounds

def _weights(rows, cols, seed, outliers=True):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(rows, cols, generator=g) * 0.02
    if outliers:
        mask = torch.rand(rows, cols, generator=g) < 0.01
        w = torch.where(mask, w * 20, w)
    return w.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_roundtrip_error_bound_without_double_quant():
    wb = _weights(64, 512, 4)
    qt = nf4.quantize(wb, dq_blocksize=0)
    w = bf16_bits_to_f32(wb).astype(np.float64)
    wh = bf16_bits_to_f32(nf4.dequantize(qt)).astype(np.float64)
    m = np.repeat(qt["absmax"].reshape(64, 8), 64, axis=1).astype(np.float64)
    half_gap = np.diff(nf4.nf4_levels().astype(np.float64)).max() / 2
    assert abs(half_gap - 0.1519) < 1e-3
    bound = m * (half_gap + 2.0 ** -22) + 2.0 ** -8 * np.abs(wh) + 1e-45
    assert np.all(np.abs(w - wh) <= bound)
    # the bound is reasonably tight: some element comes within half of it
    assert np.max(np.abs(w - wh) / bound) > 0.5


def test_roundtrip_error_bound_with_double_quant():
    wb = _weights(128, 1024, 5)
    qt = nf4.quantize(wb, dq_blocksize=256)
    assert qt["mean_exact"]
    w = bf16_bits_to_f32(wb).astype(np.float64)
    wh = bf16_bits_to_f32(nf4.dequantize(qt)).astype(np.float64)
    nb = 1024 // 64
    m = qt["absmax"].astype(np.float64)
    mh = nf4.absmax_hat(qt).astype(np.float64)
    step = np.repeat(qt["step"], 256)[:m.size].astype(np.float64)
    # second level: |m - m_hat| <= step/2 plus a few ulps of the fp32 arithmetic
    ulp = np.spacing(np.abs(mh).astype(np.float32) + np.float32(step)).astype(np.float64)
    assert np.all(np.abs(m - mh) <= step / 2 + 2 * ulp)
    codes = nf4.unpack_nibbles(qt["packed"]).reshape(128, 1024)
    qv = np.abs(nf4.nf4_levels()[codes].astype(np.float64))
    M = np.repeat(m.reshape(128, nb), 64, axis=1)
    dM = np.repeat(np.abs(m - mh).reshape(128, nb), 64, axis=1)
    half_gap = np.diff(nf4.nf4_levels().astype(np.float64)).max() / 2
    bound = M * (half_gap + 2.0 ** -22) + qv * dM + 2.0 ** -8 * np.abs(wh) + 1e-45
    assert np.all(np.abs(w - wh) <= bound)


# --------------------------------------------------------------------------- double quant

def test_mean_is_the_exact_sum_over_count():
    rng = np.random.default_rng(6)
    a = bf16_bits_to_f32(f32_to_bf16_bits((rng.random(1000) * 0.1 + 0.01).astype(np.float32)))
    S, exact = nf4.exact_sum_f64(a)
    assert exact
    assert Fraction(S) == sum(Fraction(float(v)) for v in a)
    code, step, mean, ex = nf4.double_quantize(a)
    assert ex and mean == np.float32(S / a.size)


def test_exact_sum_detects_inexact_case():
    a = np.array([1.0, 2.0 ** -60, 3.0], dtype=np.float32)
    S, exact = nf4.exact_sum_f64(a)
    assert not exact
    assert S == 4.0


def test_double_quant_codes_range_and_extremes():
    rng = np.random.default_rng(7)
    a = (rng.random(1000) * 0.05 + 0.02).astype(np.float32)
    code, step, mean, _ = nf4.double_quantize(a, 256)
    assert step.shape == (4,)
    assert code.min() >= -127 and code.max() <= 127
    c = (a - mean).astype(np.float32)
    for g in range(4):
        cg = c[g * 256:(g + 1) * 256]
        i = int(np.argmax(np.abs(cg)))
        assert abs(int(code[g * 256 + i])) == 127
        # nearest multiple of the step: |c - code*step| <= step/2 (+ rounding)
        kg = code[g * 256:(g + 1) * 256].astype(np.float64)
        assert np.all(np.abs(cg.astype(np.float64) - kg * step[g]) <= step[g] * (0.5 + 1e-6))


def test_double_quant_exact_when_values_on_grid():
    mean = np.float32(0.25)
    stepv = np.float32(2.0 ** -10)
    k = np.arange(-127, 128, dtype=np.int64)
    a = (mean + (k * stepv).astype(np.float32)).astype(np.float32)
    a = np.concatenate([a, [mean]]).astype(np.float32)  # 256 values, mean exactly 0.25
    code, step, m, _ = nf4.double_quantize(a, 256)
    assert m == mean and step[0] == np.float32(np.float32(127 * stepv) / np.float32(127))
    assert np.array_equal(nf4.double_dequantize(code, step, m, 256), a)


def test_zero_and_constant_absmax_give_zero_step():
    a = np.full(300, 0.5, dtype=np.float32)
    code, step, mean, _ = nf4.double_quantize(a, 256)
    assert np.all(step == 0) and np.all(code == 0) and mean == np.float32(0.5)
    assert np.all(nf4.double_dequantize(code, step, mean, 256) == 0.5)


def test_all_zero_weight_matrix():
    qt = nf4.quantize(np.zeros((2, 128), dtype=np.uint16))
    assert np.all(qt["packed"] == 0x77)
    assert np.all(bf16_bits_to_f32(nf4.dequantize(qt)) == 0)


# --------------------------------------------------------------------------- pages' figures

def test_constant_storage_matches_pages_double_quant_saving():
    g = json.load(open(GOLDEN))
    before = nf4.constant_bits_per_param(8192, 8192, 64, 0)
    after = nf4.constant_bits_per_param(8192, 8192, 64, 256)
    assert before == 0.5
    assert abs(after - (8 / 64 + 32 / (64 * 256) + 32 / 8192 ** 2)) < 1e-12
    saving = before - after
    assert round(saving, 2) == g["dq_saving_bits_per_param"]["value"]
    gb = saving * g["dq_saving_65b_gigabytes"]["params"] / 8 / 1e9
    assert round(gb) == g["dq_saving_65b_gigabytes"]["value"]


def test_quantized_arrays_have_the_counted_sizes():
    qt = nf4.quantize(_weights(8, 4096, 8, outliers=False))
    n = 8 * 4096
    assert qt["packed"].size == n // 2
    assert qt["code"].size == n // 64 and qt["step"].size == (n // 64 + 255) // 256
    bits = (qt["code"].nbytes * 8 + qt["step"].nbytes * 8 + 32) / n
    assert bits == nf4.constant_bits_per_param(8, 4096)


# --------------------------------------------------------------------------- FP4 comparison table

def test_fp4_table_is_the_e2m1_value_set_scaled_to_unit_range():
    """E2M1 has 16 encodings, 15 distinct values: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}
    (the format's definition, written out); scaled by 1/6 and ascending, with
    the 16th entry repeating +1 and the zero (+0) at index 7."""
    v = nf4.e2m1_values()
    assert v.size == 16 and np.unique(v).size == 15
    spec = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert sorted(set(np.abs(v).tolist())) == spec
    q = nf4.fp4_levels()
    assert q.dtype == np.float32 and q.shape == (16,)
    want = np.array([-x / 6 for x in reversed(spec[1:])] + [x / 6 for x in spec] + [1.0], dtype=np.float32)
    assert np.array_equal(q.view(np.uint32), want.view(np.uint32))
    assert q[nf4.ZERO_CODE].view(np.uint32) == 0  # +0
    assert np.all(np.diff(q[:15].astype(np.float64)) > 0) and q[14] == q[15] == 1.0
    assert np.array_equal(q[:15], -q[14::-1])  # symmetric


def test_fp4_nearest_code_is_brute_force_argmin():
    q = nf4.fp4_levels().astype(np.float64)
    x = np.linspace(-1.0, 1.0, 200_001).astype(np.float32)
    mids = ((q[:-1] + q[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, np.nextafter(mids, np.float32(2)), np.nextafter(mids, np.float32(-2))])
    x = x[np.abs(x) <= 1.0]  # quotients w / absmax never leave [-1, 1]
    d = np.abs(x.astype(np.float64)[:, None] - q[None, :])
    brute = np.argmin(d, axis=1)  # first minimum: ties to the lower index
    got = nf4.nearest_code(x, nf4.fp4_levels())
    assert np.array_equal(got, brute)
    assert got.max() == 14  # the repeated +1 is never chosen


def test_fp4_round_trip_error_bound():
    """|w - w_hat| <= m g/2 + 2^-8 |w_hat| with g the largest FP4 level gap
    (1/3, between 2/3 and 1), without double quantization."""
    from bit_nf4_quantized_38_b300.workloads import bf16_bits, normal_with_outliers_bf16
    W = bf16_bits(normal_with_outliers_bf16((64, 1024), 0.02, 0.001, 20.0, 3))
    qt = nf4.quantize(W, dq_blocksize=0, quant_type=nf4.QT_FP4)
    wh = bf16_bits_to_f32(nf4.dequantize(qt)).astype(np.float64)
    w = bf16_bits_to_f32(W).astype(np.float64)
    m = np.repeat(qt["absmax"].reshape(64, 16), 64, axis=1).astype(np.float64)
    q = nf4.fp4_levels().astype(np.float64)
    g = np.max(np.diff(q[:15]))
    assert abs(g - 1 / 3) < 1e-7
    assert np.all(np.abs(w - wh) <= m * g / 2 * (1 + 1e-6) + 2.0 ** -8 * np.abs(wh))


# --------------------------------------------------------------------------- E4M3 second level (R21)

def test_e4m3_table_is_the_format_definition():
    """Closed-form facts of E4M3 (sign, 4-bit exponent with bias 7, 3-bit
    mantissa, subnormals at exponent 0, no infinities, one NaN per sign)."""
    v = nf4.e4m3_values()
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.isfinite(v).sum() == 254
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                          # 0x00 .. 0x7E strictly increasing
    assert pos[0] == 0.0 and pos[0x7E] == 448.0 and pos[0x08] == 2.0 ** -6
    assert np.array_equal(pos[:8], np.arange(8) * 2.0 ** -9)  # subnormals
    assert pos[0x38] == 1.0 and pos[0x30] == 0.5 and pos[0x7D] == 416.0
    assert np.array_equal(-v[0x80:0xFF], pos)                 # sign bit
    # 3 mantissa bits: within every binade the 8 values are evenly spaced
    for e in range(1, 16):
        seg = pos[8 * e:8 * e + 8] if e < 15 else pos[0x78:0x7F]
        assert np.allclose(np.diff(seg), 2.0 ** (e - 7) / 8)


def test_e4m3_coding_is_brute_force_nearest_with_even_ties():
    """Every code is the nearest E4M3 value (argmin over all finite values),
    an exact tie going to the even byte; checked on random values, all the
    exact midpoints between neighbours and their fp32 neighbours, and the
    saturating range."""
    pos = nf4.e4m3_values()[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(21)
    x = np.concatenate([
        rng.uniform(-460, 460, 4000), rng.uniform(-1, 1, 4000) * 2.0 ** rng.integers(-12, 9, 4000),
        mids, -mids, np.nextafter(mids.astype(np.float32), 0), np.nextafter(mids.astype(np.float32), 1000),
        [0.0, 448.0, 449.0, 463.9, 464.0, 1e30, -1e30]]).astype(np.float32)
    got = nf4.e4m3_codes(x)
    a = np.abs(x.astype(np.float64))
    d = np.abs(a[:, None] - pos[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # tie rule: the even byte among the nearest ones
    expect = np.array([np.flatnonzero(c)[np.argmin(np.flatnonzero(c) % 2)] if c.sum() > 1 else np.flatnonzero(c)[0]
                       for c in cand])
    expect = np.where(a >= 448.0, 0x7E, expect)  # saturation (fp64 distances to 1e30 all round alike)
    expect = np.where(np.signbit(x), expect | 0x80, expect)
    assert np.array_equal(got, expect.astype(np.uint8))
    # hand cases from the definition
    assert list(nf4.e4m3_codes(np.array([1.0625, 1.1875, 432.0, 7.5 * 2 ** -9, 1.5 * 2 ** -9, -0.0], np.float32))) == \
        [0x38, 0x3A, 0x7E, 0x08, 0x02, 0x80]


def test_e4m3_double_quant_round_trip_bound():
    """|m - m_hat| <= half an E4M3 spacing of the quotient times the step, plus
    the fp32 roundings; the group maximum codes to 448 exactly."""
    rng = np.random.default_rng(22)
    a = (rng.random(1000) * 0.05 + 0.02).astype(np.float32)
    code, step, mean, _ = nf4.double_quantize(a, 256, nf4.DQ_E4M3)
    assert not np.any(code.view(np.uint8) & 0x7F == 0x7F)
    vals = nf4.dq_code_values(code, nf4.DQ_E4M3)
    assert np.abs(vals).max() <= 448.0
    c = (a - mean).astype(np.float32).astype(np.float64)
    st = np.repeat(step, 256)[:a.size].astype(np.float64)
    for g in range(4):
        i = g * 256 + int(np.argmax(np.abs(c[g * 256:(g + 1) * 256])))
        assert abs(vals[i]) == 448.0
    q = c / st
    spacing = np.where(np.abs(q) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6))) - 3))
    mh = nf4.double_dequantize(code, step, mean, 256, nf4.DQ_E4M3).astype(np.float64)
    ulp = np.spacing(np.abs(mh).astype(np.float32) + np.float32(step.max())).astype(np.float64)
    assert np.all(np.abs(a - mh) <= st * (spacing / 2 + 2.0 ** -20) + 2 * ulp)


def test_e4m3_double_quant_exact_on_grid_and_zero_step():
    mean = np.float32(0.25)
    stv = np.float32(2.0 ** -12)
    pos = nf4.e4m3_values()[:0x7F]
    ks = np.concatenate([-pos[::-1], pos])[::2]  # E4M3 values, -448 .. 448
    a = (mean + (ks * stv).astype(np.float32)).astype(np.float32)
    a = np.concatenate([a, np.full(256 - a.size, mean)]).astype(np.float32)
    code, step, m, _ = nf4.double_quantize_codes(a, mean, 256, nf4.DQ_E4M3) + (mean, None)
    assert step[0] == np.float32(np.float32(448 * stv) / np.float32(448))
    assert np.array_equal(nf4.double_dequantize(code, step, mean, 256, nf4.DQ_E4M3), a)
    z = np.full(300, 0.5, dtype=np.float32)
    code, step, mean, _ = nf4.double_quantize(z, 256, nf4.DQ_E4M3)
    assert np.all(step == 0) and np.all(code == 0)
