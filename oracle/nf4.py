"""NF4 quantization with double quantization -- CPU oracle (test infrastructure only).

What the pages fix:
  * 4-bit NormalFloat (NF4) is a 4-bit data type that is information-
    theoretically optimal for normally distributed weights and beats 4-bit
    integers and 4-bit floats (arXiv 2305.14314 abstract page, innovation (a);
    QLoRA news write-up, list of innovations, first item).
  * Quantization is blockwise with one quantization constant per block, and
    double quantization quantizes those constants, saving about 0.37 bit per
    parameter, about 3 GB for a 65B model (news write-up, "Double
    Quantization" item; Finnish summary, item (2)).

Readings taken where the pages are silent:
  R1 Codebook.  "Quantiles of N(0,1) normalised to [-1, 1] with an exact zero":
     16 levels with both endpoints and an exact zero cannot be symmetric, so
     the positive side gets 8 levels and the negative side 7.  The positive
     levels are the standard-normal quantiles at 8 probabilities equally
     spaced from DELTA down towards 1/2 (9 points, the 1/2 end dropped), the
     negative levels are the negated quantiles at 7 probabilities equally
     spaced from DELTA towards 1/2 (8 points, the 1/2 end dropped), zero is
     added, and everything is divided by the quantile at DELTA so the
     endpoints are exactly -1 and +1.  DELTA = 1 - (1/32 + 1/30)/2, the mean
     of the outermost tail probabilities of symmetric 16- and 15-level
     quantile grids.  The levels are built in fp64 and rounded once to fp32;
     those 16 fp32 values are the codebook.
  R2 Block size 64 over consecutive elements of a row-major matrix (every row
     length is a multiple of 64, so blocks never straddle rows).
  R3 The code of an element is the index of the nearest codebook level to
     x = fl32(w / absmax); an exact tie goes to the lower index.  An all-zero
     block (absmax 0) codes every element as the zero level (index 7).
  R4 Nibble packing: element 2j goes to the high nibble of byte j.
  R5 Double quantization: the second level is a symmetric linear int8 code of
     the mean-subtracted block absmax values in groups of 256 consecutive
     blocks: mu = fl32(S / n_b) with S the fp64 sum of all block absmax values
     (exact for real weights, checked); c = fl32(absmax - mu);
     step = fl32(max|c| / 127) per group; code = clamp(rne(fl32(c / step)),
     -127, 127) (0 when step is 0).  Decode: fl32(fl32(code * step) + mu),
     with no fused multiply-add.
  R6 Dequantized weight: w_hat = bf16_rne(fl32(q[code] * absmax_hat)).
  R21 The second-level code may instead be an 8-bit float (the pages only
     say the constants are quantized): E4M3, the plainest 8-bit float that
     keeps 3 mantissa bits (1 sign bit, 4 exponent bits with bias 7,
     subnormals m * 2^-9 at exponent 0, largest finite 448, no infinities;
     bytes 0x7F/0xFF are NaN and never produced).  Same groups and mu as R5;
     step = fl32(max|c| / 448); code = the E4M3 value nearest to
     fl32(c / step), ties to the even code (mantissa bit 0 clear), magnitudes
     above 448 saturating to 448, the sign of the quotient kept (a negative
     quotient that rounds to zero is byte 0x80); decode
     fl32(fl32(value(code) * step) + mu).
  R17 FP4 (the 4-bit float the pages say NF4 beats; its format is not on the
     pages): the plainest 4-bit float, E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6
     and negatives), scaled by 1/6 to [-1, 1]; codes index the ascending
     table of its 15 distinct values (zero at 7, as for NF4), the 16th entry
     repeating +1.  Coding, packing, double quantization and dequantization
     are the same as for NF4 with this table.

Parity: the codebook, coding, packing, DQ and dequantization are pinned by
tests against closed forms, brute force and error bounds; the exact codebook
digits, R3's tie rule, R4's order and R5's int8-linear second level are
conventions (no page prints them): parity unpinned for those choices as such,
they are fixed by reading.
"""
import math

import numpy as np
from scipy.special import ndtri

from .bf16 import bf16_bits_to_f32, f32_to_bf16_bits

BLOCKSIZE = 64
DQ_BLOCKSIZE = 256
DQ_INT8, DQ_E4M3 = 0, 1  # second-level codes (R5, R21)
ZERO_CODE = 7

# R1: outer probability of the asymmetric quantile grid.
DELTA = 1.0 - 0.5 * (1.0 / 32.0 + 1.0 / 30.0)


def normal_quantile(p):
    """Standard normal quantile Phi^-1(p) in fp64 (scipy's ndtri)."""
    return ndtri(np.asarray(p, dtype=np.float64))


def nf4_probabilities():
    """Probabilities whose quantiles give the positive and negative levels (R1)."""
    pos = np.linspace(DELTA, 0.5, 9)[:-1]  # 8 values, DELTA first
    neg = np.linspace(DELTA, 0.5, 8)[:-1]  # 7 values, DELTA first
    return pos, neg


def nf4_levels_f64():
    """The 16 NF4 levels in fp64, ascending (R1)."""
    pos_p, neg_p = nf4_probabilities()
    z_max = normal_quantile(DELTA)
    pos = normal_quantile(pos_p) / z_max
    neg = -normal_quantile(neg_p) / z_max
    levels = np.sort(np.concatenate([neg, [0.0], pos]))
    return levels


def nf4_levels():
    """The NF4 codebook: the fp64 levels rounded once to fp32 (R1)."""
    return nf4_levels_f64().astype(np.float32)


QT_NF4, QT_FP4 = 0, 1


def e2m1_values():
    """Every value of the 4-bit float E2M1 (1 sign, 2 exponent, 1 mantissa
    bit, exponent bias 1, no infinities or NaN): exponent field 0 gives the
    subnormals 0 and 0.5; field e > 0 gives 2^(e-1) (1 + m/2).  16 encodings."""
    vals = []
    for s in (0, 1):
        for e in range(4):
            for m in (0, 1):
                mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
                vals.append(-mag if s else mag)
    return np.array(vals, dtype=np.float64)


def fp4_levels():
    """The FP4 comparison code table (reading R17): the distinct E2M1 values
    divided by the largest magnitude (6) so the endpoints are -1 and +1,
    ascending (15 values, one zero at index 7), rounded once to fp32, with a
    16th entry repeating +1 (the nearest-level rule with ties to the lower
    index never picks it)."""
    v = e2m1_values()
    distinct = np.unique(v) + 0.0  # -0 and +0 compare equal: one zero, made +0
    lv = (distinct / np.max(np.abs(distinct))).astype(np.float32)
    return np.concatenate([lv, lv[-1:]])


def code_levels(quant_type=QT_NF4):
    """The 16-entry level table a quant type's 4-bit codes index."""
    if quant_type == QT_NF4:
        return nf4_levels()
    if quant_type == QT_FP4:
        return fp4_levels()
    raise ValueError(f"quant type {quant_type}")


def nf4_midpoints(levels=None):
    """Decision thresholds t_j = (q_j + q_{j+1}) / 2 of the fp32 code table, exact in fp64."""
    q = (nf4_levels() if levels is None else np.asarray(levels, np.float32)).astype(np.float64)
    return (q[:-1] + q[1:]) / 2.0


def nearest_code(x, levels=None):
    """Index of the nearest fp32 level to each fp32 x (ties to the lower index, R3).

    code = #{ j : x > t_j } over the 15 exact fp64 midpoints (NF4 by default).
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    t = nf4_midpoints(levels)
    return (x[..., None] > t).sum(axis=-1).astype(np.uint8)


def block_absmax(w_f32, blocksize=BLOCKSIZE):
    """Per-block max |w| over consecutive groups of `blocksize` in each row (R2).

    w_f32: (rows, cols) float32 with cols % blocksize == 0.
    Returns float32 (rows, cols // blocksize).
    """
    rows, cols = w_f32.shape
    assert cols % blocksize == 0
    return np.abs(w_f32.reshape(rows, cols // blocksize, blocksize)).max(axis=2)


def nf4_codes(w_f32, absmax, blocksize=BLOCKSIZE, rows_per_chunk=512, levels=None):
    """NF4 code of every element, given its block's absmax (R3).

    x = fl32(w / absmax) as an IEEE single division; all-zero blocks code to 7.
    Rows are processed in chunks only to bound memory.
    """
    rows, cols = w_f32.shape
    nb = cols // blocksize
    out = np.empty((rows, cols), dtype=np.uint8)
    for r0 in range(0, rows, rows_per_chunk):
        r1 = min(rows, r0 + rows_per_chunk)
        w3 = w_f32[r0:r1].reshape(r1 - r0, nb, blocksize)
        m = absmax[r0:r1].reshape(r1 - r0, nb, 1).astype(np.float32)
        zero = m == 0
        safe = np.where(zero, np.float32(1.0), m)
        x = (w3 / safe).astype(np.float32)
        codes = nearest_code(x, levels)
        codes = np.where(zero, np.uint8(ZERO_CODE), codes)
        out[r0:r1] = codes.reshape(r1 - r0, cols)
    return out


def pack_nibbles(codes):
    """Pack codes two per byte, element 2j in the high nibble of byte j (R4)."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1)
    assert c.size % 2 == 0
    return ((c[0::2] << 4) | c[1::2]).astype(np.uint8)


def unpack_nibbles(packed):
    """Inverse of pack_nibbles."""
    p = np.asarray(packed, dtype=np.uint8).reshape(-1)
    out = np.empty(p.size * 2, dtype=np.uint8)
    out[0::2] = p >> 4
    out[1::2] = p & 0x0F
    return out


def exact_sum_f64(values_f32):
    """fp64 sum of non-negative fp32 values, and whether fp64 holds it exactly.

    The sum is computed exactly in integer arithmetic (every fp32 value is an
    integer multiple of 2**g for the smallest exponent g present) and then
    rounded once to fp64.  When the exact sum fits in 53 bits, every order of
    fp64 summation gives this same value.
    """
    v = np.asarray(values_f32, dtype=np.float32).reshape(-1)
    nz = v[v != 0].astype(np.float64)
    if nz.size == 0:
        return 0.0, True
    mant, expo = np.frexp(nz)  # nz = mant * 2**expo, 0.5 <= mant < 1
    k = (mant * 2.0 ** 24).astype(np.int64)  # exact: fp32 has 24 significant bits
    e = expo.astype(np.int64) - 24
    g = int(e.min())
    span = int(e.max()) - g
    if span + 24 + math.ceil(math.log2(nz.size + 1)) <= 62:
        total = int(np.sum(k << (e - g)))
    else:
        total = sum(int(ki) << int(ei - g) for ki, ei in zip(k, e))
    tz = (total & -total).bit_length() - 1
    exact = (total >> tz).bit_length() <= 53
    return math.ldexp(float(total), g) if exact else float(
        math.fsum(nz.tolist())), exact


def e4m3_values():
    """Values of the 256 E4M3 bytes (R21), fp64: sign * 2^(e-7) * (1 + m/8) for
    exponent field e > 0, sign * m * 2^-9 for e = 0; NaN for 0x7F and 0xFF."""
    v = np.empty(256, dtype=np.float64)
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        mag = math.ldexp(1.0 + m / 8.0, e - 7) if e else math.ldexp(float(m), -9)
        v[b] = math.nan if (e == 15 and m == 7) else (-mag if s else mag)
    return v


def e4m3_codes(x):
    """E4M3 byte of each fp32 x (R21): nearest value, ties to the even code,
    saturating at 448, sign of x kept."""
    x = np.asarray(x, dtype=np.float32).reshape(-1)
    pos = e4m3_values()[:0x7F]  # 0x00 .. 0x7E: 0 .. 448, strictly increasing
    a = np.abs(x.astype(np.float64))
    hi = np.clip(np.searchsorted(pos, a, side="left"), 0, 0x7E)  # first value >= a (or the top)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - pos[lo], pos[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(a >= pos[0x7E], 0x7E, np.where(pick_hi, hi, lo)).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def dq_code_values(code, dq_type=DQ_INT8):
    """Values of second-level code bytes (int8 storage): the int8 itself, or the E4M3 value."""
    code = np.asarray(code, dtype=np.int8).reshape(-1)
    if dq_type == DQ_E4M3:
        return e4m3_values()[code.view(np.uint8)].astype(np.float32)
    return code.astype(np.float32)


def double_quantize(absmax, dq_blocksize=DQ_BLOCKSIZE, dq_type=DQ_INT8):
    """Second-level code of the mean-subtracted block absmax values (R5, or R21 for E4M3).

    absmax: float32 vector of n_b block absmax values in block order
    (row-major over (row, block-in-row)).
    Returns (code int8[n_b], step float32[n_2], mean float32, mean_exact bool).
    """
    a = np.asarray(absmax, dtype=np.float32).reshape(-1)
    n_b = a.size
    S, exact = exact_sum_f64(a)
    mean = dq_mean_from_sum(S, n_b)
    code, step = double_quantize_codes(a, mean, dq_blocksize, dq_type)
    return code, step, mean, exact


def dq_mean_from_sum(S, n_b):
    """mu = fl32(S / n_b): the fp64 sum of all block absmax values over their count (R5)."""
    return np.float32(float(S) / float(n_b))


def double_quantize_codes(absmax, mean, dq_blocksize=DQ_BLOCKSIZE, dq_type=DQ_INT8):
    """The second-level codes and steps of consecutive block absmax values,
    given the mean mu (R5; R21 for E4M3): groups of dq_blocksize start at the
    first value.  Returns (code int8[n] -- E4M3 bytes viewed as int8 --,
    step float32[ceil(n / dq_blocksize)])."""
    a = np.asarray(absmax, dtype=np.float32).reshape(-1)
    n_b = a.size
    mean = np.float32(mean)
    c = (a - mean).astype(np.float32)
    n_2 = (n_b + dq_blocksize - 1) // dq_blocksize
    code = np.zeros(n_b, dtype=np.int8)
    step = np.zeros(n_2, dtype=np.float32)
    for g in range(n_2):
        cg = c[g * dq_blocksize:(g + 1) * dq_blocksize]
        a2 = np.float32(np.abs(cg).max())
        st = np.float32(a2 / np.float32(448.0 if dq_type == DQ_E4M3 else 127.0))
        step[g] = st
        if st == 0:
            continue
        x = (cg / st).astype(np.float32)
        if dq_type == DQ_E4M3:
            code[g * dq_blocksize:(g + 1) * dq_blocksize] = e4m3_codes(x).view(np.int8)
        else:
            code[g * dq_blocksize:(g + 1) * dq_blocksize] = np.clip(np.rint(x), -127, 127).astype(np.int8)
    return code, step


def double_dequantize(code, step, mean, dq_blocksize=DQ_BLOCKSIZE, dq_type=DQ_INT8):
    """absmax_hat = fl32(fl32(value(code) * step) + mean), no FMA (R5, R21)."""
    code = np.asarray(code, dtype=np.int8).reshape(-1)
    st = np.repeat(np.asarray(step, dtype=np.float32), dq_blocksize)[:code.size]
    prod = (dq_code_values(code, dq_type) * st).astype(np.float32)
    return (prod + np.float32(mean)).astype(np.float32)


def dequantize_codes(codes, absmax_hat, blocksize=BLOCKSIZE, levels=None):
    """w_hat = bf16_rne(fl32(q[code] * absmax_hat)) (R6); returns bf16 bits, same shape as codes."""
    rows, cols = codes.shape
    q = nf4_levels() if levels is None else np.asarray(levels, np.float32)
    vals = q[codes.astype(np.int64)].reshape(rows, cols // blocksize, blocksize)
    prod = (vals * absmax_hat.reshape(rows, cols // blocksize, 1).astype(np.float32)).astype(np.float32)
    return f32_to_bf16_bits(prod.reshape(rows, cols))


def quantize(w_bits, blocksize=BLOCKSIZE, dq_blocksize=DQ_BLOCKSIZE, quant_type=QT_NF4, dq_type=DQ_INT8):
    """Quantize a bf16 (rows, cols) weight matrix given as uint16 bit patterns.

    Returns a dict with: rows, cols, blocksize, dq_blocksize, quant_type,
    packed (uint8, rows*cols/2), absmax (float32, n_b), and, when
    dq_blocksize > 0, code (int8, n_b), step (float32, n_2), mean (float32),
    mean_exact (bool), dq_type.  quant_type selects the code table (NF4, or FP4
    for comparison); dq_type the second-level code (int8, or E4M3).
    """
    w_bits = np.asarray(w_bits, dtype=np.uint16)
    rows, cols = w_bits.shape
    w = bf16_bits_to_f32(w_bits)
    absmax = block_absmax(w, blocksize)
    codes = nf4_codes(w, absmax, blocksize, levels=code_levels(quant_type))
    out = dict(rows=rows, cols=cols, blocksize=blocksize, dq_blocksize=dq_blocksize, quant_type=quant_type,
               packed=pack_nibbles(codes), absmax=absmax.reshape(-1))
    if dq_blocksize:
        code, step, mean, exact = double_quantize(absmax.reshape(-1), dq_blocksize, dq_type)
        out.update(code=code, step=step, mean=mean, mean_exact=exact, dq_type=dq_type)
    return out


def absmax_hat(qt):
    """The block constants the dequantizer uses: decoded DQ values, or the fp32 absmax."""
    if qt["dq_blocksize"]:
        return double_dequantize(qt["code"], qt["step"], qt["mean"], qt["dq_blocksize"],
                                 qt.get("dq_type", DQ_INT8))
    return np.asarray(qt["absmax"], dtype=np.float32)


def dequantize(qt, rows=None):
    """Dequantize a quantized tensor to bf16 bits (rows x cols), optionally only some rows."""
    R, C, bs = qt["rows"], qt["cols"], qt["blocksize"]
    codes = unpack_nibbles(qt["packed"]).reshape(R, C)
    mh = absmax_hat(qt).reshape(R, C // bs)
    if rows is not None:
        codes, mh = codes[rows], mh[rows]
    return dequantize_codes(codes, mh, bs, levels=code_levels(qt.get("quant_type", QT_NF4)))


def constant_bits_per_param(rows, cols, blocksize=BLOCKSIZE, dq_blocksize=DQ_BLOCKSIZE):
    """Bits of quantization constants per parameter, counted from the stored arrays.

    Without DQ: one fp32 absmax per block.  With DQ: one int8 code per block,
    one fp32 step per group of dq_blocksize blocks, one fp32 mean per tensor.
    """
    n = rows * cols
    n_b = n // blocksize
    if not dq_blocksize:
        return 32.0 * n_b / n
    n_2 = (n_b + dq_blocksize - 1) // dq_blocksize
    return (8.0 * n_b + 32.0 * n_2 + 32.0) / n
