"""The E4M3 forward and dX of the frozen-NF4 linear -- CPU oracle (test infrastructure only).

What the pages fix: the QLoRA project page's configuration example sets the
compute dtype of the 4-bit layer (bnb_4bit_compute_dtype = bfloat16); the
layer computes Y = X W_hat^T + s (X A) B (QLoRA abstract; LoRA tutorial,
h = W x + dW x).  The pages say nothing about 8-bit floats.

Reading R22 (the FP8 variant of that compute dtype; plainest choices):
  * operands in E4M3 (R21: nearest value, ties to the even code, saturating
    at 448, the sign kept);
  * the weight before its bf16 rounding, fl32(q[code] * m_hat), scaled by one
    power of two 2^E for the whole tensor: the largest with
    max |m_hat| * 2^E <= 448 (E = 0 when that maximum is 0; exact scaling);
  * X per row m by the same rule: E_m the largest integer with
    amax_m * 2^E_m <= 448 (0 for an all-zero row), codes of x * 2^E_m (exact
    scaling) -- a power of two rather than amax / 448, so that every scaling
    is exact and no division rounds;
  * Y[m] = 2^(-E_m - E) * (Xq Wq^T) + s (X A) B -- the main product of the
    E4M3 values exactly (fp64 here, fp32 accumulation on the GPU), the LoRA
    term in the same precision as the bf16 forward.
Reading R24 (the backward, QLoRA abstract: gradients flow through the frozen
4-bit weight into the adapters): the dX product dY W_hat takes the same E4M3
weight Wq (same E) and dY coded per row by the X-row rule; G = dY B^T comes
from the bf16 dY, so dX[m] = 2^(-E_m - E) (dYq Wq) + s G A^T; dA and dB are
the bf16 backward's (no 8-bit operand enters them).
Parity: the quantized operands are pinned by the E4M3 coder's own pins and by
closed-form checks of the scale rules; the product is a library matmul.
"""
import math

import numpy as np

from . import nf4
from .bf16 import bf16_bits_to_f32, bf16_bits_to_f64


def weight_exponent(maxm):
    """E of R22: the largest integer with maxm * 2^E <= 448 (0 for maxm = 0),
    clamped to [-60, 60]."""
    maxm = float(np.float32(maxm))
    if not maxm > 0:
        return 0
    mf, ef = math.frexp(maxm)          # maxm = mf 2^ef, mf in [0.5, 1)
    f, e = 2.0 * mf, ef - 1            # maxm = f 2^e, f in [1, 2)
    return max(-60, min(60, (8 if f <= 1.75 else 7) - e))


def weight_products_f32(qt):
    """fl32(q[code] * m_hat) for every weight element (rows x cols float32)."""
    R, C, bs = qt["rows"], qt["cols"], qt["blocksize"]
    codes = nf4.unpack_nibbles(qt["packed"]).reshape(R, C)
    q = nf4.code_levels(qt.get("quant_type", nf4.QT_NF4))
    mh = np.repeat(nf4.absmax_hat(qt).reshape(R, C // bs), bs, axis=1).astype(np.float32)
    return (q[codes.astype(np.int64)] * mh).astype(np.float32)


def weight_e4m3(qt):
    """(E, Wq as fp64 values R x C) of R22."""
    E = weight_exponent(np.abs(nf4.absmax_hat(qt)).max())
    scaled = (weight_products_f32(qt) * np.float32(math.ldexp(1.0, E))).astype(np.float32)
    return E, nf4.e4m3_values()[nf4.e4m3_codes(scaled)].reshape(scaled.shape)


def rows_e4m3(x_bits):
    """(row exponents E_m int[M], Xq fp64 values M x K) of R22."""
    x = bf16_bits_to_f32(np.asarray(x_bits, dtype=np.uint16))
    Em = np.array([weight_exponent(a) for a in np.abs(x).max(axis=1)], dtype=np.int64)
    xs = (x * np.ldexp(np.float32(1.0), Em).astype(np.float32)[:, None]).astype(np.float32)
    return Em, nf4.e4m3_values()[nf4.e4m3_codes(xs)].reshape(x.shape)


def lora_forward_e4m3(x_bits, qt, a_bits, b_bits, s):
    """Y (fp64, M x N) of R22, and (E, E_m, row factors 2^(-E_m - E))."""
    E, wq = weight_e4m3(qt)
    Em, xq = rows_e4m3(x_bits)
    rs = np.ldexp(1.0, -Em - E)
    x = bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16))
    lora = float(s) * ((x @ bf16_bits_to_f64(a_bits)) @ bf16_bits_to_f64(b_bits))
    return rs[:, None] * (xq @ wq.T) + lora, (E, Em, rs)


def lora_backward_e4m3(dy_bits, qt, a_bits, b_bits, s):
    """dX (fp64, M x K) of R24, and (E, E_m of the dY rows, row factors 2^(-E_m - E))."""
    E, wq = weight_e4m3(qt)
    Em, dyq = rows_e4m3(dy_bits)
    rs = np.ldexp(1.0, -Em - E)
    dy = bf16_bits_to_f64(np.asarray(dy_bits, dtype=np.uint16))
    lora = float(s) * ((dy @ bf16_bits_to_f64(b_bits).T) @ bf16_bits_to_f64(a_bits).T)
    return rs[:, None] * (dyq @ wq) + lora, (E, Em, rs)
