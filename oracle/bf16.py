"""bfloat16 <-> float32 conversions for the oracle (test infrastructure only).

bfloat16 is the compute dtype of the method ("QLoRA" project description page,
configuration example: 4-bit compute dtype torch.bfloat16).  numpy has no
bfloat16 type, so bf16 values are carried as their uint16 bit patterns.

Rounding is IEEE-754 round-to-nearest, ties-to-even, to an 8-bit significand
(1 implicit + 7 stored bits) with the fp32 exponent range.  Only finite inputs
are handled (the method's inputs are finite).

Pinned in tests against torch's own float32 -> bfloat16 conversion (a library
routine) on every tie class and on random values.
"""
import numpy as np


def f32_to_bf16_bits(x):
    """Round float32 values to bfloat16 (RNE); return uint16 bit patterns."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    # Keep the top 16 bits; the discarded low half decides the rounding.
    low = u & 0xFFFF
    keep = u >> 16
    lsb = keep & 1
    round_up = (low > 0x8000) | ((low == 0x8000) & (lsb == 1))
    out = keep + round_up.astype(np.uint64)
    return out.astype(np.uint16)


def bf16_bits_to_f32(b):
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b):
    return bf16_bits_to_f32(b).astype(np.float64)


def f64_to_bf16_bits_via_f32(x):
    """Round an fp64 value to fp32 (RNE) and then to bf16 (RNE)."""
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float64).astype(np.float32))
