"""Pins of the E4M3-forward oracle (oracle/fp8.py) against closed forms and a
brute-force restatement on tiny inputs."""
import math

import numpy as np
import pytest

from oracle import fp8, linear, nf4
from oracle.bf16 import bf16_bits_to_f32, f32_to_bf16_bits


def _bits(a):
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_weight_exponent_is_the_largest_fitting_power_of_two():
    rng = np.random.default_rng(31)
    vals = np.concatenate([rng.random(2000) * 10.0 ** rng.integers(-6, 6, 2000), [448.0, 1.75, 1.7500001, 224.0,
                                                                                     0.0123, 1e-30]])
    for m in vals.astype(np.float32):
        E = fp8.weight_exponent(m)
        if E == 60:  # clamped: any larger power would still fit
            assert float(m) * 2.0 ** 60 <= 448.0
            continue
        assert float(m) * 2.0 ** E <= 448.0 < float(m) * 2.0 ** (E + 1)
    assert fp8.weight_exponent(448.0) == 0 and fp8.weight_exponent(1.75) == 8 and fp8.weight_exponent(0.0) == 0


def test_row_codes_use_the_top_binade_and_bound_the_error():
    rng = np.random.default_rng(32)
    x = (rng.standard_normal((6, 256)) * 10.0 ** rng.integers(-3, 3, (6, 1))).astype(np.float32)
    x[5] = 0.0
    xb = _bits(x)
    xf = bf16_bits_to_f32(xb).astype(np.float64)
    Em, xq = fp8.rows_e4m3(xb)
    assert Em[5] == 0 and np.all(xq[5] == 0)
    for m in range(5):
        amax = np.abs(xf[m]).max()
        assert amax * 2.0 ** Em[m] <= 448.0 < amax * 2.0 ** (Em[m] + 1)
        assert 224.0 <= np.abs(xq[m]).max() <= 448.0
        # half an E4M3 spacing (3 mantissa bits, subnormal spacing 2^-9) of the exactly scaled value
        qv = xf[m] * 2.0 ** Em[m]
        sp = np.where(np.abs(qv) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(qv), 2 ** -6))) - 3))
        assert np.all(np.abs(xq[m] - qv) <= sp / 2)


def _e4m3_brute(v):
    """Nearest finite E4M3 value by a plain loop over all 254 finite codes (ties: even code)."""
    vals = nf4.e4m3_values()
    best, bc = None, None
    a = abs(float(v))
    if a >= 448.0:
        return math.copysign(448.0, v)
    for c in range(0x7F):
        d = abs(vals[c] - a)
        if best is None or d < best or (d == best and c % 2 == 0):
            best, bc = d, c
    return math.copysign(vals[bc], v) if not (vals[bc] == 0 and not math.copysign(1, v) < 0) else vals[bc]


def test_forward_matches_a_plain_loop_on_a_tiny_case():
    rng = np.random.default_rng(33)
    M, K, N, r, s = 3, 64, 5, 2, 0.5
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qt = nf4.quantize(_bits(W))
    X = _bits(rng.standard_normal((M, K)))
    A, B = _bits(rng.standard_normal((K, r)) * 0.3), _bits(rng.standard_normal((r, N)) * 0.1)
    Y, (E, Em, rs) = fp8.lora_forward_e4m3(X, qt, A, B, s)
    # plain restatement
    q = nf4.nf4_levels()
    codes = nf4.unpack_nibbles(qt["packed"]).reshape(N, K)
    mh = nf4.absmax_hat(qt).reshape(N, K // 64)
    maxm = max(abs(float(v)) for v in mh.ravel())
    E2 = 0
    while maxm * 2.0 ** (E2 + 1) <= 448.0:
        E2 += 1
    while maxm * 2.0 ** E2 > 448.0:
        E2 -= 1
    assert E == E2
    xf = bf16_bits_to_f32(X)
    for m in range(M):
        amax = max(abs(float(v)) for v in xf[m])
        em = 0
        while amax * 2.0 ** (em + 1) <= 448.0:
            em += 1
        while amax * 2.0 ** em > 448.0:
            em -= 1
        assert em == Em[m]
        for n in range(N):
            acc = 0.0
            for k in range(K):
                wv = _e4m3_brute(float(np.float32(np.float32(q[codes[n, k]]) * np.float32(mh[n, k // 64]))) * 2.0 ** E)
                xv = _e4m3_brute(float(xf[m, k]) * 2.0 ** em)
                acc += wv * xv
            lora = s * sum(sum(float(xf[m, k]) * float(bf16_bits_to_f32(A)[k, j]) for k in range(K))
                           * float(bf16_bits_to_f32(B)[j, n]) for j in range(r))
            ref = 2.0 ** (-em - E) * acc + lora
            assert abs(Y[m, n] - ref) <= 1e-12 * (abs(ref) + 1)


def test_e4m3_forward_stays_near_the_bf16_forward():
    """The E4M3 operands keep 3 mantissa bits (relative rounding <= 2^-4 each):
    on normal data the forward stays within a few percent of the bf16 one."""
    rng = np.random.default_rng(34)
    M, K, N, r = 64, 512, 96, 16
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qt = nf4.quantize(_bits(W))
    X = _bits(rng.standard_normal((M, K)))
    A, B = _bits(rng.standard_normal((K, r)) * 0.25), _bits(rng.standard_normal((r, N)) * 0.01)
    Y8, _ = fp8.lora_forward_e4m3(X, qt, A, B, 1.0)
    Y16, _ = linear.lora_forward(X, nf4.dequantize(qt), A, B, 1.0)
    rel = np.linalg.norm(Y8 - Y16) / np.linalg.norm(Y16)
    assert 1e-4 < rel < 0.06


def test_backward_matches_a_plain_loop_on_a_tiny_case():
    """dX of R24 restated element by element: the same E4M3 weight (E from
    max |m_hat|), dY rows coded by the X-row rule, G from the bf16 dY."""
    rng = np.random.default_rng(35)
    M, K, N, r, s = 3, 64, 6, 2, 0.75
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qt = nf4.quantize(_bits(W))
    dY = _bits(rng.standard_normal((M, N)) * 3.0)
    A, B = _bits(rng.standard_normal((K, r)) * 0.3), _bits(rng.standard_normal((r, N)) * 0.1)
    dX, (E, Em, rs) = fp8.lora_backward_e4m3(dY, qt, A, B, s)
    q = nf4.nf4_levels()
    codes = nf4.unpack_nibbles(qt["packed"]).reshape(N, K)
    mh = nf4.absmax_hat(qt).reshape(N, K // 64)
    maxm = max(abs(float(v)) for v in mh.ravel())
    E2 = 0
    while maxm * 2.0 ** (E2 + 1) <= 448.0:
        E2 += 1
    while maxm * 2.0 ** E2 > 448.0:
        E2 -= 1
    assert E == E2
    dyf, af, bf = bf16_bits_to_f32(dY), bf16_bits_to_f32(A), bf16_bits_to_f32(B)
    for m in range(M):
        amax = max(abs(float(v)) for v in dyf[m])
        em = 0
        while amax * 2.0 ** (em + 1) <= 448.0:
            em += 1
        while amax * 2.0 ** em > 448.0:
            em -= 1
        assert em == Em[m]
        g = [sum(float(dyf[m, n]) * float(bf[j, n]) for n in range(N)) for j in range(r)]
        for k in range(K):
            acc = 0.0
            for n in range(N):
                wv = _e4m3_brute(float(np.float32(np.float32(q[codes[n, k]]) * np.float32(mh[n, k // 64]))) * 2.0 ** E)
                acc += _e4m3_brute(float(dyf[m, n]) * 2.0 ** em) * wv
            ref = 2.0 ** (-em - E) * acc + s * sum(g[j] * float(af[k, j]) for j in range(r))
            assert abs(dX[m, k] - ref) <= 1e-12 * (abs(ref) + 1)


def test_e4m3_backward_stays_near_the_bf16_backward():
    rng = np.random.default_rng(36)
    M, K, N, r = 64, 256, 192, 16
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qt = nf4.quantize(_bits(W))
    dY, X = _bits(rng.standard_normal((M, N))), _bits(rng.standard_normal((M, K)))
    A, B = _bits(rng.standard_normal((K, r)) * 0.25), _bits(rng.standard_normal((r, N)) * 0.01)
    dX8, _ = fp8.lora_backward_e4m3(dY, qt, A, B, 1.0)
    dX16 = linear.lora_backward(dY, X, nf4.dequantize(qt), A, B, 1.0)[0]
    rel = np.linalg.norm(dX8 - dX16) / np.linalg.norm(dX16)
    assert 1e-4 < rel < 0.06
