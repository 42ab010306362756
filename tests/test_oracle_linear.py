"""Pins for the fp64 LoRA-linear oracle: finite differences, the merge identity
the LoRA tutorial states, the W_B = 0 start, one-hot inputs, and the pages'
parameter-count figures (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import linear

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


def _tiny(seed, M=3, K=64, N=5, r=2):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((N, K)) * 0.1
    A = rng.standard_normal((K, r))
    B = rng.standard_normal((r, N))
    R = rng.standard_normal((M, N))
    return X, W, A, B, R


def _loss(X, W, A, B, R, s):
    Y, _ = linear.lora_forward(X, W, A, B, s)
    return float(np.sum(Y * R))


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_central_finite_differences(seed):
    X, W, A, B, R = _tiny(seed)
    s = 0.75
    dX, dA, dB, _ = linear.lora_backward(R, X, W, A, B, s)
    h = 0.5  # the loss is linear in each argument: differences are exact up to rounding
    for name, P, grad in (("X", X, dX), ("A", A, dA), ("B", B, dB)):
        fd = np.zeros_like(P)
        for idx in np.ndindex(P.shape):
            Pp = P.copy(); Pp[idx] += h
            Pm = P.copy(); Pm[idx] -= h
            args = {"X": X, "A": A, "B": B}
            args[name] = Pp
            lp = _loss(args["X"], W, args["A"], args["B"], R, s)
            args[name] = Pm
            lm = _loss(args["X"], W, args["A"], args["B"], R, s)
            fd[idx] = (lp - lm) / (2 * h)
        assert np.allclose(fd, grad, rtol=1e-10, atol=1e-10), name


@pytest.mark.parametrize("seed", [3, 4])
def test_adapter_grads_alone_match_central_finite_differences(seed):
    """lora_adapter_grads (no weight argument) against finite differences of
    the full layer's loss in A and B, and lora_xa against one-hot X rows."""
    X, W, A, B, R = _tiny(seed, M=4, K=64, N=6, r=3)
    s = 1.25
    dA, dB, XA = linear.lora_adapter_grads(R, X, A, B, s)
    h = 0.5
    for name, P, grad in (("A", A, dA), ("B", B, dB)):
        fd = np.zeros_like(P)
        for idx in np.ndindex(P.shape):
            Pp = P.copy(); Pp[idx] += h
            Pm = P.copy(); Pm[idx] -= h
            if name == "A":
                lp, lm = _loss(X, W, Pp, B, R, s), _loss(X, W, Pm, B, R, s)
            else:
                lp, lm = _loss(X, W, A, Pp, R, s), _loss(X, W, A, Pm, R, s)
            fd[idx] = (lp - lm) / (2 * h)
        assert np.allclose(fd, grad, rtol=1e-10, atol=1e-10), name
    # XA: one-hot token rows read out rows of A
    E = np.zeros((3, 64)); E[np.arange(3), [1, 17, 63]] = 1.0
    assert np.array_equal(linear.lora_xa(E, A), A[[1, 17, 63]])
    assert np.allclose(XA, linear.lora_xa(X, A), rtol=0, atol=0)


def test_frozen_weight_gets_no_gradient_and_dW_would_be_nonzero():
    # dX uses W; W itself receives nothing (only dX, dA, dB are returned)
    X, W, A, B, R = _tiny(2)
    out = linear.lora_backward(R, X, W, A, B, 1.0)
    assert len(out) == 4


def test_forward_equals_merged_dense_weight():
    X, W, A, B, _ = _tiny(3, M=4, K=128, N=7, r=4)
    s = 2.0
    Y, _ = linear.lora_forward(X, W, A, B, s)
    Wm = linear.merged_weight(W, A, B, s)
    assert np.allclose(Y, X @ Wm.T, rtol=1e-12, atol=1e-12)


def test_zero_B_gives_plain_linear_and_zero_dA():
    X, W, A, B, R = _tiny(4)
    B0 = np.zeros_like(B)
    Y, _ = linear.lora_forward(X, W, A, B0, 3.0)
    assert np.array_equal(Y, X @ W.T)
    dX, dA, dB, G = linear.lora_backward(R, X, W, A, B0, 3.0)
    assert np.all(dA == 0) and np.all(G == 0)
    assert np.allclose(dX, R @ W)
    assert np.any(dB != 0)


def test_one_hot_tokens_read_out_weight_columns():
    rng = np.random.default_rng(5)
    N, K, r = 6, 64, 2
    W = rng.standard_normal((N, K))
    A = rng.standard_normal((K, r)); B = np.zeros((r, N))
    ks = [0, 5, 63]
    X = np.zeros((3, K)); X[np.arange(3), ks] = 1.0
    Y, _ = linear.lora_forward(X, W, A, B, 1.0)
    for m, k in enumerate(ks):
        assert np.array_equal(Y[m], W[:, k])
    # one-hot dY reads out weight rows through dX
    dY = np.zeros((2, N)); dY[0, 1] = 1.0; dY[1, 4] = 1.0
    dX, _, _, _ = linear.lora_backward(dY, X[:2], W, A, B, 1.0)
    assert np.array_equal(dX[0], W[1]) and np.array_equal(dX[1], W[4])


def test_bf16_bit_inputs_are_widened_exactly():
    bits = np.array([[0x3F80, 0xC000]], dtype=np.uint16)  # 1.0, -2.0
    assert np.array_equal(linear.as_f64(bits), np.array([[1.0, -2.0]]))


def test_pages_lora_parameter_counts():
    g = json.load(open(GOLDEN))
    ex = g["lora_factor_example"]
    assert ex["A"] * ex["B"] == ex["delta_w_params"]
    assert linear.lora_param_count([(ex["A"], ex["B"])], ex["r"]) == ex["factor_params"]
    # reading: LoRA on the q and v projections of all 32 layers of LLaMA-7B, bf16
    n = linear.lora_param_count([(4096, 4096), (4096, 4096)] * 32, 8)
    mb = n * 2 / 2 ** 20
    assert round(mb) == g["lora_7b_rank8_megabytes"]["value"]
