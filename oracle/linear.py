"""Frozen-NF4 linear layer with a LoRA adapter, forward and backward -- CPU oracle.

TEST INFRASTRUCTURE ONLY.

What the pages fix (LoRA tutorial, Lit-LLaMA, Chinese translation, sections
on the weight update and on parameter efficiency; arXiv 2305.14314 abstract):
  * the layer output is h = W x + dW x with dW = W_A W_B, the original weights
    frozen and only W_A, W_B trained, a scale alpha on the low-rank branch;
  * W_B starts at zero so dW = 0 at the start of training;
  * merging W' = W + W_A W_B gives the same output with no extra cost;
  * QLoRA back-propagates through the frozen 4-bit weights into the adapters.

Row-major notation used here (tokens are rows):  X is M x K, the frozen
weight W_hat is N x K (out x in, dequantized NF4, bf16), A is K x r, B is
r x N, s = alpha / r.  Then the pages' W_B corresponds to A^T and W_A to B^T:

    Y  = X W_hat^T + s (X A) B
    G  = dY B^T
    dX = dY W_hat + s G A^T
    dA = s X^T G
    dB = s (X A)^T dY
    (no gradient for W_hat: it is frozen)

Everything is computed in fp64 from the exact bf16 input values; the
intermediate X A is not rounded.  Pinned by tests with fp64 central finite
differences of <Y, R> (the loss is bilinear, so the differences are exact up
to rounding), by the merge identity, by the W_B = 0 special case and by
one-hot inputs.
"""
import numpy as np

from .bf16 import bf16_bits_to_f64


def as_f64(a):
    """bf16 bit patterns (uint16) -> fp64; fp32/fp64 arrays pass through."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def lora_forward(X, W_hat, A, B, s):
    """Y = X W_hat^T + s (X A) B in fp64; returns (Y, XA)."""
    X, W_hat, A, B = map(as_f64, (X, W_hat, A, B))
    XA = X @ A
    Y = X @ W_hat.T + float(s) * (XA @ B)
    return Y, XA


def lora_backward(dY, X, W_hat, A, B, s):
    """Gradients of <Y, dY> w.r.t. X, A, B in fp64; returns (dX, dA, dB, G)."""
    dY, X, W_hat, A, B = map(as_f64, (dY, X, W_hat, A, B))
    s = float(s)
    G = dY @ B.T
    dX = dY @ W_hat + s * (G @ A.T)
    dA = s * (X.T @ G)
    dB = s * ((X @ A).T @ dY)
    return dX, dA, dB, G


def lora_xa(X, A):
    """XA = X A in fp64: the adapter's down-projection on its own (no weight)."""
    X, A = map(as_f64, (X, A))
    return X @ A


def lora_adapter_grads(dY, X, A, B, s):
    """The adapter gradients on their own, without the frozen weight, in fp64:
    G = dY B^T, dA = s X^T G, dB = s (X A)^T dY.  Returns (dA, dB, XA).
    Pinned separately from lora_backward by finite differences of <Y, dY>."""
    dY, X, A, B = map(as_f64, (dY, X, A, B))
    s = float(s)
    XA = X @ A
    G = dY @ B.T
    return s * (X.T @ G), s * (XA.T @ dY), XA


def merged_weight(W_hat, A, B, s):
    """W' = W_hat + s (A B)^T: the merged dense weight (fp64)."""
    W_hat, A, B = map(as_f64, (W_hat, A, B))
    return W_hat + float(s) * (A @ B).T


def lora_param_count(shapes, r):
    """Trainable adapter parameters for a list of (out, in) linear shapes at rank r."""
    return sum(r * (n_out + n_in) for n_out, n_in in shapes)


def linear_flops(M, N, K, r):
    """Algorithmic flops of one forward + backward: 4MNK + 6Mr(N+K)."""
    return 4 * M * N * K + 6 * M * r * (N + K)
