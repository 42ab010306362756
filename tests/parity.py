"""Tolerance check shared by the GPU parity tests (not a test module).

The path's stated tolerance for GEMM outputs and gradients (fp32 accumulation,
checked against the fp64 oracle on the same dequantized weights): relative
Frobenius error <= 5e-3 and, per element, |err| <= 1e-2 (|ref| + rms(ref)).
Every check records its margins (the measured error as a fraction of each
bound); the session prints the worst ones at the end.
"""
import numpy as np

REL_FRO = 5e-3
ELEM = 1e-2

MARGINS = []  # (check name, relative Frobenius error / REL_FRO, worst element error / bound)


def assert_close(name, got, want, rel_fro=REL_FRO, elem=ELEM):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, f"{name}: shape {got.shape} != {want.shape}"
    diff = got - want
    rel = np.linalg.norm(diff) / max(np.linalg.norm(want), 1e-300)
    rms = np.sqrt(np.mean(want ** 2))
    worst = float(np.max(np.abs(diff) / (elem * (np.abs(want) + rms)))) if want.size else 0.0
    MARGINS.append((name, rel / rel_fro, worst))
    assert rel <= rel_fro, f"{name}: relative Frobenius error {rel:.3e}"
    assert worst <= 1.0, f"{name}: element error {worst:.3f} of the bound"
    return rel, worst
