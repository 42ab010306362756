"""The allocation-free quantize entry point (nf4_quantize_noalloc).

It exists for callers that cannot allocate scratch memory per call -- code
under a memory plan fixed up front, code embedded in a host runtime that owns
every allocation, code that must avoid cudaMalloc's implicit synchronisation.  It must
give exactly what nf4_quantize gives with a caller-provided workspace, call
after call, since every call reuses the same built-in scratch array.  This
file is collected last so that a run stopping at its first failure has run
every other test already; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ql():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_38_b300 import qlora
    return qlora


def _quantize_noalloc_abi(ql, W, dq):
    """Call the C entry point directly through ctypes (no workspace argument)."""
    q = ql.NF4Tensor.empty(W.shape[0], W.shape[1], W.device, dq)
    s = q.struct()
    rc = ql.lib.nf4_quantize_noalloc(ctypes.c_void_p(W.data_ptr()), ctypes.byref(s),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == ql.QL_OK, ql.lib.ql_last_error().decode()
    return q


def _same(a, b):
    for f in ("packed", "absmax", "absmax_code", "dq_step", "dq_mean"):
        x, y = getattr(a, f), getattr(b, f)
        assert (x is None) == (y is None), f
        if x is not None:
            assert torch.equal(x, y), f


@pytest.mark.parametrize("dq", [256, 0])
def test_noalloc_quantize_matches_workspace_quantize_on_consecutive_calls(ql, dq):
    from bit_nf4_quantized_38_b300.workloads import normal_bf16, normal_with_outliers_bf16
    dev = torch.device("cuda")
    W1 = normal_with_outliers_bf16((2048, 4096), 0.02, 0.001, 20.0, seed=31).to(dev)
    W2 = normal_bf16((1032, 576), 0.05, seed=32).to(dev)   # different size: the array keeps old contents
    ref1 = ql.nf4_quantize(W1, dq_blocksize=dq)
    ref2 = ql.nf4_quantize(W2, dq_blocksize=dq)
    got1 = _quantize_noalloc_abi(ql, W1, dq)
    got2 = _quantize_noalloc_abi(ql, W2, dq)
    got1b = _quantize_noalloc_abi(ql, W1, dq)
    torch.cuda.synchronize()
    ql.device_status()
    _same(got1, ref1)
    _same(got2, ref2)
    _same(got1b, ref1)


def test_noalloc_rejects_weights_beyond_its_scratch(ql):
    buf = ctypes.c_void_p(0x10000)
    s = ql.NF4Struct(1 << 16, 1 << 13, 64, 256, buf, None, buf, buf, buf)  # 8 Mi blocks > 4 Mi
    assert ql.lib.nf4_quantize_noalloc(buf, ctypes.byref(s), None) == ql.QL_ERR_UNSUPPORTED
    assert "scratch" in ql.lib.ql_last_error().decode()
