"""Host-side checks of libqlora that need no GPU: the library loads, exports
every symbol include/qlora.h declares, builds the same NF4 codebook as the
oracle, sizes workspaces, and rejects bad arguments before any launch."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import nf4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ql():
    from bit_nf4_quantized_38_b300 import qlora
    return qlora


def _declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"QL_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


def test_library_exports_every_declared_symbol(ql):
    names = _declared_symbols()
    assert {"nf4_quantize", "nf4_dequantize", "qlora_linear_fwd", "qlora_linear_bwd"} <= set(names)
    for n in names:
        assert hasattr(ql.lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", ql.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)", out))
    assert set(names) <= exported


def test_codebook_matches_oracle_bit_for_bit(ql):
    lib_levels = np.array(ql.nf4_codebook(), dtype=np.float32)
    assert np.array_equal(lib_levels.view(np.uint32), nf4.nf4_levels().view(np.uint32))


def test_workspace_sizes(ql):
    assert ql.workspace_size(ql.OP_QUANTIZE, 0, 4096, 4096, 0) >= 4096 * 4096 // 64 * 4
    assert ql.workspace_size(ql.OP_DEQUANTIZE, 0, 4096, 4096, 0) == 0
    assert ql.workspace_size(99) == 2 ** 64 - 1
    # up to 32 tokens take the decode path and its workspace
    fwd = lambda M: ql.workspace_size(ql.OP_LINEAR_FWD, M, 5120, 5120, 64)
    assert fwd(17) == fwd(32) == fwd(16) == fwd(1) and fwd(33) != fwd(32)
    # the E4M3 calls keep two halves, each holding the M x K (forward) or
    # M x N (backward) codes
    assert ql.workspace_size(ql.OP_LINEAR_FWD_FP8, 4096, 1024, 4096, 64) >= 2 * 4096 * 4096
    assert ql.workspace_size(ql.OP_LINEAR_BWD_FP8, 4096, 1024, 4096, 64) >= 2 * 4096 * 1024


def test_quantize_rejects_bad_arguments_on_host(ql):
    lib = ql.lib
    buf = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    s = ql.NF4Struct(64, 100, 64, 256, buf, None, buf, buf, buf)
    assert lib.nf4_quantize(buf, ctypes.byref(s), buf, 1 << 20, None) == ql.QL_ERR_UNSUPPORTED
    assert "multiple of 64" in lib.ql_last_error().decode()
    s = ql.NF4Struct(64, 128, 32, 256, buf, None, buf, buf, buf)
    assert lib.nf4_quantize(buf, ctypes.byref(s), buf, 1 << 20, None) == ql.QL_ERR_UNSUPPORTED
    s = ql.NF4Struct(64, 128, 64, 128, buf, None, buf, buf, buf)
    assert lib.nf4_quantize(buf, ctypes.byref(s), buf, 1 << 20, None) == ql.QL_ERR_UNSUPPORTED
    s = ql.NF4Struct(0, 128, 64, 256, buf, None, buf, buf, buf)
    assert lib.nf4_quantize(buf, ctypes.byref(s), buf, 1 << 20, None) == ql.QL_ERR_INVALID
    s = ql.NF4Struct(64, 128, 64, 256, buf, None, buf, buf, buf)
    assert lib.nf4_quantize(None, ctypes.byref(s), buf, 1 << 20, None) == ql.QL_ERR_INVALID
    assert lib.nf4_quantize(ctypes.c_void_p(0x10002), ctypes.byref(s), buf, 1 << 20, None) == ql.QL_ERR_MISALIGNED
    assert lib.nf4_quantize(buf, ctypes.byref(s), buf, 16, None) == ql.QL_ERR_UNSUPPORTED
    s = ql.NF4Struct(64, 128, 64, 0, buf, None, None, None, None)  # dq off needs absmax
    assert lib.nf4_quantize(buf, ctypes.byref(s), buf, 1 << 20, None) == ql.QL_ERR_INVALID
    assert lib.nf4_quantize(buf, None, buf, 1 << 20, None) == ql.QL_ERR_INVALID
    s = ql.NF4Struct(64, 128, 64, 256, buf, None, buf, buf, buf, ql.QL_NF4, 2)  # unknown second-level code
    assert lib.nf4_quantize(buf, ctypes.byref(s), buf, 1 << 20, None) == ql.QL_ERR_UNSUPPORTED
    assert "dq_type" in lib.ql_last_error().decode()
    s = ql.NF4Struct(64, 128, 64, 0, buf, buf, None, None, None, ql.QL_NF4, 7)  # ignored without double quant
    assert lib.nf4_dequantize(ctypes.byref(s), None, None) == ql.QL_ERR_INVALID  # fails on the null output instead


def _fake_pointers_only_without_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("passes fake device pointers: host-side checks, run where there is no GPU")


def test_linear_calls_reject_bad_arguments_on_host(ql):
    """Every case fails the host-side checks, so no CUDA call is made."""
    _fake_pointers_only_without_gpu()
    lib, E = ql.lib, ql
    p, odd, ws_odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10002), ctypes.c_void_p(0x10010)
    big = 1 << 40

    def W(rows=256, cols=512, dq=256):
        return ql.NF4Struct(rows, cols, 64, dq, p, None if dq else p, p, p, p)

    def fwd(X=p, M=64, w=None, A=p, B=p, r=16, Y=p, XA=None, ws=p, wsb=big):
        w = w or W()
        return lib.qlora_linear_fwd(X, M, ctypes.byref(w), A, B, r, 1.0, Y, XA, ws, wsb, None)

    def bwd(dY=p, X=p, XA=None, M=64, w=None, A=p, B=p, r=16, dX=p, dA=p, dB=p, ws=p, wsb=big):
        w = w or W()
        return lib.qlora_linear_bwd(dY, X, XA, M, ctypes.byref(w), A, B, r, 1.0, dX, dA, dB, ws, wsb, None)

    for M in (64, 4):  # the tensor-core path and the decode path
        assert fwd(X=None, M=M) == E.QL_ERR_INVALID
        assert fwd(Y=None, M=M) == E.QL_ERR_INVALID
        assert fwd(A=odd, M=M) == E.QL_ERR_MISALIGNED
        assert fwd(XA=odd, M=M) == E.QL_ERR_MISALIGNED
        assert fwd(r=12, M=M) == E.QL_ERR_UNSUPPORTED
        assert "rank 12" in lib.ql_last_error().decode()
        assert fwd(w=W(rows=100), M=M) == E.QL_ERR_UNSUPPORTED
        assert "multiple of 8" in lib.ql_last_error().decode()
        assert fwd(w=W(cols=100), M=M) == E.QL_ERR_UNSUPPORTED
        assert fwd(w=W(dq=128), M=M) == E.QL_ERR_UNSUPPORTED
        assert fwd(ws=None, M=M) == E.QL_ERR_INVALID
        assert fwd(ws=ws_odd, M=M) == E.QL_ERR_MISALIGNED
        need = ql.workspace_size(ql.OP_LINEAR_FWD, M, 256, 512, 16)
        assert need > 0 and fwd(wsb=need - 1, M=M) == E.QL_ERR_UNSUPPORTED
    assert fwd(M=0) == E.QL_ERR_INVALID
    assert fwd(M=-3) == E.QL_ERR_INVALID
    assert lib.qlora_linear_fwd(p, 64, None, p, p, 16, 1.0, p, None, p, big, None) == E.QL_ERR_INVALID

    assert bwd(dA=None) == E.QL_ERR_INVALID
    assert bwd(dX=odd) == E.QL_ERR_MISALIGNED
    assert bwd(XA=odd) == E.QL_ERR_MISALIGNED
    assert bwd(r=0) == E.QL_ERR_UNSUPPORTED
    assert bwd(M=0) == E.QL_ERR_INVALID
    assert bwd(w=W(rows=0)) == E.QL_ERR_INVALID
    need = ql.workspace_size(ql.OP_LINEAR_BWD, 64, 256, 512, 16)
    assert need > 0 and bwd(wsb=need - 1) == E.QL_ERR_UNSUPPORTED

    # the E4M3 backward: the same checks, and N a multiple of 16 (TMA rows of dY codes)
    def bwd8(dY=p, X=p, XA=None, M=64, w=None, A=p, B=p, r=16, dX=p, dA=p, dB=p, ws=p, wsb=big):
        w = w or W()
        return lib.qlora_linear_bwd_fp8(dY, X, XA, M, ctypes.byref(w), A, B, r, 1.0, dX, dA, dB, ws, wsb, None)

    assert bwd8(dB=None) == E.QL_ERR_INVALID
    assert bwd8(dY=odd) == E.QL_ERR_MISALIGNED
    assert bwd8(r=24) == E.QL_ERR_UNSUPPORTED
    assert bwd8(w=W(rows=264)) == E.QL_ERR_UNSUPPORTED
    assert "multiple of 16" in lib.ql_last_error().decode()
    need = ql.workspace_size(ql.OP_LINEAR_BWD_FP8, 64, 256, 512, 16)
    assert need >= 64 * 256 and bwd8(wsb=need - 1) == E.QL_ERR_UNSUPPORTED  # holds the M x N dY codes


def test_dequantize_and_noalloc_reject_bad_arguments_on_host(ql):
    _fake_pointers_only_without_gpu()
    lib, E = ql.lib, ql
    p, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10002)
    s = ql.NF4Struct(256, 512, 64, 256, p, None, p, p, p)
    assert lib.nf4_dequantize(ctypes.byref(s), None, None) == E.QL_ERR_INVALID
    assert lib.nf4_dequantize(ctypes.byref(s), odd, None) == E.QL_ERR_MISALIGNED
    s_bad = ql.NF4Struct(256, 512, 64, 256, p, None, None, p, p)
    assert lib.nf4_dequantize(ctypes.byref(s_bad), p, None) == E.QL_ERR_INVALID
    # the built-in scratch holds 4 Mi blocks of 64: one block more is refused
    too_big = ql.NF4Struct((1 << 22) // 64 + 1, 64 * 64, 64, 256, p, None, p, p, p)
    assert lib.nf4_quantize_noalloc(p, ctypes.byref(too_big), None) == E.QL_ERR_UNSUPPORTED
    assert "scratch" in lib.ql_last_error().decode()
    assert lib.nf4_quantize_noalloc(p, None, None) == E.QL_ERR_INVALID


def test_selftest_wait_rejects_bad_limits_on_host(ql):
    for limit in (0, -5, 2_000_000_001):
        assert ql.lib.ql_selftest_wait(limit, None) == ql.QL_ERR_INVALID
        assert "limit" in ql.lib.ql_last_error().decode()


def test_quotient_without_division_is_exact_on_all_bf16_pairs(tmp_path):
    """The quantizer replaces w / m by a reciprocal and one FMA correction; this
    checks that sequence against IEEE division for every pair of bf16 values
    with |w| <= m the kernel's fast path accepts (exhaustive, ~5e8 pairs)."""
    src = os.path.join(ROOT, "tests", "native", "quotient_check.c")
    exe = str(tmp_path / "quotient_check")
    subprocess.run(["gcc", "-O2", "-mfma", "-ffp-contract=off", "-o", exe, src, "-lm"], check=True)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout
    assert "bad 0" in p.stdout


def test_division_free_coding_is_exact_on_all_bf16_pairs(tmp_path):
    """The quantizer codes each element without a division: the cell from an
    approximate quotient, the decision from the sign of w - m u (plus
    m delta when needed).  Checked against the code of the IEEE quotient for
    every pair of bf16 values with |w| <= m in the fast path's range, with the
    reciprocal perturbed up to two ulps either way (exhaustive, ~2.5e9
    cases), on the NF4 codebook of the oracle."""
    from oracle import nf4
    src = os.path.join(ROOT, "tests", "native", "coding_check.c")
    exe = str(tmp_path / "coding_check")
    subprocess.run(["gcc", "-O2", "-mfma", "-ffp-contract=off", "-fopenmp", "-o", exe, src, "-lm"], check=True)
    levels = [float(v).hex() for v in nf4.nf4_levels()]
    p = subprocess.run([exe, *levels], capture_output=True, text=True, timeout=900)
    assert p.returncode == 0, p.stdout
    assert "bad 0" in p.stdout
    assert "one_fma 1" in p.stdout  # the NF4 table takes the one-FMA decision


def test_merge_rejects_bad_arguments_on_host(ql):
    _fake_pointers_only_without_gpu()
    lib, E = ql.lib, ql
    p, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10002)
    s = ql.NF4Struct(256, 512, 64, 256, p, None, p, p, p)
    assert lib.qlora_merge(ctypes.byref(s), None, p, 16, 1.0, p, None) == E.QL_ERR_INVALID
    assert lib.qlora_merge(ctypes.byref(s), p, p, 16, 1.0, odd, None) == E.QL_ERR_MISALIGNED
    assert lib.qlora_merge(ctypes.byref(s), p, p, 12, 1.0, p, None) == E.QL_ERR_UNSUPPORTED
    assert "rank 12" in lib.ql_last_error().decode()
    bad = ql.NF4Struct(100, 512, 64, 256, p, None, p, p, p)
    assert lib.qlora_merge(ctypes.byref(bad), p, p, 16, 1.0, p, None) == E.QL_ERR_UNSUPPORTED


def test_fp4_table_matches_oracle_bit_for_bit(ql):
    lib_levels = np.array(ql.codebook(ql.QL_FP4), dtype=np.float32)
    assert np.array_equal(lib_levels.view(np.uint32), nf4.fp4_levels().view(np.uint32))
    with pytest.raises(ql.QLError):
        ql.codebook(7)


def test_division_free_coding_is_exact_on_the_fp4_table(tmp_path):
    """The same exhaustive check as for NF4, on the FP4 comparison table."""
    src = os.path.join(ROOT, "tests", "native", "coding_check.c")
    exe = str(tmp_path / "coding_check")
    subprocess.run(["gcc", "-O2", "-mfma", "-ffp-contract=off", "-fopenmp", "-o", exe, src, "-lm"], check=True)
    p = subprocess.run([exe, *[float(v).hex() for v in nf4.fp4_levels()]], capture_output=True, text=True,
                       timeout=900)
    assert p.returncode == 0, p.stdout
    assert "bad 0" in p.stdout


def test_unknown_quant_type_is_rejected_on_host(ql):
    _fake_pointers_only_without_gpu()
    p = ctypes.c_void_p(0x10000)
    s = ql.NF4Struct(256, 512, 64, 256, p, None, p, p, p, 5)
    assert ql.lib.nf4_dequantize(ctypes.byref(s), p, None) == ql.QL_ERR_UNSUPPORTED
    assert "quant_type 5" in ql.lib.ql_last_error().decode()


def test_quantize_host_rejects_bad_arguments_on_host(ql):
    _fake_pointers_only_without_gpu()
    lib, E = ql.lib, ql
    p = ctypes.c_void_p(0x10000)
    s = ql.NF4Struct(256, 512, 64, 256, p, None, p, p, p)
    need = ql.workspace_size(ql.OP_QUANTIZE_HOST, 0, 256, 512, 0)
    assert need > ql.workspace_size(ql.OP_QUANTIZE, 0, 256, 512, 0)
    assert lib.nf4_quantize_host(None, ctypes.byref(s), p, need, None, None) == E.QL_ERR_INVALID
    assert lib.nf4_quantize_host(p, ctypes.byref(s), p, need - 1, None, None) == E.QL_ERR_UNSUPPORTED
    assert lib.nf4_quantize_host(p, ctypes.byref(s), ctypes.c_void_p(0x10010), need, None, None) == \
        E.QL_ERR_MISALIGNED
