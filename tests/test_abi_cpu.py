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
