"""Python binding of libqlora (the C ABI declared in include/qlora.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch provides device memory and the current stream.  Importing
this module raises ImportError when the library has not been built; there is
no other code path.
"""
import ctypes
import os
from dataclasses import dataclass

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libqlora.so")

QL_OK, QL_ERR_INVALID, QL_ERR_UNSUPPORTED, QL_ERR_MISALIGNED, QL_ERR_CUDA, QL_ERR_TIMEOUT = range(6)
QL_NF4, QL_FP4 = 0, 1
QL_DQ_INT8, QL_DQ_E4M3 = 0, 1  # second-level codes (ql_nf4_tensor.dq_type)
(OP_QUANTIZE, OP_DEQUANTIZE, OP_LINEAR_FWD, OP_LINEAR_BWD, OP_QUANTIZE_HOST, OP_LINEAR_FWD_FP8,
 OP_LINEAR_BWD_FP8) = range(7)

_c_i64, _c_i32, _c_f32, _c_p, _c_sz = (ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                       ctypes.c_void_p, ctypes.c_size_t)


class NF4Struct(ctypes.Structure):
    _fields_ = [("rows", _c_i64), ("cols", _c_i64), ("blocksize", _c_i32), ("dq_blocksize", _c_i32),
                ("packed", _c_p), ("absmax", _c_p), ("absmax_code", _c_p), ("dq_step", _c_p),
                ("dq_mean", _c_p), ("quant_type", _c_i32), ("dq_type", _c_i32)]


_SIGNATURES = {
    "ql_workspace_size": (_c_sz, [ctypes.c_int, _c_i64, _c_i64, _c_i64, _c_i32]),
    "ql_nf4_codebook": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float)]),
    "ql_codebook": (ctypes.c_int, [_c_i32, ctypes.POINTER(ctypes.c_float)]),
    "nf4_quantize": (ctypes.c_int, [_c_p, ctypes.POINTER(NF4Struct), _c_p, _c_sz, _c_p]),
    "nf4_quantize_noalloc": (ctypes.c_int, [_c_p, ctypes.POINTER(NF4Struct), _c_p]),
    "nf4_quantize_host": (ctypes.c_int, [_c_p, ctypes.POINTER(NF4Struct), _c_p, _c_sz, _c_p, _c_p]),
    "nf4_quantize_shard_begin": (ctypes.c_int, [_c_p, ctypes.POINTER(NF4Struct), _c_p, _c_sz, _c_p]),
    "nf4_quantize_shard_end": (ctypes.c_int, [ctypes.POINTER(NF4Struct), _c_p, _c_sz, _c_i64, _c_p]),
    "nf4_dequantize": (ctypes.c_int, [ctypes.POINTER(NF4Struct), _c_p, _c_p]),
    "qlora_linear_fwd": (ctypes.c_int, [_c_p, _c_i64, ctypes.POINTER(NF4Struct), _c_p, _c_p, _c_i32,
                                        _c_f32, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "qlora_linear_fwd_fp8": (ctypes.c_int, [_c_p, _c_i64, ctypes.POINTER(NF4Struct), _c_p, _c_p, _c_i32,
                                            _c_f32, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "qlora_linear_bwd": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, ctypes.POINTER(NF4Struct), _c_p,
                                        _c_p, _c_i32, _c_f32, _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "qlora_linear_bwd_fp8": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, ctypes.POINTER(NF4Struct), _c_p,
                                            _c_p, _c_i32, _c_f32, _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "qlora_merge": (ctypes.c_int, [ctypes.POINTER(NF4Struct), _c_p, _c_p, _c_i32, _c_f32, _c_p, _c_p]),
    "ql_get_device_status": (ctypes.c_int, [_c_p]),
    "ql_selftest_wait": (ctypes.c_int, [ctypes.c_int64, _c_p]),
    "ql_last_error": (ctypes.c_char_p, []),
    "ql_launch_count": (ctypes.c_uint64, []),
    "ql_timing_start": (ctypes.c_int, [ctypes.c_int]),
    "ql_timing_stop": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_double)]),
    "ql_spans_start": (ctypes.c_int, [_c_p, ctypes.c_int]),
    "ql_spans_stop": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m bit_nf4_quantized_38_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class QLError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libqlora error {code}: {msg}")
        self.code = code


def _check(rc):
    if rc != QL_OK:
        raise QLError(rc, lib.ql_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def workspace_size(op, M=0, N=0, K=0, r=0):
    return int(lib.ql_workspace_size(op, M, N, K, r))


def nf4_codebook():
    buf = (ctypes.c_float * 16)()
    _check(lib.ql_nf4_codebook(buf))
    return [float(v) for v in buf]


def codebook(quant_type=QL_NF4):
    """The 16 levels of a code table (QL_NF4 or QL_FP4), ascending."""
    buf = (ctypes.c_float * 16)()
    _check(lib.ql_codebook(int(quant_type), buf))
    return [float(v) for v in buf]


def device_status(stream=None):
    """QL_OK, or raises QLError(QL_ERR_TIMEOUT) if a kernel gave up waiting."""
    _check(lib.ql_get_device_status(_stream(stream)))


def selftest_wait(limit_ns, stream=None):
    """Launch the failure-path self-test: a kernel whose bounded wait runs out
    after `limit_ns`; device_status() afterwards raises QL_ERR_TIMEOUT."""
    _check(lib.ql_selftest_wait(int(limit_ns), _stream(stream)))


def launch_count():
    """Kernels the library has launched in this process."""
    return int(lib.ql_launch_count())


def timing_start(capacity):
    """Bracket the next `capacity` tensor-core GEMM launches with CUDA events."""
    _check(lib.ql_timing_start(int(capacity)))


def timing_stop():
    """Returns (summed GEMM milliseconds, launches, summed algorithmic flops)."""
    ms, n, fl = ctypes.c_float(), ctypes.c_int(), ctypes.c_double()
    _check(lib.ql_timing_stop(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(fl)))
    return float(ms.value), int(n.value), float(fl.value)


def spans_start(buf):
    """Record the first-start / last-end %globaltimer of the next len(buf) // 2
    tensor-core GEMM launches into the int64 CUDA tensor `buf` (see
    ql_spans_start); the pairs are initialised here on the current stream."""
    if buf.dtype != torch.int64 or not buf.is_cuda or buf.numel() % 2:
        raise ValueError("buf must be an even-length int64 CUDA tensor")
    v = buf.view(-1, 2)
    v[:, 0].fill_(-1)  # UINT64_MAX as int64
    v[:, 1].fill_(0)
    _check(lib.ql_spans_start(_ptr(buf), buf.numel() // 2))


def spans_stop():
    """Returns (recorded launches, their summed algorithmic flops)."""
    n, fl = ctypes.c_int(), ctypes.c_double()
    _check(lib.ql_spans_stop(ctypes.byref(n), ctypes.byref(fl)))
    return int(n.value), float(fl.value)


def _workspace(nbytes, device, ws):
    if nbytes == 0:
        return None, 0
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws, ws.numel()


@dataclass
class NF4Tensor:
    """Device storage of an NF4 weight (layout as ql_nf4_tensor in include/qlora.h)."""
    rows: int
    cols: int
    packed: torch.Tensor
    absmax: torch.Tensor = None
    absmax_code: torch.Tensor = None
    dq_step: torch.Tensor = None
    dq_mean: torch.Tensor = None
    blocksize: int = 64
    dq_blocksize: int = 256
    quant_type: int = QL_NF4
    dq_type: int = QL_DQ_INT8

    @classmethod
    def empty(cls, rows, cols, device, dq_blocksize=256, blocksize=64, quant_type=QL_NF4, dq_type=QL_DQ_INT8):
        n_b = rows * cols // blocksize
        t = cls(rows, cols, torch.empty(rows * cols // 2, dtype=torch.uint8, device=device),
                blocksize=blocksize, dq_blocksize=dq_blocksize, quant_type=quant_type, dq_type=dq_type)
        if dq_blocksize:
            t.absmax_code = torch.empty(n_b, dtype=torch.int8, device=device)
            t.dq_step = torch.empty((n_b + dq_blocksize - 1) // dq_blocksize, dtype=torch.float32,
                                    device=device)
            t.dq_mean = torch.empty(1, dtype=torch.float32, device=device)
        else:
            t.absmax = torch.empty(n_b, dtype=torch.float32, device=device)
        return t

    def struct(self):
        return NF4Struct(self.rows, self.cols, self.blocksize, self.dq_blocksize,
                         _ptr(self.packed), _ptr(self.absmax), _ptr(self.absmax_code),
                         _ptr(self.dq_step), _ptr(self.dq_mean), self.quant_type, self.dq_type)

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in
                   (self.packed, self.absmax, self.absmax_code, self.dq_step, self.dq_mean)
                   if t is not None)


def nf4_quantize(W, dq_blocksize=256, blocksize=64, out=None, ws=None, stream=None, quant_type=QL_NF4,
                 dq_type=QL_DQ_INT8):
    """Quantize a bf16 (rows x cols) CUDA tensor to NF4 (or FP4) codes (+ double
    quant with int8 or E4M3 second-level codes)."""
    _need(W, torch.bfloat16, "W")
    rows, cols = W.shape
    q = out if out is not None else NF4Tensor.empty(rows, cols, W.device, dq_blocksize, blocksize, quant_type,
                                                    dq_type)
    ws, nbytes = _workspace(workspace_size(OP_QUANTIZE, 0, rows, cols, 0), W.device, ws)
    s = q.struct()
    _check(lib.nf4_quantize(_ptr(W), ctypes.byref(s), _ptr(ws), nbytes, _stream(stream)))
    return q


def nf4_quantize_noalloc(W, dq_blocksize=256, blocksize=64, out=None, stream=None):
    """nf4_quantize without a workspace: the scratch is the library's built-in
    array (for callers that cannot allocate per call; see include/qlora.h)."""
    _need(W, torch.bfloat16, "W")
    rows, cols = W.shape
    q = out if out is not None else NF4Tensor.empty(rows, cols, W.device, dq_blocksize, blocksize)
    s = q.struct()
    _check(lib.nf4_quantize_noalloc(_ptr(W), ctypes.byref(s), _stream(stream)))
    return q


def nf4_quantize_host(W_host, device, dq_blocksize=256, blocksize=64, out=None, ws=None, stream=None,
                      copy_stream=None, quant_type=QL_NF4, dq_type=QL_DQ_INT8):
    """Quantize a bf16 (rows x cols) CPU tensor into NF4 on `device` while it
    streams to the GPU (quantize-on-load; see include/qlora.h).  Pinned
    memory lets the copies overlap the kernels.  Keep W_host alive and
    unchanged until `stream` has passed the call."""
    if W_host.is_cuda or W_host.dtype != torch.bfloat16 or not W_host.is_contiguous():
        raise ValueError("W_host must be a contiguous bf16 CPU tensor")
    rows, cols = W_host.shape
    device = torch.device(device)
    q = out if out is not None else NF4Tensor.empty(rows, cols, device, dq_blocksize, blocksize, quant_type, dq_type)
    ws, nbytes = _workspace(workspace_size(OP_QUANTIZE_HOST, 0, rows, cols, 0), device, ws)
    s = q.struct()
    st = _stream(stream)
    cst = st if copy_stream is None else ctypes.c_void_p(copy_stream.cuda_stream)
    _check(lib.nf4_quantize_host(ctypes.c_void_p(W_host.data_ptr()), ctypes.byref(s), _ptr(ws), nbytes, cst, st))
    return q


def nf4_quantize_shard_begin(W_shard, dq_blocksize=256, blocksize=64, out=None, ws=None, stream=None):
    """First half of a row-sharded quantization (see include/qlora.h).
    Returns (q_shard, ws, partial_sum) where partial_sum is a float64 CUDA
    view of the shard's absmax sum at the head of ws."""
    _need(W_shard, torch.bfloat16, "W_shard")
    rows, cols = W_shard.shape
    q = out if out is not None else NF4Tensor.empty(rows, cols, W_shard.device, dq_blocksize, blocksize)
    ws, nbytes = _workspace(workspace_size(OP_QUANTIZE, 0, rows, cols, 0), W_shard.device, ws)
    s = q.struct()
    _check(lib.nf4_quantize_shard_begin(_ptr(W_shard), ctypes.byref(s), _ptr(ws), nbytes, _stream(stream)))
    return q, ws, ws[:8].view(torch.float64)


def nf4_quantize_shard_end(q, ws, total_blocks, stream=None):
    """Second half: the double-quant codes of this shard with mu taken from the
    (all-reduced) sum at the head of ws over `total_blocks` blocks."""
    s = q.struct()
    _check(lib.nf4_quantize_shard_end(ctypes.byref(s), _ptr(ws), ws.numel(), int(total_blocks),
                                      _stream(stream)))
    return q


def nf4_dequantize(q, out=None, stream=None):
    if out is None:
        out = torch.empty(q.rows, q.cols, dtype=torch.bfloat16, device=q.packed.device)
    _need(out, torch.bfloat16, "out", (q.rows, q.cols))
    s = q.struct()
    _check(lib.nf4_dequantize(ctypes.byref(s), _ptr(out), _stream(stream)))
    return out


def qlora_linear_fwd(X, q, A, B, scale, Y=None, XA=None, ws=None, stream=None, want_xa=True):
    """Y = X W_hat^T + scale (X A) B; returns (Y, XA or None)."""
    M, K = X.shape
    r = A.shape[1]
    _need(X, torch.bfloat16, "X", (M, q.cols))
    _need(A, torch.bfloat16, "A", (q.cols, r))
    _need(B, torch.bfloat16, "B", (r, q.rows))
    if Y is None:
        Y = torch.empty(M, q.rows, dtype=torch.bfloat16, device=X.device)
    _need(Y, torch.bfloat16, "Y", (M, q.rows))
    if XA is None and want_xa:
        XA = torch.empty(M, r, dtype=torch.bfloat16, device=X.device)
    if XA is not None:
        _need(XA, torch.bfloat16, "XA", (M, r))
    ws, nbytes = _workspace(workspace_size(OP_LINEAR_FWD, M, q.rows, q.cols, r), X.device, ws)
    s = q.struct()
    _check(lib.qlora_linear_fwd(_ptr(X), M, ctypes.byref(s), _ptr(A), _ptr(B), r, float(scale),
                                _ptr(Y), _ptr(XA), _ptr(ws), nbytes, _stream(stream)))
    return Y, XA


def qlora_linear_fwd_fp8(X, q, A, B, scale, Y=None, XA=None, ws=None, stream=None, want_xa=True):
    """qlora_linear_fwd with the main product on E4M3 operands (see
    include/qlora.h); returns (Y, XA or None)."""
    M, K = X.shape
    r = A.shape[1]
    _need(X, torch.bfloat16, "X", (M, q.cols))
    _need(A, torch.bfloat16, "A", (q.cols, r))
    _need(B, torch.bfloat16, "B", (r, q.rows))
    if Y is None:
        Y = torch.empty(M, q.rows, dtype=torch.bfloat16, device=X.device)
    _need(Y, torch.bfloat16, "Y", (M, q.rows))
    if XA is None and want_xa:
        XA = torch.empty(M, r, dtype=torch.bfloat16, device=X.device)
    if XA is not None:
        _need(XA, torch.bfloat16, "XA", (M, r))
    ws, nbytes = _workspace(workspace_size(OP_LINEAR_FWD_FP8, M, q.rows, q.cols, r), X.device, ws)
    s = q.struct()
    _check(lib.qlora_linear_fwd_fp8(_ptr(X), M, ctypes.byref(s), _ptr(A), _ptr(B), r, float(scale),
                                    _ptr(Y), _ptr(XA), _ptr(ws), nbytes, _stream(stream)))
    return Y, XA


def qlora_linear_bwd(dY, X, XA, q, A, B, scale, dX=None, dA=None, dB=None, ws=None, stream=None):
    """Returns (dX bf16, dA fp32, dB fp32)."""
    return _linear_bwd(lib.qlora_linear_bwd, OP_LINEAR_BWD, dY, X, XA, q, A, B, scale, dX, dA, dB, ws, stream)


def qlora_linear_bwd_fp8(dY, X, XA, q, A, B, scale, dX=None, dA=None, dB=None, ws=None, stream=None):
    """The backward with the dX main product on E4M3 operands; returns (dX bf16, dA fp32, dB fp32)."""
    return _linear_bwd(lib.qlora_linear_bwd_fp8, OP_LINEAR_BWD_FP8, dY, X, XA, q, A, B, scale, dX, dA, dB, ws,
                       stream)


def _linear_bwd(fn, op, dY, X, XA, q, A, B, scale, dX, dA, dB, ws, stream):
    M = X.shape[0]
    r = A.shape[1]
    _need(dY, torch.bfloat16, "dY", (M, q.rows))
    _need(X, torch.bfloat16, "X", (M, q.cols))
    _need(A, torch.bfloat16, "A", (q.cols, r))
    _need(B, torch.bfloat16, "B", (r, q.rows))
    if XA is not None:
        _need(XA, torch.bfloat16, "XA", (M, r))
    dev = X.device
    dX = torch.empty(M, q.cols, dtype=torch.bfloat16, device=dev) if dX is None else dX
    dA = torch.empty(q.cols, r, dtype=torch.float32, device=dev) if dA is None else dA
    dB = torch.empty(r, q.rows, dtype=torch.float32, device=dev) if dB is None else dB
    _need(dX, torch.bfloat16, "dX", (M, q.cols))
    _need(dA, torch.float32, "dA", (q.cols, r))
    _need(dB, torch.float32, "dB", (r, q.rows))
    ws, nbytes = _workspace(workspace_size(op, M, q.rows, q.cols, r), dev, ws)
    s = q.struct()
    _check(fn(_ptr(dY), _ptr(X), _ptr(XA), M, ctypes.byref(s), _ptr(A), _ptr(B), r, float(scale), _ptr(dX),
              _ptr(dA), _ptr(dB), _ptr(ws), nbytes, _stream(stream)))
    return dX, dA, dB


def qlora_merge(q, A, B, scale, out=None, stream=None):
    """W' = bf16(w_hat + scale (A B)^T): the merged dense bf16 weight (rows x cols)."""
    r = A.shape[1]
    _need(A, torch.bfloat16, "A", (q.cols, r))
    _need(B, torch.bfloat16, "B", (r, q.rows))
    if out is None:
        out = torch.empty(q.rows, q.cols, dtype=torch.bfloat16, device=A.device)
    _need(out, torch.bfloat16, "out", (q.rows, q.cols))
    s = q.struct()
    _check(lib.qlora_merge(ctypes.byref(s), _ptr(A), _ptr(B), r, float(scale), _ptr(out), _stream(stream)))
    return out
