// C entry points of libqlora: argument checks, workspace layout, dispatch.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>

#include "common.cuh"
#include "linear.cuh"
#include "merge.cuh"

namespace ql {

namespace {
thread_local char g_msg[512] = "";
std::atomic<uint64_t> g_launches{0};
__device__ int g_status;
}  // namespace

int set_error(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int check_cuda(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return QL_OK;
  return set_error(QL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int *device_status_ptr() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
  return static_cast<int *>(p);
}

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int check_tensor(const ql_nf4_tensor *q, const char *fn, bool need_absmax_dq_off) {
  if (!q) return set_error(QL_ERR_INVALID, "%s: null nf4 tensor", fn);
  if (q->rows <= 0 || q->cols <= 0)
    return set_error(QL_ERR_INVALID, "%s: non-positive weight shape %lld x %lld", fn,
                     (long long)q->rows, (long long)q->cols);
  if (q->blocksize != 64) return set_error(QL_ERR_UNSUPPORTED, "%s: blocksize %d (only 64)", fn, q->blocksize);
  if (q->dq_blocksize != 0 && q->dq_blocksize != 256)
    return set_error(QL_ERR_UNSUPPORTED, "%s: dq_blocksize %d (only 0 or 256)", fn, q->dq_blocksize);
  if (q->cols % 64) return set_error(QL_ERR_UNSUPPORTED, "%s: cols %lld not a multiple of 64", fn, (long long)q->cols);
  if (q->quant_type != QL_NF4 && q->quant_type != QL_FP4)
    return set_error(QL_ERR_UNSUPPORTED, "%s: quant_type %d (0 = NF4, 1 = FP4)", fn, q->quant_type);
  if (!q->packed) return set_error(QL_ERR_INVALID, "%s: null packed", fn);
  if (!aligned(q->packed, 16)) return set_error(QL_ERR_MISALIGNED, "%s: packed not 16-byte aligned", fn);
  if (q->dq_blocksize) {
    if (q->dq_type != QL_DQ_INT8 && q->dq_type != QL_DQ_E4M3)
      return set_error(QL_ERR_UNSUPPORTED, "%s: dq_type %d (0 = int8, 1 = E4M3)", fn, q->dq_type);
    if (!q->absmax_code || !q->dq_step || !q->dq_mean)
      return set_error(QL_ERR_INVALID, "%s: null double-quant array", fn);
    if (!aligned(q->absmax_code, 16) || !aligned(q->dq_step, 16) || !aligned(q->dq_mean, 4))
      return set_error(QL_ERR_MISALIGNED, "%s: double-quant array misaligned", fn);
  } else if (need_absmax_dq_off) {
    if (!q->absmax) return set_error(QL_ERR_INVALID, "%s: null absmax", fn);
    if (!aligned(q->absmax, 16)) return set_error(QL_ERR_MISALIGNED, "%s: absmax not 16-byte aligned", fn);
  }
  return QL_OK;
}

// quantize workspace: [fp64 sum | pad to 256][fp32 absmax n_b (double quant only)]
size_t quantize_ws(int64_t N, int64_t K) { return 256 + round_up((size_t)(N * K / 64) * 4, 256); }

// quantize-on-load: rows per staging chunk (about 16 MB of bf16) and the
// workspace, [quantize workspace][chunk 0][chunk 1]
int64_t host_chunk_rows(int64_t N, int64_t K) {
  const int64_t rows = std::max<int64_t>(1, ((int64_t)8 << 20) / std::max<int64_t>(K, 1));
  return std::min(rows, std::max<int64_t>(N, 1));
}
size_t quantize_host_ws(int64_t N, int64_t K) {
  return quantize_ws(N, K) + 2 * round_up((size_t)(host_chunk_rows(N, K) * K * 2), 256);
}

}  // namespace
}  // namespace ql

using namespace ql;

extern "C" size_t ql_workspace_size(int op, int64_t M, int64_t N, int64_t K, int32_t r) {
  switch (op) {
    case QL_OP_QUANTIZE: return quantize_ws(N, K);
    case QL_OP_DEQUANTIZE: return 0;
    case QL_OP_LINEAR_FWD: return linear_fwd_ws(M, N, K, r);
    case QL_OP_LINEAR_BWD: return linear_bwd_ws(M, N, K, r);
    case QL_OP_QUANTIZE_HOST: return quantize_host_ws(N, K);
    case QL_OP_LINEAR_FWD_FP8: return linear_fwd_fp8_ws(M, N, K, r);
    case QL_OP_LINEAR_BWD_FP8: return linear_bwd_fp8_ws(M, N, K, r);
    default: return (size_t)-1;
  }
}

extern "C" const char *ql_last_error(void) { return g_msg; }

extern "C" uint64_t ql_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int ql_get_device_status(ql_stream_t stream) {
  int rc = check_cuda(cudaStreamSynchronize(stream), "ql_get_device_status: synchronize");
  if (rc) return rc;
  int v = 0;
  rc = check_cuda(cudaMemcpyFromSymbol(&v, g_status, sizeof(int)), "ql_get_device_status: read");
  if (rc) return rc;
  if (v != kStatusOk) {
    int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof(int));
    return set_error(QL_ERR_TIMEOUT, "a kernel gave up waiting (status %d)", v);
  }
  return QL_OK;
}

namespace {

int check_quant_ws(const ql_nf4_tensor *q, void *ws, size_t ws_bytes, const char *fn) {
  if (!ws) return set_error(QL_ERR_INVALID, "%s: null workspace", fn);
  if (!aligned(ws, 256)) return set_error(QL_ERR_MISALIGNED, "%s: workspace not 256-byte aligned", fn);
  if (ws_bytes < quantize_ws(q->rows, q->cols))
    return set_error(QL_ERR_UNSUPPORTED, "%s: workspace %zu < %zu bytes", fn, ws_bytes,
                     quantize_ws(q->rows, q->cols));
  return QL_OK;
}

// First-level quantization: codes, block absmax (into the workspace when
// double quantization follows) and the fp64 absmax sum at the workspace head.
int quantize_first(const uint16_t *W, const ql_nf4_tensor *q, void *ws, size_t ws_bytes, cudaStream_t st,
                   const char *fn) {
  int rc = check_tensor(q, fn, true);
  if (rc) return rc;
  if (!W) return set_error(QL_ERR_INVALID, "%s: null W", fn);
  if (!aligned(W, 16)) return set_error(QL_ERR_MISALIGNED, "%s: W not 16-byte aligned", fn);
  rc = check_quant_ws(q, ws, ws_bytes, fn);
  if (rc) return rc;
  note_other_call(st);
  double *sum = static_cast<double *>(ws);
  float *absmax = q->dq_blocksize ? reinterpret_cast<float *>(static_cast<char *>(ws) + 256) : q->absmax;
  rc = check_cuda(cudaMemsetAsync(sum, 0, sizeof(double), st), "quantize: clear sum");
  if (rc) return rc;
  return check_cuda(launch_quantize(W, q->rows, q->cols, q->quant_type, q->packed, absmax, sum, st),
                    "quantize: launch");
}

// Second level: mu = fl32(S / total_blocks) from the fp64 sum at the
// workspace head, then the codes and steps of this tensor's blocks.
int quantize_second(const ql_nf4_tensor *q, void *ws, int64_t total_blocks, cudaStream_t st) {
  if (!q->dq_blocksize) return QL_OK;
  const int64_t n_b = q->rows * q->cols / 64;
  float *absmax = reinterpret_cast<float *>(static_cast<char *>(ws) + 256);
  return check_cuda(launch_double_quant(absmax, n_b, total_blocks, q->dq_blocksize, q->dq_type, static_cast<double *>(ws),
                                        q->absmax_code, q->dq_step, q->dq_mean, st),
                    "quantize: double-quant launch");
}

}  // namespace

extern "C" int nf4_quantize(const uint16_t *W, const ql_nf4_tensor *q, void *ws, size_t ws_bytes,
                            ql_stream_t stream) {
  g_msg[0] = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc = quantize_first(W, q, ws, ws_bytes, st, "nf4_quantize");
  if (rc) return rc;
  return quantize_second(q, ws, q->rows * q->cols / 64, st);
}

extern "C" int nf4_quantize_shard_begin(const uint16_t *W, const ql_nf4_tensor *q, void *ws, size_t ws_bytes,
                                        ql_stream_t stream) {
  g_msg[0] = 0;
  return quantize_first(W, q, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), "nf4_quantize_shard_begin");
}

extern "C" int nf4_quantize_shard_end(const ql_nf4_tensor *q, void *ws, size_t ws_bytes, int64_t total_blocks,
                                      ql_stream_t stream) {
  g_msg[0] = 0;
  const char *fn = "nf4_quantize_shard_end";
  int rc = check_tensor(q, fn, true);
  if (rc) return rc;
  rc = check_quant_ws(q, ws, ws_bytes, fn);
  if (rc) return rc;
  const int64_t n_b = q->rows * q->cols / 64;
  if (total_blocks < n_b)
    return set_error(QL_ERR_INVALID, "%s: total_blocks %lld < the shard's %lld blocks", fn, (long long)total_blocks,
                     (long long)n_b);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  note_other_call(st);
  return quantize_second(q, ws, total_blocks, st);
}

extern "C" int nf4_dequantize(const ql_nf4_tensor *q, uint16_t *W_out, ql_stream_t stream) {
  g_msg[0] = 0;
  int rc = check_tensor(q, "nf4_dequantize", true);
  if (rc) return rc;
  if (!W_out) return set_error(QL_ERR_INVALID, "nf4_dequantize: null output");
  if (!aligned(W_out, 16)) return set_error(QL_ERR_MISALIGNED, "nf4_dequantize: output not 16-byte aligned");
  note_other_call(reinterpret_cast<cudaStream_t>(stream));
  return check_cuda(launch_dequantize(*q, W_out, reinterpret_cast<cudaStream_t>(stream)),
                    "nf4_dequantize: launch");
}

extern "C" int qlora_linear_fwd(const uint16_t *X, int64_t M, const ql_nf4_tensor *W, const uint16_t *A,
                                const uint16_t *B, int32_t r, float scale, uint16_t *Y, uint16_t *XA_out,
                                void *ws, size_t ws_bytes, ql_stream_t stream) {
  g_msg[0] = 0;
  int rc = check_tensor(W, "qlora_linear_fwd", true);
  if (rc) return rc;
  LinearArgs a{};
  a.X = X; a.M = M; a.W = *W; a.A = A; a.B = B; a.r = r; a.scale = scale;
  a.Y = Y; a.XA = XA_out; a.ws = ws; a.ws_bytes = ws_bytes;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return linear_fwd(a);
}

extern "C" int qlora_linear_fwd_fp8(const uint16_t *X, int64_t M, const ql_nf4_tensor *W, const uint16_t *A,
                                    const uint16_t *B, int32_t r, float scale, uint16_t *Y, uint16_t *XA_out,
                                    void *ws, size_t ws_bytes, ql_stream_t stream) {
  g_msg[0] = 0;
  int rc = check_tensor(W, "qlora_linear_fwd_fp8", true);
  if (rc) return rc;
  LinearArgs a{};
  a.X = X; a.M = M; a.W = *W; a.A = A; a.B = B; a.r = r; a.scale = scale;
  a.Y = Y; a.XA = XA_out; a.ws = ws; a.ws_bytes = ws_bytes;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return linear_fwd_fp8(a);
}

extern "C" int qlora_linear_bwd(const uint16_t *dY, const uint16_t *X, const uint16_t *XA, int64_t M,
                                const ql_nf4_tensor *W, const uint16_t *A, const uint16_t *B, int32_t r,
                                float scale, uint16_t *dX, float *dA, float *dB, void *ws, size_t ws_bytes,
                                ql_stream_t stream) {
  g_msg[0] = 0;
  int rc = check_tensor(W, "qlora_linear_bwd", true);
  if (rc) return rc;
  LinearArgs a{};
  a.dY = dY; a.X = X; a.XA_in = XA; a.M = M; a.W = *W; a.A = A; a.B = B; a.r = r; a.scale = scale;
  a.dX = dX; a.dA = dA; a.dB = dB; a.ws = ws; a.ws_bytes = ws_bytes;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return linear_bwd(a);
}

extern "C" int qlora_linear_bwd_fp8(const uint16_t *dY, const uint16_t *X, const uint16_t *XA, int64_t M,
                                const ql_nf4_tensor *W, const uint16_t *A, const uint16_t *B, int32_t r,
                                float scale, uint16_t *dX, float *dA, float *dB, void *ws, size_t ws_bytes,
                                ql_stream_t stream) {
  g_msg[0] = 0;
  int rc = check_tensor(W, "qlora_linear_bwd_fp8", true);
  if (rc) return rc;
  LinearArgs a{};
  a.dY = dY; a.X = X; a.XA_in = XA; a.M = M; a.W = *W; a.A = A; a.B = B; a.r = r; a.scale = scale;
  a.dX = dX; a.dA = dA; a.dB = dB; a.ws = ws; a.ws_bytes = ws_bytes;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return linear_bwd_fp8(a);
}

extern "C" int qlora_merge(const ql_nf4_tensor *W, const uint16_t *A, const uint16_t *B, int32_t r, float scale,
                           uint16_t *W_out, ql_stream_t stream) {
  g_msg[0] = 0;
  const char *fn = "qlora_merge";
  int rc = check_tensor(W, fn, true);
  if (rc) return rc;
  if (!A || !B || !W_out) return set_error(QL_ERR_INVALID, "%s: null A, B or W_out", fn);
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(W_out, 16))
    return set_error(QL_ERR_MISALIGNED, "%s: A, B or W_out not 16-byte aligned", fn);
  if (r != 8 && r != 16 && r != 32 && r != 64 && r != 128)
    return set_error(QL_ERR_UNSUPPORTED, "%s: rank %d (8, 16, 32, 64 or 128)", fn, r);
  if (W->rows % 8) return set_error(QL_ERR_UNSUPPORTED, "%s: N = %lld not a multiple of 8", fn, (long long)W->rows);
  if (W->rows > ((int64_t)1 << 30) || W->cols > ((int64_t)1 << 30))
    return set_error(QL_ERR_UNSUPPORTED, "%s: dimension above 2^30", fn);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  note_other_call(st);
  return launch_merge(*W, A, B, r, scale, W_out, st);
}

extern "C" int nf4_quantize_host(const uint16_t *W_host, const ql_nf4_tensor *q, void *ws, size_t ws_bytes,
                                 ql_stream_t copy_stream, ql_stream_t stream) {
  g_msg[0] = 0;
  const char *fn = "nf4_quantize_host";
  int rc = check_tensor(q, fn, true);
  if (rc) return rc;
  if (!W_host) return set_error(QL_ERR_INVALID, "%s: null W_host", fn);
  if (!ws) return set_error(QL_ERR_INVALID, "%s: null workspace", fn);
  if (!aligned(ws, 256)) return set_error(QL_ERR_MISALIGNED, "%s: workspace not 256-byte aligned", fn);
  const int64_t N = q->rows, K = q->cols;
  if (ws_bytes < quantize_host_ws(N, K))
    return set_error(QL_ERR_UNSUPPORTED, "%s: workspace %zu < %zu bytes", fn, ws_bytes, quantize_host_ws(N, K));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t cst = reinterpret_cast<cudaStream_t>(copy_stream);
  note_other_call(st);
  char *base = static_cast<char *>(ws);
  double *sum = reinterpret_cast<double *>(base);
  float *absmax = q->dq_blocksize ? reinterpret_cast<float *>(base + 256) : q->absmax;
  const int64_t crows = host_chunk_rows(N, K);
  const size_t cbytes = round_up((size_t)(crows * K * 2), 256);
  uint16_t *stage[2] = {reinterpret_cast<uint16_t *>(base + quantize_ws(N, K)),
                        reinterpret_cast<uint16_t *>(base + quantize_ws(N, K) + cbytes)};
  cudaEvent_t ev[5] = {};
  for (auto &e : ev) {
    rc = check_cuda(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "nf4_quantize_host: event");
    if (rc) break;
  }
  // ev[0]: work queued on `stream` before this call (it may still use ws);
  // ev[1 + h]: chunk in staging buffer h copied; ev[3 + h]: chunk in h coded
  if (!rc) rc = check_cuda(cudaMemsetAsync(sum, 0, sizeof(double), st), "nf4_quantize_host: clear sum");
  if (!rc) rc = check_cuda(cudaEventRecord(ev[0], st), "nf4_quantize_host: record");
  if (!rc) rc = check_cuda(cudaStreamWaitEvent(cst, ev[0], 0), "nf4_quantize_host: wait");
  for (int64_t r0 = 0, c = 0; !rc && r0 < N; r0 += crows, ++c) {
    const int h = (int)(c & 1);
    const int64_t rows = std::min(crows, N - r0);
    if (c >= 2) rc = check_cuda(cudaStreamWaitEvent(cst, ev[3 + h], 0), "nf4_quantize_host: wait");
    if (!rc)
      rc = check_cuda(cudaMemcpyAsync(stage[h], W_host + r0 * K, (size_t)(rows * K * 2), cudaMemcpyHostToDevice, cst),
                      "nf4_quantize_host: copy");
    if (!rc) rc = check_cuda(cudaEventRecord(ev[1 + h], cst), "nf4_quantize_host: record");
    if (!rc) rc = check_cuda(cudaStreamWaitEvent(st, ev[1 + h], 0), "nf4_quantize_host: wait");
    if (!rc)
      rc = check_cuda(launch_quantize(stage[h], rows, K, q->quant_type, q->packed + r0 * (K / 2),
                                      absmax + r0 * (K / 64), sum, st),
                      "nf4_quantize_host: launch");
    if (!rc) rc = check_cuda(cudaEventRecord(ev[3 + h], st), "nf4_quantize_host: record");
  }
  if (!rc && q->dq_blocksize)
    rc = check_cuda(launch_double_quant(absmax, N * K / 64, N * K / 64, q->dq_blocksize, q->dq_type, sum, q->absmax_code,
                                        q->dq_step, q->dq_mean, st),
                    "nf4_quantize_host: double-quant launch");
  for (auto &e : ev)
    if (e) cudaEventDestroy(e);  // released once recorded work completes
  return rc;
}
