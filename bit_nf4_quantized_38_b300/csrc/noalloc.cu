// nf4_quantize without a caller-provided workspace.
//
// Some callers cannot hand the library a scratch buffer: code that runs
// where device allocation is not allowed or not wanted -- inside a host
// runtime that owns every allocation, under a memory planner that fixed every
// buffer up front, or on a latency-critical path where cudaMalloc's implicit
// device synchronisation is unacceptable -- and thin C callers that have no
// allocator of their own.  For them the quantizer's scratch (an fp64 sum and
// the fp32 block absmax values) lives in one file-scope device array of fixed
// size, which every GPU that loads the library keeps until the process exits.
#include <mutex>

#include "common.cuh"

namespace ql {
namespace {

// 256 bytes for the fp64 sum, then room for kNoAllocMaxBlocks fp32 absmax
// values: 4 Mi blocks of 64 = 256 Mi parameters (every LLaMA-65B weight fits).
constexpr int64_t kNoAllocMaxBlocks = int64_t(1) << 22;
constexpr size_t kNoAllocBytes = 256 + (size_t)kNoAllocMaxBlocks * 4;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the host-side name is only a stand-in, never a device address).
int scratch_address(void **out) {
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "nf4_quantize_noalloc: current device");
  if (rc) return rc;
  if (dev < 0 || dev >= 64) return set_error(QL_ERR_UNSUPPORTED, "nf4_quantize_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    rc = check_cuda(cudaGetSymbolAddress(&p, g_noalloc_scratch), "nf4_quantize_noalloc: scratch address");
    if (rc) return rc;
    addr[dev] = p;
  }
  *out = addr[dev];
  return QL_OK;
}

}  // namespace
}  // namespace ql

using namespace ql;

extern "C" int nf4_quantize_noalloc(const uint16_t *W, const ql_nf4_tensor *q, ql_stream_t stream) {
  if (!q) return set_error(QL_ERR_INVALID, "nf4_quantize_noalloc: null nf4 tensor");
  if (q->rows > 0 && q->cols > 0 && q->rows * (q->cols / 64) > kNoAllocMaxBlocks)
    return set_error(QL_ERR_UNSUPPORTED,
                     "nf4_quantize_noalloc: %lld x %lld weight has %lld blocks; the built-in scratch holds at most "
                     "%lld (use nf4_quantize with a workspace)",
                     (long long)q->rows, (long long)q->cols, (long long)(q->rows * (q->cols / 64)),
                     (long long)kNoAllocMaxBlocks);
  void *ws = nullptr;
  int rc = scratch_address(&ws);
  if (rc) return rc;
  // Same checks and launch sequence as nf4_quantize; the fp64 sum at the head
  // of the scratch is cleared by nf4_quantize on every call.
  return nf4_quantize(W, q, ws, kNoAllocBytes, stream);
}
