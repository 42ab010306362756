// Self-test of the library's failure path.  Every wait in the library's
// kernels is bounded by wall time; when one gives up, the kernel records it in
// the device status word and returns instead of hanging, and the host learns
// of it from ql_get_device_status.  This entry point exercises that path on
// purpose: one CTA waits on a barrier that nothing will ever complete, with
// the caller's limit, so the status word must read "timed out" afterwards
// while the context stays usable.
#include "common.cuh"
#include "linear.cuh"
#include "ptx.cuh"

namespace ql {
namespace {

__global__ void __launch_bounds__(32) k_selftest_wait(uint64_t limit_ns, int *status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);  // one arrival expected; none ever comes
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncwarp();
  ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

}  // namespace
}  // namespace ql

using namespace ql;

extern "C" int ql_selftest_wait(int64_t limit_ns, ql_stream_t stream) {
  if (limit_ns <= 0 || limit_ns > 2000000000ll)
    return set_error(QL_ERR_INVALID, "ql_selftest_wait: limit %lld ns outside (0, 2 s]", (long long)limit_ns);
  int *status = device_status_ptr();
  if (!status) return set_error(QL_ERR_CUDA, "ql_selftest_wait: no device status word");
  note_other_call(reinterpret_cast<cudaStream_t>(stream));
  k_selftest_wait<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>((uint64_t)limit_ns, status);
  count_launch();
  return check_cuda(cudaGetLastError(), "ql_selftest_wait launch");
}
