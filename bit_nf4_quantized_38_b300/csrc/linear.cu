#include "linear.cuh"

namespace ql {
size_t linear_fwd_ws(int64_t, int64_t, int64_t, int32_t) { return 0; }
size_t linear_bwd_ws(int64_t, int64_t, int64_t, int32_t) { return 0; }
int linear_fwd(const LinearArgs &) { return set_error(QL_ERR_UNSUPPORTED, "qlora_linear_fwd: not built yet"); }
int linear_bwd(const LinearArgs &) { return set_error(QL_ERR_UNSUPPORTED, "qlora_linear_bwd: not built yet"); }
}  // namespace ql
