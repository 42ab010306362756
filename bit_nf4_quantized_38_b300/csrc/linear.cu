// Forward and backward of the frozen-NF4 linear with a LoRA adapter:
// argument checks, workspace layout and the launch sequence on one stream.
//
// forward  (M tokens):
//   1. XA = X A                      split-reduction side GEMM + finalize
//   2. Bt = bf16(s B^T), zero-padded  pack
//   3. Y  = X W_hat^T + XA Bt^T       tensor-core GEMM, LoRA as extra K-steps
// backward:
//   1. XA (copied from the forward, or recomputed)
//   2. Gs = bf16(s dY B^T)            side GEMM + finalize
//   3. Ap = A, zero-padded            pack
//   4. dX = dY W_hat + Gs Ap^T        tensor-core GEMM (W_hat^T tiles)
//   5. dA = X^T Gs                    side GEMM + finalize
//   6. dB = s XA^T dY                 side GEMM + finalize
#include <algorithm>

#include "decode.cuh"
#include "linear.cuh"
#include "tc_gemm.cuh"

namespace ql {
namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }
int padded_rank(int r) { return std::max(64, (r + 63) / 64 * 64); }
bool rank_ok(int r) { return r == 8 || r == 16 || r == 32 || r == 64 || r == 128; }
bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct FwdLayout {
  size_t xa_pad, bt_pad, part, total;
  int splits;
};
FwdLayout fwd_layout(int64_t M, int64_t N, int64_t K, int r) {
  FwdLayout L{};
  const int rp = padded_rank(r);
  L.splits = skinny_splits(M, r, K);
  size_t off = 0;
  L.xa_pad = off; off += up256((size_t)M * rp * 2);
  L.bt_pad = off; off += up256((size_t)N * rp * 2);
  L.part = off; off += up256((size_t)L.splits * M * r * 4);
  L.total = off;
  return L;
}

struct BwdLayout {
  size_t xa_pad, gs_pad, a_pad, part, total;
  int s_xa, s_g, s_da, s_db;
};
BwdLayout bwd_layout(int64_t M, int64_t N, int64_t K, int r) {
  BwdLayout L{};
  const int rp = padded_rank(r);
  L.s_xa = skinny_splits(M, r, K);
  L.s_g = skinny_splits(M, r, N);
  L.s_da = skinny_splits(K, r, M);
  L.s_db = skinny_splits(r, N, M);
  size_t part = std::max({(size_t)L.s_xa * M * r, (size_t)L.s_g * M * r, (size_t)L.s_da * K * r,
                          (size_t)L.s_db * r * N}) * 4;
  size_t off = 0;
  L.xa_pad = off; off += up256((size_t)M * rp * 2);
  L.gs_pad = off; off += up256((size_t)M * rp * 2);
  L.a_pad = off; off += up256((size_t)K * rp * 2);
  L.part = off; off += up256(part);
  L.total = off;
  return L;
}

int check_common(const LinearArgs &a, const char *fn, size_t need) {
  if (a.M <= 0) return set_error(QL_ERR_INVALID, "%s: M = %lld", fn, (long long)a.M);
  if (!rank_ok(a.r)) return set_error(QL_ERR_UNSUPPORTED, "%s: rank %d (8, 16, 32, 64 or 128)", fn, a.r);
  if (a.W.rows % 8) return set_error(QL_ERR_UNSUPPORTED, "%s: N = %lld not a multiple of 8", fn, (long long)a.W.rows);
  if (a.M > (int64_t)1 << 30 || a.W.rows > (int64_t)1 << 30 || a.W.cols > (int64_t)1 << 30)
    return set_error(QL_ERR_UNSUPPORTED, "%s: dimension above 2^30", fn);
  if (need && !a.ws) return set_error(QL_ERR_INVALID, "%s: null workspace", fn);
  if (a.ws && (reinterpret_cast<uintptr_t>(a.ws) & 255))
    return set_error(QL_ERR_MISALIGNED, "%s: workspace not 256-byte aligned", fn);
  if (a.ws_bytes < need) return set_error(QL_ERR_UNSUPPORTED, "%s: workspace %zu < %zu bytes", fn, a.ws_bytes, need);
  return QL_OK;
}

#define QL_TRY(x)            \
  do {                       \
    int rc_ = (x);           \
    if (rc_) return rc_;     \
  } while (0)

}  // namespace

constexpr int64_t kDecodeMaxM = 16;  // M at or below this takes the decode path

size_t linear_fwd_ws(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M <= 0 || N <= 0 || K <= 0 || !rank_ok(r)) return 0;
  if (M <= kDecodeMaxM) return decode_ws(N, K, r);
  return fwd_layout(M, N, K, r).total;
}

size_t linear_bwd_ws(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M <= 0 || N <= 0 || K <= 0 || !rank_ok(r)) return 0;
  return bwd_layout(M, N, K, r).total;
}

int linear_fwd(const LinearArgs &a) {
  const char *fn = "qlora_linear_fwd";
  if (!a.X || !a.A || !a.B || !a.Y) return set_error(QL_ERR_INVALID, "%s: null X, A, B or Y", fn);
  if (!al16(a.X) || !al16(a.A) || !al16(a.B) || !al16(a.Y) || (a.XA && !al16(a.XA)))
    return set_error(QL_ERR_MISALIGNED, "%s: operand not 16-byte aligned", fn);
  const int64_t M = a.M, N = a.W.rows, K = a.W.cols;
  const int r = a.r, rp = padded_rank(r);
  if (M >= 1 && M <= kDecodeMaxM) {
    QL_TRY(check_common(a, fn, decode_ws(N, K, r)));
    DecodeProblem d{};
    d.X = a.X; d.M = M; d.K = K; d.N = N; d.w = nf4_view(a.W); d.A = a.A; d.B = a.B; d.r = r;
    d.scale = a.scale; d.Y = a.Y; d.XA_out = a.XA; d.ws = a.ws;
    return launch_decode(d, a.stream);
  }
  const FwdLayout L = fwd_layout(M, N, K, r);
  QL_TRY(check_common(a, fn, L.total));
  char *ws = static_cast<char *>(a.ws);
  uint16_t *xa_pad = reinterpret_cast<uint16_t *>(ws + L.xa_pad);
  uint16_t *bt_pad = reinterpret_cast<uint16_t *>(ws + L.bt_pad);
  float *part = reinterpret_cast<float *>(ws + L.part);
  cudaStream_t st = a.stream;

  QL_TRY(launch_skinny(SkinnyProblem{a.X, K, false, a.A, r, false, M, r, K, L.splits, part}, st));
  QL_TRY(launch_finalize_bf16(part, L.splits, M, r, 1.0f, xa_pad, rp, a.XA, st));
  QL_TRY(launch_pack_transpose(a.B, r, N, a.scale, bt_pad, rp, st));
  GemmProblem g{};
  g.trans = false;
  g.A = a.X; g.M = M; g.Kred = K;
  g.A2 = xa_pad; g.B2 = bt_pad; g.r = r; g.rp = rp;
  g.w = nf4_view(a.W);
  g.out = a.Y; g.Nout = N;
  return launch_nf4_gemm(g, st);
}

int linear_bwd(const LinearArgs &a) {
  const char *fn = "qlora_linear_bwd";
  if (!a.dY || !a.X || !a.A || !a.B || !a.dX || !a.dA || !a.dB)
    return set_error(QL_ERR_INVALID, "%s: null operand", fn);
  if (!al16(a.dY) || !al16(a.X) || !al16(a.A) || !al16(a.B) || !al16(a.dX) || !al16(a.dA) || !al16(a.dB) ||
      (a.XA_in && !al16(a.XA_in)))
    return set_error(QL_ERR_MISALIGNED, "%s: operand not 16-byte aligned", fn);
  const int64_t M = a.M, N = a.W.rows, K = a.W.cols;
  const int r = a.r, rp = padded_rank(r);
  const BwdLayout L = bwd_layout(M, N, K, r);
  QL_TRY(check_common(a, fn, L.total));
  char *ws = static_cast<char *>(a.ws);
  uint16_t *xa_pad = reinterpret_cast<uint16_t *>(ws + L.xa_pad);
  uint16_t *gs_pad = reinterpret_cast<uint16_t *>(ws + L.gs_pad);
  uint16_t *a_pad = reinterpret_cast<uint16_t *>(ws + L.a_pad);
  float *part = reinterpret_cast<float *>(ws + L.part);
  cudaStream_t st = a.stream;

  // 1. XA, zero-padded to rp columns
  if (a.XA_in) {
    QL_TRY(launch_pack_pad(a.XA_in, M, r, xa_pad, rp, st));
  } else {
    QL_TRY(launch_skinny(SkinnyProblem{a.X, K, false, a.A, r, false, M, r, K, L.s_xa, part}, st));
    QL_TRY(launch_finalize_bf16(part, L.s_xa, M, r, 1.0f, xa_pad, rp, nullptr, st));
  }
  // 2. Gs = bf16(s dY B^T)
  QL_TRY(launch_skinny(SkinnyProblem{a.dY, N, false, a.B, N, true, M, r, N, L.s_g, part}, st));
  QL_TRY(launch_finalize_bf16(part, L.s_g, M, r, a.scale, gs_pad, rp, nullptr, st));
  // 3-4. dX = dY W_hat + Gs A^T
  QL_TRY(launch_pack_pad(a.A, K, r, a_pad, rp, st));
  GemmProblem g{};
  g.trans = true;
  g.A = a.dY; g.M = M; g.Kred = N;
  g.A2 = gs_pad; g.B2 = a_pad; g.r = r; g.rp = rp;
  g.w = nf4_view(a.W);
  g.out = a.dX; g.Nout = K;
  QL_TRY(launch_nf4_gemm(g, st));
  // 5. dA = X^T Gs
  QL_TRY(launch_skinny(SkinnyProblem{a.X, K, true, gs_pad, rp, false, K, r, M, L.s_da, part}, st));
  QL_TRY(launch_finalize_f32(part, L.s_da, K, r, 1.0f, a.dA, st));
  // 6. dB = s XA^T dY
  QL_TRY(launch_skinny(SkinnyProblem{xa_pad, rp, true, a.dY, N, false, r, N, M, L.s_db, part}, st));
  return launch_finalize_f32(part, L.s_db, r, N, a.scale, a.dB, st);
}

}  // namespace ql
