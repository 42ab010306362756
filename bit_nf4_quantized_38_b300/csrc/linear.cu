// Forward and backward of the frozen-NF4 linear with a LoRA adapter:
// argument checks, workspace layout and the launch sequence on one stream.
//
// forward, M > 32 tokens (2 launches; 3 for M <= 128):
//   1. XA = X A  -> XA_out (bf16) and XAs = bf16(s XA)     LoRA kernel
//   2. Y  = X W_hat^T + XAs B                             tensor-core GEMM,
//                                                          LoRA as extra K-steps
//      (M <= 128: the few-token kernel, skinny.cu, and its fixup kernel)
// forward, M <= 32: the decode path (decode.cu).
// backward (4 launches, 5 when XA must be recomputed):
//   0. XA = X A                                            (only without XA)
//   1. Gs = bf16(s dY B^T)                                  LoRA kernel
//   2. dX = dY W_hat + Gs A^T                               tensor-core GEMM
//   3. dA = X^T Gs                                          LoRA kernel
//   4. dB = s XA^T dY                                       LoRA kernel (stores dB^T's transpose)
#include <algorithm>
#include <mutex>
#include <unordered_map>
#include <utility>
#include <vector>

#include "decode.cuh"
#include "fp8.cuh"
#include "linear.cuh"
#include "tc_gemm.cuh"

namespace ql {
namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }
bool rank_ok(int r) { return r == 8 || r == 16 || r == 32 || r == 64 || r == 128; }
bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// forward workspace: XAs [M][r] bf16; backward: Gs [M][r] + recomputed XA [M][r];
// with M <= 128 tokens either also holds the fp32 partials of the GEMM (the
// forward's few-token kernel, the backward's split over the reduction).
// Training workspaces have two halves; successive calls on a stream
// alternate between them (see next_ws_half).
size_t part_bytes(int64_t M, int64_t Nout, int64_t Kred) {
  const int s = gemm_splits(M, Nout, Kred);
  return s > 1 ? up256((size_t)s * M * Nout * 4) : 0;
}
size_t fwd_part_bytes(int64_t M, int64_t N, int64_t K, int r) { return up256(skinny_part_bytes(M, N, K, r)); }
size_t fwd_half(int64_t M, int64_t N, int64_t K, int r) {  // s XA bf16 [M][r], partials
  return up256((size_t)M * r * 2) + fwd_part_bytes(M, N, K, r);
}
size_t bwd_half(int64_t M, int64_t N, int64_t K, int r) {  // s G, XA: bf16 [M][r] each, partials
  return 2 * up256((size_t)M * r * 2) + part_bytes(M, K, N);
}
size_t fwd_ws(int64_t M, int64_t N, int64_t K, int r) { return 2 * fwd_half(M, N, K, r); }
size_t bwd_ws(int64_t M, int64_t N, int64_t K, int r) { return 2 * bwd_half(M, N, K, r); }

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

// M at or below this takes the decode path (the weight-streaming kernel with
// 8, 16 or 32 token columns); above it the few-token tensor-core kernel
constexpr int64_t kDecodeMaxM = 32;

// ---------------------------------------------------------------------------
// What the previous library call on a stream may still be reading or writing.
//
// Within a call the kernels are programmatic dependents of one another, and
// so is the first kernel of a linear call of the one before it.  When that
// first kernel's inputs are disjoint from everything the previous linear
// call writes (its outputs and its workspace), it may read and compute while
// that call's last kernels still run, and waits only before its first store:
// every kernel older than the previous call has completed by the time the
// previous call lets a dependent start (a call's kernels let dependents start
// only after waiting for their own predecessor), and a kernel launched
// without programmatic dependence in between makes the hardware fall back to
// full ordering.  The decode kernel may also store early, into workspace and
// outputs that the previous call neither reads nor writes.
struct Range {
  uintptr_t lo, hi;
};
//
// A decode call whose finishing kernel lets dependents launch before it has
// waited for its own predecessor (`early_dependents`) relies on the next
// call's stream CTAs being too large to share an SM with its stream CTAs
// (which fill every SM), so that the call before it has completed by the time
// the next call's CTAs run.  That holds only for a decode call after it; any
// other call after it waits for it in full.
struct PrevCall {
  bool linear = false;  // a linear call (its kernels let dependents start early)
  bool early_dependents = false;  // a decode call that let dependents launch before its own wait
  std::vector<Range> writes, reads;
  int decode_half = 0;  // workspace half of the stream's last decode call
};
// Keyed by (device, stream): the legacy and per-thread default stream handles
// are the same value on every device.
struct StreamKey {
  int dev;
  cudaStream_t st;
  bool operator==(const StreamKey &o) const { return dev == o.dev && st == o.st; }
};
struct StreamKeyHash {
  size_t operator()(const StreamKey &k) const {
    return std::hash<const void *>()(static_cast<const void *>(k.st)) * 31u + (size_t)k.dev;
  }
};
std::mutex g_prev_mu;
std::unordered_map<StreamKey, PrevCall, StreamKeyHash> g_prev;

StreamKey key_of(cudaStream_t st) {
  int dev = 0;
  cudaGetDevice(&dev);
  return StreamKey{dev, st};
}

Range range(const void *p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}

// True if early modes are allowed after the stream's previous call for a call
// of the given kind (see PrevCall).
bool early_ok(const PrevCall &pc, bool decode_next) { return pc.linear && (decode_next || !pc.early_dependents); }

// True if the stream's previous call was a linear call whose writes miss all of `reads`.
bool reads_clear_of_previous(cudaStream_t st, const std::vector<Range> &reads, bool decode_next = false) {
  std::lock_guard<std::mutex> lock(g_prev_mu);
  auto it = g_prev.find(key_of(st));
  if (it == g_prev.end() || !early_ok(it->second, decode_next)) return false;
  for (const Range &r : reads)
    for (const Range &w : it->second.writes)
      if (r.lo < w.hi && w.lo < r.hi) return false;
  return true;
}

// True if the stream's previous call was a linear call that neither reads
// nor writes any of `writes`.
bool writes_clear_of_previous(cudaStream_t st, const std::vector<Range> &writes, bool decode_next = false) {
  std::lock_guard<std::mutex> lock(g_prev_mu);
  auto it = g_prev.find(key_of(st));
  if (it == g_prev.end() || !early_ok(it->second, decode_next)) return false;
  for (const Range &r : writes) {
    for (const Range &w : it->second.writes)
      if (r.lo < w.hi && w.lo < r.hi) return false;
    for (const Range &w : it->second.reads)
      if (r.lo < w.hi && w.lo < r.hi) return false;
  }
  return true;
}

void note_call(cudaStream_t st, bool linear, std::vector<Range> writes, std::vector<Range> reads = {},
               bool early_dependents = false) {
  std::lock_guard<std::mutex> lock(g_prev_mu);
  PrevCall &pc = g_prev[key_of(st)];
  pc.linear = linear;
  pc.early_dependents = early_dependents;
  pc.writes = std::move(writes);
  pc.reads = std::move(reads);
}

// Linear calls on a stream alternate between the two halves of their
// workspace, so a call never writes the half its predecessor may still use.
int next_ws_half(cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_prev_mu);
  PrevCall &pc = g_prev[key_of(st)];
  pc.decode_half ^= 1;
  return pc.decode_half;
}

void weight_ranges(const ql_nf4_tensor &W, std::vector<Range> &out) {
  const int64_t n_b = W.rows * W.cols / 64;
  out.push_back(range(W.packed, (size_t)(W.rows * W.cols / 2)));
  if (W.dq_blocksize) {
    out.push_back(range(W.absmax_code, (size_t)n_b));
    out.push_back(range(W.dq_step, (size_t)((n_b + 255) / 256) * 4));
    out.push_back(range(W.dq_mean, 4));
  } else {
    out.push_back(range(W.absmax, (size_t)n_b * 4));
  }
}

}  // namespace

void note_other_call(cudaStream_t st) { note_call(st, false, {}); }

size_t linear_fwd_ws(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M <= 0 || N <= 0 || K <= 0 || !rank_ok(r)) return 0;
  if (M <= kDecodeMaxM) return decode_ws(N, K, r);
  return fwd_ws(M, N, K, r);
}

size_t linear_bwd_ws(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M <= 0 || N <= 0 || K <= 0 || !rank_ok(r)) return 0;
  return bwd_ws(M, N, K, r);
}

int linear_fwd(const LinearArgs &a) {
  const char *fn = "qlora_linear_fwd";
  if (!a.X || !a.A || !a.B || !a.Y) return set_error(QL_ERR_INVALID, "%s: null X, A, B or Y", fn);
  if (!al16(a.X) || !al16(a.A) || !al16(a.B) || !al16(a.Y) || (a.XA && !al16(a.XA)))
    return set_error(QL_ERR_MISALIGNED, "%s: operand not 16-byte aligned", fn);
  const int64_t M = a.M, N = a.W.rows, K = a.W.cols;
  const int r = a.r;
  if (M >= 1 && M <= kDecodeMaxM) {
    QL_TRY(check_common(a, fn, decode_ws(N, K, r)));
    DecodeProblem d{};
    d.X = a.X; d.M = M; d.K = K; d.N = N; d.w = nf4_view(a.W); d.A = a.A; d.B = a.B; d.r = r;
    d.scale = a.scale; d.Y = a.Y; d.XA_out = a.XA; d.ws = a.ws;
    d.half = next_ws_half(a.stream);
    std::vector<Range> reads;
    weight_ranges(a.W, reads);
    d.w_early = reads_clear_of_previous(a.stream, reads, true);
    const std::vector<Range> xab = {range(a.X, (size_t)(M * K * 2)), range(a.A, (size_t)(K * r * 2)),
                                    range(a.B, (size_t)(r * N * 2))};
    d.x_early = d.w_early && reads_clear_of_previous(a.stream, xab, true);
    reads.insert(reads.end(), xab.begin(), xab.end());
    const size_t half = decode_ws_half(N, r);
    const Range wsr = range(static_cast<char *>(a.ws) + (d.half ? half : 0), half);
    std::vector<Range> outs = {range(a.Y, (size_t)(M * N * 2))};
    if (a.XA) outs.push_back(range(a.XA, (size_t)(M * r * 2)));
    d.ws_early = writes_clear_of_previous(a.stream, {wsr}, true);
    outs.push_back(wsr);
    bool early_dependents = false;
    const int rc = launch_decode(d, a.stream, &early_dependents);
    // recorded even when the launch failed part-way: the next call then waits in full
    note_call(a.stream, rc == QL_OK, std::move(outs), std::move(reads), early_dependents);
    return rc;
  }
  QL_TRY(check_common(a, fn, fwd_ws(M, N, K, r)));
  cudaStream_t st = a.stream;
  const size_t half = fwd_half(M, N, K, r);
  char *wsh = static_cast<char *>(a.ws) + (next_ws_half(st) ? half : 0);
  uint16_t *xas = reinterpret_cast<uint16_t *>(wsh);
  float *part = fwd_part_bytes(M, N, K, r) ? reinterpret_cast<float *>(wsh + up256((size_t)M * r * 2)) : nullptr;

  const std::vector<Range> xa_reads = {range(a.X, (size_t)(M * K * 2)), range(a.A, (size_t)(K * r * 2))};
  std::vector<Range> xa_writes = {range(wsh, half)};
  if (a.XA) xa_writes.push_back(range(a.XA, (size_t)(M * r * 2)));
  std::vector<Range> reads = xa_reads;
  reads.push_back(range(a.B, (size_t)(r * N * 2)));
  weight_ranges(a.W, reads);
  const bool early = reads_clear_of_previous(st, reads);
  std::vector<Range> main_reads = {range(a.X, (size_t)(M * K * 2))};
  weight_ranges(a.W, main_reads);
  const bool gemm_early = reads_clear_of_previous(st, main_reads);
  const bool free_ = reads_clear_of_previous(st, xa_reads) && writes_clear_of_previous(st, xa_writes);
  std::vector<Range> writes = xa_writes;
  writes.push_back(range(a.Y, (size_t)(M * N * 2)));
  note_call(st, true, std::move(writes), reads);

  LoraProblem L{};
  L.A = a.X; L.a_mn = false; L.B = a.A; L.b_mn = true;  // X [M][K], A [K][r]
  L.P = M; L.Q = r; L.T = K; L.mode = 0; L.scale = a.scale;
  L.out = xas; L.ldo = r; L.out2 = a.XA; L.ldo2 = r;
  L.dep = free_ ? kDepFree : (early ? kDepStores : kDepStart);
  QL_TRY(launch_lora(L, st));
  GemmProblem g{};
  g.trans = false;
  g.A = a.X; g.M = M; g.Kred = K;
  g.A2 = xas; g.B2 = a.B; g.r = r;
  g.w = nf4_view(a.W);
  g.out = a.Y; g.Nout = N;
  g.early_main = gemm_early;
  g.part = part;
  return launch_nf4_gemm(g, st);
}

// E4M3 forward workspace: two halves (calls on a stream alternate), each
// [partial maxima of |m_hat| | pad to 1 KB][row exponents M int32][X codes
// M x K bytes][XAs M x r bf16]
size_t fp8_fwd_half(int64_t M, int64_t K, int32_t r) {
  return 1024 + up256((size_t)M * 4) + up256((size_t)M * K) + up256((size_t)M * r * 2);
}
size_t linear_fwd_fp8_ws(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M <= 0 || N <= 0 || K <= 0 || !rank_ok(r)) return 0;
  return 2 * fp8_fwd_half(M, K, r);
}

// Forward with E4M3 main steps (3 launches, in stream order):
//   1. X codes e4m3(x 2^E_m) with the row exponents, and max |m_hat| partials  (k_prep_e4m3)
//   2. XA = X A -> XA_out, and XAs = bf16(fl32(s XA) 2^(E_m + E))              LoRA kernel
//   3. Y = 2^(-E_m - E) (X_e4m3 . W_e4m3^T + XAs B)                            CTA-pair GEMM
// When X and the weight are not written by the previous call on the stream,
// and this call's workspace half is not touched by it, the operand kernel and
// the LoRA kernel's main loop run alongside that call's GEMM (its last wave
// leaves SMs idle); the LoRA kernel stores once the operand kernel (and so
// the previous call) has completed, and the GEMM follows it.
int linear_fwd_fp8(const LinearArgs &a) {
  const char *fn = "qlora_linear_fwd_fp8";
  if (!a.X || !a.A || !a.B || !a.Y) return set_error(QL_ERR_INVALID, "%s: null X, A, B or Y", fn);
  if (!al16(a.X) || !al16(a.A) || !al16(a.B) || !al16(a.Y) || (a.XA && !al16(a.XA)))
    return set_error(QL_ERR_MISALIGNED, "%s: operand not 16-byte aligned", fn);
  const int64_t M = a.M, N = a.W.rows, K = a.W.cols;
  const int r = a.r;
  QL_TRY(check_common(a, fn, linear_fwd_fp8_ws(M, N, K, r)));
  cudaStream_t st = a.stream;
  const size_t half = fp8_fwd_half(M, K, r);
  char *ws = static_cast<char *>(a.ws) + (next_ws_half(st) ? half : 0);
  float *wpart = reinterpret_cast<float *>(ws);
  int *rows = reinterpret_cast<int *>(ws + 1024);
  uint8_t *xq = reinterpret_cast<uint8_t *>(ws + 1024 + up256((size_t)M * 4));
  uint16_t *xas = reinterpret_cast<uint16_t *>(ws + 1024 + up256((size_t)M * 4) + up256((size_t)M * K));
  const NF4View w = nf4_view(a.W);

  std::vector<Range> prep_reads = {range(a.X, (size_t)(M * K * 2))};
  weight_ranges(a.W, prep_reads);
  const bool prep_free = reads_clear_of_previous(st, prep_reads) && writes_clear_of_previous(st, {range(ws, half)});
  const bool lora_early = reads_clear_of_previous(st, {range(a.X, (size_t)(M * K * 2)), range(a.A, (size_t)(K * r * 2))});
  std::vector<Range> reads = prep_reads;
  reads.push_back(range(a.A, (size_t)(K * r * 2)));
  reads.push_back(range(a.B, (size_t)(r * N * 2)));
  std::vector<Range> writes = {range(ws, half), range(a.Y, (size_t)(M * N * 2))};
  if (a.XA) writes.push_back(range(a.XA, (size_t)(M * r * 2)));
  note_call(st, true, std::move(writes), reads);

  int nwpart = 0;
  // the codes in pair-swapped order, matching the GEMM's weight rows
  QL_TRY(check_cuda(launch_prep_e4m3(a.X, M, K, w, xq, rows, wpart, &nwpart, prep_free, true, st),
                    "qlora_linear_fwd_fp8: operand codes"));
  LoraProblem L{};
  L.A = a.X; L.a_mn = false; L.B = a.A; L.b_mn = true;  // X [M][K], A [K][r]
  L.P = M; L.Q = r; L.T = K; L.mode = 0; L.scale = a.scale;
  L.out = xas; L.ldo = r; L.out2 = a.XA; L.ldo2 = r;
  L.row_exp = rows;
  L.wmax = wpart;
  L.nwpart = nwpart;
  // reads X and A alongside the operand kernel (and the previous call's
  // GEMM, when the operand kernel runs free); stores, and reads the scales,
  // after the operand kernel completes
  L.dep = (prep_free && lora_early) ? kDepStores : kDepStart;
  QL_TRY(launch_lora(L, st));
  GemmProblem g{};
  g.trans = false;
  g.A = reinterpret_cast<const uint16_t *>(xq); g.M = M; g.Kred = K;
  g.A2 = xas; g.B2 = a.B; g.r = r;
  g.w = w;
  g.out = a.Y; g.Nout = N;
  g.fp8 = true;
  g.row_exp = rows;
  g.wmax = wpart;
  g.nwpart = nwpart;
  // The main loop reads the X codes, the weight and the |m_hat| partials:
  // written by the operand kernel, which completed before the LoRA kernel
  // (a dependent that waits for it before letting this GEMM start) did; the
  // LoRA kernel itself writes only XAs, read after the wait.
  g.early_main = true;
  return launch_nf4_gemm(g, st);
}

// E4M3 backward workspace: two halves (calls on a stream alternate), each
// [partial maxima of |m_hat| | pad to 1 KB][row exponents of dY, M int32]
// [dY codes M x N bytes][Gs' M x r bf16][G M x r bf16][XA M x r bf16 (recomputed
// when the caller passes none)]
size_t fp8_bwd_half(int64_t M, int64_t N, int32_t r) {
  return 1024 + up256((size_t)M * 4) + up256((size_t)M * N) + 3 * up256((size_t)M * r * 2);
}
size_t linear_bwd_fp8_ws(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M <= 0 || N <= 0 || K <= 0 || !rank_ok(r)) return 0;
  return 2 * fp8_bwd_half(M, N, r);
}

// Backward with E4M3 main steps in dX (5 or 6 launches, in stream order):
//   1. dY codes e4m3(dy 2^E_m) with the row exponents, and max |m_hat|  (k_prep_e4m3)
//   (XA = X A, when the caller passes no saved XA)                       LoRA kernel
//   2. G = dY B^T -> G16 = bf16(G) and Gs' = bf16(fl32(s G) 2^(E_m + E)) LoRA kernel
//   3. dX = 2^(-E_m - E) (dY_e4m3 . W_e4m3 + Gs' A^T)                     CTA-pair GEMM
//   4. dA = s X^T G16 and dB = s XA^T dY (as in the bf16 backward)       one LoRA launch
// As in the E4M3 forward, the kernels before the GEMM read and compute
// alongside the previous call's last kernels when their inputs and this
// call's workspace half are clear of that call.
int linear_bwd_fp8(const LinearArgs &a) {
  const char *fn = "qlora_linear_bwd_fp8";
  if (!a.dY || !a.X || !a.A || !a.B || !a.dX || !a.dA || !a.dB)
    return set_error(QL_ERR_INVALID, "%s: null operand", fn);
  if (!al16(a.dY) || !al16(a.X) || !al16(a.A) || !al16(a.B) || !al16(a.dX) || !al16(a.dA) || !al16(a.dB) ||
      (a.XA_in && !al16(a.XA_in)))
    return set_error(QL_ERR_MISALIGNED, "%s: operand not 16-byte aligned", fn);
  const int64_t M = a.M, N = a.W.rows, K = a.W.cols;
  const int r = a.r;
  QL_TRY(check_common(a, fn, linear_bwd_fp8_ws(M, N, K, r)));
  if (N % 16)  // rows of dY codes are TMA rows: a multiple of 16 bytes
    return set_error(QL_ERR_UNSUPPORTED, "%s: N = %lld not a multiple of 16", fn, (long long)N);
  cudaStream_t st = a.stream;
  const size_t half = fp8_bwd_half(M, N, r);
  char *ws = static_cast<char *>(a.ws) + (next_ws_half(st) ? half : 0);
  std::vector<Range> prep_reads = {range(a.dY, (size_t)(M * N * 2))};
  weight_ranges(a.W, prep_reads);
  const bool prep_free = reads_clear_of_previous(st, prep_reads) && writes_clear_of_previous(st, {range(ws, half)});
  std::vector<Range> lora_reads = {range(a.dY, (size_t)(M * N * 2)), range(a.X, (size_t)(M * K * 2)),
                                   range(a.A, (size_t)(K * r * 2)), range(a.B, (size_t)(r * N * 2))};
  if (a.XA_in) lora_reads.push_back(range(a.XA_in, (size_t)(M * r * 2)));
  const bool lora_early = prep_free && reads_clear_of_previous(st, lora_reads);
  std::vector<Range> reads = lora_reads;
  weight_ranges(a.W, reads);
  note_call(st, true,
            {range(a.dX, (size_t)(M * K * 2)), range(a.dA, (size_t)(K * r * 4)), range(a.dB, (size_t)(r * N * 4)),
             range(ws, half)},
            std::move(reads));
  float *wpart = reinterpret_cast<float *>(ws);
  int *rows = reinterpret_cast<int *>(ws + 1024);
  uint8_t *dyq = reinterpret_cast<uint8_t *>(ws + 1024 + up256((size_t)M * 4));
  uint16_t *gs8 = reinterpret_cast<uint16_t *>(ws + 1024 + up256((size_t)M * 4) + up256((size_t)M * N));
  uint16_t *g16 = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(gs8) + up256((size_t)M * r * 2));
  uint16_t *xa_tmp = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(g16) + up256((size_t)M * r * 2));
  const NF4View w = nf4_view(a.W);
  int nwpart = 0;
  QL_TRY(check_cuda(launch_prep_e4m3(a.dY, M, N, w, dyq, rows, wpart, &nwpart, prep_free, false, st),
                    "qlora_linear_bwd_fp8: operand codes"));
  // the LoRA kernels before the GEMM read inputs only and store after their
  // predecessor completes (the operand kernel, whose completion implies the
  // previous call's)
  const int lora_dep = lora_early ? kDepStores : kDepStart;
  const uint16_t *xa = a.XA_in;
  if (!xa) {  // XA = X A (fp32 accumulation, bf16)
    LoraProblem L{};
    L.A = a.X; L.a_mn = false; L.B = a.A; L.b_mn = true;
    L.P = M; L.Q = r; L.T = K; L.mode = 0; L.scale = 1.0f; L.out = xa_tmp; L.ldo = r;
    L.dep = lora_dep;
    QL_TRY(launch_lora(L, st));
    xa = xa_tmp;
  }
  {  // G16 = bf16(dY B^T), Gs' = bf16(fl32(s G) 2^(E_m + E)): dY [M][N], B [r][N]
    LoraProblem L{};
    L.A = a.dY; L.a_mn = false; L.B = a.B; L.b_mn = false;
    L.P = M; L.Q = r; L.T = N; L.mode = 0; L.scale = a.scale; L.out = gs8; L.ldo = r;
    L.out2 = g16; L.ldo2 = r;
    L.row_exp = rows;
    L.wmax = wpart;
    L.nwpart = nwpart;
    L.dep = lora_dep;
    QL_TRY(launch_lora(L, st));
  }
  {  // dX = 2^(-E_m - E) (dY_e4m3 W_e4m3 + Gs' A^T)
    GemmProblem g{};
    g.trans = true;
    g.A = reinterpret_cast<const uint16_t *>(dyq); g.M = M; g.Kred = N;
    g.A2 = gs8; g.B2 = a.A; g.r = r;
    g.w = w;
    g.out = a.dX; g.Nout = K;
    g.fp8 = true;
    g.row_exp = rows;
    g.wmax = wpart;
    g.nwpart = nwpart;
    // the main loop reads the dY codes, the weight and max |m_hat|, written
    // by the operand kernel, which completed before the G kernel (a
    // dependent that waits for it at its start) let this GEMM launch
    g.early_main = true;
    QL_TRY(launch_nf4_gemm(g, st));
  }
  // dA = s X^T G16 (X [M][K], G16 [M][r] read MN-major); dB = s XA^T dY, stored
  // transposed; their inputs were complete before the dX GEMM let them start
  LoraProblem LA{};
  LA.A = a.X; LA.a_mn = true; LA.B = g16; LA.b_mn = true;
  LA.P = K; LA.Q = r; LA.T = M; LA.mode = 1; LA.scale = a.scale; LA.out = a.dA; LA.ldo = r;
  LA.dep = kDepExit;
  LoraProblem LB{};
  LB.A = a.dY; LB.a_mn = true; LB.B = xa; LB.b_mn = true;
  LB.P = N; LB.Q = r; LB.T = M; LB.mode = 2; LB.scale = a.scale; LB.out = a.dB; LB.ldo = N;
  LB.dep = kDepExit;
  return launch_lora2(LA, LB, st);
}

int linear_bwd(const LinearArgs &a) {
  const char *fn = "qlora_linear_bwd";
  if (!a.dY || !a.X || !a.A || !a.B || !a.dX || !a.dA || !a.dB)
    return set_error(QL_ERR_INVALID, "%s: null operand", fn);
  if (!al16(a.dY) || !al16(a.X) || !al16(a.A) || !al16(a.B) || !al16(a.dX) || !al16(a.dA) || !al16(a.dB) ||
      (a.XA_in && !al16(a.XA_in)))
    return set_error(QL_ERR_MISALIGNED, "%s: operand not 16-byte aligned", fn);
  const int64_t M = a.M, N = a.W.rows, K = a.W.cols;
  const int r = a.r;
  QL_TRY(check_common(a, fn, bwd_ws(M, N, K, r)));
  cudaStream_t st = a.stream;
  const size_t half = bwd_half(M, N, K, r);
  char *ws = static_cast<char *>(a.ws) + (next_ws_half(st) ? half : 0);
  uint16_t *gs = reinterpret_cast<uint16_t *>(ws);
  uint16_t *xa_tmp = reinterpret_cast<uint16_t *>(ws + up256((size_t)M * r * 2));
  float *part = part_bytes(M, K, N) ? reinterpret_cast<float *>(ws + 2 * up256((size_t)M * r * 2)) : nullptr;

  std::vector<Range> reads = {range(a.dY, (size_t)(M * N * 2)), range(a.X, (size_t)(M * K * 2)),
                             range(a.A, (size_t)(K * r * 2)), range(a.B, (size_t)(r * N * 2))};
  if (a.XA_in) reads.push_back(range(a.XA_in, (size_t)(M * r * 2)));
  weight_ranges(a.W, reads);
  // The first kernel (the XA recompute, or G) and G read only inputs (X and
  // A; dY and B) and write only this call's workspace half: when those are
  // clear of the previous call they read, compute and store alongside it.
  const std::vector<Range> x_a = {range(a.X, (size_t)(M * K * 2)), range(a.A, (size_t)(K * r * 2))};
  const std::vector<Range> dy_b = {range(a.dY, (size_t)(M * N * 2)), range(a.B, (size_t)(r * N * 2))};
  const bool half_clear = writes_clear_of_previous(st, {range(ws, half)});
  const bool g_early = reads_clear_of_previous(st, dy_b);
  const bool x_early = reads_clear_of_previous(st, x_a);
  std::vector<Range> main_reads = {range(a.dY, (size_t)(M * N * 2))};
  weight_ranges(a.W, main_reads);
  const bool gemm_early = reads_clear_of_previous(st, main_reads);
  note_call(st, true,
            {range(a.dX, (size_t)(M * K * 2)), range(a.dA, (size_t)(K * r * 4)), range(a.dB, (size_t)(r * N * 4)),
             range(ws, half)},
            reads);

  const uint16_t *xa = a.XA_in;
  if (!xa) {  // 0. XA = X A
    LoraProblem L{};
    L.A = a.X; L.a_mn = false; L.B = a.A; L.b_mn = true;
    L.P = M; L.Q = r; L.T = K; L.mode = 0; L.scale = 1.0f; L.out = xa_tmp; L.ldo = r;
    L.dep = (x_early && half_clear) ? kDepFree : (x_early ? kDepStores : kDepStart);
    QL_TRY(launch_lora(L, st));
    xa = xa_tmp;
  }
  {  // 1. Gs = bf16(s dY B^T): dY [M][N], B [r][N]
    LoraProblem L{};
    L.A = a.dY; L.a_mn = false; L.B = a.B; L.b_mn = false;
    L.P = M; L.Q = r; L.T = N; L.mode = 0; L.scale = a.scale; L.out = gs; L.ldo = r;
    // the first kernel of the call, or the second after the recompute above
    // (which writes nothing G touches)
    L.dep = (g_early && half_clear && (a.XA_in || x_early)) ? kDepFree
            : (g_early && a.XA_in)                          ? kDepStores
                                                            : kDepStart;
    QL_TRY(launch_lora(L, st));
  }
  {  // 2. dX = dY W_hat + Gs A^T
    GemmProblem g{};
    g.trans = true;
    g.A = a.dY; g.M = M; g.Kred = N;
    g.A2 = gs; g.B2 = a.A; g.r = r;
    g.w = nf4_view(a.W);
    g.out = a.dX; g.Nout = K;
    g.early_main = gemm_early;
    g.part = part;
    QL_TRY(launch_nf4_gemm(g, st));
  }
  // 3. dA = X^T Gs (X [M][K] and Gs [M][r] read MN-major) and 4. dB = s XA^T dY,
  // computed as dB^T = s dY^T XA and stored transposed: one launch.  Their
  // inputs (X, Gs, dY, XA) were all complete before the dX GEMM let them
  // start, so they run alongside it and wait for it only at exit.
  LoraProblem LA{};
  LA.A = a.X; LA.a_mn = true; LA.B = gs; LA.b_mn = true;
  LA.P = K; LA.Q = r; LA.T = M; LA.mode = 1; LA.scale = 1.0f; LA.out = a.dA; LA.ldo = r;
  LA.dep = kDepExit;
  LoraProblem LB{};
  LB.A = a.dY; LB.a_mn = true; LB.B = xa; LB.b_mn = true;
  LB.P = N; LB.Q = r; LB.T = M; LB.mode = 2; LB.scale = a.scale; LB.out = a.dB; LB.ldo = N;
  LB.dep = kDepExit;
  return launch_lora2(LA, LB, st);
}

}  // namespace ql
