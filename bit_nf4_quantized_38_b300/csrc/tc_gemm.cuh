// Launch interfaces of the tensor-core GEMM and the LoRA side kernels (internal).
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace ql {

// Device view of an NF4 weight (the arrays of ql_nf4_tensor).
struct NF4View {
  const uint8_t *packed;
  const int8_t *code;
  const float *step;
  const float *mean;
  const float *absmax;
  int64_t rows, cols;
  int dq;
  int qt;   // quant type: the code table the codes index
  int dqt;  // second-level code (QL_DQ_INT8 or QL_DQ_E4M3)
};

inline NF4View nf4_view(const ql_nf4_tensor &t) {
  return NF4View{t.packed, t.absmax_code, t.dq_step, t.dq_mean, t.absmax, t.rows, t.cols, t.dq_blocksize != 0,
                 t.quant_type, t.dq_type};
}

// out[M][Nout] = A[M][Kred] . op(W_hat) + A2[M][r] . op2(B2)
//   trans = false: op(W_hat) = W_hat^T (Nout = W rows, Kred = W cols);
//                  B2 is stored [r][Nout] (the LoRA B), op2 = identity
//   trans = true : op(W_hat) = W_hat   (Nout = W cols, Kred = W rows);
//                  B2 is stored [Nout][r] (the LoRA A), op2 = transpose
// The LoRA operands are read by TMA with zero fill beyond r, in ceil(r/64)
// extra K-steps of 64.
struct GemmProblem {
  bool trans;
  const uint16_t *A;
  int64_t M, Kred;
  const uint16_t *A2;
  const uint16_t *B2;
  int r;   // LoRA rank
  NF4View w;
  uint16_t *out;
  int64_t Nout;
  // A and the weight are written by no kernel that may still be running
  // (the previous library call writes neither): the CTA-pair kernel then
  // starts its main loop before its predecessor completes.
  bool early_main = false;
  // fp32 partial buffer, or null: for the forward form with M <= 128 the
  // few-token kernel's shares (skinny_part_bytes); for the transposed form
  // the single-CTA kernel split over the reduction (M <= 128:
  // gemm_splits(M, Nout, Kred) x M x Nout floats)
  float *part = nullptr;
  // E4M3 main steps (forward form; CTA-pair kernel): A holds the E4M3 codes
  // of X [M][Kred] bytes (row m scaled by 2^row_exp[m]), A2 the LoRA operand
  // already multiplied by 2^(row_exp[m] + E), and the output row m is
  // multiplied by 2^(-row_exp[m] - E); wmax points at nwpart partial maxima
  // of |m_hat| whose largest is the weight's, E = e4m3_weight_exponent(it).
  bool fp8 = false;
  const int *row_exp = nullptr;
  const float *wmax = nullptr;
  int nwpart = 0;
};
int launch_nf4_gemm(const GemmProblem &g, cudaStream_t st);
// Splits over the reduction of a GEMM with M <= 128 tokens (1 otherwise): as
// many as make the tiles x splits about one CTA per SM of a 148-SM GPU, at
// most 16 and at most one per 64-wide K-step.
constexpr int kSplitTarget = 148;
int gemm_splits(int64_t M, int64_t Nout, int64_t Kred);

// 2-D bf16 tensor map [outer][inner] (inner contiguous), box [box_outer][64],
// 128-byte swizzle, zero fill outside the tensor.
int make_tmap(CUtensorMap *tm, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_outer);

// 2-D tensor map over packed NF4 bytes [rows][row_bytes], box [box_rows][128
// bytes] (four 64-element blocks of each row), 128-byte swizzle (16-byte
// piece j of row i stored at j xor (i mod 8)), zero fill.
int make_tmap_packed(CUtensorMap *tm, const uint8_t *ptr, uint64_t row_bytes, uint64_t rows, uint32_t box_rows);

// Few-token forward (16 < M <= 128): the transposed product on the tensor
// cores, weight rows as the MMA M dimension and tokens as N, split over all
// SMs by a stream-K partition of (128-row tile, K-step) units; fp32 partials
// of tiles that several CTAs share are summed in a fixed order by a second
// kernel.  `g.part` holds skinny_part_bytes(...) bytes.  Forward form only.
constexpr int64_t kSkinnyMaxM = 128;
size_t skinny_part_bytes(int64_t M, int64_t Nout, int64_t Kred, int r);
int launch_nf4_skinny(const GemmProblem &g, unsigned long long *span, cudaStream_t st);

// ---------------------------------------------------------------- LoRA side (tensor cores)
// out = scale * (A op . B op^T) over a reduction index t:
//   A operand [P][T] stored K-major (a_mn = false) or as [T][P] (a_mn = true),
//   B operand [Q][T] stored K-major (b_mn = false) or as [T][Q] (b_mn = true);
//   mode 0: bf16 out[p][q] = bf16(scale v), and out2[p][q] = bf16(v) if set;
//   mode 1: fp32 out[p][q] = scale v;  mode 2: fp32 out[q][p] = scale v.
// Q <= 128.
struct LoraProblem {
  const uint16_t *A;
  bool a_mn;
  const uint16_t *B;
  bool b_mn;
  int64_t P, Q, T;
  int mode;
  float scale;
  void *out;
  int64_t ldo;
  uint16_t *out2;
  int64_t ldo2;
  // mode 0 only: multiply row p of `out` by 2^(row_exp[p] + E), E =
  // e4m3_weight_exponent of the largest of the nwpart partial maxima at wmax
  // (after the scale; exact)
  const int *row_exp = nullptr;
  const float *wmax = nullptr;
  int nwpart = 0;
  // Ordering against the previous kernel in the stream (programmatic
  // dependent launch):
  //   kDepStart  wait for it before reading anything (the default);
  //   kDepStores the inputs are not written by any kernel still running: read
  //              and compute alongside it, wait for it before the first store;
  //   kDepExit   the inputs were complete before it let this kernel start and
  //              this kernel writes nothing it reads: run alongside it; one CTA
  //              waits for it before exiting (so completion still implies its
  //              completion);
  //   kDepFree   no kernel still running writes what this kernel reads, or
  //              reads or writes what it writes: run and store alongside it;
  //              one CTA waits for it before exiting, so that this grid still
  //              completes after it (the other CTAs leave their SMs at once).
  int dep = 0;
};
constexpr int kDepStart = 0, kDepStores = 1, kDepExit = 2, kDepFree = 3;
int launch_lora(const LoraProblem &L, cudaStream_t st);
// L0 and L1 in one launch when their operand layouts and width class agree
// (else two launches); both must be independent of each other.
int launch_lora2(const LoraProblem &L0, const LoraProblem &L1, cudaStream_t st);
int lora_splits(int64_t P, int64_t T);

}  // namespace ql
