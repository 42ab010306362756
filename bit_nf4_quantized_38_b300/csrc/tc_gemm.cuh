// Launch interfaces of the tensor-core GEMM and the LoRA side kernels (internal).
#pragma once
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
};

inline NF4View nf4_view(const ql_nf4_tensor &t) {
  return NF4View{t.packed, t.absmax_code, t.dq_step, t.dq_mean, t.absmax, t.rows, t.cols, t.dq_blocksize != 0};
}

// out[M][Nout] = A[M][Kred] . op(W_hat) + A2[M][rp] . B2[Nout][rp]^T
//   trans = false: op(W_hat) = W_hat^T (Nout = W rows, Kred = W cols)
//   trans = true : op(W_hat) = W_hat   (Nout = W cols, Kred = W rows)
// A2 / B2 are the LoRA operands, zero-padded to rp (a multiple of 64) columns.
struct GemmProblem {
  bool trans;
  const uint16_t *A;
  int64_t M, Kred;
  const uint16_t *A2;
  const uint16_t *B2;
  int r;   // LoRA rank
  int rp;  // r padded to a multiple of 64
  NF4View w;
  uint16_t *out;
  int64_t Nout;
};
int launch_nf4_gemm(const GemmProblem &g, cudaStream_t st);

// ---------------------------------------------------------------- LoRA side
// Partial products over splits of the reduction index t:
//   part[s][p][q] = sum_{t in split s} L(p, t) R(t, q)
// L is stored [p][t] (l_tp = false) or [t][p] (l_tp = true), R is stored
// [t][q] (r_qt = false) or [q][t] (r_qt = true); all bf16 row-major with
// leading dimensions ldl / ldr (elements).
struct SkinnyProblem {
  const uint16_t *L;
  int64_t ldl;
  bool l_tp;
  const uint16_t *R;
  int64_t ldr;
  bool r_qt;
  int64_t P, Q, T;
  int splits;
  float *part;  // [splits][P][Q]
};
int launch_skinny(const SkinnyProblem &s, cudaStream_t st);
int skinny_splits(int64_t P, int64_t Q, int64_t T);

// out_pad[P][qp] = bf16(scale * sum_s part[s]) for q < Q, zero for Q <= q < qp;
// out[P][Q] (optional) = the same values unpadded.
int launch_finalize_bf16(const float *part, int splits, int64_t P, int64_t Q, float scale, uint16_t *out_pad,
                         int qp, uint16_t *out, cudaStream_t st);
// out[P][Q] = scale * sum_s part[s] (fp32)
int launch_finalize_f32(const float *part, int splits, int64_t P, int64_t Q, float scale, float *out,
                        cudaStream_t st);
// Bt[n][j] = bf16(scale * B[j][n]) for j < r, 0 for r <= j < rp   (B is r x N)
int launch_pack_transpose(const uint16_t *B, int r, int64_t N, float scale, uint16_t *Bt, int rp,
                          cudaStream_t st);
// Ap[k][j] = A[k][j] for j < r, 0 for r <= j < rp                  (A is K x r)
int launch_pack_pad(const uint16_t *A, int64_t K, int r, uint16_t *Ap, int rp, cudaStream_t st);

}  // namespace ql
