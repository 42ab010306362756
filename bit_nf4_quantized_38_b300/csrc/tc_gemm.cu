// Dequant-in-the-mainloop tensor-core GEMM for the QLoRA linear (sm_103a).
//
//   forward  : Y  = [X  | XA] . [W_hat | s B^T]^T      (B tile rows = W rows)
//   backward : dX = [dY | sG] . [W_hat ; A^T]           (B tile = W_hat^T)
//
// The frozen weight W_hat is never materialised: converter warps expand the
// packed NF4 nibbles of each 64-element block through a 16-entry bf16 table
// (the block's 16 possible values q[c] * absmax_hat, rounded once) straight
// into the 128-byte-swizzled shared-memory tile the tensor core reads.  The
// LoRA branch rides along as extra K-steps whose operands TMA loads directly.
//
// One CTA computes a 128 x 256 output tile with tcgen05.mma (M=128, N=256,
// K=16 per instruction) into a TMEM accumulator of 256 columns:
//   warp 0      TMA producer (X / dY tiles; LoRA tiles)
//   warp 1      TMEM allocation and the single MMA-issuing thread
//   warps 2-5   converters during the main loop, then the epilogue
// A 4-stage ring of {A 16 KB, B 32 KB} tiles is handed between the roles with
// mbarriers (full: TMA bytes + 128 converter arrivals; empty: MMA commit).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "ptx.cuh"
#include "tc_gemm.cuh"
#include "convert.cuh"
#include "fp8.cuh"

namespace ql {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int CONV_THREADS = 128;
constexpr int TMEM_COLS = 256;
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

struct GemmArgs {
  int M;            // output rows
  int Nout;         // output columns
  int ksteps_main;  // 64-wide reduction steps through the NF4 weight
  int ksteps_lora;  // 64-wide reduction steps through the LoRA operands
  NF4View w;
  uint16_t *out;
  int64_t ldo;
  int *status;
  // Optional span record (null when off): [0] earliest CTA start after the
  // dependency wait, [1] latest CTA end, in %globaltimer nanoseconds.
  unsigned long long *span;
  // The main-loop operands (A and the weight) are not written by any kernel
  // that may still run: start the main loop at once and wait for the
  // previous kernel only before the LoRA steps (pair kernel; see there).
  int early_main;
  float *part;  // single-CTA kernel split over K (gridDim.z > 1): fp32 partials [splits][M][ldo]
  // E4M3 main steps (CTA-pair kernel, kFp8): per X row its exponent E_m; the
  // partial maxima of |m_hat| (the weight's maximum is the largest of the
  // nwpart), from which the converters take the weight's exponent E; the
  // epilogue multiplies row m by 2^(-E_m - E)
  const int *row_exp;
  const float *wmax;
  int nwpart;
  float q[16];
};

// The raw inputs of one 64-element row-block, loaded ahead of their use: no
// value is computed from them at load time, so the loads stay in flight
// until the conversion (a computation -- or a register copy -- would wait for
// them there).
struct RowBlockSrc {
  uint4 p0, p1;
  float s;   // absmax (no double quantization) or the step of the block's group
  int code;  // second-level code byte (double quantization)
  bool valid;
};

__device__ __forceinline__ void load_rowblock(const NF4View &w, int64_t n, int64_t kb, RowBlockSrc &r) {
  r.valid = n < w.rows && kb < w.cols / 64;
  if (r.valid) {
    const uint8_t *src = w.packed + n * (w.cols >> 1) + kb * 32;
    r.p0 = ptx::ldg_nc_v4(src);
    r.p1 = ptx::ldg_nc_v4(src + 16);
    const int64_t b = n * (w.cols >> 6) + kb;
    if (w.dq) {
      r.code = __ldg(w.code + b);
      r.s = __ldg(w.step + (b >> 8));
    } else {
      r.s = __ldg(w.absmax + b);
    }
  }
}

// The block constant m_hat of a loaded row-block (0 outside the weight);
// `mean` = the tensor's mu (double quantization).
__device__ __forceinline__ float rowblock_mhat(const RowBlockSrc &r, const NF4View &w, float mean) {
  if (!r.valid) return 0.0f;
  return w.dq ? __fadd_rn(__fmul_rn(dq_code_value((int8_t)r.code, w.dqt), r.s), mean) : r.s;
}

template <bool kTrans>
__global__ void __launch_bounds__(THREADS, 1)
k_nf4_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
           const __grid_constant__ CUtensorMap tmB2, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 2);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto full = [&](int s) { return ptx::smem_u32(&bars[s]); };
  auto empty = [&](int s) { return ptx::smem_u32(&bars[STAGES + s]); };
  const uint32_t accf = ptx::smem_u32(&bars[2 * STAGES]);
  const uint32_t drainb = ptx::smem_u32(&bars[2 * STAGES + 1]);  // MMAs in flight after an abort

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  // Split over the reduction (few output tiles, M <= 128): CTA z takes main
  // K-steps [kq0, kq0 + nmain) and the last one also the LoRA steps; each
  // stores its fp32 partial tile, and k_splitk_sum adds them in split order.
  const int sp = blockIdx.z, nsplit = gridDim.z;
  const int kq0 = (int)((int64_t)sp * p.ksteps_main / nsplit);
  const int nmain = (int)((int64_t)(sp + 1) * p.ksteps_main / nsplit) - kq0;
  const int nsteps = nmain + (sp == nsplit - 1 ? p.ksteps_lora : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full(s), 1 + CONV_THREADS);
      ptx::mbar_init(empty(s), 1);
    }
    ptx::mbar_init(accf, 1);
    ptx::mbar_init(drainb, 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmA2);
    ptx::prefetch_tmap(&tmB2);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched as a programmatic dependent: the setup above overlaps the
  // previous kernel; its outputs (the LoRA operand) are read only from here on
  ptx::griddep_wait();
  ptx::griddep_launch();
  if (p.span && threadIdx.x == 0) atomicMin(p.span, (unsigned long long)ptx::globaltimer());

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      for (int ks = 0; ks < nsteps; ++ks) {
        const int s = ks % STAGES;
        const uint32_t ph = (ks / STAGES) & 1;
        if (!ptx::mbar_wait(empty(s), ph ^ 1, abort, p.status)) break;
        const uint32_t a_dst = sbase + s * STAGE_BYTES;
        if (ks < nmain) {
          ptx::mbar_arrive_expect_tx(full(s), A_BYTES);
          ptx::tma_load_2d(a_dst, &tmA, full(s), (kq0 + ks) * BK, m0);
        } else {
          const int kl = ks - nmain;
          ptx::mbar_arrive_expect_tx(full(s), A_BYTES + B_BYTES);
          ptx::tma_load_2d(a_dst, &tmA2, full(s), kl * BK, m0);
          if (kTrans) {  // LoRA A stored [k][j]: K-major rows of the output columns
            ptx::tma_load_2d(a_dst + A_BYTES, &tmB2, full(s), kl * BK, n0);
          } else {       // LoRA B stored [j][n]: MN-major, four 64-column atoms
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              ptx::tma_load_2d(a_dst + A_BYTES + 8192 * i, &tmB2, full(s), n0 + 64 * i, kl * BK);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_mn = ptx::idesc_bf16(BM, BN, true);
      constexpr uint32_t idesc_kmaj = ptx::idesc_bf16(BM, BN, false);
      bool ok = true;
      for (int ks = 0; ks < nsteps; ++ks) {
        const int s = ks % STAGES;
        const uint32_t ph = (ks / STAGES) & 1;
        if (!ptx::mbar_wait(full(s), ph, abort, p.status)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t a_addr = sbase + s * STAGE_BYTES;
        const uint32_t b_addr = a_addr + A_BYTES;
        const bool lora = ks >= nmain;
        const uint64_t a_desc = ptx::desc_sw128(a_addr, 16, 1024);
        // K-major B: rows of 128 B, 8-row atoms 1024 B apart.  MN-major B
        // (W_hat^T for dX, the LoRA B for the forward): atoms of 64 output
        // columns x 8 reduction rows; 8 K-atoms (1024 B apart) per 8 KB
        // MN-atom column.
        const bool bmn = kTrans != lora;
        const uint64_t b_desc = bmn ? ptx::desc_sw128(b_addr, 8192, 1024) : ptx::desc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // K advance of 16 elements: +32 B inside the swizzled row (K-major)
          // or two 8-row K-atoms = +2048 B (MN-major)
          const uint64_t ad = a_desc + (uint64_t)(kk * 2);
          const uint64_t bd = b_desc + (uint64_t)(bmn ? kk * 128 : kk * 2);
          ptx::mma_bf16(tmem, ad, bd, bmn ? idesc_mn : idesc_kmaj, (ks > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(empty(s));
      }
      if (ok) {
        ptx::mma_commit(accf);
      } else {  // gave up: let the MMAs already issued finish before TMEM is freed
        ptx::mma_commit(drainb);
        drain_wait(drainb, 0);
      }
    }
  } else {
    // ---------------------------------------------------------------- converters
    const int ct = threadIdx.x - 64;  // 0..127
    float q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = p.q[i];
    // the two row-blocks this thread expands in every stage
    int64_t rb_n[2], rb_kb0[2];
    uint32_t rb_dst[2], rb_swz[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = ct + h * 128;
      if (!kTrans) {
        rb_n[h] = n0 + i;  // weight row = output column
        rb_kb0[h] = 0;     // + ks
        rb_dst[h] = (uint32_t)i * 128u;
        rb_swz[h] = (uint32_t)(i & 7);
      } else {
        const int nl = i & 63, kbl = i >> 6;
        rb_n[h] = nl;                  // + 64 ks: weight row = reduction index
        rb_kb0[h] = (n0 >> 6) + kbl;   // weight column block = output columns / 64
        rb_dst[h] = (uint32_t)((kbl * 8 + (nl >> 3)) * 1024 + (nl & 7) * 128);
        rb_swz[h] = (uint32_t)(nl & 7);
      }
    }
    const float mean = p.w.dq ? __ldg(p.w.mean) : 0.0f;
    auto fetch = [&](int ks, RowBlockSrc (&r)[2]) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!kTrans) load_rowblock(p.w, rb_n[h], rb_kb0[h] + ks, r[h]);
        else load_rowblock(p.w, rb_n[h] + (int64_t)ks * 64, rb_kb0[h], r[h]);
      }
    };
    auto body = [&](int ks, RowBlockSrc (&cur)[2]) -> bool {
      const int s = ks % STAGES;
      const uint32_t ph = (ks / STAGES) & 1;
      if (!ptx::mbar_wait(empty(s), ph ^ 1, abort, p.status)) return false;
      if (ks < nmain) {
        const uint32_t b_addr = sbase + s * STAGE_BYTES + A_BYTES;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (cur[h].valid)
            convert_rowblock(cur[h].p0, cur[h].p1, rowblock_mhat(cur[h], p.w, mean), q, b_addr + rb_dst[h], rb_swz[h]);
          else
            zero_row(b_addr + rb_dst[h]);
        }
        ptx::fence_proxy_async_smem();
      }
      ptx::mbar_arrive(full(s));
      return true;
    };
    // Two register sets taking steps in turn, each loaded two steps ahead of
    // its use (no copies between them).
    RowBlockSrc sa[2], sb[2];
    if (nmain > 0) fetch(kq0, sa);
    if (nmain > 1) fetch(kq0 + 1, sb);
    for (int ks = 0; ks < nsteps; ks += 2) {
      if (!body(ks, sa)) break;
      if (ks + 2 < nmain) fetch(kq0 + ks + 2, sa);
      if (ks + 1 >= nsteps || !body(ks + 1, sb)) break;
      if (ks + 3 < nmain) fetch(kq0 + ks + 3, sb);
    }
    // ---------------------------------------------------------------- epilogue
    if (!*abort && ptx::mbar_wait(accf, 0, abort, p.status)) {
      ptx::tc_fence_after();
      const int qd = warp & 3;  // TMEM lane quarter this warp may access
      const int row = m0 + qd * 32 + lane;
      uint16_t *orow = p.out + (int64_t)row * p.ldo;
      float *prow = nsplit > 1 ? p.part + ((int64_t)sp * p.M + row) * p.ldo : nullptr;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(c * 32), r);
        ptx::tmem_wait_ld();
        if (row < p.M) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int col = n0 + c * 32 + j * 8;
            if (col + 8 <= p.Nout) {
              if (prow) {  // fp32 partial of this split
                float4 *dst = reinterpret_cast<float4 *>(prow + col);
                dst[0] = make_float4(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1]),
                                     __uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3]));
                dst[1] = make_float4(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5]),
                                     __uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]));
              } else {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1]));
                v.y = pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3]));
                v.z = pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5]));
                v.w = pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]));
                *reinterpret_cast<uint4 *>(orow + col) = v;
              }
            }
          }
        }
      }
    }
  }
  // after an abort, copies already issued into the ring are given time to land
  if (*abort && threadIdx.x == 0) settle();
  ptx::tc_fence_before();
  __syncthreads();
  if (p.span && threadIdx.x == 0) atomicMax(p.span + 1, (unsigned long long)ptx::globaltimer());
  if (warp == 1) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// out = bf16(sum over the splits of part[s]) in split order (fixed, so the
// result is deterministic); 8 outputs per thread.  A programmatic dependent
// of the split GEMM: waits for it before reading.
__global__ void __launch_bounds__(256) k_splitk_sum(const float *__restrict__ part, int nsplit, int64_t n8,
                                                    uint16_t *__restrict__ out) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    float4 a = __ldcg(reinterpret_cast<const float4 *>(part) + 2 * i);
    float4 b = __ldcg(reinterpret_cast<const float4 *>(part) + 2 * i + 1);
    for (int s = 1; s < nsplit; ++s) {
      const float4 *ps = reinterpret_cast<const float4 *>(part + (int64_t)s * n8 * 8) + 2 * i;
      const float4 x = __ldcg(ps), y = __ldcg(ps + 1);
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
      b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
    }
    reinterpret_cast<uint4 *>(out)[i] =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

// ---------------------------------------------------------------------------- CTA-pair kernel
//
// A cluster of two CTAs on two SMs computes a (NACC x 256) x 256 output tile
// with pair MMAs (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16): the
// even CTA issues them; each CTA holds 128 A rows per accumulator and HALF of
// the 256 B rows, and the tensor cores of the pair exchange the B halves.  So
// every dequantized weight element is converted once and consumed by
// NACC x 256 token rows, and each SM reads only its own A and B halves from
// shared memory.  With NACC = 2 each CTA keeps two accumulators (2 x 256 TMEM
// columns).
//   warp 0     TMA producer: this CTA's A tiles (and LoRA B half); completion
//              is counted on the even CTA's `full` barrier
//   warp 1     TMEM allocation; in the even CTA, the MMA-issuing thread
//   warps 2-9  two converter groups of 4 warps taking alternate stages (each
//              has two MMA steps of time to load and expand its row-blocks),
//              then the epilogue (group g drains accumulator g)
namespace pairk {
constexpr int BMH = 128;  // A rows per CTA per accumulator
constexpr int BNH = 128;  // B rows per CTA (half of N = 256)
constexpr int BK = 64, STAGES = 4, THREADS = 320, GROUP_WARPS = 4;
template <int NACC>
struct Geo {
  static constexpr int A_ONE = BMH * BK * 2;  // 16 KB
  static constexpr int A_BYTES = NACC * A_ONE;
  static constexpr int B_BYTES = BNH * BK * 2;  // 16 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = NACC * 256;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 256;
};
}  // namespace pairk

// With kFp8 the main steps are E4M3 x E4M3 products on kind::f8f6f4: A = X
// (forward) or dY (dX) quantized per row to E4M3 (the same 128-byte smem rows
// now hold 128 reduction elements, so a step covers K = 128 with the same four
// MMA instructions of K = 32), B = the weight converted to E4M3 with a
// power-of-two scale 2^E; the LoRA steps stay bf16 into the same accumulator
// with their A operand (XAs, or s G) already multiplied by 2^(E_m + E), and
// the epilogue multiplies each row by 2^(-E_m - E) (exact).  In the dX form
// each converter thread writes one 128-byte row: the E4M3 values of weight
// row n (a reduction index) over this CTA's 128 output columns, which the
// tensor core reads as an MN-major B operand (one 128-column atom, 8-row
// groups 1 KB apart, 32 reduction rows = 4 KB per instruction).
template <bool kTrans, int NACC, bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pairk::THREADS, 1)
k_nf4_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                const __grid_constant__ CUtensorMap tmB2, const GemmArgs p) {
  using G = pairk::Geo<NACC>;
  constexpr int PSTAGES = pairk::STAGES, PBK = pairk::BK, BMH = pairk::BMH, BNH = pairk::BNH,
                GROUP_WARPS = pairk::GROUP_WARPS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + PSTAGES * G::STAGE_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * PSTAGES + 2);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *dep_seen = reinterpret_cast<volatile int *>(tmem_slot + 2);  // gate CTA: predecessor done
  float *wmax_s = reinterpret_cast<float *>(tmem_slot + 3);                  // E4M3: max |m_hat|
  auto full = [&](int s) { return ptx::smem_u32(&bars[s]); };
  auto empty = [&](int s) { return ptx::smem_u32(&bars[PSTAGES + s]); };
  const uint32_t accf = ptx::smem_u32(&bars[2 * PSTAGES]);
  const uint32_t drainb = ptx::smem_u32(&bars[2 * PSTAGES + 1]);  // MMAs in flight after an abort

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = ptx::cluster_ctarank();
  const int n0 = (blockIdx.x >> 1) * 256;          // pair's first output column
  const int mrow0 = blockIdx.y * (NACC * 256);     // pair's first output row
  const int nsteps = p.ksteps_main + p.ksteps_lora;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      ptx::mbar_init(full(s), 2 + 2 * GROUP_WARPS);  // 2 producers + one group's warps in each CTA
      ptx::mbar_init(empty(s), 1);
    }
    ptx::mbar_init(accf, 1);
    ptx::mbar_init(drainb, 1);
    *abort = 0;
    *dep_seen = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmA2);
    ptx::prefetch_tmap(&tmB2);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), G::TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  if constexpr (kFp8) {
    // max |m_hat| from the operand kernel's partials: that kernel completed
    // before this grid could launch (its dependent, the LoRA kernel, waits
    // for it before letting this GEMM start), so they may be read here
    if (warp == 2) {
      const float m = wmax_of_warp(p.wmax, p.nwpart);
      if (lane == 0) *wmax_s = m;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the previous kernel, whose
  // output (the LoRA operand) is read only after griddep_wait.
  //  - Default: wait here, then let dependents launch.
  //  - early_main: the main loop reads only operands no running kernel
  //    writes, so it starts at once; the producer waits before the first LoRA
  //    step, and the epilogue (after the last MMA) follows that wait.  This
  //    GEMM's main loop thus runs in the SMs the previous GEMM's last wave
  //    leaves idle.  Dependents may launch once every CTA has started, except
  //    that the gate CTA (block 0, 0) lets them launch only after one of its
  //    threads has seen the previous kernel complete: so, as with the
  //    default, no kernel of the next call starts before every kernel older
  //    than this one's predecessor has completed.  (Each thread of the gate
  //    CTA triggers only after that wait: idle lanes wait themselves, the
  //    working roles trigger once they see `dep_seen`.)
  const bool gate = p.early_main && blockIdx.x == 0 && blockIdx.y == 0;
  bool triggered = false;
  if (!p.early_main) {
    ptx::griddep_wait();
    ptx::griddep_launch();
    triggered = true;
  } else if (!gate) {
    ptx::griddep_launch();
    triggered = true;
  } else if ((warp == 0 && lane != 0) || (warp == 1 && lane != 0)) {
    ptx::griddep_wait();
    if (warp == 0 && lane == 1) *dep_seen = 1;
    ptx::griddep_launch();
    triggered = true;
  }
  // gate CTA, working threads: trigger once the predecessor is known complete
  auto poll_trigger = [&]() {
    if (!triggered && *dep_seen) {
      ptx::griddep_launch();
      triggered = true;
    }
  };
  if (p.span && threadIdx.x == 0) atomicMin(p.span, (unsigned long long)ptx::globaltimer());

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      bool waited = !p.early_main;
      for (int ks = 0; ks < nsteps; ++ks) {
        const int s = ks % PSTAGES;
        const uint32_t ph = (ks / PSTAGES) & 1;
        if (!ptx::mbar_wait_cluster(empty(s), ph ^ 1, abort, p.status)) break;
        const uint32_t a_dst = sbase + s * G::STAGE_BYTES;
        const uint32_t lead_full = ptx::mapa(full(s), 0);
        const bool lora = ks >= p.ksteps_main;
        if (lora && !waited) {  // early_main: the LoRA operand is the previous kernel's output
          ptx::griddep_wait();
          waited = true;
          ptx::griddep_launch();
          triggered = true;
        }
        poll_trigger();
        ptx::mbar_arrive_expect_tx_cluster(lead_full, G::A_BYTES + (lora ? G::B_BYTES : 0));
        // x in elements of the operand: bf16 (64 per step) or E4M3 bytes (128)
        const int x = lora ? (ks - p.ksteps_main) * PBK : ks * (kFp8 ? 2 * PBK : PBK);
#pragma unroll
        for (int a = 0; a < NACC; ++a)
          ptx::tma_load_2d_pair(a_dst + a * G::A_ONE, lora ? &tmA2 : &tmA, lead_full, x,
                                mrow0 + a * 256 + (int)crank * BMH);
        if (lora) {
          if (kTrans) {  // LoRA A stored [k][j]: K-major rows of this CTA's output columns
            ptx::tma_load_2d_pair(a_dst + G::A_BYTES, &tmB2, lead_full, x, n0 + (int)crank * BNH);
          } else {       // LoRA B stored [j][n]: MN-major, two 64-column atoms
            ptx::tma_load_2d_pair(a_dst + G::A_BYTES, &tmB2, lead_full, n0 + (int)crank * BNH, x);
            ptx::tma_load_2d_pair(a_dst + G::A_BYTES + 8192, &tmB2, lead_full, n0 + (int)crank * BNH + 64, x);
          }
        }
      }
      // a CTA that gave up before its LoRA steps still completes after its predecessor
      if (!waited) ptx::griddep_wait();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA (even CTA)
    if (lane == 0 && crank == 0) {
      constexpr uint32_t idesc_mn = ptx::idesc_bf16(256, 256, true);
      constexpr uint32_t idesc_kmaj = ptx::idesc_bf16(256, 256, false);
      bool ok = true;
      for (int ks = 0; ks < nsteps; ++ks) {
        const int s = ks % PSTAGES;
        const uint32_t ph = (ks / PSTAGES) & 1;
        if (!ptx::mbar_wait_cluster(full(s), ph, abort, p.status)) { ok = false; break; }
        ptx::tc_fence_after();
        poll_trigger();
        const uint32_t a_addr = sbase + s * G::STAGE_BYTES;
        const uint32_t b_addr = a_addr + G::A_BYTES;
        const bool bmn = kTrans != (ks >= p.ksteps_main);
        // K-major B half: 128 rows of 128 B.  MN-major B half (W_hat^T, or
        // the LoRA B in the forward): 2 MN-atoms of 64 output columns, 8 KB
        // apart, each 8 K-atoms of 8 reduction rows, 1 KB apart.
        const bool e4m3 = kFp8 && ks < p.ksteps_main;
        // (an E4M3 MN-major half is one 128-column atom: no second atom, LBO 0)
        const uint64_t b_desc = bmn ? ptx::desc_sw128(b_addr, e4m3 ? 0 : 8192, 1024) : ptx::desc_sw128(b_addr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < PBK / 16; ++kk) {
          // K-major: 32 bytes per instruction either way (16 bf16 or 32 E4M3
          // elements); MN-major: 16 bf16 reduction rows (2 KB) or 32 E4M3
          // rows (4 KB)
          const uint64_t bd = b_desc + (uint64_t)(bmn ? kk * (e4m3 ? 256 : 128) : kk * 2);
#pragma unroll
          for (int a = 0; a < NACC; ++a) {
            const uint64_t ad = ptx::desc_sw128(a_addr + a * G::A_ONE, 16, 1024) + (uint64_t)(kk * 2);
            if (e4m3)
              ptx::mma_e4m3_pair(tmem + a * 256, ad, bd, ptx::idesc_e4m3(256, 256, bmn),
                                 (ks > 0 || kk > 0) ? 1u : 0u);
            else
              ptx::mma_bf16_pair(tmem + a * 256, ad, bd, bmn ? idesc_mn : idesc_kmaj,
                                 (ks > 0 || kk > 0) ? 1u : 0u);
          }
        }
        ptx::mma_commit_pair(empty(s));
      }
      if (ok) {
        ptx::mma_commit_pair(accf);
      } else {  // gave up: let the MMAs already issued finish before TMEM is freed
        ptx::mma_commit_pair(drainb);
        drain_wait(drainb, 0);
      }
    }
  } else {
    // ---------------------------------------------------------------- converters
    const int grp = (warp - 2) / GROUP_WARPS;              // stages ks = grp, grp + 2, ...
    const int ct = ((warp - 2) % GROUP_WARPS) * 32 + lane;  // this thread's row-block, 0..127
    float q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = p.q[i];
    int64_t rb_n, rb_kb0;
    uint32_t rb_dst, rb_swz;
    if (!kTrans) {
      rb_n = n0 + (int)crank * BNH + ct;  // weight row = output column
      rb_kb0 = 0;                         // + ks
      rb_dst = (uint32_t)ct * 128u;
      rb_swz = (uint32_t)(ct & 7);
    } else if (kFp8) {
      rb_n = ct;                                          // + 128 ks: the reduction row
      rb_kb0 = (n0 + (int)crank * BNH) >> 6;              // + h: output columns / 64
      rb_dst = (uint32_t)ct * 128u;
      rb_swz = (uint32_t)(ct & 7);
    } else {
      const int nl = ct & 63, kbl = ct >> 6;
      rb_n = nl;                                          // + 64 ks
      rb_kb0 = ((n0 + (int)crank * BNH) >> 6) + kbl;      // output columns / 64
      rb_dst = (uint32_t)((kbl * 8 + (nl >> 3)) * 1024 + (nl & 7) * 128);
      rb_swz = (uint32_t)(nl & 7);
    }
    // E4M3: the weight's power-of-two scale 2^E (the largest with
    // max |m_hat| 2^E <= 448), applied exactly to every block constant
    const float s2e = kFp8 ? e4m3_weight_scale(*wmax_s) : 1.0f;
    constexpr int RB = kFp8 ? 2 : 1;  // row-blocks per thread per step (K = 128 per E4M3 step)
    const float mean = p.w.dq ? __ldg(p.w.mean) : 0.0f;
    auto fetch = [&](int ks, RowBlockSrc (&r)[RB]) {
#pragma unroll
      for (int h = 0; h < RB; ++h) {
        if (kTrans) load_rowblock(p.w, rb_n + (int64_t)ks * 64 * RB, rb_kb0 + h, r[h]);
        else load_rowblock(p.w, rb_n, rb_kb0 + RB * ks + h, r[h]);
      }
    };
    auto body = [&](int ks, RowBlockSrc (&cur)[RB]) -> bool {
      const int s = ks % PSTAGES;
      const uint32_t ph = (ks / PSTAGES) & 1;
      poll_trigger();
      if (!ptx::mbar_wait_cluster(empty(s), ph ^ 1, abort, p.status)) return false;
      if (ks < p.ksteps_main) {
        const uint32_t b_addr = sbase + s * G::STAGE_BYTES + G::A_BYTES;
        if (kFp8) {
#pragma unroll
          for (int h = 0; h < RB; ++h)  // an invalid row-block has zero codes and constant: zero bytes
            // forward: the reduction runs along the row, and the X codes
            // carry the same pair order, so the pairs may stay swapped; dX:
            // the row runs along the output columns, so in order
            convert_rowblock_e4m3<kTrans>(cur[h].p0, cur[h].p1, __fmul_rn(rowblock_mhat(cur[h], p.w, mean), s2e), q,
                                  b_addr + rb_dst, h, rb_swz);
        } else {
          if (cur[0].valid) convert_rowblock(cur[0].p0, cur[0].p1, rowblock_mhat(cur[0], p.w, mean), q, b_addr + rb_dst, rb_swz);
          else zero_row(b_addr + rb_dst);
        }
        ptx::fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(full(s), 0));
      return true;
    };
    // This group takes stages grp, grp + 2, ...: register sets take them in
    // turn, each loaded as many of the group's stages ahead of its use as
    // there are sets (no copies between them, so the loads stay in flight
    // that long): two for bf16, three for E4M3, whose steps convert twice the
    // elements (a third bf16 set measured no faster on the power-capped 33B
    // step).
    if constexpr (kFp8) {
      RowBlockSrc sa[RB], sb[RB], sc[RB];
      if (grp < p.ksteps_main) fetch(grp, sa);
      if (grp + 2 < p.ksteps_main) fetch(grp + 2, sb);
      if (grp + 4 < p.ksteps_main) fetch(grp + 4, sc);
      for (int ks = grp; ks < nsteps; ks += 6) {
        if (!body(ks, sa)) break;
        if (ks + 6 < p.ksteps_main) fetch(ks + 6, sa);
        if (ks + 2 >= nsteps || !body(ks + 2, sb)) break;
        if (ks + 8 < p.ksteps_main) fetch(ks + 8, sb);
        if (ks + 4 >= nsteps || !body(ks + 4, sc)) break;
        if (ks + 10 < p.ksteps_main) fetch(ks + 10, sc);
      }
    } else {
      RowBlockSrc sa[RB], sb[RB];
      if (grp < p.ksteps_main) fetch(grp, sa);
      if (grp + 2 < p.ksteps_main) fetch(grp + 2, sb);
      for (int ks = grp; ks < nsteps; ks += 4) {
        if (!body(ks, sa)) break;
        if (ks + 4 < p.ksteps_main) fetch(ks + 4, sa);
        if (ks + 2 >= nsteps || !body(ks + 2, sb)) break;
        if (ks + 6 < p.ksteps_main) fetch(ks + 6, sb);
      }
    }
    // ---------------------------------------------------------------- epilogue
    if (!*abort && ptx::mbar_wait_cluster(accf, 0, abort, p.status)) {
      ptx::tc_fence_after();
      const int qd = warp & 3;  // TMEM lane quarter this warp may access
      const int acc = NACC == 2 ? grp : 0;
      const int c_begin = NACC == 2 ? 0 : grp * 4, c_end = NACC == 2 ? 8 : grp * 4 + 4;
      const int row = mrow0 + acc * 256 + (int)crank * BMH + qd * 32 + lane;
      uint16_t *orow = p.out + (int64_t)row * p.ldo;
      const float rs = kFp8 && row < p.M ? e4m3_row_factor(__ldg(p.row_exp + row), *wmax_s) : 1.0f;
#pragma unroll 1
      for (int c = c_begin; c < c_end; ++c) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * 256 + c * 32), r);
        ptx::tmem_wait_ld();
        if (row < p.M) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int col = n0 + c * 32 + j * 8;
            if (col + 8 <= p.Nout) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = kFp8 ? __fmul_rn(__uint_as_float(r[8 * j + e]), rs)
                                                      : __uint_as_float(r[8 * j + e]);
              uint4 v;
              v.x = pack_bf16x2(f[0], f[1]);
              v.y = pack_bf16x2(f[2], f[3]);
              v.z = pack_bf16x2(f[4], f[5]);
              v.w = pack_bf16x2(f[6], f[7]);
              *reinterpret_cast<uint4 *>(orow + col) = v;
            }
          }
        }
      }
    }
  }
  // gate CTA: a thread that has not triggered yet exits only after the predecessor
  if (!triggered) ptx::griddep_wait();
  // after an abort, copies already issued into the ring are given time to land
  if (*abort && threadIdx.x == 0) settle();
  ptx::tc_fence_before();
  __syncthreads();
  if (p.span && threadIdx.x == 0) atomicMax(p.span + 1, (unsigned long long)ptx::globaltimer());
  ptx::cluster_sync();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem, G::TMEM_COLS);
}

// ---------------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

int gemm_splits(int64_t M, int64_t Nout, int64_t Kred) {
  if (M > 128) return 1;
  const int64_t tiles = (Nout + BN - 1) / BN, ks = (Kred + BK - 1) / BK;
  int64_t s = (kSplitTarget + tiles - 1) / tiles;
  s = std::min<int64_t>(s, 16);
  s = std::min<int64_t>(s, ks);
  return (int)std::max<int64_t>(s, 1);
}

int make_tmap(CUtensorMap *tm, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return QL_OK;
}

int make_tmap_packed(CUtensorMap *tm, const uint8_t *ptr, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(QL_ERR_CUDA, "cuTensorMapEncodeTiled (packed) failed (%d)", (int)r);
  return QL_OK;
}

namespace {

template <bool kTrans, int NACC, bool kFp8>
int launch_pair(const GemmProblem &g, unsigned long long *span, cudaStream_t st) {
  using Gm = pairk::Geo<NACC>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    int rc = check_cuda(cudaFuncSetAttribute(k_nf4_gemm_pair<kTrans, NACC, kFp8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Gm::SMEM),
                        "tensor-core pair GEMM: shared-memory attribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  CUtensorMap tA, tA2, tB2;
  // E4M3 A: the per-row codes [M][K] bytes, 128-byte rows of the box
  int rc = kFp8 ? make_tmap_packed(&tA, reinterpret_cast<const uint8_t *>(g.A), (uint64_t)g.Kred, (uint64_t)g.M,
                                   pairk::BMH)
                : make_tmap(&tA, g.A, (uint64_t)g.Kred, (uint64_t)g.M, pairk::BMH);
  if (!rc) rc = make_tmap(&tA2, g.A2, (uint64_t)g.r, (uint64_t)g.M, pairk::BMH);
  if (!rc)
    rc = kTrans ? make_tmap(&tB2, g.B2, (uint64_t)g.r, (uint64_t)g.Nout, pairk::BNH)
                : make_tmap(&tB2, g.B2, (uint64_t)g.Nout, (uint64_t)g.r, 64);
  if (rc) return rc;
  GemmArgs a{};
  a.M = (int)g.M;
  a.Nout = (int)g.Nout;
  a.ksteps_main = (int)((g.Kred + (kFp8 ? 2 * BK : BK) - 1) / (kFp8 ? 2 * BK : BK));
  a.ksteps_lora = (g.r + BK - 1) / BK;
  a.w = g.w;
  a.out = g.out;
  a.ldo = g.Nout;
  a.status = device_status_ptr();
  a.span = span;
  a.early_main = g.early_main ? 1 : 0;
  a.row_exp = g.row_exp;
  a.wmax = g.wmax;
  a.nwpart = g.nwpart;
  const Codebook &cb = codebook(g.w.qt);
  for (int i = 0; i < 16; ++i) a.q[i] = cb.q[i];
  dim3 grid((unsigned)(2 * ((g.Nout + 255) / 256)), (unsigned)((g.M + NACC * 256 - 1) / (NACC * 256)));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(pairk::THREADS);
  cfg.dynamicSmemBytes = Gm::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_nf4_gemm_pair<kTrans, NACC, kFp8>, tA, tA2, tB2, a);
  count_launch();
  return check_cuda(e, "tensor-core pair GEMM launch");
}

template <bool kTrans>
int launch(const GemmProblem &g, unsigned long long *span, cudaStream_t st) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    int rc = check_cuda(cudaFuncSetAttribute(k_nf4_gemm<kTrans>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES),
                        "tensor-core GEMM: shared-memory attribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  CUtensorMap tA, tA2, tB2;
  int rc = make_tmap(&tA, g.A, (uint64_t)g.Kred, (uint64_t)g.M, BM);
  if (!rc) rc = make_tmap(&tA2, g.A2, (uint64_t)g.r, (uint64_t)g.M, BM);
  if (!rc)
    rc = kTrans ? make_tmap(&tB2, g.B2, (uint64_t)g.r, (uint64_t)g.Nout, BN)
                : make_tmap(&tB2, g.B2, (uint64_t)g.Nout, (uint64_t)g.r, 64);
  if (rc) return rc;
  GemmArgs a{};
  a.M = (int)g.M;
  a.Nout = (int)g.Nout;
  a.ksteps_main = (int)((g.Kred + BK - 1) / BK);
  a.ksteps_lora = (g.r + BK - 1) / BK;
  a.w = g.w;
  a.out = g.out;
  a.ldo = g.Nout;
  a.status = device_status_ptr();
  a.span = span;
  const Codebook &cb = codebook(g.w.qt);
  for (int i = 0; i < 16; ++i) a.q[i] = cb.q[i];
  const int nsplit = g.part ? gemm_splits(g.M, g.Nout, g.Kred) : 1;
  a.part = nsplit > 1 ? g.part : nullptr;
  dim3 grid((unsigned)((g.Nout + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM), (unsigned)nsplit);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_nf4_gemm<kTrans>, tA, tA2, tB2, a);
  count_launch();
  rc = check_cuda(e, "tensor-core GEMM launch");
  if (rc || nsplit == 1) return rc;
  const int64_t n8 = g.M * g.Nout / 8;
  cudaLaunchConfig_t sc{};
  sc.gridDim = dim3((unsigned)std::min<int64_t>((n8 + 255) / 256, 148 * 8));
  sc.blockDim = dim3(256);
  sc.stream = st;
  sc.attrs = attr;
  sc.numAttrs = 1;
  e = cudaLaunchKernelEx(&sc, k_splitk_sum, (const float *)g.part, nsplit, n8, g.out);
  count_launch();
  return check_cuda(e, "split-K sum launch");
}

struct Timing {
  bool on = false;
  int capacity = 0, used = 0;
  std::vector<cudaEvent_t> ev;
  std::vector<double> flops;
};
thread_local Timing g_timing;

// Span records of the GEMM launches (ql_spans_start / ql_spans_stop).
struct Spans {
  bool on = false;
  unsigned long long *buf = nullptr;
  int capacity = 0, used = 0;
  double flops = 0.0;
};
thread_local Spans g_spans;

}  // namespace

int launch_nf4_gemm(const GemmProblem &g, cudaStream_t st) {
  Timing &t = g_timing;
  const bool timed = t.on && t.used < t.capacity;
  if (timed) cudaEventRecord(t.ev[2 * t.used], st);
  Spans &sp = g_spans;
  unsigned long long *span = (sp.on && sp.used < sp.capacity) ? sp.buf + 2 * sp.used : nullptr;
  int rc;
  if (g.fp8) {
    if (!g.row_exp || !g.wmax || g.nwpart < 1) return set_error(QL_ERR_INVALID, "E4M3 GEMM: scales missing");
    if (g.trans)
      rc = g.M <= 256 ? launch_pair<true, 1, true>(g, span, st) : launch_pair<true, 2, true>(g, span, st);
    else
      rc = g.M <= 256 ? launch_pair<false, 1, true>(g, span, st) : launch_pair<false, 2, true>(g, span, st);
  } else if (!g.trans && g.M <= kSkinnyMaxM && g.part) {
    rc = launch_nf4_skinny(g, span, st);
  } else if (g.M <= 128) {
    rc = g.trans ? launch<true>(g, span, st) : launch<false>(g, span, st);
  } else if (g.M <= 256) {
    rc = g.trans ? launch_pair<true, 1, false>(g, span, st) : launch_pair<false, 1, false>(g, span, st);
  } else {
    rc = g.trans ? launch_pair<true, 2, false>(g, span, st) : launch_pair<false, 2, false>(g, span, st);
  }
  const double flops = 2.0 * (double)g.M * (double)g.Nout * (double)(g.Kred + g.r);
  if (timed && rc == QL_OK) {
    cudaEventRecord(t.ev[2 * t.used + 1], st);
    t.flops[t.used] = flops;
    ++t.used;
  }
  if (span && rc == QL_OK) {
    ++sp.used;
    sp.flops += flops;
  }
  return rc;
}

}  // namespace ql

extern "C" int ql_timing_start(int capacity) {
  using namespace ql;
  Timing &t = g_timing;
  if (t.on) return set_error(QL_ERR_INVALID, "ql_timing_start: timing already on");
  if (capacity <= 0) return set_error(QL_ERR_INVALID, "ql_timing_start: capacity %d", capacity);
  t.ev.assign(2 * (size_t)capacity, nullptr);
  t.flops.assign((size_t)capacity, 0.0);
  for (auto &e : t.ev) {
    int rc = check_cuda(cudaEventCreate(&e), "ql_timing_start: event");
    if (rc) return rc;
  }
  t.capacity = capacity;
  t.used = 0;
  t.on = true;
  return QL_OK;
}

extern "C" int ql_timing_stop(float *total_ms, int *launches, double *flops) {
  using namespace ql;
  Timing &t = g_timing;
  if (!t.on) return set_error(QL_ERR_INVALID, "ql_timing_stop: timing is off");
  int rc = QL_OK;
  float sum = 0.0f;
  double fl = 0.0;
  for (int i = 0; i < t.used && !rc; ++i) {
    float ms = 0.0f;
    rc = check_cuda(cudaEventSynchronize(t.ev[2 * i + 1]), "ql_timing_stop: synchronize");
    if (!rc) rc = check_cuda(cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]), "ql_timing_stop: elapsed");
    sum += ms;
    fl += t.flops[i];
  }
  for (auto &e : t.ev)
    if (e) cudaEventDestroy(e);
  if (total_ms) *total_ms = sum;
  if (launches) *launches = t.used;
  if (flops) *flops = fl;
  t = Timing{};
  return rc;
}

extern "C" int ql_spans_start(uint64_t *device_buffer, int capacity) {
  using namespace ql;
  Spans &sp = g_spans;
  if (sp.on) return set_error(QL_ERR_INVALID, "ql_spans_start: span recording already on");
  if (!device_buffer || capacity <= 0)
    return set_error(QL_ERR_INVALID, "ql_spans_start: null buffer or capacity %d", capacity);
  if (reinterpret_cast<uintptr_t>(device_buffer) & 7)
    return set_error(QL_ERR_MISALIGNED, "ql_spans_start: buffer not 8-byte aligned");
  sp = Spans{};
  sp.on = true;
  sp.buf = reinterpret_cast<unsigned long long *>(device_buffer);
  sp.capacity = capacity;
  return QL_OK;
}

extern "C" int ql_spans_stop(int *launches, double *flops) {
  using namespace ql;
  Spans &sp = g_spans;
  if (!sp.on) return set_error(QL_ERR_INVALID, "ql_spans_stop: span recording is off");
  if (launches) *launches = sp.used;
  if (flops) *flops = sp.flops;
  sp = Spans{};
  return QL_OK;
}
