// LoRA side products of the QLoRA linear on the tensor cores (LoRA tutorial:
// dW = W_A W_B with rank r; QLoRA abstract: gradients flow into the adapters
// only):
//   XA  = X A             (P = M tokens, Q = r, reduce over K)
//   Gs  = s dY B^T        (P = M,        Q = r, reduce over N)
//   dA  = X^T Gs          (P = K,        Q = r, reduce over M)
//   dB^T = s dY^T XA      (P = N,        Q = r, reduce over M; stored as dB)
// Each has a small side (r <= 128) and a long reduction.  One tcgen05 kernel
// serves all four: a 128 x NQ tile (NQ = 64 or 128, r zero-padded by TMA) per
// CTA, A and B operands loaded by TMA straight from their stored layout
// (K-major or MN-major, 128-byte swizzle, zero fill outside the tensor), the
// reduction split across a cluster of CTAs whose fp32 tiles are summed in
// fixed CTA order through distributed shared memory, and the scale and
// conversion fused into that reduction.  No partial buffer, no extra launch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "tc_gemm.cuh"
#include "fp8.cuh"

namespace ql {
namespace {

constexpr int LBP = 128, LBT = 64, LSTAGES = 4, LTHREADS = 128;

struct LoraTcArgs {
  int64_t P, Q, T;
  int mode;  // 0: bf16 out[p][q] = bf16(scale v) (+ out2 = bf16(v)); 1: fp32 out[p][q]; 2: fp32 out[q][p]
  float scale;
  void *out;
  int64_t ldo;
  uint16_t *out2;
  int64_t ldo2;
  const int *row_exp;  // mode 0: out[p][q] = bf16(fl32(scale v) 2^(row_exp[p] + E)) when set
  const float *wmax;   // E = e4m3_weight_exponent(the largest of wmax[0, nwpart))
  int nwpart;
  int dep;  // kDepStart, kDepStores or kDepExit (see LoraProblem)
  int *status;
};

template <int NQ>
struct LGeo {
  static constexpr int A_BYTES = LBP * LBT * 2;  // 16 KB
  static constexpr int B_BYTES = NQ * LBT * 2;   // 8 or 16 KB
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int TILE_LD = NQ + 4;         // fp32 row stride of the epilogue tile
  static constexpr size_t SMEM = (size_t)LSTAGES * STAGE + 1024 + 256;
  static_assert(LBP * TILE_LD * 4 <= LSTAGES * STAGE, "epilogue tile must fit in the stage ring");
};

template <bool A_MN, bool B_MN, int NQ>
__global__ void __launch_bounds__(LTHREADS, 1)
k_lora_tc(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
          const __grid_constant__ LoraTcArgs a0, const __grid_constant__ CUtensorMap tmA1,
          const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ LoraTcArgs a1, int ctas0) {
  // Two independent products can share one launch: CTAs [0, ctas0) work on
  // the first, the rest on the second (same operand layouts and cluster size).
  const bool second = (int)blockIdx.x >= ctas0;
  const LoraTcArgs &a = second ? a1 : a0;
  const CUtensorMap *tmA = second ? &tmA1 : &tmA0;
  const CUtensorMap *tmB = second ? &tmB1 : &tmB0;
  const int bid = second ? (int)blockIdx.x - ctas0 : (int)blockIdx.x;
  using G = LGeo<NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LSTAGES * G::STAGE);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * LSTAGES + 1);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto full = [&](int s) { return ptx::smem_u32(&bars[s]); };
  auto empty = [&](int s) { return ptx::smem_u32(&bars[LSTAGES + s]); };
  const uint32_t accf = ptx::smem_u32(&bars[2 * LSTAGES]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = ptx::cluster_ctarank(), csize = ptx::cluster_nctarank();
  const int64_t p0 = (int64_t)(bid / (int)csize) * LBP;
  const int64_t nT = (a.T + LBT - 1) / LBT;
  const int64_t ks0 = (int64_t)crank * nT / csize, ks1 = (int64_t)(crank + 1) * nT / csize;
  const int nsteps = (int)(ks1 - ks0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < LSTAGES; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), 1);
    }
    ptx::mbar_init(accf, 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(tmA);
    ptx::prefetch_tmap(tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), NQ);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent; where it waits for the previous
  // kernel depends on a.dep (see LoraProblem).  Dependents are let in only
  // once this kernel has waited, except after kDepExit and kDepFree (whose
  // dependent waits for this grid to complete before touching anything).
  if (a.dep == kDepStart) ptx::griddep_wait();
  if (a.dep != kDepStores) ptx::griddep_launch();

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA
    for (int i = 0; i < nsteps; ++i) {
      const int s = i % LSTAGES;
      const uint32_t ph = (i / LSTAGES) & 1;
      if (!ptx::mbar_wait(empty(s), ph ^ 1, abort, a.status)) break;
      const uint32_t a_dst = sbase + s * G::STAGE, b_dst = a_dst + G::A_BYTES;
      const int t0 = (int)((ks0 + i) * LBT);
      ptx::mbar_arrive_expect_tx(full(s), G::STAGE);
      if (!A_MN) {
        ptx::tma_load_2d(a_dst, tmA, full(s), t0, (int)p0);  // rows p, inner t
      } else {
        ptx::tma_load_2d(a_dst, tmA, full(s), (int)p0, t0);  // rows t, inner p: two 64-wide atoms
        ptx::tma_load_2d(a_dst + 8192, tmA, full(s), (int)p0 + 64, t0);
      }
      if (!B_MN) {
        ptx::tma_load_2d(b_dst, tmB, full(s), t0, 0);
      } else {
#pragma unroll
        for (int j = 0; j < NQ / 64; ++j) ptx::tma_load_2d(b_dst + 8192 * j, tmB, full(s), 64 * j, t0);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA
    constexpr uint32_t idesc = ptx::idesc_bf16(LBP, NQ, B_MN, A_MN);
    bool ok = true;
    for (int i = 0; i < nsteps; ++i) {
      const int s = i % LSTAGES;
      const uint32_t ph = (i / LSTAGES) & 1;
      if (!ptx::mbar_wait(full(s), ph, abort, a.status)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t a_addr = sbase + s * G::STAGE, b_addr = a_addr + G::A_BYTES;
      // K-major: rows of 128 B, 8-row atoms 1 KB apart, K advance +32 B.
      // MN-major: 64-wide atoms 8 KB apart, 8-row K groups 1 KB apart, K advance +2 KB.
      const uint64_t ad = A_MN ? ptx::desc_sw128(a_addr, 8192, 1024) : ptx::desc_sw128(a_addr, 16, 1024);
      const uint64_t bd = B_MN ? ptx::desc_sw128(b_addr, 8192, 1024) : ptx::desc_sw128(b_addr, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < LBT / 16; ++kk)
        ptx::mma_bf16(tmem, ad + (uint64_t)(A_MN ? kk * 128 : kk * 2), bd + (uint64_t)(B_MN ? kk * 128 : kk * 2),
                      idesc, (i > 0 || kk > 0) ? 1u : 0u);
      ptx::mma_commit(empty(s));
    }
    if (ok && nsteps > 0) ptx::mma_commit(accf);
  }

  // ---------------------------------------------------------------- epilogue
  // accumulator (128 lanes x NQ columns) -> fp32 tile in the stage ring
  float *tile = reinterpret_cast<float *>(smem);
  const int row = warp * 32 + lane;
  bool have = nsteps > 0 && !*abort && ptx::mbar_wait(accf, 0, abort, a.status);
  have = __all_sync(0xffffffffu, have);  // tcgen05.ld is warp-collective
  if (have) ptx::tc_fence_after();
#pragma unroll 1
  for (int c = 0; c < NQ / 32; ++c) {
    uint32_t r[32];
    if (have) {
      ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c * 32), r);
      ptx::tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
    }
    float4 *dst = reinterpret_cast<float4 *>(tile + row * G::TILE_LD + c * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                           __uint_as_float(r[4 * i + 3]));
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (a.dep == kDepStores) {  // the first global store follows
    ptx::griddep_wait();
    ptx::griddep_launch();
  }
  // E4M3 scaling: E from the operand kernel's partial maxima (complete: this
  // grid has waited for its predecessor by now, in every mode that scales)
  __shared__ int e_w;
  if (a.row_exp) {
    if (warp == 0) {
      const float m = wmax_of_warp(a.wmax, a.nwpart);
      if (lane == 0) e_w = e4m3_weight_exponent(m);
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- cluster reduction
  // CTA c finishes rows [c*128/S, (c+1)*128/S) of the tile, adding the S
  // partial tiles in CTA order.
  const int r0 = (int)(crank * LBP / csize), r1 = (int)((crank + 1) * LBP / csize);
  const int nrows = r1 - r0, chunks = NQ / 4;
  const uint32_t tile_addr = ptx::smem_u32(tile);
  for (int idx = threadIdx.x; idx < nrows * chunks; idx += LTHREADS) {
    int rr, c4;
    if (a.mode == 2) {  // transposed store: consecutive threads -> consecutive p
      rr = r0 + idx % nrows;
      c4 = idx / nrows;
    } else {
      rr = r0 + idx / chunks;
      c4 = idx % chunks;
    }
    const uint32_t off = (uint32_t)((rr * G::TILE_LD + 4 * c4) * 4);
    float4 v[8];  // every CTA's partial loaded before adding (cluster size <= 8)
#pragma unroll
    for (uint32_t cc = 0; cc < 8; ++cc)
      v[cc] = cc < csize ? ptx::ld_shared_cluster_v4(ptx::mapa(tile_addr + off, cc)) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (uint32_t cc = 0; cc < 8; ++cc)
      if (cc < csize) {
        sum.x += v[cc].x; sum.y += v[cc].y; sum.z += v[cc].z; sum.w += v[cc].w;
      }
    const int64_t p = p0 + rr;
    if (p >= a.P) continue;
    const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t q = 4 * c4 + e;
      if (q >= a.Q) break;
      float sv = __fmul_rn(vals[e], a.scale);
      if (a.mode == 0) {
        if (a.row_exp) sv = __fmul_rn(sv, __uint_as_float((uint32_t)(__ldg(a.row_exp + p) + e_w + 127) << 23));
        static_cast<uint16_t *>(a.out)[p * a.ldo + q] = (uint16_t)(pack_bf16x2(sv, 0.f) & 0xFFFFu);
        if (a.out2) a.out2[p * a.ldo2 + q] = (uint16_t)(pack_bf16x2(vals[e], 0.f) & 0xFFFFu);
      } else if (a.mode == 1) {
        static_cast<float *>(a.out)[p * a.ldo + q] = sv;
      } else {
        static_cast<float *>(a.out)[q * a.ldo + p] = sv;
      }
    }
  }
  // keep this CTA's tile alive until every CTA of the cluster has read it
  ptx::cluster_sync();
  if (warp == 1) ptx::tmem_dealloc(tmem, NQ);
  // kDepExit and kDepFree: one CTA waits for the previous grid before exiting,
  // so this grid completes after it; the others leave their SMs at once
  if ((a.dep == kDepExit || a.dep == kDepFree) && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0)
    ptx::griddep_wait();
}

template <bool A_MN, bool B_MN, int NQ>
int prepare(const LoraProblem &L, CUtensorMap *tA, CUtensorMap *tB, LoraTcArgs *a) {
  // A operand: K-major [P][T] (box 64 x 128) or MN-major [T][P] (box 64 x 64)
  int rc = A_MN ? make_tmap(tA, L.A, (uint64_t)L.P, (uint64_t)L.T, 64)
                : make_tmap(tA, L.A, (uint64_t)L.T, (uint64_t)L.P, LBP);
  // B operand: K-major [Q][T] (box 64 x NQ) or MN-major [T][Q] (box 64 x 64)
  if (!rc)
    rc = B_MN ? make_tmap(tB, L.B, (uint64_t)L.Q, (uint64_t)L.T, 64)
              : make_tmap(tB, L.B, (uint64_t)L.T, (uint64_t)L.Q, NQ);
  if (rc) return rc;
  *a = LoraTcArgs{};
  a->P = L.P; a->Q = L.Q; a->T = L.T; a->mode = L.mode; a->scale = L.scale;
  a->out = L.out; a->ldo = L.ldo; a->out2 = L.out2; a->ldo2 = L.ldo2;
  a->row_exp = L.row_exp;
  a->wmax = L.wmax;
  a->nwpart = L.nwpart;
  a->dep = L.dep;
  a->status = device_status_ptr();
  return QL_OK;
}

// One launch for L0 and, if given, L1 (same layouts and width class).
template <bool A_MN, bool B_MN, int NQ>
int launch_t(const LoraProblem &L0, const LoraProblem *L1, cudaStream_t st) {
  using G = LGeo<NQ>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    int rc = check_cuda(cudaFuncSetAttribute(k_lora_tc<A_MN, B_MN, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)G::SMEM),
                        "LoRA kernel: shared-memory attribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  CUtensorMap tA0, tB0, tA1, tB1;
  LoraTcArgs a0, a1;
  int rc = prepare<A_MN, B_MN, NQ>(L0, &tA0, &tB0, &a0);
  if (!rc && L1) rc = prepare<A_MN, B_MN, NQ>(*L1, &tA1, &tB1, &a1);
  if (rc) return rc;
  if (!L1) {
    tA1 = tA0; tB1 = tB0; a1 = a0;
  }
  const int64_t tiles0 = (L0.P + LBP - 1) / LBP, tiles1 = L1 ? (L1->P + LBP - 1) / LBP : 0;
  int S = lora_splits(L0.P + (L1 ? L1->P : 0), L1 ? std::min(L0.T, L1->T) : L0.T);
  const int ctas0 = (int)(tiles0 * S);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((tiles0 + tiles1) * S));
  cfg.blockDim = dim3(LTHREADS);
  cfg.dynamicSmemBytes = G::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_lora_tc<A_MN, B_MN, NQ>, tA0, tB0, a0, tA1, tB1, a1, ctas0);
  count_launch();
  return check_cuda(e, "LoRA kernel launch");
}

template <bool A_MN, bool B_MN>
int launch_ab(const LoraProblem &L, const LoraProblem *L1, cudaStream_t st) {
  return L.Q <= 64 ? launch_t<A_MN, B_MN, 64>(L, L1, st) : launch_t<A_MN, B_MN, 128>(L, L1, st);
}

}  // namespace

int lora_splits(int64_t P, int64_t T) {
  // As many splits as keep every CTA in one wave (two CTAs per SM on 148
  // SMs), at most 8 (the portable cluster size).
  const int64_t tiles = (P + LBP - 1) / LBP, nT = (T + LBT - 1) / LBT;
  int64_t S = (2 * 148) / tiles;
  S = std::min<int64_t>(S, 8);
  S = std::min<int64_t>(S, std::max<int64_t>(1, nT));
  return (int)std::max<int64_t>(S, 1);
}

int launch_lora(const LoraProblem &L, cudaStream_t st) {
  if (L.a_mn) return L.b_mn ? launch_ab<true, true>(L, nullptr, st) : launch_ab<true, false>(L, nullptr, st);
  return L.b_mn ? launch_ab<false, true>(L, nullptr, st) : launch_ab<false, false>(L, nullptr, st);
}

int launch_lora2(const LoraProblem &L0, const LoraProblem &L1, cudaStream_t st) {
  const bool same = L0.a_mn == L1.a_mn && L0.b_mn == L1.b_mn && (L0.Q <= 64) == (L1.Q <= 64);
  if (!same) {
    int rc = launch_lora(L0, st);
    return rc ? rc : launch_lora(L1, st);
  }
  if (L0.a_mn) return L0.b_mn ? launch_ab<true, true>(L0, &L1, st) : launch_ab<true, false>(L0, &L1, st);
  return L0.b_mn ? launch_ab<false, true>(L0, &L1, st) : launch_ab<false, false>(L0, &L1, st);
}

}  // namespace ql
