// Few-token forward of the QLoRA linear on the tensor cores (16 < M <= 128
// tokens: prefill and batched generation with the frozen 4-bit weight).
//
//   Y = X W_hat^T + XAs B        (XAs = bf16(s X A), made by the LoRA kernel)
//
// With so few tokens the weight stream is the cost (0.52 bytes per weight
// against 2M flops per weight), so the product is computed transposed: a
// 128-row tile of W_hat is the MMA's M side and the M tokens (padded to Mp, a
// multiple of 32) its N side, Y^T tile = W_hat tile . X^T, so no tensor-core
// work is spent on padding 32 tokens up to 128.  The LoRA term rides along as
// ceil(r/64) extra K-steps with A = B^T (an MN-major TMA tile of the stored B)
// and B = XAs.
//
// Work split: the units (tile, K-step) of all tiles, the LoRA steps counted
// as steps of their tile, are cut into G equal contiguous ranges, one per
// CTA (one CTA per SM), so every SM streams the same share of the weight
// whatever the shape.  A tile that one CTA covers whole is stored as bf16 by
// that CTA; every other CTA stores the fp32 sum of its share of a tile, and
// k_skinny_fixup adds the shares of each tile in CTA order (deterministic).
//
// Roles (12 warps):
//   warp 0      TMA of the packed weight in chunks of 128 rows x 128 bytes (4
//               K-steps; whole 128-byte lines of each row, which the memory
//               system serves far better than 32-byte pieces) into a 4-stage
//               ring (64 KB in flight per SM)
//   warp 11     gathers the block constants (codes and steps) of runs of 16
//               K-steps by cp.async into 4 staging buffers, runs ahead
//   warp 1      TMEM allocation (two accumulators of Mp columns, so the next
//               segment's MMAs overlap the previous segment's epilogue) and
//               the single MMA-issuing thread, which waits on one barrier per
//               step (a wait costs far more than an MMA issue once MMAs are in
//               flight, and these MMAs are small)
//   warp 2      TMA of the X tile (or the LoRA tiles) of each step
//   warps 3-10  four converter groups of 2 warps taking K-steps in turn:
//               each thread computes the m_hat of two row-blocks (rows r and
//               r + 64) from the staged constants and expands both,
//               interleaved, from the packed ring into the 128-byte-swizzled
//               A tile of the
//               {A, X} ring (as deep as 128 KB allows); at the end
//               of every segment (one tile's share) each group drains half of
//               the accumulator columns
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "convert.cuh"
#include "ptx.cuh"
#include "tc_gemm.cuh"

namespace ql {
namespace {

constexpr int TBM = 128;                   // weight rows per tile (MMA M)
constexpr int TBK = 64;                    // reduction per step
constexpr int ASTAGES = 4;                 // ring of A tiles (converted W_hat, or LoRA B^T)
constexpr int MAX_XSTAGES = 16;            // ring of X tiles: as many as fit in XRING_BYTES
constexpr int PSTAGES = 4;                 // ring of packed weight chunks
constexpr int A_BYTES = TBM * TBK * 2;     // 16 KB
constexpr int XRING_BYTES = 64 * 1024;     // X ring: 16 stages at Mp = 32 ... 4 at Mp = 128
constexpr int PCHUNK = 4;                  // K-steps per packed chunk (128 bytes of each row)
constexpr int P_BYTES = TBM * TBK / 2 * PCHUNK;  // 16 KB packed chunk
constexpr int THREADS = 384;
constexpr int CONV_WARP0 = 3;
constexpr int SCALE_WARP = 11;
constexpr int NGROUPS = 4;                 // converter groups, taking K-steps in turn
constexpr int GROUP_THREADS = 64;          // 2 warps; each thread expands 2 row-blocks per step
constexpr int CONV_THREADS = NGROUPS * GROUP_THREADS;
constexpr int RUN = 16;                    // K-steps of block constants gathered at once
constexpr int SBUF = 4;                    // runs of block constants in flight
constexpr int SBUF_BYTES = TBM * 64;       // per row: 16 words (codes and steps, or absmax)
constexpr int NBARS = 2 * ASTAGES + 2 * MAX_XSTAGES + 2 * PSTAGES + 5 + 2 * SBUF;
constexpr size_t SMEM = (size_t)ASTAGES * A_BYTES + XRING_BYTES + (size_t)PSTAGES * P_BYTES +
                        (size_t)SBUF * SBUF_BYTES + 1024 + 512;
constexpr int kCtas = 148;                 // CTAs of the stream-K split (one per SM)

struct SkinnyArgs {
  int M, Mp, Nout;
  int ksm, ksl, upt;  // main steps, LoRA steps, steps per tile
  int tiles, G;
  int64_t U;          // tiles * upt
  NF4View w;
  uint16_t *out;
  float *part;        // [G + tiles - 1][Mp][128] fp32 shares
  int *status;
  unsigned long long *span;
  int early_main;     // X and the weight are final: start before the predecessor completes
  uint32_t tmem_cols;
  int xstages;        // X ring depth
  uint32_t x_bytes;   // X tile: Mp x 128 B
  float q[16];
};

// CTA that owns unit u under the split [c U / G, (c + 1) U / G).
__host__ __device__ __forceinline__ int owner_of(int64_t u, int64_t U, int G) {
  return (int)(((u + 1) * (int64_t)G - 1) / U);
}

// A run: `len` consecutive main K-steps kf.. of tile t (len = 0: none left).
struct Run {
  int t, kf, len;
};

// Position (tile t, step k) in a CTA's run of units, advanced one unit at a time.
struct Cursor {
  int t, k;
  __device__ __forceinline__ void next(int upt) {
    if (++k == upt) {
      k = 0;
      ++t;
    }
  }
};

// Ring slot and phase bit, advanced one use at a time.
struct Slot {
  int s;
  uint32_t ph;
  __device__ __forceinline__ void next(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// The CTA's main steps cut into runs of at most RUN steps within one tile,
// in order (LoRA steps skipped).
struct RunCursor {
  int gs;
  Cursor c;
  __device__ __forceinline__ Run next(int nsteps, int ksm, int upt) {
    while (gs < nsteps && c.k >= ksm) {
      c.next(upt);
      ++gs;
    }
    Run r{c.t, c.k, 0};
    if (gs >= nsteps) return r;
    r.len = min(min(RUN, ksm - c.k), nsteps - gs);
    for (int i = 0; i < r.len; ++i) c.next(upt);
    gs += r.len;
    return r;
  }
};

__global__ void __launch_bounds__(THREADS, 1)
k_nf4_skinny(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmX,
             const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmXA,
             const __grid_constant__ SkinnyArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t xbase = sbase + ASTAGES * A_BYTES;           // X tiles
  const uint32_t pbase = xbase + XRING_BYTES;                 // packed chunks
  const uint32_t stage_base = pbase + PSTAGES * P_BYTES;      // runs of block constants
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + ASTAGES * A_BYTES + XRING_BYTES + PSTAGES * P_BYTES +
                                                SBUF * SBUF_BYTES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
  auto afull = [&](int s) { return bar(s); };
  auto aempty = [&](int s) { return bar(ASTAGES + s); };
  auto xfull = [&](int s) { return bar(2 * ASTAGES + s); };
  auto xempty = [&](int s) { return bar(2 * ASTAGES + MAX_XSTAGES + s); };
  constexpr int PB = 2 * ASTAGES + 2 * MAX_XSTAGES;
  auto pfull = [&](int s) { return bar(PB + s); };
  auto pempty = [&](int s) { return bar(PB + PSTAGES + s); };
  auto accf = [&](int a) { return bar(PB + 2 * PSTAGES + a); };
  auto tfree = [&](int a) { return bar(PB + 2 * PSTAGES + 2 + a); };
  const uint32_t drainb = bar(PB + 2 * PSTAGES + 4);
  auto sfull = [&](int b) { return bar(PB + 2 * PSTAGES + 5 + b); };
  auto sempty = [&](int b) { return bar(PB + 2 * PSTAGES + 5 + SBUF + b); };
  const int xstages = p.xstages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t u0 = (int64_t)blockIdx.x * p.U / p.G, u1 = (int64_t)(blockIdx.x + 1) * p.U / p.G;
  const int nsteps = (int)(u1 - u0);
  const int t0 = (int)(u0 / p.upt), k0 = (int)(u0 - (int64_t)t0 * p.upt);

  if (threadIdx.x == 0) {
    for (int s = 0; s < ASTAGES; ++s) {
      ptx::mbar_init(afull(s), GROUP_THREADS);  // the converting (or LoRA-loading) group
      ptx::mbar_init(aempty(s), 1);
    }
    for (int s = 0; s < MAX_XSTAGES; ++s) {
      ptx::mbar_init(xfull(s), 1);
      ptx::mbar_init(xempty(s), 1);
    }
    for (int s = 0; s < PSTAGES; ++s) {
      ptx::mbar_init(pfull(s), 1);
      ptx::mbar_init(pempty(s), PCHUNK * GROUP_THREADS);  // see the converters' release
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(accf(a), 1);
      ptx::mbar_init(tfree(a), CONV_THREADS);
    }
    ptx::mbar_init(drainb, 1);
    for (int b = 0; b < SBUF; ++b) {
      ptx::mbar_init(sfull(b), 32);  // one arrival per scale-warp lane once its copies land
      ptx::mbar_init(sempty(b), CONV_THREADS);
    }
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmP);
    ptx::prefetch_tmap(&tmX);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmXA);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent.  Without early_main everything
  // waits for the predecessor here; with it only the LoRA loads (XAs is the
  // predecessor's output) and the stores wait.
  if (!p.early_main) ptx::griddep_wait();
  ptx::griddep_launch();
  if (p.span && threadIdx.x == 0) atomicMin(p.span, (unsigned long long)ptx::globaltimer());

  if (warp == 0) {
    // ---------------------------------------------------------- packed weight
    if (lane == 0) {
      // one copy per chunk (tile t, K-steps 4q .. 4q + 3) the CTA's main steps touch
      Cursor c{t0, k0};
      Slot ps{0, 0};
      int ct = -1, cq = -1;
      for (int gs = 0; gs < nsteps; ++gs, c.next(p.upt)) {
        if (c.k >= p.ksm || (c.t == ct && c.k / PCHUNK == cq)) continue;
        ct = c.t;
        cq = c.k / PCHUNK;
        if (!ptx::mbar_wait(pempty(ps.s), ps.ph ^ 1, abort, p.status)) break;
        ptx::mbar_arrive_expect_tx(pfull(ps.s), P_BYTES);
        ptx::tma_load_2d(pbase + ps.s * P_BYTES, &tmP, pfull(ps.s), cq * PCHUNK * 32, ct * TBM);
        ps.next(PSTAGES);
      }
    }
  } else if (warp == SCALE_WARP) {
    // ---------------------------------------------------------- block constants
    // Gathers, for every run, per row (lane l: rows l + 32 i) the code words
    // covering the run's code bytes and the one or two step values they fall
    // under (or the run's absmax values without double quantization) into
    // staging buffer rn mod SBUF by cp.async; the buffer's barrier completes
    // when the copies land.  The converters compute m_hat from it.
    const int kbr = (int)(p.w.cols >> 6);
    const int64_t n_b = (int64_t)p.Nout * kbr;
    RunCursor rc{0, Cursor{t0, k0}};
    for (int rn = 0;; ++rn) {
      const Run r = rc.next(nsteps, p.ksm, p.upt);
      if (r.len == 0) break;
      const int b = rn % SBUF;
      if (!ptx::mbar_wait(sempty(b), ((rn / SBUF) & 1) ^ 1, abort, p.status)) break;
      const uint32_t sb = stage_base + (uint32_t)b * SBUF_BYTES;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = lane + 32 * i;
        const int64_t n = (int64_t)r.t * TBM + rl;
        if (n >= p.Nout) continue;
        const uint32_t dst = sb + (uint32_t)rl * 64u;
        const int64_t b0 = n * kbr + r.kf;
        if (p.w.dq) {
          const int64_t w0 = b0 >> 2, w1 = (b0 + r.len - 1) >> 2;
          for (int64_t w = w0; w <= w1; ++w)
            ptx::cp_async4(dst + 4u * (uint32_t)(w - w0), p.w.code + 4 * w, (int)(n_b - 4 * w < 4 ? n_b - 4 * w : 4));
          ptx::cp_async4(dst + 24u, p.w.step + (b0 >> 8), 4);
          ptx::cp_async4(dst + 28u, p.w.step + ((b0 + r.len - 1) >> 8), 4);
        } else {
          for (int j = 0; j < r.len; ++j) ptx::cp_async4(dst + 4u * (uint32_t)j, p.w.absmax + b0 + j, 4);
        }
      }
      ptx::cp_async_arrive(sfull(b));
    }
    ptx::cp_async_wait<0>();
  } else if (warp == 2) {
    // ---------------------------------------------------------- X / XAs tiles
    if (lane == 0) {
      bool waited = !p.early_main;
      Cursor c{t0, k0};
      Slot sx{0, 0};
      for (int gs = 0; gs < nsteps; ++gs, c.next(p.upt), sx.next(xstages)) {
        if (!ptx::mbar_wait(xempty(sx.s), sx.ph ^ 1, abort, p.status)) break;
        const uint32_t dst = xbase + sx.s * p.x_bytes;
        ptx::mbar_arrive_expect_tx(xfull(sx.s), p.x_bytes);
        if (c.k < p.ksm) {
          ptx::tma_load_2d(dst, &tmX, xfull(sx.s), c.k * TBK, 0);
        } else {
          if (!waited) {  // XAs is the predecessor's output
            ptx::griddep_wait();
            waited = true;
          }
          ptx::tma_load_2d(dst, &tmXA, xfull(sx.s), (c.k - p.ksm) * TBK, 0);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc_main = ptx::idesc_bf16(TBM, p.Mp, false, false);
      const uint32_t idesc_lora = ptx::idesc_bf16(TBM, p.Mp, false, true);
      bool ok = true;
      Cursor c{t0, k0};
      Slot sa{0, 0}, sx{0, 0};
      for (int gs = 0; gs < nsteps; ++gs, c.next(p.upt), sa.next(ASTAGES), sx.next(xstages)) {
        const int j = c.t - t0, acc = j & 1;
        const bool first = c.k == 0 || gs == 0, last = c.k == p.upt - 1 || gs == nsteps - 1;
        if (first && j >= 2) {  // the epilogue of segment j - 2 has read this accumulator
          if (!ptx::mbar_wait(tfree(acc), ((j - 2) >> 1) & 1, abort, p.status)) { ok = false; break; }
          ptx::tc_fence_after();
        }
        // afull(s) also implies xfull: the group arrives after the X tile landed
        if (!ptx::mbar_wait(afull(sa.s), sa.ph, abort, p.status)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t a_addr = sbase + sa.s * A_BYTES, x_addr = xbase + sx.s * p.x_bytes;
        const uint32_t d = tmem + (uint32_t)(acc * p.Mp);
        const bool lora = c.k >= p.ksm;
        // A: the converted W_hat tile (K-major rows of 128 B) or B^T (MN-major:
        // two 64-row atoms 8 KB apart, 8-rank groups 1 KB apart); B: X or XAs.
        const uint64_t a_desc = lora ? ptx::desc_sw128(a_addr, 8192, 1024) : ptx::desc_sw128(a_addr, 16, 1024);
        const uint64_t b_desc = ptx::desc_sw128(x_addr, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < TBK / 16; ++kk)
          ptx::mma_bf16(d, a_desc + (uint64_t)(lora ? kk * 128 : kk * 2), b_desc + (uint64_t)(kk * 2),
                        lora ? idesc_lora : idesc_main, (first && kk == 0) ? 0u : 1u);
        ptx::mma_commit(aempty(sa.s));
        ptx::mma_commit(xempty(sx.s));
        if (last) ptx::mma_commit(accf(acc));
      }
      if (!ok) {  // gave up: let the MMAs already issued finish before TMEM is freed
        ptx::mma_commit(drainb);
        drain_wait(drainb, 0);
      }
    }
  } else {
    // ---------------------------------------------------------- converters + epilogue
    const int cw = warp - CONV_WARP0;
    const int g = cw >> 1;                   // group: K-steps gs with gs mod NGROUPS = g
    const int row = (cw & 1) * 32 + lane;    // expands row-blocks row and row + 64
    const int qd = warp & 3;                 // TMEM lane quarter for the epilogue
    const int eh = cw >> 2;                  // epilogue: half of the accumulator columns
    float q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = p.q[i];
    // packed chunk: rows of 128 bytes (4 K-steps), 16-byte pieces swizzled by
    // row mod 8 (the same for rows row and row + 64)
    const uint32_t prow_off = (uint32_t)row * 128u, psw = (uint32_t)(row & 7);
    // last unit of the CTA: main steps of tile tl end before kl_end
    const int64_t ul = u1 - 1;
    const int tl = (int)(ul / p.upt), kl_end = min((int)(ul - (int64_t)tl * p.upt) + 1, p.ksm);
    int ct = -1, cq = -1;  // chunk of the current main step
    const int kbr = (int)(p.w.cols >> 6);
    const float mean = p.w.dq ? __ldg(p.w.mean) : 0.0f;
    bool stores_ok = !p.early_main;
    Cursor c{t0, k0};
    Slot sa{0, 0}, ps{0, 0}, sx{0, 0};
    // the run of block constants the current main step belongs to
    RunCursor rc{0, Cursor{t0, k0}};
    Run run = rc.next(nsteps, p.ksm, p.upt);
    int rn = 0, rj = 0;
    int64_t rb0[2] = {0, 0};  // the two rows' first blocks of the run
    // m_hat of row-block rj of the run, for the row staged at `sb`
    auto mhat_of = [&](uint32_t sb, int64_t b0) {
      if (p.w.dq) {
        const int off = (int)(b0 & 3) + rj;  // byte of the staged code words
        const uint32_t word = ptx::lds32(sb + 4u * (uint32_t)(off >> 2));
        const float code = dq_code_value((int8_t)(word >> (8 * (off & 3))), p.w.dqt);
        const bool second = ((b0 + rj) >> 8) != (b0 >> 8);
        return __fadd_rn(__fmul_rn(code, __uint_as_float(ptx::lds32(sb + (second ? 28u : 24u)))), mean);
      }
      return __uint_as_float(ptx::lds32(sb + 4u * (uint32_t)rj));
    };
#pragma unroll 1
    for (int gs = 0; gs < nsteps; ++gs, c.next(p.upt), sa.next(ASTAGES), sx.next(xstages)) {
      const bool main_step = c.k < p.ksm;
      const uint32_t sb = stage_base + (uint32_t)(rn % SBUF) * SBUF_BYTES + (uint32_t)row * 64u;
      if (main_step && rj == 0) {
        if (!ptx::mbar_wait(sfull(rn % SBUF), (rn / SBUF) & 1, abort, p.status)) break;
        rb0[0] = ((int64_t)run.t * TBM + row) * kbr + run.kf;
        rb0[1] = rb0[0] + 64 * (int64_t)kbr;
      }
      if (main_step && (c.t != ct || c.k / PCHUNK != cq)) {  // the next chunk's stage
        if (ct >= 0) ps.next(PSTAGES);
        ct = c.t;
        cq = c.k / PCHUNK;
      }
      if ((gs & (NGROUPS - 1)) == g) {
        if (main_step) {
          if (!ptx::mbar_wait(pfull(ps.s), ps.ph, abort, p.status)) break;
          const uint32_t src = pbase + ps.s * P_BYTES + prow_off;
          const uint32_t j0 = (uint32_t)(2 * (c.k % PCHUNK));
          const uint32_t o0 = ((j0 ^ psw) << 4), o1 = (((j0 + 1) ^ psw) << 4);
          const uint4 a0 = ptx::lds128(src + o0), a1 = ptx::lds128(src + o1);
          const uint4 b0 = ptx::lds128(src + 64 * 128 + o0), b1 = ptx::lds128(src + 64 * 128 + o1);
          const float ma = mhat_of(sb, rb0[0]), mb = mhat_of(sb + 64 * 64, rb0[1]);
          if (!ptx::mbar_wait(aempty(sa.s), sa.ph ^ 1, abort, p.status)) break;
          const uint32_t dst = sbase + sa.s * A_BYTES + (uint32_t)row * 128u;
          const int64_t n = (int64_t)c.t * TBM + row;
          if (n + 64 < p.Nout) {
            convert_rowblock2(a0, a1, ma, b0, b1, mb, q, dst, dst + 64 * 128, (uint32_t)(row & 7));
          } else {
            if (n < p.Nout) convert_rowblock(a0, a1, ma, q, dst, (uint32_t)(row & 7));
            else zero_row(dst);
            zero_row(dst + 64 * 128);
          }
          ptx::fence_proxy_async_smem();
          // The chunk's stage is free after its steps in this CTA's range are
          // converted: each such step's group arrives once per thread, and the
          // last one also for the chunk's steps outside the range, so every
          // chunk completes PCHUNK x GROUP_THREADS arrivals.
          const int kfirst = max(cq * PCHUNK, c.t == t0 ? k0 : 0);
          const int klast = min(cq * PCHUNK + PCHUNK, c.t == tl ? kl_end : p.ksm) - 1;
          ptx::mbar_arrive_cnt(pempty(ps.s), c.k == klast ? 1u + (uint32_t)(PCHUNK - (klast - kfirst + 1)) : 1u);
          if (!ptx::mbar_wait(xfull(sx.s), sx.ph, abort, p.status)) break;
          ptx::mbar_arrive(afull(sa.s));
        } else {
          // LoRA step: A = B^T, B stored [r][N]: two MN-major atoms of 64
          // weight rows x 64 ranks, loaded by one thread of the group
          if (!ptx::mbar_wait(aempty(sa.s), sa.ph ^ 1, abort, p.status)) break;
          if (!ptx::mbar_wait(xfull(sx.s), sx.ph, abort, p.status)) break;
          if ((cw & 1) == 0 && lane == 0) {
            const uint32_t a_dst = sbase + sa.s * A_BYTES;
            const int l = c.k - p.ksm;
            ptx::mbar_arrive_expect_tx(afull(sa.s), A_BYTES);
            ptx::tma_load_2d(a_dst, &tmB, afull(sa.s), c.t * TBM, l * TBK);
            ptx::tma_load_2d(a_dst + 8192, &tmB, afull(sa.s), c.t * TBM + 64, l * TBK);
          } else {
            ptx::mbar_arrive(afull(sa.s));
          }
        }
      }
      if (main_step) {
        if (++rj == run.len) {  // done with this run's staging buffer
          ptx::mbar_arrive(sempty(rn % SBUF));
          ++rn;
          rj = 0;
          run = rc.next(nsteps, p.ksm, p.upt);
        }
      }
      if (c.k != p.upt - 1 && gs != nsteps - 1) continue;
      // ------------------------------------------------------ epilogue of segment j
      const int t = c.t, j = t - t0, acc = j & 1;
      if (!ptx::mbar_wait(accf(acc), (j >> 1) & 1, abort, p.status)) break;
      ptx::tc_fence_after();
      if (!stores_ok) {
        ptx::griddep_wait();
        stores_ok = true;
      }
      const int64_t ua = (int64_t)t * p.upt;
      const bool whole = owner_of(ua, p.U, p.G) == owner_of(ua + p.upt - 1, p.U, p.G);
      const int i = qd * 32 + lane;
      const int64_t n = (int64_t)t * TBM + i;
      const int half = p.Mp >> 1, c0 = eh * half;
      float *prow = p.part + ((int64_t)(blockIdx.x + t) * p.Mp) * TBM + i;
#pragma unroll 1
      for (int cc = 0; cc < half; cc += 16) {
        uint32_t r[16];
        ptx::tmem_ld_32x32b_x16(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * p.Mp + c0 + cc), r);
        ptx::tmem_wait_ld();
        if (n < p.Nout) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int m = c0 + cc + e;
            if (m < p.M) {
              if (whole) p.out[(int64_t)m * p.Nout + n] = (uint16_t)(pack_bf16x2(__uint_as_float(r[e]), 0.0f) & 0xFFFFu);
              else prow[(int64_t)m * TBM] = __uint_as_float(r[e]);
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tfree(acc));
    }
  }
  // after an abort, copies already issued into the rings are given time to land
  if (*abort && threadIdx.x == 0) settle();
  ptx::tc_fence_before();
  __syncthreads();
  if (p.span && threadIdx.x == 0) atomicMax(p.span + 1, (unsigned long long)ptx::globaltimer());
  if (warp == 1) ptx::tmem_dealloc(tmem, p.tmem_cols);
}

// Y[m][n] = bf16(sum of the fp32 shares of tile n / 128 in CTA order), for
// the tiles that more than one CTA shares; 8 outputs per thread.  The shares
// are loaded 8 at a time before they are added (in CTA order), so the loads
// overlap.  A programmatic dependent of k_nf4_skinny: waits for it before
// reading.
__global__ void __launch_bounds__(128) k_skinny_fixup(const float *__restrict__ part, int64_t U, int G, int upt,
                                                      int tiles, int M, int Mp, int Nout, uint16_t *__restrict__ out) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int64_t items = (int64_t)tiles * M * (TBM / 8);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += stride) {
    const int i8 = (int)(it % (TBM / 8));
    const int64_t rest = it / (TBM / 8);
    const int m = (int)(rest % M), t = (int)(rest / M);
    const int64_t n = (int64_t)t * TBM + i8 * 8;
    if (n >= Nout) continue;
    const int64_t ua = (int64_t)t * upt;
    const int cf = owner_of(ua, U, G), cl = owner_of(ua + upt - 1, U, G);
    if (cf == cl) continue;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    for (int c0 = cf; c0 <= cl; c0 += 8) {
      float4 x[8], y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c0 + i <= cl) {
          const float4 *ps = reinterpret_cast<const float4 *>(part + ((int64_t)(c0 + i + t) * Mp + m) * TBM + i8 * 8);
          x[i] = __ldcg(ps);
          y[i] = __ldcg(ps + 1);
        }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c0 + i <= cl) {
          if (c0 + i == cf) {
            a = x[i];
            b = y[i];
          } else {
            a.x += x[i].x; a.y += x[i].y; a.z += x[i].z; a.w += x[i].w;
            b.x += y[i].x; b.y += y[i].y; b.z += y[i].z; b.w += y[i].w;
          }
        }
    }
    *reinterpret_cast<uint4 *>(out + (int64_t)m * Nout + n) =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

struct Geometry {
  int Mp, ksm, ksl, upt, tiles, G;
  int64_t U;
};
// cta_cap: CTAs the split may use (at most kCtas)
Geometry geometry(int64_t M, int64_t Nout, int64_t Kred, int r, int cta_cap = kCtas) {
  Geometry g{};
  g.Mp = (int)((M + 31) / 32 * 32);
  g.ksm = (int)((Kred + TBK - 1) / TBK);
  g.ksl = (r + TBK - 1) / TBK;
  g.upt = g.ksm + g.ksl;
  g.tiles = (int)((Nout + TBM - 1) / TBM);
  g.U = (int64_t)g.tiles * g.upt;
  g.G = (int)std::min<int64_t>(g.U, std::min(cta_cap, kCtas));
  return g;
}

}  // namespace

size_t skinny_part_bytes(int64_t M, int64_t Nout, int64_t Kred, int r) {
  if (M <= 0 || M > kSkinnyMaxM) return 0;
  const Geometry g = geometry(M, Nout, Kred, r);
  return (size_t)(g.G + g.tiles - 1) * (size_t)g.Mp * TBM * 4;
}

int launch_nf4_skinny(const GemmProblem &gp, unsigned long long *span, cudaStream_t st) {
  if (gp.trans || gp.M <= 0 || gp.M > kSkinnyMaxM || !gp.part)
    return set_error(QL_ERR_INVALID, "few-token GEMM: forward form with 1..128 tokens and a partial buffer only");
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    int rc = check_cuda(cudaFuncSetAttribute(k_nf4_skinny, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM),
                        "few-token GEMM: shared-memory attribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  // With early_main this kernel runs alongside the LoRA kernel that makes XAs
  // (one CTA per split of its reduction): leave it those SMs, so that no CTA
  // of this kernel (which fills an SM) waits for it to finish.  The partial
  // buffer, sized for kCtas CTAs, has room for any smaller split.
  const int cap = gp.early_main ? kCtas - lora_splits(gp.M, gp.Kred) * (int)((gp.M + 127) / 128) : kCtas;
  const Geometry geo = geometry(gp.M, gp.Nout, gp.Kred, gp.r, cap);
  CUtensorMap tP, tX, tB, tXA;
  int rc = make_tmap_packed(&tP, gp.w.packed, (uint64_t)gp.Kred / 2, (uint64_t)gp.Nout, TBM);
  if (!rc) rc = make_tmap(&tX, gp.A, (uint64_t)gp.Kred, (uint64_t)gp.M, (uint32_t)geo.Mp);
  if (!rc) rc = make_tmap(&tB, gp.B2, (uint64_t)gp.Nout, (uint64_t)gp.r, 64);
  if (!rc) rc = make_tmap(&tXA, gp.A2, (uint64_t)gp.r, (uint64_t)gp.M, (uint32_t)geo.Mp);
  if (rc) return rc;
  SkinnyArgs a{};
  a.M = (int)gp.M;
  a.Mp = geo.Mp;
  a.Nout = (int)gp.Nout;
  a.ksm = geo.ksm;
  a.ksl = geo.ksl;
  a.upt = geo.upt;
  a.tiles = geo.tiles;
  a.G = geo.G;
  a.U = geo.U;
  a.w = gp.w;
  a.out = gp.out;
  a.part = gp.part;
  a.status = device_status_ptr();
  a.span = span;
  a.early_main = gp.early_main ? 1 : 0;
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * geo.Mp)) cols <<= 1;
  a.tmem_cols = cols;
  a.x_bytes = (uint32_t)(geo.Mp * TBK * 2);
  a.xstages = std::min<int>(MAX_XSTAGES, XRING_BYTES / (int)a.x_bytes);
  const Codebook &cb = codebook(gp.w.qt);
  for (int i = 0; i < 16; ++i) a.q[i] = cb.q[i];

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)geo.G);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_nf4_skinny, tP, tX, tB, tXA, a);
  count_launch();
  rc = check_cuda(e, "few-token GEMM launch");
  if (rc) return rc;
  const int64_t items = (int64_t)geo.tiles * gp.M * (TBM / 8);
  cudaLaunchConfig_t fc{};
  fc.gridDim = dim3((unsigned)std::min<int64_t>((items + 127) / 128, 148 * 16));
  fc.blockDim = dim3(128);
  fc.stream = st;
  fc.attrs = attr;
  fc.numAttrs = 1;
  e = cudaLaunchKernelEx(&fc, k_skinny_fixup, (const float *)gp.part, geo.U, geo.G, geo.upt, geo.tiles, (int)gp.M,
                         geo.Mp, (int)gp.Nout, gp.out);
  count_launch();
  return check_cuda(e, "few-token GEMM fixup launch");
}

}  // namespace ql
