// Device helpers shared by the tensor-core GEMM kernels (internal): the
// in-shared-memory dequantizer of one 64-element row-block and the bounded
// waits used after an abort.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace ql {

// 8 bf16 values of one 16-byte smem chunk from 8 packed nibbles, through the
// 16-entry table held as low-byte (TL) and high-byte (TH) planes.  Byte j of
// `w` holds element 2j in its high nibble and element 2j+1 in its low nibble.
__device__ __forceinline__ void lookup8(uint32_t w, const uint32_t (&TL)[4], const uint32_t (&TH)[4],
                                        uint32_t &o0, uint32_t &o1, uint32_t &o2, uint32_t &o3) {
  using ptx::prmt;
  // selector: the low 3 bits of every nibble pick a byte among 8 entries
  const uint32_t s = w & 0x77777777u;
  // second-level selector: byte i from the first (entries 0-7) or second
  // (entries 8-15) half, by bit 3 of nibble i
  const uint32_t s2 = ((w >> 1) & 0x44444444u) | 0x32103210u;
  {
    uint32_t L = prmt(prmt(TL[0], TL[1], s), prmt(TL[2], TL[3], s), s2);
    uint32_t H = prmt(prmt(TH[0], TH[1], s), prmt(TH[2], TH[3], s), s2);
    // L, H bytes hold elements (1, 0, 3, 2); interleave to bf16 pairs (0,1), (2,3)
    o0 = prmt(L, H, 0x4051u);
    o1 = prmt(L, H, 0x6273u);
  }
  {
    const uint32_t sh = s >> 16, s2h = s2 >> 16;
    uint32_t L = prmt(prmt(TL[0], TL[1], sh), prmt(TL[2], TL[3], sh), s2h);
    uint32_t H = prmt(prmt(TH[0], TH[1], sh), prmt(TH[2], TH[3], sh), s2h);
    o2 = prmt(L, H, 0x4051u);
    o3 = prmt(L, H, 0x6273u);
  }
}

// One 64-element row-block: 32 packed bytes and the block constant -> one
// 128-byte row of a 128B-swizzled tile at `dst` (chunk j stored at j ^ swz).
__device__ __forceinline__ void convert_rowblock(const uint4 &p0, const uint4 &p1, float mhat,
                                                 const float (&q)[16], uint32_t dst, uint32_t swz) {
  uint32_t P[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) P[k] = pack_bf16x2(__fmul_rn(q[2 * k], mhat), __fmul_rn(q[2 * k + 1], mhat));
  uint32_t TL[4], TH[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    TL[i] = ptx::prmt(P[2 * i], P[2 * i + 1], 0x6420u);
    TH[i] = ptx::prmt(P[2 * i], P[2 * i + 1], 0x7531u);
  }
  const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t o0, o1, o2, o3;
    lookup8(words[j], TL, TH, o0, o1, o2, o3);
    ptx::sts128(dst + (((uint32_t)j ^ swz) << 4), o0, o1, o2, o3);
  }
}

// Two row-blocks at once (independent instruction streams interleaved, for
// latency hiding); both rows have the same swizzle phase `swz`.
__device__ __forceinline__ void convert_rowblock2(const uint4 &a0, const uint4 &a1, float ma, const uint4 &b0,
                                                  const uint4 &b1, float mb, const float (&q)[16], uint32_t dst_a,
                                                  uint32_t dst_b, uint32_t swz) {
  uint32_t TLa[4], THa[4], TLb[4], THb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t pa0 = pack_bf16x2(__fmul_rn(q[4 * i], ma), __fmul_rn(q[4 * i + 1], ma));
    const uint32_t pa1 = pack_bf16x2(__fmul_rn(q[4 * i + 2], ma), __fmul_rn(q[4 * i + 3], ma));
    const uint32_t pb0 = pack_bf16x2(__fmul_rn(q[4 * i], mb), __fmul_rn(q[4 * i + 1], mb));
    const uint32_t pb1 = pack_bf16x2(__fmul_rn(q[4 * i + 2], mb), __fmul_rn(q[4 * i + 3], mb));
    TLa[i] = ptx::prmt(pa0, pa1, 0x6420u);
    THa[i] = ptx::prmt(pa0, pa1, 0x7531u);
    TLb[i] = ptx::prmt(pb0, pb1, 0x6420u);
    THb[i] = ptx::prmt(pb0, pb1, 0x7531u);
  }
  const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t o0, o1, o2, o3, e0, e1, e2, e3;
    lookup8(wa[j], TLa, THa, o0, o1, o2, o3);
    lookup8(wb[j], TLb, THb, e0, e1, e2, e3);
    const uint32_t off = ((uint32_t)j ^ swz) << 4;
    ptx::sts128(dst_a + off, o0, o1, o2, o3);
    ptx::sts128(dst_b + off, e0, e1, e2, e3);
  }
}

// 8 E4M3 bytes (elements i = 0..7 in bytes 0..7 of lo, hi) from the 8 codes
// in nibbles 0..7 of `s`, through the 16-byte table T (entry c in byte c % 4
// of T[c / 4]): bits 0-2 of a code pick a byte among 8, bit 3 the table half.
// A byte permute reads only the low 16 bits (4 selectors) of its selector
// word, so both halves share one masked word and one final-selector word.
__device__ __forceinline__ void lut8_e4m3(uint32_t s, const uint32_t (&T)[4], uint32_t &lo, uint32_t &hi) {
  using ptx::prmt;
  const uint32_t sel = s & 0x77777777u;                      // byte index within a table half
  const uint32_t fin = ((s >> 1) & 0x44444444u) | 0x32103210u;  // which half, per element
  const uint32_t sel_h = sel >> 16, fin_h = fin >> 16;
  lo = prmt(prmt(T[0], T[1], sel), prmt(T[2], T[3], sel), fin);
  hi = prmt(prmt(T[0], T[1], sel_h), prmt(T[2], T[3], sel_h), fin_h);
}

// One 64-element row-block to E4M3: the block's table holds
// e4m3(fl32(q[c] * mE)) with mE = m_hat * 2^E (exact scaling), so an element
// becomes e4m3(fl32(q[c] * m_hat) * 2^E); its 64 bytes are 16-byte pieces
// 4h .. 4h + 3 of the 128-byte swizzled row at `row_addr` (piece j stored at
// j ^ swz): h = 0 for the first 64 K-elements of a 128-wide step, 1 for the
// second.  kInOrder: byte i holds element i; otherwise the bytes of each pair
// come out swapped (element 2j + 1 at byte 2j), which saves the nibble swap
// and is exact wherever the other operand carries the same order along the
// reduction (a dot product does not depend on the order of its terms).
template <bool kInOrder>
__device__ __forceinline__ void convert_rowblock_e4m3(const uint4 &p0, const uint4 &p1, float mE,
                                                      const float (&q)[16], uint32_t row_addr, int h, uint32_t swz) {
  uint32_t T[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    T[i] = ptx::cvt_e4m3x2(__fmul_rn(q[4 * i], mE), __fmul_rn(q[4 * i + 1], mE)) |
           (ptx::cvt_e4m3x2(__fmul_rn(q[4 * i + 2], mE), __fmul_rn(q[4 * i + 3], mE)) << 16);
  const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint32_t w = words[2 * jj + t];
      // byte j of w holds element 2j (high nibble) and 2j + 1 (low): swapped,
      // nibble i holds element i
      const uint32_t sw = kInOrder ? (((w >> 4) & 0x0F0F0F0Fu) | ((w << 4) & 0xF0F0F0F0u)) : w;
      lut8_e4m3(sw, T, o[2 * t], o[2 * t + 1]);
    }
    ptx::sts128(row_addr + ((((uint32_t)(4 * h + jj)) ^ swz) << 4), o[0], o[1], o[2], o[3]);
  }
}

// Wait for phase `parity` of a barrier for at most `limit_ns`, ignoring the
// abort flag (used only after an abort, for work already in flight).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = 100000000ull) {
  const uint64_t t0 = ptx::globaltimer();
#pragma unroll 1
  while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer() - t0 < limit_ns) {
  }
}

// After an abort: a fixed 50 us pause so that tensor copies already issued
// into shared memory land before the CTA exits (their barriers may never
// complete, since the other roles stopped arriving on them).
__device__ __forceinline__ void settle() {
  const uint64_t t0 = ptx::globaltimer();
#pragma unroll 1
  while (ptx::globaltimer() - t0 < 50000ull) {
  }
}

__device__ __forceinline__ void zero_row(uint32_t dst) {
#pragma unroll
  for (int j = 0; j < 8; ++j) ptx::sts128(dst + (j << 4), 0, 0, 0, 0);
}

}  // namespace ql
