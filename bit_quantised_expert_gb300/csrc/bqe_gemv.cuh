// bqe_gemv.cuh — the per-format dequant-GEMV inner loops of the decode
// layer: one warp, one 32-row panel of a weight tile in shared memory, one
// 256-column group, all activation rows of the item at once on the tensor
// cores (mma.sync m16n8k16: the weights are decoded in registers straight
// into the A fragments, so the skinny product needs no shared-memory operand
// staging), fp32 accumulation.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>

#include "bqe_internal.cuh"

namespace bqe {

__device__ __forceinline__ float ue8m0_f32(uint32_t e) {
  return e == 0 ? __int_as_float(0x00400000) : __int_as_float((int)(e << 23));
}

__device__ __forceinline__ float2 e2m1x2_f32(uint32_t byte) {
  __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)byte, __NV_E2M1);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Four E2M1 pairs of one 32-bit word -> four f16x2 (exact; the low nibble of
// each byte is the lower half), by the hardware E2M1x2 -> f16x2 conversion.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                                uint32_t& h3) {
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

__device__ __forceinline__ float silu_f(float t) { return t / (1.0f + expf(-t)); }

// Activation rows of an item: f16 x 2^s in the format's column order (W1/W3)
// or the f16 hi/lo records of h (W2).
enum { kActF16 = 1, kActH16 = 3 };
__host__ __device__ inline int act_mode(int phase) { return phase == 0 ? kActF16 : kActH16; }

// Bytes of one staged activation row (one bulk copy) ...
__host__ __device__ inline int act_row_bytes(int amode, int fmt, int kc) {
  return amode == kActF16 ? f16_len(fmt, kc) * 2 : (int)h16_rec_bytes(fmt, kc);
}
// ... and the distance between two staged rows in shared memory: x rows sit
// 64 bytes past a multiple of 128, so that the 16-byte B loads of two rows
// (one quarter-warp) fall in different banks (NVFP4: 32 bytes, see below).
__host__ __device__ inline int act_row_stride(int amode, int fmt, int kc) {
  const int b = act_row_bytes(amode, fmt, kc);
  // NVFP4 reads 8-byte B pieces (half-warps over four rows): 32 bytes apart
  return amode == kActF16 ? ((b + 127) & ~127) + (fmt == BQE_FMT_NVFP4 ? 32 : 64) : (b + 15) & ~15;
}

// ----------------------------------------------------------------------------
// Group loops: one warp, one 32-row panel (two m16 tiles), one 256-column
// group, all rows of the item in one pass.  The weights are
// decoded straight into the A fragments of mma.sync m16n8k16 (f16 inputs,
// fp32 accumulation; every decoded value is an exact f16); the activation
// rows are the B columns: row n of x in column n (W1/W3), or h of row r as two
// columns, 2r (hi) and 2r + 1 (lo) (W2, h = hi + lo to about 2^-22 of the
// group's largest value), four rows per MMA.  Thread (gq = lane / 4, tq =
// lane % 4) holds rows gq, gq + 8 of each m16 tile.  The K order inside a k16
// step is free as long as A and B follow the same one: each format takes the
// order in which its codes decode cheapest (the staged rows follow it), and
// its block scale multiplies the fp32 accumulators once per block.
// ----------------------------------------------------------------------------
// d += a b on the tensor cores (m16n8k16, row.col, f16 x f16 -> f32)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// (a & b) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hadd2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
constexpr uint32_t kF16x2One024 = 0x64006400u;  // (1024, 1024): a code c in its mantissa reads 1024 + c

// MXFP4: thread tq takes byte-word tq of a row's 16-byte block (columns 8 tq
// .. 8 tq + 7), natural column order: k16 step s of block b meets x columns
// 32 b + 8 tq + 4 s .. + 3, one 16-byte load of B per block.
template <int NJ>
__device__ __forceinline__ void mma_mxfp4(const uint8_t* tile, int nb, int grp, const uint8_t* const (&bv)[NJ],
                                          int lane, float (&acc)[NJ][2][4]) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll 2
  for (int bi = 0; bi < 8; ++bi) {
    const int b = grp * 8 + bi;
    uint4 bx[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) bx[j] = *reinterpret_cast<const uint4*>(bv[j] + (b * 32 + 8 * tq) * 2);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int r0 = 16 * mt + gq;
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(tile + b * 512 + r0 * 16 + 4 * tq);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(tile + b * 512 + (r0 + 8) * 16 + 4 * tq);
      const float s0 = ue8m0_f32(tile[nb * 512 + b * 32 + r0]), s1 = ue8m0_f32(tile[nb * 512 + b * 32 + r0 + 8]);
      uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
      e2m1x8_to_f16x2(w0, p0, p1, p2, p3);
      e2m1x8_to_f16x2(w1, q0, q1, q2, q3);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16(d, p0, q0, p1, q1, bx[j].x, bx[j].y);
        mma_f16(d, p2, q2, p3, q3, bx[j].z, bx[j].w);
        acc[j][mt][0] = fmaf(d[0], s0, acc[j][mt][0]);
        acc[j][mt][1] = fmaf(d[1], s0, acc[j][mt][1]);
        acc[j][mt][2] = fmaf(d[2], s1, acc[j][mt][2]);
        acc[j][mt][3] = fmaf(d[3], s1, acc[j][mt][3]);
      }
    }
  }
}

// MXFP4 with one activation row (W1/W3 at M = 1): block bi of the group's 8
// meets B column bi (x of the block's 32 columns in that column, zero in the
// others), so each block's dot products collect in an accumulator column of
// their own and the E8M0 scales multiply once per task instead of once per
// block; the row sums are then the scaled columns added across the four
// threads of a row.  Output as mma_group_nj's (row 0 of outv).
__device__ __forceinline__ void mma_mxfp4_r1(const uint8_t* tile, int nb, int grp, const uint8_t* xrow, int lane,
                                             float* outv) {
  const int gq = lane >> 2, tq = lane & 3;
  // x of block gq of the group, columns 8 tq .. 8 tq + 7 (natural order)
  const uint4 xg = *reinterpret_cast<const uint4*>(xrow + ((grp * 8 + gq) * 32 + 8 * tq) * 2);
  float d[2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) d[mt][0] = d[mt][1] = d[mt][2] = d[mt][3] = 0.f;
#pragma unroll 2
  for (int bi = 0; bi < 8; ++bi) {
    const int b = grp * 8 + bi;
    const bool on = gq == bi;
    const uint32_t x0 = on ? xg.x : 0u, x1 = on ? xg.y : 0u, x2 = on ? xg.z : 0u, x3 = on ? xg.w : 0u;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int r0 = 16 * mt + gq;
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(tile + b * 512 + r0 * 16 + 4 * tq);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(tile + b * 512 + (r0 + 8) * 16 + 4 * tq);
      uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
      e2m1x8_to_f16x2(w0, p0, p1, p2, p3);
      e2m1x8_to_f16x2(w1, q0, q1, q2, q3);
      mma_f16(d[mt], p0, q0, p1, q1, x0, x1);
      mma_f16(d[mt], p2, q2, p3, q3, x2, x3);
    }
  }
  // thread (gq, tq) holds columns (blocks) 2 tq, 2 tq + 1 of rows r0 and r0 + 8
  const uint8_t* sc = tile + nb * 512;
  const int c0 = (grp * 8 + 2 * tq) * 32;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = 16 * mt + gq;
    float v0 = d[mt][0] * ue8m0_f32(sc[c0 + r0]);
    v0 = fmaf(d[mt][1], ue8m0_f32(sc[c0 + 32 + r0]), v0);
    float v1 = d[mt][2] * ue8m0_f32(sc[c0 + r0 + 8]);
    v1 = fmaf(d[mt][3], ue8m0_f32(sc[c0 + 32 + r0 + 8]), v1);
    v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
    v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
    if (tq == 0) {
      outv[r0] = v0;
      outv[r0 + 8] = v1;
    }
  }
}

// MXFP4 W2 with one activation row: the h record's hi and lo halves of
// block bq (of four) meet B columns 2 bq and 2 bq + 1; two passes cover the
// group's eight blocks, each in accumulators of its own, and the E8M0 scales
// multiply once per task.  rec: the row's h record (hi | 64 B | lo | 2^-s of
// each 256 columns), flen its halves per part.
__device__ __forceinline__ void mma_mxfp4_r1_hl(const uint8_t* tile, int nb, int grp, const uint8_t* rec, int flen,
                                                int lane, float* outv) {
  const int gq = lane >> 2, tq = lane & 3;
  const uint8_t* src = rec + ((gq & 1) ? 2 * flen + 64 : 0);  // B column gq: hi (even) or lo (odd)
  const uint4 xa = *reinterpret_cast<const uint4*>(src + ((grp * 8 + (gq >> 1)) * 32 + 8 * tq) * 2);
  const uint4 xb = *reinterpret_cast<const uint4*>(src + ((grp * 8 + 4 + (gq >> 1)) * 32 + 8 * tq) * 2);
  float d[2][2][4];
#pragma unroll
  for (int ps = 0; ps < 2; ++ps)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) d[ps][mt][0] = d[ps][mt][1] = d[ps][mt][2] = d[ps][mt][3] = 0.f;
#pragma unroll
  for (int ps = 0; ps < 2; ++ps) {
    const uint4 xg = ps ? xb : xa;
#pragma unroll 2
    for (int bq = 0; bq < 4; ++bq) {
      const int b = grp * 8 + 4 * ps + bq;
      const bool on = (gq >> 1) == bq;
      const uint32_t x0 = on ? xg.x : 0u, x1 = on ? xg.y : 0u, x2 = on ? xg.z : 0u, x3 = on ? xg.w : 0u;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int r0 = 16 * mt + gq;
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(tile + b * 512 + r0 * 16 + 4 * tq);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(tile + b * 512 + (r0 + 8) * 16 + 4 * tq);
        uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
        e2m1x8_to_f16x2(w0, p0, p1, p2, p3);
        e2m1x8_to_f16x2(w1, q0, q1, q2, q3);
        mma_f16(d[ps][mt], p0, q0, p1, q1, x0, x1);
        mma_f16(d[ps][mt], p2, q2, p3, q3, x2, x3);
      }
    }
  }
  // thread (gq, tq) holds hi and lo of block tq of each pass, rows r0, r0 + 8
  const uint8_t* sc = tile + nb * 512;
  const int ca = (grp * 8 + tq) * 32, cb = ca + 4 * 32;
  const float us = reinterpret_cast<const float*>(rec + 4 * flen + 64)[grp];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = 16 * mt + gq;
    float v0 = (d[0][mt][0] + d[0][mt][1]) * ue8m0_f32(sc[ca + r0]);
    v0 = fmaf(d[1][mt][0] + d[1][mt][1], ue8m0_f32(sc[cb + r0]), v0);
    float v1 = (d[0][mt][2] + d[0][mt][3]) * ue8m0_f32(sc[ca + r0 + 8]);
    v1 = fmaf(d[1][mt][2] + d[1][mt][3], ue8m0_f32(sc[cb + r0 + 8]), v1);
    v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
    v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
    if (tq == 0) {
      outv[r0] = v0 * us;
      outv[r0 + 8] = v1 * us;
    }
  }
}

// Two E2M1 code bytes (the low 16 bits of w) -> two f16x2, and two E4M3
// scale bytes (the low 16 bits of s) -> one f16x2, by the hardware conversions.
__device__ __forceinline__ void e2m1x4_to_f16x2(uint32_t w, uint32_t& h0, uint32_t& h1) {
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %2;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1; }"
      : "=r"(h0), "=r"(h1)
      : "r"(w));
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t s) {
  uint32_t h;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.rn.f16x2.e4m3x2 %0, lo; }" : "=r"(h) : "r"(s));
  return h;
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// NVFP4 (16-column blocks = one k16 step): thread tq takes code bytes 2 tq,
// 2 tq + 1 of a row's 8 (columns 4 tq .. 4 tq + 3), natural column order; the
// block's E4M3 scale multiplies the decoded pair in f16, exactly (an E2M1
// value times an E4M3 value has at most 6 significant bits and stays within
// f16's normal range), so the scale rides in A and the accumulators need
// none.  Even and odd blocks accumulate separately (two MMA chains).
template <int NJ>
__device__ __forceinline__ void mma_nvfp4(const uint8_t* tile, int nb, int grp, const uint8_t* const (&bv)[NJ],
                                          int lane, float (&acc)[NJ][2][4]) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = 16 * mt + gq;
    float d[NJ][2][4];
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) d[j][h][0] = d[j][h][1] = d[j][h][2] = d[j][h][3] = 0.f;
#pragma unroll 4
    for (int bi = 0; bi < 16; ++bi) {
      const int b = grp * 16 + bi;
      const uint32_t c0 = *reinterpret_cast<const uint16_t*>(tile + b * 256 + r0 * 8 + 2 * tq);
      const uint32_t c1 = *reinterpret_cast<const uint16_t*>(tile + b * 256 + (r0 + 8) * 8 + 2 * tq);
      const uint32_t sc = e4m3x2_to_f16x2((uint32_t)tile[nb * 256 + b * 32 + r0] |
                                          ((uint32_t)tile[nb * 256 + b * 32 + r0 + 8] << 8));
      const uint32_t s0 = __byte_perm(sc, sc, 0x1010), s1 = __byte_perm(sc, sc, 0x3232);
      uint32_t p0, p1, q0, q1;
      e2m1x4_to_f16x2(c0, p0, p1);
      e2m1x4_to_f16x2(c1, q0, q1);
      p0 = hmul2u(p0, s0);
      p1 = hmul2u(p1, s0);
      q0 = hmul2u(q0, s1);
      q1 = hmul2u(q1, s1);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const uint2 x = *reinterpret_cast<const uint2*>(bv[j] + (b * 16 + 4 * tq) * 2);
        mma_f16(d[j][bi & 1], p0, q0, p1, q1, x.x, x.y);
      }
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][mt][e] += d[j][0][e] + d[j][1][e];
  }
}

// Q2_0: the codes of columns p and 8 + p of a 16-column word (bits 2p and
// 16 + 2p) as f16 (2q - 3).  With the pair at bits 2P, 16 + 2P (P = 1..4;
// pairs 0 and 5..7 are shifted there first) lop3 places it in the mantissa
// of 1024 (1024 + 4^P q, exact), and one fma scales by 2 4^-P and subtracts
// 2^(11 - 2P) + 3: exact, the constants being f16 numbers.
template <int P>
__device__ __forceinline__ uint32_t q2_pair(uint32_t w) {
  constexpr uint32_t kMul[5] = {0u, 0x38003800u, 0x30003000u, 0x28002800u, 0x20002000u};  // 2 4^-P
  constexpr uint32_t kAdd[5] = {0u, 0xE006E006u, 0xD818D818u, 0xD060D060u, 0xC980C980u};  // -(2^(11-2P) + 3)
  return hfma2u(and_or(w, 0x00030003u << (2 * P), kF16x2One024), kMul[P], kAdd[P]);
}
// the eight pairs of one word, pair p in a[p]
__device__ __forceinline__ void q2_pairs(uint32_t w, uint32_t (&a)[8]) {
  const uint32_t wl = w << 2, wr = w >> 8;
  a[0] = q2_pair<1>(wl);
  a[1] = q2_pair<1>(w);
  a[2] = q2_pair<2>(w);
  a[3] = q2_pair<3>(w);
  a[4] = q2_pair<4>(w);
  a[5] = q2_pair<1>(wr);
  a[6] = q2_pair<2>(wr);
  a[7] = q2_pair<3>(wr);
}

// Q2_0 (64-column blocks): thread tq takes word tq of a row's 16 code bytes
// (columns 16 tq .. + 15 of the block); step s of the block = pairs 2s, 2s + 1,
// the B rows in P order (positions 16 tq + 4 s .. + 3).
template <int NJ>
__device__ __forceinline__ void mma_q2_0(const uint8_t* tile, int nb, int grp, const uint8_t* const (&bv)[NJ],
                                         int lane, float (&acc)[NJ][2][4]) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll 1
  for (int bi = 0; bi < 4; ++bi) {
    const int b = grp * 4 + bi;
    uint4 bx[NJ][2];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      bx[j][0] = *reinterpret_cast<const uint4*>(bv[j] + (b * 64 + 16 * tq) * 2);
      bx[j][1] = *reinterpret_cast<const uint4*>(bv[j] + (b * 64 + 16 * tq + 8) * 2);
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int r0 = 16 * mt + gq;
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(tile + b * 512 + r0 * 16 + 4 * tq);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(tile + b * 512 + (r0 + 8) * 16 + 4 * tq);
      const float d0 = __half2float(*reinterpret_cast<const __half*>(tile + nb * 512 + (b * 32 + r0) * 2));
      const float d1 = __half2float(*reinterpret_cast<const __half*>(tile + nb * 512 + (b * 32 + r0 + 8) * 2));
      uint32_t a[8], c[8];
      q2_pairs(w0, a);
      q2_pairs(w1, c);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16(d, a[0], c[0], a[1], c[1], bx[j][0].x, bx[j][0].y);
        mma_f16(d, a[2], c[2], a[3], c[3], bx[j][0].z, bx[j][0].w);
        mma_f16(d, a[4], c[4], a[5], c[5], bx[j][1].x, bx[j][1].y);
        mma_f16(d, a[6], c[6], a[7], c[7], bx[j][1].z, bx[j][1].w);
        acc[j][mt][0] = fmaf(d[0], d0, acc[j][mt][0]);
        acc[j][mt][1] = fmaf(d[1], d0, acc[j][mt][1]);
        acc[j][mt][2] = fmaf(d[2], d1, acc[j][mt][2]);
        acc[j][mt][3] = fmaf(d[3], d1, acc[j][mt][3]);
      }
    }
  }
}

// Q3_K, one 16-column sub-block of one row: low code bits w (16 x 2 bits,
// columns 0..7 in the low half), high bits h16 (bit c = column c), sub-scale
// s.  Pair p (columns p, 8 + p) as f16 s (q - 4): the two low bits moved to
// bits 6..7 and the high bit to bit 8 of each half give 1024 + 64 q, and one
// fma with (s / 64, -20 s) (f16 numbers) leaves s (q - 4) exactly (|.| <= 252).
__device__ __forceinline__ void q3k_pairs(uint32_t w, uint32_t h16, int s, uint32_t (&a)[8]) {
  const uint32_t hs = __byte_perm(h16, 0u, 0x4140);  // columns 0..7 -> bits 0..7, 8..15 -> bits 16..23
  const __half sh = __int2half_rn(s);
  const __half2 m2 = __half2half2(__hmul(sh, __ushort_as_half(0x2400)));  // s / 64
  const __half2 c2 = __half2half2(__hmul(sh, __ushort_as_half(0xCD00)));  // -20 s
  const uint32_t mu = *reinterpret_cast<const uint32_t*>(&m2), cu = *reinterpret_cast<const uint32_t*>(&c2);
  const uint32_t lo[8] = {w << 6, w << 4, w << 2, w, w >> 2, w >> 4, w >> 6, w >> 8};
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t t = and_or(lo[p], 0x00C000C0u, kF16x2One024);
    a[p] = hfma2u(and_or(hs << (8 - p), 0x01000100u, t), mu, cu);
  }
}

// Q3_K (256-column blocks): thread tq takes sub-blocks tq, 4 + tq, 8 + tq,
// 12 + tq (word tq of each 16-byte piece of low bits; the high bits of
// sub-block j are half-word j of the 32 high-bit bytes); the sub-scales are
// in A, the block's d on the accumulators.  B rows in P order.
template <int NJ>
__device__ __forceinline__ void mma_q3k(const uint8_t* tile, int nb, int grp, const uint8_t* const (&bv)[NJ],
                                        int lane, float (&acc)[NJ][2][4]) {
  const int gq = lane >> 2, tq = lane & 3;
  const int b = grp;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    float dd[NJ][4];
#pragma unroll
    for (int j = 0; j < NJ; ++j) dd[j][0] = dd[j][1] = dd[j][2] = dd[j][3] = 0.f;
    const int r0 = 16 * mt + gq;
    const uint8_t* sc0 = tile + nb * 3072 + (b * 32 + r0) * 12;
    const uint8_t* sc1 = tile + nb * 3072 + (b * 32 + r0 + 8) * 12;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      const int sj = 4 * q + tq;  // this thread's sub-block
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(tile + (b * 4 + q) * 512 + r0 * 16 + 4 * tq);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(tile + (b * 4 + q) * 512 + (r0 + 8) * 16 + 4 * tq);
      const int ho = nb * 2048 + (b * 2 + (q >> 1)) * 512 + 4 * (2 * (q & 1) + (tq >> 1));
      const uint32_t h0 = (*reinterpret_cast<const uint32_t*>(tile + ho + r0 * 16) >> (16 * (tq & 1))) & 0xFFFFu;
      const uint32_t h1 = (*reinterpret_cast<const uint32_t*>(tile + ho + (r0 + 8) * 16) >> (16 * (tq & 1))) & 0xFFFFu;
      // 6-bit sub-scale sj: bits 6 sj .. of the 12 scale bytes (two bytes hold it)
      const int bit = 6 * sj, by = bit >> 3, sb = bit & 7;
      const int s0 = (int)(((uint32_t)sc0[by] | ((uint32_t)(by < 11 ? sc0[by + 1] : 0) << 8)) >> sb) & 63;
      const int s1 = (int)(((uint32_t)sc1[by] | ((uint32_t)(by < 11 ? sc1[by + 1] : 0) << 8)) >> sb) & 63;
      uint32_t a[8], c[8];
      q3k_pairs(w0, h0, s0, a);
      q3k_pairs(w1, h1, s1, c);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const uint4 x0 = *reinterpret_cast<const uint4*>(bv[j] + (b * 256 + 64 * q + 16 * tq) * 2);
        const uint4 x1 = *reinterpret_cast<const uint4*>(bv[j] + (b * 256 + 64 * q + 16 * tq + 8) * 2);
        mma_f16(dd[j], a[0], c[0], a[1], c[1], x0.x, x0.y);
        mma_f16(dd[j], a[2], c[2], a[3], c[3], x0.z, x0.w);
        mma_f16(dd[j], a[4], c[4], a[5], c[5], x1.x, x1.y);
        mma_f16(dd[j], a[6], c[6], a[7], c[7], x1.z, x1.w);
      }
    }
    const float d0 = __half2float(*reinterpret_cast<const __half*>(tile + nb * 3456 + (b * 32 + r0) * 2));
    const float d1 = __half2float(*reinterpret_cast<const __half*>(tile + nb * 3456 + (b * 32 + r0 + 8) * 2));
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      acc[j][mt][0] = fmaf(dd[j][0], d0, acc[j][mt][0]);
      acc[j][mt][1] = fmaf(dd[j][1], d0, acc[j][mt][1]);
      acc[j][mt][2] = fmaf(dd[j][2], d1, acc[j][mt][2]);
      acc[j][mt][3] = fmaf(dd[j][3], d1, acc[j][mt][3]);
    }
  }
}

// TQ1: five base-3 digits of the two code bytes in v = (1024 + B_lo, 1024 +
// B_hi) as f16x2 (t = digit - 1), in f16 arithmetic: one fma with (1/3 in
// f16, 682.5) rounds to 1024 + floor(B / 3) for every byte 0..242, a second
// leaves digit - 2048 (exact), an add of 2047 gives t; four rounds, then the
// last quotient is the fifth digit.
__device__ __forceinline__ void tq1_digits(uint32_t v, uint32_t (&a)[5]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const uint32_t q = hfma2u(v, 0x35553555u, 0x61556155u);    // 1024 + floor(B / 3)
    a[r] = hadd2u(hfma2u(q, 0xC200C200u, v), 0x67FF67FFu);    // (v - 3 q) + 2047
    v = q;
  }
  a[4] = hadd2u(v, 0xE401E401u);                              // - 1025
}

// TQ1 (256-column blocks): thread tq takes 13 code bytes of a row: word tq of
// each of the three 16-byte pieces (bytes 16 q + 4 tq .. + 3) and byte 48 + tq;
// bytes paired two by two in the halves of an f16x2 give five digit pairs
// each (the last byte alone), 35 pairs = 18 k16 steps (T order of the B rows).
template <int NJ>
__device__ __forceinline__ void mma_tq1(const uint8_t* tile, int nb, int grp, const uint8_t* const (&bv)[NJ],
                                        int lane, float (&acc)[NJ][2][4]) {
  const int gq = lane >> 2, tq = lane & 3;
  const int b = grp;
  const uint32_t tsel = 0x5450u + (uint32_t)tq;  // byte tq, then 0x64, 0x00, 0x64
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = 16 * mt + gq;
    float dd[NJ][4];
#pragma unroll
    for (int j = 0; j < NJ; ++j) dd[j][0] = dd[j][1] = dd[j][2] = dd[j][3] = 0.f;
    uint32_t w0[3], w1[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      w0[q] = *reinterpret_cast<const uint32_t*>(tile + (b * 3 + q) * 512 + r0 * 16 + 4 * tq);
      w1[q] = *reinterpret_cast<const uint32_t*>(tile + (b * 3 + q) * 512 + (r0 + 8) * 16 + 4 * tq);
    }
    const uint2 t0 = *reinterpret_cast<const uint2*>(tile + nb * 1536 + (b * 32 + r0) * 8);
    const uint2 t1 = *reinterpret_cast<const uint2*>(tile + nb * 1536 + (b * 32 + r0 + 8) * 8);
    uint32_t ca = 0, cc = 0;  // pair carried to the next step (rows r0, r0 + 8)
    uint4 bx[NJ];
#pragma unroll
    for (int beta = 0; beta < 7; ++beta) {
      uint32_t v0, v1;
      if (beta < 6) {
        const uint32_t sel = (beta & 1) ? 0x5352u : 0x5150u;
        v0 = __byte_perm(w0[beta >> 1], 0x64006400u, sel);
        v1 = __byte_perm(w1[beta >> 1], 0x64006400u, sel);
      } else {
        v0 = __byte_perm(t0.x, 0x64006400u, tsel);
        v1 = __byte_perm(t1.x, 0x64006400u, tsel);
      }
      uint32_t a[5], c[5];
      tq1_digits(v0, a);
      tq1_digits(v1, c);
      // pairs 5 beta .. 5 beta + 4; step s takes pairs 2s, 2s + 1
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const int pi = 5 * beta + k;
        if ((pi & 1) == 0) {
          ca = a[k];
          cc = c[k];
          if (pi == 34) {  // the last pair meets the zero pair 35 (step 17: the B loaded for step 16)
#pragma unroll
            for (int j = 0; j < NJ; ++j) mma_f16(dd[j], ca, cc, 0u, 0u, bx[j].z, bx[j].w);
          }
        } else {
          const int s = pi >> 1;
          if ((s & 1) == 0) {
#pragma unroll
            for (int j = 0; j < NJ; ++j)
              bx[j] = *reinterpret_cast<const uint4*>(bv[j] + (b * 288 + (s >> 1) * 32 + tq * 8) * 2);
#pragma unroll
            for (int j = 0; j < NJ; ++j) mma_f16(dd[j], ca, cc, a[k], c[k], bx[j].x, bx[j].y);
          } else {
#pragma unroll
            for (int j = 0; j < NJ; ++j) mma_f16(dd[j], ca, cc, a[k], c[k], bx[j].z, bx[j].w);
          }
        }
      }
    }
    const float d0 = __half2float(__ushort_as_half((unsigned short)(t0.y & 0xFFFFu)));
    const float d1 = __half2float(__ushort_as_half((unsigned short)(t1.y & 0xFFFFu)));
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      acc[j][mt][0] = fmaf(dd[j][0], d0, acc[j][mt][0]);
      acc[j][mt][1] = fmaf(dd[j][1], d0, acc[j][mt][1]);
      acc[j][mt][2] = fmaf(dd[j][2], d1, acc[j][mt][2]);
      acc[j][mt][3] = fmaf(dd[j][3], d1, acc[j][mt][3]);
    }
  }
}

// B column pointers of the thread and the group loop of the format, then the
// partial sums of each (row, weight row) into outv[r * 32 + weight row].
template <int NJ, int FS>
__device__ __forceinline__ void mma_group_nj(int R, int fmt, const uint8_t* tile, int kc, int nb, int grp,
                                             const uint8_t* act, int rstr, int lane, float* outv, bool hl) {
  const int gq = lane >> 2, tq = lane & 3;
  const int flen = f16_len(fmt, kc);
  const uint8_t* bv[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    // B column gq: x row gq (W1/W3); hi (gq even) or lo of row 4 j + gq / 2 (W2).
    // Columns past the item's rows repeat its last row: their results are dropped.
    const int r = hl ? min(4 * j + (gq >> 1), R - 1) : min(gq, R - 1);
    bv[j] = act + r * rstr + (hl && (gq & 1) ? 2 * flen + 64 : 0);
  }
  float acc[NJ][2][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) acc[j][mt][0] = acc[j][mt][1] = acc[j][mt][2] = acc[j][mt][3] = 0.f;
  // (an instance carries only its formats' loops)
  switch (fmt) {
    case BQE_FMT_MXFP4:
      if (fs_has<FS>(BQE_FMT_MXFP4)) mma_mxfp4<NJ>(tile, nb, grp, bv, lane, acc);
      break;
    case BQE_FMT_Q2_0:
      if (fs_has<FS>(BQE_FMT_Q2_0)) mma_q2_0<NJ>(tile, nb, grp, bv, lane, acc);
      break;
    case BQE_FMT_Q3_K:
      if (fs_has<FS>(BQE_FMT_Q3_K)) mma_q3k<NJ>(tile, nb, grp, bv, lane, acc);
      break;
    case BQE_FMT_TQ1:
      if (NJ == 1 && fs_has<FS>(BQE_FMT_TQ1))
        mma_tq1<1>(tile, nb, grp, reinterpret_cast<const uint8_t* const(&)[1]>(bv), lane,
                   reinterpret_cast<float(&)[1][2][4]>(acc));
      break;
    case BQE_FMT_NVFP4:
      if (fs_has<FS>(BQE_FMT_NVFP4)) mma_nvfp4<NJ>(tile, nb, grp, bv, lane, acc);
      break;
    default: break;
  }
  if (!hl) {
    // thread tq holds x rows 2 tq, 2 tq + 1
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = 2 * tq + (e & 1), wr = 16 * mt + gq + 8 * (e >> 1);
        if (r < R) outv[r * 32 + wr] = acc[0][mt][e];
      }
  } else {
    // thread tq holds hi and lo of row 4 j + tq; the group's 2^-s removed here
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int r = 4 * j + tq;
      if (r < R) {
        const float us = reinterpret_cast<const float*>(act + r * rstr + 4 * flen + 64)[grp];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          outv[r * 32 + 16 * mt + gq] = (acc[j][mt][0] + acc[j][mt][1]) * us;
          outv[r * 32 + 16 * mt + gq + 8] = (acc[j][mt][2] + acc[j][mt][3]) * us;
        }
      }
    }
  }
}

// The loop of one task: R <= 8 rows (RC == 1: one row).
template <int RC, int FS>
__device__ __forceinline__ void consume_mma(int R, int fmt, const uint8_t* tile, int kc, int nb, int grp,
                                            const uint8_t* act, int lane, float* outv, int amode) {
  const int rstr = act_row_stride(amode, fmt, kc);
  const bool hl = amode == kActH16;
  if (fs_has<FS>(BQE_FMT_MXFP4) && fmt == BQE_FMT_MXFP4 && (RC == 1 || R == 1)) {
    if (!hl)
      mma_mxfp4_r1(tile, nb, grp, act, lane, outv);
    else
      mma_mxfp4_r1_hl(tile, nb, grp, act, f16_len(fmt, kc), lane, outv);
  } else if (RC == 1 || !hl || R <= 4) {
    mma_group_nj<1, FS>(RC == 1 ? 1 : R, fmt, tile, kc, nb, grp, act, rstr, lane, outv, hl);
  } else if (fs_has<FS>(BQE_FMT_TQ1) && fmt == BQE_FMT_TQ1) {
    // W2 rows 0..3, then 4..: ternary codes decoded twice (two MMAs per step
    // would not fit this kernel's register budget)
    mma_group_nj<1, FS>(4, fmt, tile, kc, nb, grp, act, rstr, lane, outv, true);
    mma_group_nj<1, FS>(R - 4, fmt, tile, kc, nb, grp, act + 4 * rstr, rstr, lane, outv + 4 * 32, true);
  } else {
    mma_group_nj<2, FS>(R, fmt, tile, kc, nb, grp, act, rstr, lane, outv, hl);
  }
}

}  // namespace bqe
