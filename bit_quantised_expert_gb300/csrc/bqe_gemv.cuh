// bqe_gemv.cuh — the per-format dequant-GEMV group kernels of the decode
// layer: one lane = one weight row, one 256-column group of a tile in shared
// memory, R <= 4 activation rows at a time, fp32 accumulation.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>

#include "bqe_internal.cuh"

namespace bqe {

// ---------------------------------------------------------------------------
// per-format group kernels: one lane = one weight row, 256 columns, R rows of
// activations; acc[r] accumulates the row's dot products (two halves kept in
// a float2 for the packed FMA, added at the end).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

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

// a0 += lo(w) * lo(x), a1 += hi(w) * hi(x): f16 inputs, exact f32 products,
// f32 accumulation (mixed-precision FMA of sm_100+).
__device__ __forceinline__ void fma_f16x2_f32(uint32_t w, uint32_t x, float& a0, float& a1) {
  asm("{ .reg .f16 wl, wh, xl, xh; mov.b32 {wl, wh}, %2; mov.b32 {xl, xh}, %3;\n"
      "  fma.rn.f32.f16 %0, wl, xl, %0; fma.rn.f32.f16 %1, wh, xh, %1; }"
      : "+f"(a0), "+f"(a1)
      : "r"(w), "r"(x));
}

template <int R>
__device__ __forceinline__ void group_mxfp4(const uint8_t* tile, int nb, int grp, const float* act, int kc, int lane,
                                            float2 (&acc)[R]) {
#pragma unroll 2
  for (int bi = 0; bi < 8; ++bi) {
    const int b = grp * 8 + bi;
    const uint4 c4 = *reinterpret_cast<const uint4*>(tile + b * 512 + lane * 16);
    const float sc = ue8m0_f32(tile[nb * 512 + b * 32 + lane]);
    float2 bs[R][2];  // two independent chains per row
#pragma unroll
    for (int r = 0; r < R; ++r) bs[r][0] = bs[r][1] = f2(0.f, 0.f);
    const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t h0, h1, h2, h3;
      e2m1x8_to_f16x2(wd[w], h0, h1, h2, h3);
      const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
      const float2 v1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
      const float2 v2 = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      const float2 v3 = __half22float2(*reinterpret_cast<const __half2*>(&h3));
      const int k = grp * 256 + bi * 32 + w * 8;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4 xa = *reinterpret_cast<const float4*>(act + r * kc + k);
        const float4 xb = *reinterpret_cast<const float4*>(act + r * kc + k + 4);
        bs[r][0] = __ffma2_rn(v0, f2(xa.x, xa.y), bs[r][0]);
        bs[r][1] = __ffma2_rn(v1, f2(xa.z, xa.w), bs[r][1]);
        bs[r][0] = __ffma2_rn(v2, f2(xb.x, xb.y), bs[r][0]);
        bs[r][1] = __ffma2_rn(v3, f2(xb.z, xb.w), bs[r][1]);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
      acc[r] = __ffma2_rn(f2(bs[r][0].x + bs[r][1].x, bs[r][0].y + bs[r][1].y), f2(sc, sc), acc[r]);
  }
}

// MXFP4 group with f16 activations (act_h: R rows x kc halves, scaled by a
// power of two per row; the epilogue removes the scale).  Four accumulator
// chains per row.
template <int R>
__device__ __forceinline__ void group_mxfp4_h(const uint8_t* tile, int nb, int grp, const uint16_t* act_h, int kc,
                                              int lane, float2 (&acc)[R]) {
#pragma unroll 1
  for (int bi = 0; bi < 8; ++bi) {
    const int b = grp * 8 + bi;
    const uint4 c4 = *reinterpret_cast<const uint4*>(tile + b * 512 + lane * 16);
    const float sc = ue8m0_f32(tile[nb * 512 + b * 32 + lane]);
    float a[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) a[r][0] = a[r][1] = a[r][2] = a[r][3] = 0.f;
    const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t h0, h1, h2, h3;
      e2m1x8_to_f16x2(wd[w], h0, h1, h2, h3);
      const int k = grp * 256 + bi * 32 + w * 8;
      const int ch = (w & 1) * 2;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint4 xv = *reinterpret_cast<const uint4*>(act_h + r * kc + k);
        fma_f16x2_f32(h0, xv.x, a[r][ch], a[r][ch + 1]);
        fma_f16x2_f32(h1, xv.y, a[r][ch], a[r][ch + 1]);
        fma_f16x2_f32(h2, xv.z, a[r][ch], a[r][ch + 1]);
        fma_f16x2_f32(h3, xv.w, a[r][ch], a[r][ch + 1]);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r].x = fmaf((a[r][0] + a[r][1]) + (a[r][2] + a[r][3]), sc, acc[r].x);
  }
}

// ----------------------------------------------------------------------------
// Integer paths for the fp16-scaled formats (Q2_0, Q3_K, TQ1).  The layer
// input x of a row is staged as X_hi + X_lo / 128 with X_hi = rint(x 2^si)
// (int16, |X_hi| <= 2^14) and X_lo the int8 rounding of the remainder (so x
// is held to about 2^-21 of the row's largest value), each in a per-format
// order, plus the sums of X_hi and of X_lo over every 16 columns.  Each
// weight's integer code sits in a byte lane: dp2a adds two int16 x int8
// products and dp4a four int8 x int8 products per instruction, in exact int32
// arithmetic.  The block's offset (2q - 3, q - 4, t - 1) is applied once per
// block through the column sums, the block scale (and Q3_K sub-scale) once per
// block in fp32.
//
// Order of X ("Q order", every 16 columns): X_hi word 2k = (x_k, x_{k+4}),
// word 2k + 1 = (x_{k+8}, x_{k+12}); X_lo word k = (x_k, x_{k+4}, x_{k+8},
// x_{k+12}), k = 0..3, so that the byte lanes of (codes >> 2k) & 0x03030303
// meet their x.  Order for TQ1 ("T order", every 256 columns = 13 runs of 20
// and padding): in run m, X_hi word 2r = (x_{20m+r}, x_{20m+5+r}), word 2r + 1
// = (x_{20m+10+r}, x_{20m+15+r}); X_lo word r = (x_{20m+r}, x_{20m+5+r},
// x_{20m+10+r}, x_{20m+15+r}), r = 0..4 (slots past column 255 are zero).
// ----------------------------------------------------------------------------
constexpr int kTOrderBlock = 528;   // bytes of one 256-column block of X_hi in T order
constexpr int kTOrderBlockL = 272;  // ... of X_lo

__host__ __device__ inline int act_x_bytes(int fmt, int kc) { return (int)int_rec_hi_bytes(fmt == BQE_FMT_TQ1, kc); }
__host__ __device__ inline int act_xl_bytes(int fmt, int kc) { return (int)int_rec_lo_bytes(fmt == BQE_FMT_TQ1, kc); }

// Pointers into one staged row of the integer mode: [X_hi | X_lo | sums of
// X_hi | sums of X_lo | 2^-si of each 256 columns (4 slots)].
struct IntRow {
  const uint8_t* xh;  // X_hi of the 256-column group
  const uint8_t* xl;  // X_lo of the group
  const int* sh;      // 16 sums of X_hi
  const int* sl;      // 16 sums of X_lo
  float sc;           // 2^-si of the group: the sums below are in units of it
};
__device__ __forceinline__ IntRow int_row(const uint8_t* act, int r, int rowb, int fmt, int kc, int grp) {
  const int xb = act_x_bytes(fmt, kc), xbl = act_xl_bytes(fmt, kc);
  const uint8_t* base = act + r * rowb;
  IntRow t;
  t.xh = base + grp * (fmt == BQE_FMT_TQ1 ? kTOrderBlock : 512);
  t.xl = base + xb + grp * (fmt == BQE_FMT_TQ1 ? kTOrderBlockL : 256);
  t.sh = reinterpret_cast<const int*>(base + xb + xbl) + grp * 16;
  t.sl = reinterpret_cast<const int*>(base + xb + xbl + kc / 4) + grp * 16;
  t.sc = reinterpret_cast<const float*>(base + xb + xbl + kc / 2)[grp];
  return t;
}
// a + b / 128 in fp32 (both exact integers below 2^24 in magnitude)
__device__ __forceinline__ float hi_lo(int a, int b) { return fmaf((float)b, 0.0078125f, (float)a); }

template <int R>
__device__ __forceinline__ void group_q2_0_i(const uint8_t* tile, int nb, int grp, const uint8_t* act, int rowb,
                                             int kc, int lane, float2 (&acc)[R]) {
  IntRow row[R];
#pragma unroll
  for (int r = 0; r < R; ++r) row[r] = int_row(act, r, rowb, BQE_FMT_Q2_0, kc, grp);
#pragma unroll 1
  for (int bi = 0; bi < 4; ++bi) {
    const int b = grp * 4 + bi;
    const uint4 c4 = *reinterpret_cast<const uint4*>(tile + b * 512 + lane * 16);
    const float d = __half2float(*reinterpret_cast<const __half*>(tile + nb * 512 + (b * 32 + lane) * 2));
    const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
    int ih[R], il[R];
#pragma unroll
    for (int r = 0; r < R; ++r) ih[r] = il[r] = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {  // 16 weights: 16-column group 4 bi + w of this 256-column group
      int B[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) B[k] = (int)((wd[w] >> (2 * k)) & 0x03030303u);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int4* xp = reinterpret_cast<const int4*>(row[r].xh + (bi * 4 + w) * 32);
        const int4 xa = xp[0], xb = xp[1];
        const int4 xl = *reinterpret_cast<const int4*>(row[r].xl + (bi * 4 + w) * 16);
        const int X[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const int XL[4] = {xl.x, xl.y, xl.z, xl.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ih[r] = __dp2a_lo(X[2 * k], B[k], ih[r]);
          ih[r] = __dp2a_hi(X[2 * k + 1], B[k], ih[r]);
          il[r] = __dp4a(XL[k], B[k], il[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int4 sh = *reinterpret_cast<const int4*>(row[r].sh + bi * 4);
      const int4 sl = *reinterpret_cast<const int4*>(row[r].sl + bi * 4);
      const int Sh = (sh.x + sh.y) + (sh.z + sh.w), Sl = (sl.x + sl.y) + (sl.z + sl.w);
      // sum of (2q - 3) X, exact in each part
      acc[r].x = fmaf(d * row[r].sc, hi_lo(2 * ih[r] - 3 * Sh, 2 * il[r] - 3 * Sl), acc[r].x);
    }
  }
}

template <int R>
__device__ __forceinline__ void group_q3k_i(const uint8_t* tile, int nb, int grp, const uint8_t* act, int rowb,
                                            int kc, int lane, float2 (&acc)[R]) {
  IntRow row[R];
#pragma unroll
  for (int r = 0; r < R; ++r) row[r] = int_row(act, r, rowb, BQE_FMT_Q3_K, kc, grp);
  const int b = grp;
  uint32_t lo[16], hi[8], sc[3];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + (b * 4 + q) * 512 + lane * 16);
    lo[4 * q] = v.x; lo[4 * q + 1] = v.y; lo[4 * q + 2] = v.z; lo[4 * q + 3] = v.w;
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + nb * 2048 + (b * 2 + q) * 512 + lane * 16);
    hi[4 * q] = v.x; hi[4 * q + 1] = v.y; hi[4 * q + 2] = v.z; hi[4 * q + 3] = v.w;
  }
  const uint8_t* scp = tile + nb * 3072 + (b * 32 + lane) * 12;
#pragma unroll
  for (int i = 0; i < 3; ++i) sc[i] = *reinterpret_cast<const uint32_t*>(scp + 4 * i);
  const float d = __half2float(*reinterpret_cast<const __half*>(tile + nb * 3456 + (b * 32 + lane) * 2));
  int bh[R], bl[R];
#pragma unroll
  for (int r = 0; r < R; ++r) bh[r] = bl[r] = 0;
#pragma unroll
  for (int sj = 0; sj < 16; ++sj) {
    const int bit = 6 * sj;
    const uint64_t two = ((uint64_t)sc[bit >> 5]) | (((bit >> 5) < 2 ? (uint64_t)sc[(bit >> 5) + 1] : 0ull) << 32);
    const int s = (int)((uint32_t)(two >> (bit & 31)) & 63u);
    const uint32_t low = lo[sj];
    const uint32_t h16 = (hi[sj >> 1] >> ((sj & 1) * 16)) & 0xFFFFu;  // high bits of weights 16 sj ..
    int B[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // byte i: q of weight k + 4i = low 2 bits | 4 * high bit (the high bit placed by a byte
      // permute: selector nibble i is 4 when the bit is set, picking 0x04, else 0 picking 0x00)
      const uint32_t sel = ((h16 >> k) << 2) & 0x4444u;
      B[k] = (int)(((low >> (2 * k)) & 0x03030303u) | __byte_perm(0u, 0x04040404u, sel));
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int4* xp = reinterpret_cast<const int4*>(row[r].xh + sj * 32);
      const int4 xa = xp[0], xb = xp[1];
      const int4 xl = *reinterpret_cast<const int4*>(row[r].xl + sj * 16);
      const int X[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      const int XL[4] = {xl.x, xl.y, xl.z, xl.w};
      int th = 0, tl = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        th = __dp2a_lo(X[2 * k], B[k], th);
        th = __dp2a_hi(X[2 * k + 1], B[k], th);
        tl = __dp4a(XL[k], B[k], tl);
      }
      // s_j * sum of (q - 4) X per part; |block sums| < 2^31
      bh[r] += s * (th - 4 * row[r].sh[sj]);
      bl[r] += s * (tl - 4 * row[r].sl[sj]);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r].x = fmaf(d * row[r].sc, hi_lo(bh[r], bl[r]), acc[r].x);
}

// One 32-bit word of a TQ1 row (bytes 4m .. 4m + 3: run m of 20 columns):
// its five base-3 digits per byte, met with the T-order X of run m.
template <int R>
__device__ __forceinline__ void tq1_run(uint32_t wv, int m, const IntRow (&row)[R], int (&ih)[R], int (&il)[R]) {
  // bytes 4m, 4m+2 in the 16-bit lanes of ve; 4m+1, 4m+3 in vo
  uint32_t ve = wv & 0x00FF00FFu, vo = (wv >> 8) & 0x00FF00FFu;
  int B[5];
#pragma unroll
  for (int rd = 0; rd < 5; ++rd) {
    // digit rd of the four bytes: v / 3 per 16-bit lane ((v * 171) >> 9 for v <= 255)
    const uint32_t qe = ((ve * 171u) >> 9) & 0x007F007Fu, qo = ((vo * 171u) >> 9) & 0x007F007Fu;
    const uint32_t de = ve - 3u * qe, dq = vo - 3u * qo;
    ve = qe;
    vo = qo;
    B[rd] = (int)__byte_perm(de, dq, 0x6240);  // digits of bytes 4m, 4m+1, 4m+2, 4m+3
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int2* xp = reinterpret_cast<const int2*>(row[r].xh + m * 40);
    const int* xl = reinterpret_cast<const int*>(row[r].xl + m * 20);
#pragma unroll
    for (int rd = 0; rd < 5; ++rd) {
      const int2 v = xp[rd];
      ih[r] = __dp2a_lo(v.x, B[rd], ih[r]);
      ih[r] = __dp2a_hi(v.y, B[rd], ih[r]);
      il[r] = __dp4a(xl[rd], B[rd], il[r]);
    }
  }
}

template <int R>
__device__ __forceinline__ void group_tq1_i(const uint8_t* tile, int nb, int grp, const uint8_t* act, int rowb,
                                            int kc, int lane, float2 (&acc)[R]) {
  IntRow row[R];
#pragma unroll
  for (int r = 0; r < R; ++r) row[r] = int_row(act, r, rowb, BQE_FMT_TQ1, kc, grp);
  const int b = grp;
  const uint2 tail = *reinterpret_cast<const uint2*>(tile + nb * 1536 + (b * 32 + lane) * 8);
  const float d = __half2float(__ushort_as_half((unsigned short)(tail.y & 0xFFFFu)));
  int ih[R], il[R];
#pragma unroll
  for (int r = 0; r < R; ++r) ih[r] = il[r] = 0;
  // words 0..11 (bytes 0..47) four at a time, then word 12 (bytes 48..51;
  // byte 51 <= 2, so its higher digits are 0)
#pragma unroll 1
  for (int q = 0; q < 3; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + (b * 3 + q) * 512 + lane * 16);
    tq1_run<R>(v.x, 4 * q, row, ih, il);
    tq1_run<R>(v.y, 4 * q + 1, row, ih, il);
    tq1_run<R>(v.z, 4 * q + 2, row, ih, il);
    tq1_run<R>(v.w, 4 * q + 3, row, ih, il);
  }
  tq1_run<R>(tail.x, 12, row, ih, il);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    int Sh = 0, Sl = 0;
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const int4 a = *reinterpret_cast<const int4*>(row[r].sh + i);
      const int4 c = *reinterpret_cast<const int4*>(row[r].sl + i);
      Sh += (a.x + a.y) + (a.z + a.w);
      Sl += (c.x + c.y) + (c.z + c.w);
    }
    acc[r].x = fmaf(d * row[r].sc, hi_lo(ih[r] - Sh, il[r] - Sl), acc[r].x);  // sum of (t - 1) X, t the digit
  }
}

// Activation modes of an item: 0 fp32 rows, 1 f16 rows (x 2^s, MXFP4 W1/W3),
// 2 integer rows (X in the format's order, then the 16-column sums).
enum { kActF32 = 0, kActF16 = 1, kActInt = 2 };

// Mode of the activations of an item: integer for the fp16-scaled formats
// (both phases); for MXFP4 f16 in W1/W3 and fp32 in W2 (h stays fp32).
__host__ __device__ inline int act_mode(int phase, int fmt) {
  if (fmt != BQE_FMT_MXFP4) return kActInt;
  return phase == 0 ? kActF16 : kActF32;
}

__host__ __device__ inline int act_row_bytes(int amode, int fmt, int kc) {
  return amode == kActF32 ? kc * 4 : amode == kActF16 ? kc * 2 : (int)int_rec_bytes(fmt == BQE_FMT_TQ1, kc);
}

// nb: format blocks per tile row (kc / block width), from the stage header
template <int R>
__device__ __forceinline__ void consume_group_R(int fmt, const uint8_t* tile, int kc, int nb, int grp,
                                                const uint8_t* act, int lane, float* outv /* [r * 32 + lane] */,
                                                int amode) {
  float2 acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = f2(0.f, 0.f);
  if (amode == kActInt) {
    const int rowb = act_row_bytes(kActInt, fmt, kc);
    switch (fmt) {
      case BQE_FMT_Q2_0: group_q2_0_i<R>(tile, nb, grp, act, rowb, kc, lane, acc); break;
      case BQE_FMT_TQ1: group_tq1_i<R>(tile, nb, grp, act, rowb, kc, lane, acc); break;
      case BQE_FMT_Q3_K: group_q3k_i<R>(tile, nb, grp, act, rowb, kc, lane, acc); break;
    }
  } else if (amode == kActF16) {
    group_mxfp4_h<R>(tile, nb, grp, reinterpret_cast<const uint16_t*>(act), kc, lane, acc);
  } else {
    group_mxfp4<R>(tile, nb, grp, reinterpret_cast<const float*>(act), kc, lane, acc);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) outv[r * 32 + lane] = acc[r].x + acc[r].y;
}

template <int RC>
__device__ __forceinline__ void consume_group(int R, int fmt, const uint8_t* tile, int kc, int nb, int grp,
                                              const uint8_t* act, int lane, float* outv, int amode) {
  if (RC == 1 || R == 1) {
    consume_group_R<1>(fmt, tile, kc, nb, grp, act, lane, outv, amode);
    return;
  }
  if (RC == 2) {
    consume_group_R<(RC >= 2 ? 2 : 1)>(fmt, tile, kc, nb, grp, act, lane, outv, amode);
    return;
  }
  switch (R) {
    case 2: consume_group_R<2>(fmt, tile, kc, nb, grp, act, lane, outv, amode); break;
    case 3: consume_group_R<(RC >= 3 ? 3 : 1)>(fmt, tile, kc, nb, grp, act, lane, outv, amode); break;
    case 4: consume_group_R<(RC >= 4 ? 4 : 1)>(fmt, tile, kc, nb, grp, act, lane, outv, amode); break;
  }
}

// All R rows of one stage, RC (1 or kRowChunk) rows at a time (the weights of
// the group are decoded again for each further chunk).  A kernel instance for
// one-row calls (RC = 1) carries only the one-row inner loops, which keeps its
// code small and its register count low.
template <int RC>
__device__ __forceinline__ void consume_rows(int R, int fmt, const uint8_t* tile, int kc, int nb, int grp,
                                             const uint8_t* act, int lane, float* outv, int amode) {
  static_assert(RC == 1 || RC == 2 || RC == kRowChunk, "row chunk");
  const size_t row_bytes = (size_t)act_row_bytes(amode, fmt, kc);
  for (int r0 = 0; r0 < R; r0 += RC) {
    const int n = R - r0 < RC ? R - r0 : RC;
    consume_group<RC>(n, fmt, tile, kc, nb, grp, act + r0 * row_bytes, lane, outv + r0 * 32, amode);
  }
}

__device__ __forceinline__ float silu_f(float t) { return t / (1.0f + expf(-t)); }


}  // namespace bqe
