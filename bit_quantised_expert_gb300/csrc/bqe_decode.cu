// bqe_decode.cu — the decode expert kernels: fused dequant-GEMV over the
// distinct experts of one call (M <= 8 token rows).
//
// The layer's cost is the expert bytes each token streams (field report,
// section 2: "single-stream speed is set only by how many bytes each token
// moves").  So every byte of every selected expert is read from HBM exactly
// once per call and applied to all rows that chose the expert (section 4.2:
// one transfer serves every token of a batch; the Strata-DS post's batched
// draft verify puts up to 1 + drafts rows through one layer).
//
//   phase A  for each distinct expert u and each row i of W1/W3:
//            g = W1[i,:] x_r, v = W3[i,:] x_r for the rows r that chose u,
//            h[u, r, i] = silu(g) * v
//   phase B  for each row n of W2:  y[u, r, n] = W2_u[n,:] h[u, r, :]
//            out[m, n] = y[shared, m, n] + sum_j w[m, j] y[idx_j, r(m,j), n]
//
// Both phases run the same engine: a persistent grid with one CTA per SM;
// warp 0 streams work items (a tile of 32 weight rows x one K chunk of one
// or two matrices, plus the matching activation chunk) into a ring of
// shared-memory stages with cp.async.bulk and mbarrier completion; the
// consumer warps each take one 256-column group of one 32-row panel, one
// lane per weight row, dequantise in registers and accumulate in fp32 with
// packed f32x2 FMAs.  Partial sums over the groups of a chunk are reduced
// in shared memory; partial sums over chunks meet in the workspace, where
// the last-arriving CTA (an arrival counter, no waiting) finishes the row
// in a fixed order, so results are deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>

#include "bqe_internal.cuh"

namespace bqe {


struct StageHdr {
  uint64_t addr;  // slot base
  int u, p0, c, fmt, R, pad;
};

__host__ __device__ inline int phase_mats(int phase) { return phase == 0 ? 2 : 1; }

__host__ __device__ inline int phase_panels(const Geo& g, int phase) { return phase == 0 ? g.PA : g.PB; }

__host__ __device__ inline uint32_t stage_slot_bytes(const Geo& g, int phase) {
  return stage_bytes_for(phase_mats(phase), phase_panels(g, phase), phase == 0 ? g.kcA : g.kcB, g.M);
}

__host__ __device__ inline int phase_warps(const Geo& g, int phase) {
  return phase_mats(phase) * phase_panels(g, phase) * (phase == 0 ? g.GA : g.GB);
}

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

// 2-bit code q -> float (2q - 3), exactly, via a float whose fraction holds q:
// 1 + q/4 has the bit pattern 0x3F800000 | q << 21, and 8 (1 + q/4) - 11 = 2q - 3.
__device__ __forceinline__ float q2_val(uint32_t word, int j) {
  const float f = __uint_as_float(0x3F800000u | (((word >> (2 * j)) & 3u) << 21));
  return fmaf(8.0f, f, -11.0f);
}

template <int R>
__device__ __forceinline__ void group_q2_0(const uint8_t* tile, int nb, int grp, const float* act, int kc, int lane,
                                           float2 (&acc)[R]) {
#pragma unroll 1
  for (int bi = 0; bi < 4; ++bi) {
    const int b = grp * 4 + bi;
    const uint4 c4 = *reinterpret_cast<const uint4*>(tile + b * 512 + lane * 16);
    const float d = __half2float(*reinterpret_cast<const __half*>(tile + nb * 512 + (b * 32 + lane) * 2));
    float2 bs[R];
#pragma unroll
    for (int r = 0; r < R; ++r) bs[r] = f2(0.f, 0.f);
    const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
#pragma unroll
      for (int j = 0; j < 16; j += 4) {
        const float2 v0 = f2(q2_val(wd[w], j), q2_val(wd[w], j + 1));
        const float2 v1 = f2(q2_val(wd[w], j + 2), q2_val(wd[w], j + 3));
        const int k = grp * 256 + bi * 64 + w * 16 + j;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 xa = *reinterpret_cast<const float4*>(act + r * kc + k);
          bs[r] = __ffma2_rn(v0, f2(xa.x, xa.y), bs[r]);
          bs[r] = __ffma2_rn(v1, f2(xa.z, xa.w), bs[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = __ffma2_rn(bs[r], f2(d, d), acc[r]);
  }
}

// Five ternary digits of one byte (least significant first) -> t = digit - 1.
__device__ __forceinline__ void tq1_byte(uint32_t v, float (&t)[5]) {
#pragma unroll
  for (int r = 0; r < 5; ++r) {
    const uint32_t q = (v * 171u) >> 9;  // v / 3 for v <= 255
    t[r] = (float)((int)(v - 3u * q) - 1);
    v = q;
  }
}

template <int R>
__device__ __forceinline__ void group_tq1(const uint8_t* tile, int nb, int grp, const float* act, int kc, int lane,
                                          float2 (&acc)[R]) {
  const int b = grp;
  float2 bs[R];
#pragma unroll
  for (int r = 0; r < R; ++r) bs[r] = f2(0.f, 0.f);
  // bytes 0..47: three 16-byte pieces = 12 words = 12 x 4 bytes = 12 x 20 weights
#pragma unroll 1
  for (int q = 0; q < 3; ++q) {
    const uint4 c4 = *reinterpret_cast<const uint4*>(tile + (b * 3 + q) * 512 + lane * 16);
    const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float t[20];
#pragma unroll
      for (int by = 0; by < 4; ++by) {
        float tt[5];
        tq1_byte((wd[w] >> (8 * by)) & 0xFF, tt);
#pragma unroll
        for (int r5 = 0; r5 < 5; ++r5) t[by * 5 + r5] = tt[r5];
      }
      const int k = grp * 256 + (q * 16 + w * 4) * 5;
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int i4 = 0; i4 < 5; ++i4) {
          const float4 xa = *reinterpret_cast<const float4*>(act + r * kc + k + 4 * i4);
          bs[r] = __ffma2_rn(f2(t[4 * i4], t[4 * i4 + 1]), f2(xa.x, xa.y), bs[r]);
          bs[r] = __ffma2_rn(f2(t[4 * i4 + 2], t[4 * i4 + 3]), f2(xa.z, xa.w), bs[r]);
        }
      }
    }
  }
  // bytes 48..55: three digit bytes (weights 240..254), byte 51 (weight 255), d
  const uint2 tail = *reinterpret_cast<const uint2*>(tile + nb * 1536 + (b * 32 + lane) * 8);
  float t[16];
#pragma unroll
  for (int by = 0; by < 3; ++by) {
    float tt[5];
    tq1_byte((tail.x >> (8 * by)) & 0xFF, tt);
#pragma unroll
    for (int r5 = 0; r5 < 5; ++r5) t[by * 5 + r5] = tt[r5];
  }
  t[15] = (float)((int)((tail.x >> 24) % 3u) - 1);
  const float d = __half2float(__ushort_as_half((unsigned short)(tail.y & 0xFFFF)));
  const int k = grp * 256 + 240;
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      const float4 xa = *reinterpret_cast<const float4*>(act + r * kc + k + 4 * i4);
      bs[r] = __ffma2_rn(f2(t[4 * i4], t[4 * i4 + 1]), f2(xa.x, xa.y), bs[r]);
      bs[r] = __ffma2_rn(f2(t[4 * i4 + 2], t[4 * i4 + 3]), f2(xa.z, xa.w), bs[r]);
    }
    acc[r] = __ffma2_rn(bs[r], f2(d, d), acc[r]);
  }
}

template <int R>
__device__ __forceinline__ void group_q3k(const uint8_t* tile, int nb, int grp, const float* act, int kc, int lane,
                                          float2 (&acc)[R]) {
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
  float2 bsum[R];
#pragma unroll
  for (int r = 0; r < R; ++r) bsum[r] = f2(0.f, 0.f);
#pragma unroll 1
  for (int sj = 0; sj < 16; ++sj) {
    // 6-bit sub-scale sj at bits 6 sj .. 6 sj + 5 of the 96-bit little-endian string
    const int bit = 6 * sj;
    const uint64_t two = ((uint64_t)sc[bit >> 5]) | (((bit >> 5) < 2 ? (uint64_t)sc[(bit >> 5) + 1] : 0ull) << 32);
    const float s = (float)((uint32_t)(two >> (bit & 31)) & 63u);
    const uint32_t low = lo[sj];          // weights 16 sj .. 16 sj + 15: 2 bits each
    const uint32_t high = hi[sj >> 1] >> ((sj & 1) * 16);  // 16 high bits
    float2 ss[R];
#pragma unroll
    for (int r = 0; r < R; ++r) ss[r] = f2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      float v[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int qv = (int)(((low >> (2 * (j + jj))) & 3u) | (((high >> (j + jj)) & 1u) << 2));
        v[jj] = (float)(qv - 4);
      }
      const int k = grp * 256 + sj * 16 + j;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4 xa = *reinterpret_cast<const float4*>(act + r * kc + k);
        ss[r] = __ffma2_rn(f2(v[0], v[1]), f2(xa.x, xa.y), ss[r]);
        ss[r] = __ffma2_rn(f2(v[2], v[3]), f2(xa.z, xa.w), ss[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) bsum[r] = __ffma2_rn(ss[r], f2(s, s), bsum[r]);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = __ffma2_rn(bsum[r], f2(d, d), acc[r]);
}

template <int R>
__device__ __forceinline__ void consume_group_R(int fmt, const uint8_t* tile, int kc, int grp, const float* act,
                                                int lane, float* outv /* [r * 32 + lane] */, bool half_act) {
  float2 acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = f2(0.f, 0.f);
  const int nb = kc / fmt_bw(fmt);
  switch (fmt) {
    case BQE_FMT_MXFP4:
      if (half_act)
        group_mxfp4_h<R>(tile, nb, grp, reinterpret_cast<const uint16_t*>(act), kc, lane, acc);
      else
        group_mxfp4<R>(tile, nb, grp, act, kc, lane, acc);
      break;
    case BQE_FMT_Q2_0: group_q2_0<R>(tile, nb, grp, act, kc, lane, acc); break;
    case BQE_FMT_TQ1: group_tq1<R>(tile, nb, grp, act, kc, lane, acc); break;
    case BQE_FMT_Q3_K: group_q3k<R>(tile, nb, grp, act, kc, lane, acc); break;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) outv[r * 32 + lane] = acc[r].x + acc[r].y;
}

__device__ __forceinline__ void consume_group(int R, int fmt, const uint8_t* tile, int kc, int grp, const float* act,
                                              int lane, float* outv, bool half_act) {
  switch (R) {
    case 1: consume_group_R<1>(fmt, tile, kc, grp, act, lane, outv, half_act); break;
    case 2: consume_group_R<2>(fmt, tile, kc, grp, act, lane, outv, half_act); break;
    case 3: consume_group_R<3>(fmt, tile, kc, grp, act, lane, outv, half_act); break;
    case 4: consume_group_R<4>(fmt, tile, kc, grp, act, lane, outv, half_act); break;
  }
}

// All R rows of one stage, kRowChunk rows at a time (the weights of the group
// are decoded again for each further chunk; only rows 5..8 of a call pay it).
__device__ __forceinline__ void consume_rows(int R, int fmt, const uint8_t* tile, int kc, int grp, const uint8_t* act,
                                             int lane, float* outv, bool half_act) {
  const size_t row_bytes = (size_t)kc * (half_act ? 2 : 4);
  for (int r0 = 0; r0 < R; r0 += kRowChunk) {
    const int n = R - r0 < kRowChunk ? R - r0 : kRowChunk;
    consume_group(n, fmt, tile, kc, grp, reinterpret_cast<const float*>(act + r0 * row_bytes), lane, outv + r0 * 32,
                  half_act);
  }
}

__device__ __forceinline__ float silu_f(float t) { return t / (1.0f + expf(-t)); }

__device__ __forceinline__ long long clk() { return clock64(); }
// diagnostic counters: 0 producer waiting for a free stage, 1 producer issuing,
// 2 consumer (warp 1) waiting for a stage, 3 consumer waiting for a reduction
// buffer, 4 consumer computing, 5 epilogue waiting, 6 epilogue working,
// 7 whole CTA
__device__ __forceinline__ void dbg_add(const ExpParams& P, int phase, int slot, long long v) {
  if (P.diag && blockIdx.x < kDbgMaxCtas)
    atomicAdd((unsigned long long*)(P.ws + P.L.dbg) + ((size_t)phase * kDbgMaxCtas + blockIdx.x) * kDbgSlots + slot,
              (unsigned long long)v);
}

// ---------------------------------------------------------------------------
// the engine
// ---------------------------------------------------------------------------
// Shared-memory map of the engine (offsets in bytes):
//   0      StageHdr[16]               ring stage headers
//   512    full[16], empty[16]        ring mbarriers
//   768    rfull[kRed], rempty[kRed]  reduction-buffer mbarriers
//   896    abort flag
//   1024   RedMeta[kRed]
//   2048   red[kRed][NW][M][32] floats (consumer partial sums for the epilogue)
//   ...    ring of nstages slots
struct RedMeta {
  int u, p0, c, R;
};

template <int PHASE>
__global__ void __launch_bounds__(32 * (kMaxWarps + 2), 1) k_experts(ExpParams P) {
  const Geo& g = P.g;
  extern __shared__ __align__(128) uint8_t smem[];
  const int NW = phase_warps(g, PHASE);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t slot_bytes = stage_slot_bytes(g, PHASE);
  const int nstages = P.nstages;
  StageHdr* hdr = reinterpret_cast<StageHdr*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 512);
  uint64_t* empty = full + 16;
  uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + 768);
  uint64_t* rempty = rfull + kRed;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 896);
  RedMeta* rmeta = reinterpret_cast<RedMeta*>(smem + 1024);
  float* red = reinterpret_cast<float*>(smem + kEngineBase);
  const int red_stride = NW * g.M * 32;  // floats per reduction buffer; warp cw, row r at (cw * M + r) * 32
  uint8_t* ring = smem + kEngineBase + red_bytes_for(NW, g.M);
  int32_t* err = (int32_t*)(P.ws + P.L.err);

  const int kc = PHASE == 0 ? g.kcA : g.kcB;
  const int nch = PHASE == 0 ? g.nchA : g.nchB;
  const int P_ = phase_panels(g, PHASE);
  const int G = PHASE == 0 ? g.GA : g.GB;
  const int npan = PHASE == 0 ? g.npanA : g.npanB;
  const int per_u = (npan / P_) * nch;

  if (tid == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    for (int b = 0; b < kRed; ++b) {
      mbar_init(&rfull[b], NW);
      mbar_init(&rempty[b], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  griddep_wait();  // routing / phase A results must be complete and visible

  const int nU = *(volatile const int32_t*)(P.ws + P.L.nu);
  const int nItems = nU * per_u;
  // the work list (format, slot address, rows of every distinct expert) in
  // shared memory, so no item waits on a global load
  __shared__ int32_t s_ufmt[kMaxM * kMaxTopK + 1];
  __shared__ int32_t s_unrows[kMaxM * kMaxTopK + 1];
  __shared__ uint64_t s_uaddr[kMaxM * kMaxTopK + 1];
  __shared__ int8_t s_urows[(kMaxM * kMaxTopK + 1) * kMaxM];
  for (int u = tid; u < nU; u += blockDim.x) {
    s_ufmt[u] = ((const int32_t*)(P.ws + P.L.u_fmt))[u];
    s_unrows[u] = ((const int32_t*)(P.ws + P.L.u_nrows))[u];
    s_uaddr[u] = ((const uint64_t*)(P.ws + P.L.u_addr))[u];
    for (int r = 0; r < kMaxM; ++r) s_urows[u * kMaxM + r] = (int8_t)((const int32_t*)(P.ws + P.L.u_rows))[u * kMaxM + r];
  }
  __syncthreads();
  const float* xf = (const float*)(P.ws + P.L.xf);
  float* hbuf = (float*)(P.ws + P.L.h);

  if (warp == 0) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      int last_issued[16];
      for (int s = 0; s < 16; ++s) last_issued[s] = -1;
      long long pw = 0, pi_ = 0;
      int i = 0;
      for (int t = blockIdx.x; t < nItems; t += gridDim.x, ++i) {
        const int s = i % nstages;
        if (*abort_flag) break;
        if (i >= nstages) {
          const long long t0 = clk();
          if (!mbar_wait_bounded(&empty[s], ((i / nstages) - 1) & 1, P.limit_ns)) {
            set_error(err, BQE_ETIMEOUT, kErrWaitEmpty);
            *abort_flag = 1;
            break;
          }
          pw += clk() - t0;
        }
        const long long t1 = clk();
        if (i == P.drop_item && blockIdx.x == 0) continue;  // test hook: this stage never lands
        const int u = t / per_u, rem = t % per_u;
        const int pg = rem / nch, c = rem % nch;
        const int fmt = s_ufmt[u];
        const int R = s_unrows[u];
        const uint64_t addr = s_uaddr[u];
        StageHdr& H = hdr[s];
        H.addr = addr; H.u = u; H.p0 = pg * P_; H.c = c; H.fmt = fmt; H.R = R;
        const uint32_t tb = tile_bytes(fmt, kc);
        const uint32_t wbytes = (uint32_t)phase_mats(PHASE) * P_ * tb;
        const bool half_act = PHASE == 0 && fmt == BQE_FMT_MXFP4 && P.variant == 1;
        const uint32_t arow = (uint32_t)kc * (half_act ? 2u : 4u);
        const uint32_t abytes = (uint32_t)R * arow;
        uint8_t* dst = ring + (size_t)s * slot_bytes;
        mbar_arrive_expect_tx(&full[s], wbytes + abytes);
        const uint64_t m13 = matrix_bytes(fmt, g.I, g.H);
        if (PHASE == 0) {
          for (int j = 0; j < P_; ++j) {
            const uint64_t toff = (uint64_t)((pg * P_ + j) * nch + c) * tb;
            bulk_g2s(dst + j * tb, (const void*)(addr + toff), tb, &full[s]);                 // W1
            bulk_g2s(dst + (P_ + j) * tb, (const void*)(addr + m13 + toff), tb, &full[s]);    // W3
          }
        } else {
          for (int j = 0; j < P_; ++j) {
            const uint64_t toff = 2 * m13 + (uint64_t)((pg * P_ + j) * nch + c) * tb;
            bulk_g2s(dst + j * tb, (const void*)(addr + toff), tb, &full[s]);
          }
        }
        uint8_t* adst = dst + wbytes;
        const uint16_t* xh = (const uint16_t*)(P.ws + P.L.xh);
        for (int r = 0; r < R; ++r) {
          const void* src;
          if (PHASE == 0)
            src = half_act ? (const void*)(xh + (int64_t)s_urows[u * kMaxM + r] * g.H + (int64_t)c * kc)
                           : (const void*)(xf + (int64_t)s_urows[u * kMaxM + r] * g.H + (int64_t)c * kc);
          else
            src = hbuf + ((int64_t)u * g.M + r) * g.I + (int64_t)c * kc;
          bulk_g2s(adst + (size_t)r * arow, src, arow, &full[s]);
        }
        last_issued[s] = i;
        pi_ += clk() - t1;
      }
      dbg_add(P, PHASE, 0, pw);
      dbg_add(P, PHASE, 1, pi_);
      if (*abort_flag) {
        // drain this CTA's copies still in flight before leaving
        for (int s = 0; s < nstages; ++s)
          if (last_issued[s] >= 0) mbar_wait_bounded(&full[s], (last_issued[s] / nstages) & 1, 2000000000ull);
      }
    }
    return;
  }

  if (warp <= NW) {
    // --------------------------------- consumers ------------------------------
    const int cw = warp - 1;
    long long cwf = 0, cwr = 0, ccomp = 0;
    const int mat = cw / (P_ * G);         // 0: W1 (or W2), 1: W3
    const int pan = (cw / G) % P_;
    const int grp = cw % G;
    int i = 0;
    for (int t = blockIdx.x; t < nItems; t += gridDim.x, ++i) {
      const int s = i % nstages, b = i % kRed;
      const long long t0 = clk();
      // every lane waits; the warp proceeds only if all lanes saw the stage land
      bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (i / nstages) & 1, P.limit_ns));
      const long long t1 = clk();
      if (ok && i >= kRed)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&rempty[b], ((i / kRed) - 1) & 1, P.limit_ns));
      const long long t2 = clk();
      cwf += t1 - t0;
      cwr += t2 - t1;
      if (!ok) {
        if (lane == 0) {
          set_error(err, BQE_ETIMEOUT, kErrWaitFull);
          *abort_flag = 1;
        }
        break;
      }
      const StageHdr H = hdr[s];
      const uint32_t tb = tile_bytes(H.fmt, kc);
      const uint8_t* slot = ring + (size_t)s * slot_bytes;
      const uint8_t* tile = slot + (size_t)(mat * P_ + pan) * tb;
      const uint8_t* act = slot + (size_t)phase_mats(PHASE) * P_ * tb;
      float* rb = red + (size_t)b * red_stride;
      const bool half_act = PHASE == 0 && H.fmt == BQE_FMT_MXFP4 && P.variant == 1;
      consume_rows(H.R, H.fmt, tile, kc, grp, act, lane, rb + cw * g.M * 32, half_act);
      if (cw == 0 && lane == 0) rmeta[b] = RedMeta{H.u, H.p0, H.c, H.R};
      ccomp += clk() - t2;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[s]);  // the stage may be refilled
        mbar_arrive(&rfull[b]);  // this warp's partial sums are in red[b]
      }
    }
    if (cw == 0 && lane == 0) {
      dbg_add(P, PHASE, 2, cwf);
      dbg_add(P, PHASE, 3, cwr);
      dbg_add(P, PHASE, 4, ccomp);
    }
    return;
  }

  if (warp != NW + 1) return;
  // ------------------------------- epilogue warp --------------------------------
  int i = 0;
  long long ew = 0, eb = 0, tprev = clk();
  const long long tstart = tprev;
  for (int t = blockIdx.x; t < nItems; t += gridDim.x, ++i) {
    const int b = i % kRed;
    const long long t0 = clk();
    eb += t0 - tprev;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&rfull[b], (i / kRed) & 1, P.limit_ns))) {
      if (lane == 0) set_error(err, BQE_ETIMEOUT, kErrWaitFull);
      break;
    }
    tprev = clk();
    ew += tprev - t0;
    const RedMeta mt = rmeta[b];
    const float* rb = red + (size_t)b * red_stride;
    // partial sums of this item's chunk go to the workspace with plain stores;
    // the finalize kernel adds the chunks in a fixed order
    if (PHASE == 0) {
      const bool half_act = s_ufmt[mt.u] == BQE_FMT_MXFP4 && P.variant == 1;
      const float* xsc = (const float*)(P.ws + P.L.xsc);
      float* pa = (float*)(P.ws + P.L.pa);
      // W1 warps of panel pi are cw = pi*G + gi, W3 warps cw = (P + pi)*G + gi
      for (int r = 0; r < mt.R; ++r) {
        const float unscale = half_act ? xsc[s_urows[mt.u * kMaxM + r]] : 1.0f;  // 2^-s, exact
        for (int pi = 0; pi < P_; ++pi) {
          const int p = mt.p0 + pi;
          const int64_t base = (((int64_t)mt.u * g.npanA + p) * nch + mt.c) * 2 * g.M;
          float a0 = 0.f, a1 = 0.f;
          for (int gi = 0; gi < G; ++gi) {
            a0 += rb[((pi * G + gi) * g.M + r) * 32 + lane];
            a1 += rb[(((P_ + pi) * G + gi) * g.M + r) * 32 + lane];
          }
          pa[(base + r) * 32 + lane] = a0 * unscale;
          pa[(base + g.M + r) * 32 + lane] = a1 * unscale;
        }
      }
    } else {
      float* pb = (float*)(P.ws + P.L.pb);
      for (int pi = 0; pi < P_; ++pi) {
        const int n = (mt.p0 + pi) * 32 + lane;
        for (int r = 0; r < mt.R; ++r) {
          float y = 0.f;
          for (int gi = 0; gi < G; ++gi) y += rb[((pi * G + gi) * g.M + r) * 32 + lane];
          pb[(((int64_t)mt.u * nch + mt.c) * g.M + r) * g.H + n] = y;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rempty[b]);  // red[b] has been read
  }
  if (lane == 0) {
    const long long tend = clk();
    dbg_add(P, PHASE, 5, ew);
    dbg_add(P, PHASE, 6, eb + (tend - tprev));
    dbg_add(P, PHASE, 7, tend - tstart);
  }
}

// ---------------------------------------------------------------------------
// finalize: add the chunk partials in chunk order
//   phase A: h[u, r, i] = silu(sum_c g_c) * (sum_c u_c)
//   phase B: out[m, n] (+)= y_shared[m, n] + sum_j w[m, j] y[u(m,j), r(m,j), n]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_finalize_a(ExpParams P) {
  const Geo& g = P.g;
  griddep_wait();
  const int nU = *(volatile const int32_t*)(P.ws + P.L.nu);
  const int32_t* u_nrows = (const int32_t*)(P.ws + P.L.u_nrows);
  const float* pa = (const float*)(P.ws + P.L.pa);
  float* hbuf = (float*)(P.ws + P.L.h);
  const int nch = g.nchA;
  const int64_t n = (int64_t)nU * g.M * g.I;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int u = (int)(t / ((int64_t)g.M * g.I));
    const int r = (int)((t / g.I) % g.M);
    const int i = (int)(t % g.I);
    if (r >= u_nrows[u]) continue;
    const int p = i >> 5, lane = i & 31;
    float a0 = 0.f, a1 = 0.f;
    for (int c = 0; c < nch; ++c) {
      const int64_t base = (((int64_t)u * g.npanA + p) * nch + c) * 2 * g.M;
      a0 += pa[(base + r) * 32 + lane];
      a1 += pa[(base + g.M + r) * 32 + lane];
    }
    hbuf[((int64_t)u * g.M + r) * g.I + i] = silu_f(a0) * a1;
  }
}

__global__ void __launch_bounds__(256) k_finalize_b(ExpParams P) {
  const Geo& g = P.g;
  griddep_wait();
  const int nU = *(volatile const int32_t*)(P.ws + P.L.nu);
  const float* pb = (const float*)(P.ws + P.L.pb);
  const int32_t* cu = (const int32_t*)(P.ws + P.L.comb_u);
  const int32_t* cr = (const int32_t*)(P.ws + P.L.comb_r);
  const float* cwt = (const float*)(P.ws + P.L.comb_w);
  const int nch = g.nchB;
  if (nU == 0) return;  // the router reported an error; out is left untouched
  const int64_t n = (int64_t)g.M * g.H;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(t / g.H), col = (int)(t % g.H);
    float val = 0.f;
    for (int c = 0; c < nch; ++c) val += pb[((int64_t)c * g.M + m) * g.H + col];  // shared expert, u = 0
    for (int j = 0; j < g.K; ++j) {
      const int u = cu[m * g.K + j], r = cr[m * g.K + j];
      float yj = 0.f;
      for (int c = 0; c < nch; ++c) yj += pb[(((int64_t)u * nch + c) * g.M + r) * g.H + col];
      val = fmaf(cwt[m * g.K + j], yj, val);
    }
    float* o = P.out + t;
    *o = P.accumulate ? *o + val : val;
  }
}

int launch_finalize(const ExpParams& P, int phase, int sms, cudaStream_t st, bool pdl) {
  const int64_t n = phase == 0 ? (int64_t)P.g.U * P.g.M * P.g.I : (int64_t)P.g.M * P.g.H;
  int grid = (int)((n + 255) / 256);
  if (grid > 2 * sms) grid = 2 * sms;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = phase == 0 ? cudaLaunchKernelEx(&cfg, k_finalize_a, P) : cudaLaunchKernelEx(&cfg, k_finalize_b, P);
  return e == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

uint32_t experts_smem_bytes(const Geo& g, int phase, int* nstages_out) {
  const uint32_t base = kEngineBase + red_bytes_for(phase_warps(g, phase), g.M);
  const uint32_t slot = stage_slot_bytes(g, phase);
  int ns = (int)((kSmemBudget - base) / slot);
  if (ns > 8) ns = 8;
  if (nstages_out) *nstages_out = ns;
  return base + (uint32_t)ns * slot;
}

int launch_experts(const ExpParams& P, int phase, int grid, cudaStream_t st, bool pdl) {
  int ns = 0;
  const uint32_t smem = experts_smem_bytes(P.g, phase, &ns);
  if (ns < 2) return BQE_EUNSUPPORTED;
  // raise the kernel's dynamic shared memory limit once per device (the call is slow)
  static int limit_set[2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BQE_ECUDA;
  if (limit_set[phase][dev] < (int)smem) {
    const void* fn = phase == 0 ? (const void*)k_experts<0> : (const void*)k_experts<1>;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, fn) != cudaSuccess)
      return BQE_ECUDA;
    const int dyn_max = optin - (int)fa.sharedSizeBytes;  // dynamic + static must fit the opt-in limit
    if (dyn_max < (int)smem) return BQE_EUNSUPPORTED;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) != cudaSuccess)
      return BQE_ECUDA;
    limit_set[phase][dev] = dyn_max;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * (2 + phase_warps(P.g, phase)));  // producer + consumers + epilogue
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = phase == 0 ? cudaLaunchKernelEx(&cfg, k_experts<0>, P) : cudaLaunchKernelEx(&cfg, k_experts<1>, P);
  return e == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

}  // namespace bqe
