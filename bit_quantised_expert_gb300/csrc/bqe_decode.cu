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

constexpr int kFmtMaxBytesPerCol = 17;  // MXFP4 tile: 17 bytes per column per 32 rows

__host__ __device__ inline int phase_mats(int phase) { return phase == 0 ? 2 : 1; }

__host__ __device__ inline uint32_t stage_slot_bytes(const Geo& g, int phase) {
  const int kc = phase == 0 ? g.kcA : g.kcB;
  const int P = phase == 0 ? 1 : g.PB;
  const uint32_t w = (uint32_t)phase_mats(phase) * P * kFmtMaxBytesPerCol * kc;
  return ((w + (uint32_t)g.M * kc * 4u) + 127u) & ~127u;
}

__host__ __device__ inline int phase_warps(const Geo& g, int phase) {
  return phase == 0 ? 2 * g.GA : g.PB * g.GB;
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

template <int R>
__device__ __forceinline__ void group_mxfp4(const uint8_t* tile, int nb, int grp, const float* act, int kc, int lane,
                                            float2 (&acc)[R]) {
#pragma unroll 2
  for (int bi = 0; bi < 8; ++bi) {
    const int b = grp * 8 + bi;
    const uint4 c4 = *reinterpret_cast<const uint4*>(tile + b * 512 + lane * 16);
    const float sc = ue8m0_f32(tile[nb * 512 + b * 32 + lane]);
    float2 bs[R];
#pragma unroll
    for (int r = 0; r < R; ++r) bs[r] = f2(0.f, 0.f);
    const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 v0 = e2m1x2_f32(wd[w] & 0xFF);
      const float2 v1 = e2m1x2_f32((wd[w] >> 8) & 0xFF);
      const float2 v2 = e2m1x2_f32((wd[w] >> 16) & 0xFF);
      const float2 v3 = e2m1x2_f32(wd[w] >> 24);
      const int k = grp * 256 + bi * 32 + w * 8;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4 xa = *reinterpret_cast<const float4*>(act + r * kc + k);
        const float4 xb = *reinterpret_cast<const float4*>(act + r * kc + k + 4);
        bs[r] = __ffma2_rn(v0, f2(xa.x, xa.y), bs[r]);
        bs[r] = __ffma2_rn(v1, f2(xa.z, xa.w), bs[r]);
        bs[r] = __ffma2_rn(v2, f2(xb.x, xb.y), bs[r]);
        bs[r] = __ffma2_rn(v3, f2(xb.z, xb.w), bs[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = __ffma2_rn(bs[r], f2(sc, sc), acc[r]);
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
                                                int lane, float* outv /* [r * 32 + lane] */) {
  float2 acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = f2(0.f, 0.f);
  const int nb = kc / fmt_bw(fmt);
  switch (fmt) {
    case BQE_FMT_MXFP4: group_mxfp4<R>(tile, nb, grp, act, kc, lane, acc); break;
    case BQE_FMT_Q2_0: group_q2_0<R>(tile, nb, grp, act, kc, lane, acc); break;
    case BQE_FMT_TQ1: group_tq1<R>(tile, nb, grp, act, kc, lane, acc); break;
    case BQE_FMT_Q3_K: group_q3k<R>(tile, nb, grp, act, kc, lane, acc); break;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) outv[r * 32 + lane] = acc[r].x + acc[r].y;
}

__device__ __forceinline__ void consume_group(int R, int fmt, const uint8_t* tile, int kc, int grp, const float* act,
                                              int lane, float* outv) {
  switch (R) {
    case 1: consume_group_R<1>(fmt, tile, kc, grp, act, lane, outv); break;
    case 2: consume_group_R<2>(fmt, tile, kc, grp, act, lane, outv); break;
    case 3: consume_group_R<3>(fmt, tile, kc, grp, act, lane, outv); break;
    case 4: consume_group_R<4>(fmt, tile, kc, grp, act, lane, outv); break;
    case 5: consume_group_R<5>(fmt, tile, kc, grp, act, lane, outv); break;
    case 6: consume_group_R<6>(fmt, tile, kc, grp, act, lane, outv); break;
    case 7: consume_group_R<7>(fmt, tile, kc, grp, act, lane, outv); break;
    case 8: consume_group_R<8>(fmt, tile, kc, grp, act, lane, outv); break;
  }
}

__device__ __forceinline__ float silu_f(float t) { return t / (1.0f + expf(-t)); }

// ---------------------------------------------------------------------------
// the engine
// ---------------------------------------------------------------------------
template <int PHASE>
__global__ void __launch_bounds__(32 * (kMaxWarps + 1), 1) k_experts(ExpParams P) {
  const Geo& g = P.g;
  extern __shared__ __align__(128) uint8_t smem[];
  const int NW = phase_warps(g, PHASE);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t slot_bytes = stage_slot_bytes(g, PHASE);
  const int nstages = P.nstages;
  StageHdr* hdr = reinterpret_cast<StageHdr*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 1024);
  uint64_t* empty = full + 16;
  float* red = reinterpret_cast<float*>(smem + 2048);  // [2][kMaxWarps][kMaxM][32]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 1920);
  uint8_t* ring = smem + 2048 + 2 * kMaxWarps * kMaxM * 32 * 4;
  int32_t* err = (int32_t*)(P.ws + P.L.err);

  const int kc = PHASE == 0 ? g.kcA : g.kcB;
  const int nch = PHASE == 0 ? g.nchA : g.nchB;
  const int P_ = PHASE == 0 ? 1 : g.PB;
  const int G = PHASE == 0 ? g.GA : g.GB;
  const int npan = PHASE == 0 ? g.npanA : g.npanB;
  const int per_u = (npan / P_) * nch;

  if (tid == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  griddep_wait();  // routing / phase A results must be complete and visible

  const int nU = *(volatile const int32_t*)(P.ws + P.L.nu);
  const int nItems = nU * per_u;
  const int32_t* u_fmt = (const int32_t*)(P.ws + P.L.u_fmt);
  const uint64_t* u_addr = (const uint64_t*)(P.ws + P.L.u_addr);
  const int32_t* u_nrows = (const int32_t*)(P.ws + P.L.u_nrows);
  const int32_t* u_rows = (const int32_t*)(P.ws + P.L.u_rows);
  const float* xf = (const float*)(P.ws + P.L.xf);
  float* hbuf = (float*)(P.ws + P.L.h);

  if (warp == 0) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      int last_issued[16];
      for (int s = 0; s < 16; ++s) last_issued[s] = -1;
      int i = 0;
      for (int t = blockIdx.x; t < nItems; t += gridDim.x, ++i) {
        const int s = i % nstages;
        if (*abort_flag) break;
        if (i >= nstages) {
          if (!mbar_wait_bounded(&empty[s], ((i / nstages) - 1) & 1, P.limit_ns)) {
            set_error(err, BQE_ETIMEOUT, kErrWaitEmpty);
            *abort_flag = 1;
            break;
          }
        }
        const int u = t / per_u, rem = t % per_u;
        const int pg = rem / nch, c = rem % nch;
        const int fmt = u_fmt[u];
        const int R = u_nrows[u];
        const uint64_t addr = u_addr[u];
        StageHdr& H = hdr[s];
        H.addr = addr; H.u = u; H.p0 = pg * P_; H.c = c; H.fmt = fmt; H.R = R;
        const uint32_t tb = tile_bytes(fmt, kc);
        const uint32_t wbytes = (uint32_t)phase_mats(PHASE) * P_ * tb;
        const uint32_t abytes = (uint32_t)R * kc * 4u;
        uint8_t* dst = ring + (size_t)s * slot_bytes;
        mbar_arrive_expect_tx(&full[s], wbytes + abytes);
        const uint64_t m13 = matrix_bytes(fmt, g.I, g.H);
        if (PHASE == 0) {
          const uint64_t toff = (uint64_t)(pg * nch + c) * tb;
          bulk_g2s(dst, (const void*)(addr + toff), tb, &full[s]);
          bulk_g2s(dst + tb, (const void*)(addr + m13 + toff), tb, &full[s]);
        } else {
          for (int j = 0; j < P_; ++j) {
            const uint64_t toff = 2 * m13 + (uint64_t)((pg * P_ + j) * nch + c) * tb;
            bulk_g2s(dst + j * tb, (const void*)(addr + toff), tb, &full[s]);
          }
        }
        uint8_t* adst = dst + wbytes;
        for (int r = 0; r < R; ++r) {
          const float* src = PHASE == 0 ? xf + (int64_t)u_rows[u * kMaxM + r] * g.H + (int64_t)c * kc
                                        : hbuf + ((int64_t)u * g.M + r) * g.I + (int64_t)c * kc;
          bulk_g2s(adst + (size_t)r * kc * 4, src, (uint32_t)kc * 4u, &full[s]);
        }
        last_issued[s] = i;
      }
      if (*abort_flag) {
        // drain this CTA's copies still in flight before leaving
        for (int s = 0; s < nstages; ++s)
          if (last_issued[s] >= 0) mbar_wait_bounded(&full[s], (last_issued[s] / nstages) & 1, 2000000000ull);
      }
    }
    return;
  }

  // --------------------------------- consumers --------------------------------
  const int cw = warp - 1;
  if (cw >= NW) return;
  const int mat = PHASE == 0 ? cw / G : 0;
  const int pan = PHASE == 0 ? 0 : cw / G;
  const int grp = cw % G;
  int i = 0;
  for (int t = blockIdx.x; t < nItems; t += gridDim.x, ++i) {
    const int s = i % nstages;
    // every lane waits; the warp proceeds only if all lanes saw the stage land
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (i / nstages) & 1, P.limit_ns));
    float* rb = red + (size_t)(i & 1) * kMaxWarps * kMaxM * 32;
    const StageHdr H = hdr[s];
    if (!ok) {
      if (lane == 0) { set_error(err, BQE_ETIMEOUT, kErrWaitFull); *abort_flag = 1; }
    } else {
      const uint32_t tb = tile_bytes(H.fmt, kc);
      const uint8_t* slot = ring + (size_t)s * slot_bytes;
      const uint8_t* tile = slot + (PHASE == 0 ? mat * tb : pan * tb);
      const float* act = reinterpret_cast<const float*>(slot + (size_t)phase_mats(PHASE) * P_ * tb);
      consume_group(H.R, H.fmt, tile, kc, grp, act, lane, rb + cw * kMaxM * 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    named_bar_sync(1, NW * 32);
    if (*abort_flag) break;

    // ------------------------------ epilogues ------------------------------
    if (PHASE == 0) {
      if (cw == 0) {
        const int p = H.p0;
        const int row = p * 32 + lane;
        if (nch == 1) {
          for (int r = 0; r < H.R; ++r) {
            float gs = 0.f, us = 0.f;
            for (int gi = 0; gi < G; ++gi) {
              gs += rb[(gi * kMaxM + r) * 32 + lane];
              us += rb[((G + gi) * kMaxM + r) * 32 + lane];
            }
            hbuf[((int64_t)H.u * g.M + r) * g.I + row] = silu_f(gs) * us;
          }
        } else {
          float* pa = (float*)(P.ws + P.L.pa);
          const int64_t base = (((int64_t)H.u * g.npanA + p) * nch + H.c) * 2 * g.M;
          for (int r = 0; r < H.R; ++r) {
            float gs = 0.f, us = 0.f;
            for (int gi = 0; gi < G; ++gi) {
              gs += rb[(gi * kMaxM + r) * 32 + lane];
              us += rb[((G + gi) * kMaxM + r) * 32 + lane];
            }
            pa[(base + r) * 32 + lane] = gs;
            pa[(base + g.M + r) * 32 + lane] = us;
          }
          __threadfence();
          __syncwarp();
          unsigned int old = 0;
          unsigned int* ctr = (unsigned int*)(P.ws + P.L.ctrA) + H.u * g.npanA + p;
          if (lane == 0) old = atomicAdd(ctr, 1u);
          old = __shfl_sync(0xffffffffu, old, 0);
          if (old == (unsigned int)(nch - 1)) {
            __threadfence();
            for (int r = 0; r < H.R; ++r) {
              float gs = 0.f, us = 0.f;
              for (int c = 0; c < nch; ++c) {
                const int64_t b2 = (((int64_t)H.u * g.npanA + p) * nch + c) * 2 * g.M;
                gs += __ldcg(pa + (b2 + r) * 32 + lane);
                us += __ldcg(pa + (b2 + g.M + r) * 32 + lane);
              }
              hbuf[((int64_t)H.u * g.M + r) * g.I + row] = silu_f(gs) * us;
            }
            if (lane == 0) *ctr = 0u;
          }
        }
      }
    } else {
      if (cw < P_) {
        const int p = H.p0 + cw;
        const int n = p * 32 + lane;
        float* pb = (float*)(P.ws + P.L.pb);
        for (int r = 0; r < H.R; ++r) {
          float y = 0.f;
          for (int gi = 0; gi < G; ++gi) y += rb[((cw * G + gi) * kMaxM + r) * 32 + lane];
          pb[(((int64_t)H.u * nch + H.c) * g.M + r) * g.H + n] = y;
        }
        __threadfence();
        __syncwarp();
        unsigned int old = 0;
        unsigned int* ctr = (unsigned int*)(P.ws + P.L.ctrB) + p;
        if (lane == 0) old = atomicAdd(ctr, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == (unsigned int)(nU * nch - 1)) {
          __threadfence();
          const int32_t* cu = (const int32_t*)(P.ws + P.L.comb_u);
          const int32_t* cr = (const int32_t*)(P.ws + P.L.comb_r);
          const float* cwt = (const float*)(P.ws + P.L.comb_w);
          for (int m = 0; m < g.M; ++m) {
            float ys = 0.f;
            for (int c = 0; c < nch; ++c) ys += __ldcg(pb + (((int64_t)0 * nch + c) * g.M + m) * g.H + n);
            float val = ys;
            for (int j = 0; j < g.K; ++j) {
              const int u = cu[m * g.K + j], r = cr[m * g.K + j];
              float yj = 0.f;
              for (int c = 0; c < nch; ++c) yj += __ldcg(pb + (((int64_t)u * nch + c) * g.M + r) * g.H + n);
              val = fmaf(cwt[m * g.K + j], yj, val);
            }
            float* o = P.out + (int64_t)m * g.H + n;
            *o = P.accumulate ? *o + val : val;
          }
          if (lane == 0) *ctr = 0u;
        }
      }
    }
  }
}

uint32_t experts_smem_bytes(const Geo& g, int phase, int* nstages_out) {
  const uint32_t base = 2048 + 2 * kMaxWarps * kMaxM * 32 * 4;
  const uint32_t slot = stage_slot_bytes(g, phase);
  const uint32_t budget = 220 * 1024;
  int ns = (int)((budget - base) / slot);
  if (ns > 8) ns = 8;
  if (nstages_out) *nstages_out = ns;
  return base + (uint32_t)ns * slot;
}

int launch_experts(const ExpParams& P, int phase, int grid, cudaStream_t st, bool pdl) {
  int ns = 0;
  const uint32_t smem = experts_smem_bytes(P.g, phase, &ns);
  if (ns < 2) return BQE_EUNSUPPORTED;
  const void* fn = phase == 0 ? (const void*)k_experts<0> : (const void*)k_experts<1>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return BQE_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * (1 + phase_warps(P.g, phase)));
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
