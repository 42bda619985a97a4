// bqe_prefill.cu — the prefill path: one MoE layer over T token rows.
//
//   1. k_pf_logits   z = x Wr^T in fp32 (tiled SIMT GEMM; the top-k needs
//                    fp32 logits, as in decode)
//   2. k_pf_select   per token: sigmoid scores, biased top-k (ties to the lower
//                    expert id) or the forced choice, mixing weights, counts
//   3. k_pf_plan     per expert: validated slot, row range padded to 16, tiles
//   4. k_pf_fill     per expert: its (token, choice) pairs in token order
//   5. k_pf_gather   x rows, scaled per token by 2^s, copied into expert-grouped
//                    swizzled 16-bit tiles
//   6. k_pf_gemm<0>  per (expert tile, 64 features): gate and up rows of W1/W3
//                    dequantised in shared memory, tcgen05 MMA into tensor
//                    memory, h 2^s = silu(gate) * up 2^s written as 16-bit tiles
//   7. k_pf_gemm<1>  per (expert tile, 128 outputs): W2 the same way,
//                    y = w 2^-s (W2 h 2^s)
//   8. k_pf_combine  out[t] = y_shared + sum_j y_j in a fixed order
//
// Prefill only regroups the tokens of a layer by expert: the result per token
// is the decode layer's (the Strata 4090 post, section 5.3, requires prefill
// accelerations to leave results unchanged); the 16-bit operands of the tensor
// cores are the only difference (section 4 of the same post: tensor-core
// experts for prefill).  Operand type: fp16 by default.  x is exact in it once
// scaled by a power of two per token (max |x 2^s| in [1, 2)); TQ1 weights d t
// are exact, Q2_0 and Q3_K weights rounded to 11 bits; h carries the same
// per-token scale so it stays in range.  MXFP4 experts use bf16 (E2M1 times
// 2^(E-127) is exact there for every E).  bf16 for every expert is selectable.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bqe_gemv.cuh"
#include "bqe_prefill.cuh"
#include "bqe_umma.cuh"

namespace bqe {

enum { kErrPfProducer = 7, kErrPfDequant = 8, kErrPfMma = 9, kErrPfEpilogue = 10, kErrPfRange = 11 };

// Order of the 64 columns of a K-step in the grouped operands of an expert:
// natural, or "paired" for fp16 Q2_0 (columns j and j + 8 of every 16 next to
// each other) and Q3_K (j and j + 16 of every 32); see the dequant routines.
__host__ __device__ inline int paired_col(int fmt, int p) {  // column of K-step position p
  return fmt == BQE_FMT_Q2_0   ? 16 * (p / 16) + (p % 16) / 2 + 8 * (p % 2)
         : fmt == BQE_FMT_Q3_K ? 32 * (p / 32) + (p % 32) / 2 + 16 * (p % 2)
                               : p;
}
__host__ __device__ inline int paired_pos(int fmt, int f) {  // position of column f
  return fmt == BQE_FMT_Q2_0   ? 16 * (f / 16) + 2 * (f % 8) + (f % 16) / 8
         : fmt == BQE_FMT_Q3_K ? 32 * (f / 32) + 2 * (f % 16) + (f % 32) / 16
                               : f;
}

// ----------------------------------------------------------------------------
// 1. Router logits: z (T x E) = x (T x H, bf16) . Wr (E x H, fp32)^T, fp32.
// Tile 128 tokens x 64 experts x 32 columns, 256 threads, 8 x 4 per thread.
// ----------------------------------------------------------------------------
constexpr int kLgBM = 128, kLgBN = 64, kLgBK = 32;

__global__ void __launch_bounds__(256) k_pf_logits(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                                                   float* __restrict__ z, int T, int E, int H) {
  __shared__ __align__(16) float As[kLgBK][kLgBM];
  __shared__ __align__(16) float Bs[kLgBK][kLgBN];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.y * kLgBM, e0 = blockIdx.x * kLgBN;
  const int ty = tid / 16, tx = tid % 16;
  // loader mapping: A: token tid % 128, columns (tid / 128) * 16 .. +15;
  //                 B: expert tid % 64, columns (tid / 64) * 8 .. +7
  const int la_t = tid % kLgBM, la_k = (tid / kLgBM) * 16;
  const int lb_e = tid % kLgBN, lb_k = (tid / kLgBN) * 8;
  const bool a_ok = t0 + la_t < T, b_ok = e0 + lb_e < E;
  const uint16_t* ap = x + (int64_t)(a_ok ? t0 + la_t : 0) * H + la_k;
  const float* bp = wr + (int64_t)(b_ok ? e0 + lb_e : 0) * H + lb_k;
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  uint4 ra0 = make_uint4(0, 0, 0, 0), ra1 = ra0;
  float4 rb0 = make_float4(0.f, 0.f, 0.f, 0.f), rb1 = rb0;
  auto load = [&](int k0) {
    if (a_ok) {
      ra0 = *reinterpret_cast<const uint4*>(ap + k0);
      ra1 = *reinterpret_cast<const uint4*>(ap + k0 + 8);
    }
    if (b_ok) {
      rb0 = *reinterpret_cast<const float4*>(bp + k0);
      rb1 = *reinterpret_cast<const float4*>(bp + k0 + 4);
    }
  };
  auto bf = [](uint32_t w, int hi) { return __uint_as_float(hi ? (w & 0xFFFF0000u) : (w << 16)); };
  load(0);
  for (int k0 = 0; k0 < H; k0 += kLgBK) {
    const uint32_t aw[8] = {ra0.x, ra0.y, ra0.z, ra0.w, ra1.x, ra1.y, ra1.z, ra1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      As[la_k + 2 * i][la_t] = bf(aw[i], 0);
      As[la_k + 2 * i + 1][la_t] = bf(aw[i], 1);
    }
    Bs[lb_k + 0][lb_e] = rb0.x; Bs[lb_k + 1][lb_e] = rb0.y; Bs[lb_k + 2][lb_e] = rb0.z; Bs[lb_k + 3][lb_e] = rb0.w;
    Bs[lb_k + 4][lb_e] = rb1.x; Bs[lb_k + 5][lb_e] = rb1.y; Bs[lb_k + 6][lb_e] = rb1.z; Bs[lb_k + 7][lb_e] = rb1.w;
    __syncthreads();
    if (k0 + kLgBK < H) load(k0 + kLgBK);
#pragma unroll 8
    for (int k = 0; k < kLgBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[k][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[k][ty * 8 + 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[k][tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) z[(int64_t)t * E + e] = acc[i][j];
    }
  }
}

// ----------------------------------------------------------------------------
// 2. Selection, one warp per token.  Order: larger key s + b first, ties to
// the lower expert id (keys compared through an order-preserving uint image);
// weights w_j = s_j / sum s from the unbiased scores in the log domain (finite
// when every selected sigmoid underflows).
// ----------------------------------------------------------------------------
constexpr int kSelPerLane = 16;  // E <= 512

__global__ void __launch_bounds__(256) k_pf_select(PfParams P) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int E = P.g.E, K = P.g.K, T = P.g.T;
  if (t >= T) return;
  const float* z = (const float*)(P.ws + P.L.z) + (int64_t)t * E;
  int32_t* idx = (int32_t*)(P.ws + P.L.idx) + (int64_t)t * K;
  float* wout = (float*)(P.ws + P.L.w) + (int64_t)t * K;
  int32_t* cnt = (int32_t*)(P.ws + P.L.cnt);
  int32_t* err = (int32_t*)(P.ws + P.L.err);
  auto ord = [](float f) -> uint32_t {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  };
  {
    // per-token power of two: max |x_t| 2^s in [1, 2) (the magnitude bits of a
    // bf16 order like its value, so an integer max finds the largest |x|)
    const uint4* xr = reinterpret_cast<const uint4*>(P.x + (int64_t)t * P.g.H);
    uint32_t mx = 0;
    for (int i = lane; i < P.g.H / 8; i += 32) {
      const uint4 v = xr[i];
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) mx = max(mx, max(wv[k] & 0x7FFFu, (wv[k] >> 16) & 0x7FFFu));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    const int ex = (int)(mx >> 7);
    const int sh = ex == 0 ? 0 : min(max(127 - ex, -126), 126);
    if (lane == 0) ((float*)(P.ws + P.L.tok_sc))[t] = __int_as_float((127 - sh) << 23);
  }
  int sel = -1;      // lane j < K: the j-th choice
  float zsel = 0.f;
  if (P.forced) {
    if (lane < K) {
      sel = P.forced[(int64_t)t * K + lane];
      if (sel < 0 || sel >= E) {
        set_error(err, BQE_EDEVICE, kErrForcedIdx);
        sel = 0;
      }
      zsel = z[sel];
    }
  } else {
    uint32_t key[kSelPerLane];
#pragma unroll
    for (int i = 0; i < kSelPerLane; ++i) {
      const int e = lane + 32 * i;
      key[i] = 0u;  // 0: no expert (below every real key)
      if (e < E) key[i] = ord(1.0f / (1.0f + expf(-z[e])) + (P.bias ? P.bias[e] : 0.f));
    }
    for (int j = 0; j < K; ++j) {
      uint32_t lk = 0u;
      int li = 0x7fffffff, lc = -1;
#pragma unroll
      for (int i = 0; i < kSelPerLane; ++i)
        if (key[i] > lk) { lk = key[i]; li = lane + 32 * i; lc = i; }  // ascending e: ties keep the lower
      const uint32_t wk = __reduce_max_sync(0xffffffffu, lk);
      const int best = (int)__reduce_min_sync(0xffffffffu, (lk == wk && wk != 0u) ? (uint32_t)li : 0x7fffffffu);
#pragma unroll
      for (int i = 0; i < kSelPerLane; ++i)
        if (i == lc && li == best) key[i] = 0u;
      if (lane == j) { sel = best; zsel = z[best]; }
    }
  }
  float ls = -INFINITY;
  if (lane < K) ls = zsel < 0.f ? zsel - log1pf(expf(zsel)) : -log1pf(expf(-zsel));  // log sigmoid(z)
  float mx = ls;
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float ev = lane < K ? expf(ls - mx) : 0.f;
  float tot = ev;
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (lane < K) {
    const float w = ev / tot;
    idx[lane] = sel;
    wout[lane] = w;
    if (P.topk_idx) P.topk_idx[(int64_t)t * K + lane] = sel;
    if (P.topk_w) P.topk_w[(int64_t)t * K + lane] = w;
    atomicAdd(&cnt[sel], 1);
  }
}

// Block-wide exclusive scan of one int per thread (blockDim.x multiple of 32,
// <= 1024); returns the exclusive prefix, *total the block sum.
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int wv = lane < nw ? s_warp[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wv, o);
      if (lane >= o) wv += n;
    }
    if (lane < nw) s_warp[lane] = wv;  // inclusive warp totals
  }
  __syncthreads();
  const int before = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[nw - 1];
  return before + inc - v;
}

// ----------------------------------------------------------------------------
// 3. Plan (one CTA of 1024 threads, one group per thread; group E is the
// shared expert with all T rows).  Invalid slots raise BQE_EDEVICE and their
// group is skipped.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_pf_plan(PfParams P) {
  __shared__ int s_warp[32];
  const int G = P.g.E + 1, T = P.g.T;
  const int gi = threadIdx.x;
  int32_t* cnt = (int32_t*)(P.ws + P.L.cnt);
  int32_t* goff = (int32_t*)(P.ws + P.L.goff);
  uint64_t* gaddr = (uint64_t*)(P.ws + P.L.gaddr);
  int32_t* gfmt = (int32_t*)(P.ws + P.L.gfmt);
  int32_t* gf16 = (int32_t*)(P.ws + P.L.gf16);
  int32_t* ctr = (int32_t*)(P.ws + P.L.ctr);
  int32_t* err = (int32_t*)(P.ws + P.L.err);
  int3* tiles = (int3*)(P.ws + P.L.tile);
  int n = 0, fmt = 0;
  uint64_t addr = 0;
  if (gi < G) {
    n = gi < P.g.E ? cnt[gi] : T;
    const int slot = P.slot_table[gi];
    if (n > 0) {
      int code = 0;
      if (slot < 0 || slot >= P.pool.n_slots) {
        code = kErrSlotRange;
      } else {
        fmt = P.pool.slot_fmt[slot];
        const uint64_t off = P.pool.slot_off[slot];
        if (!fmt_ok(fmt)) {
          code = kErrSlotFmt;
        } else {
          const uint64_t bytes = 2 * matrix_bytes(fmt, P.g.I, P.g.H) + matrix_bytes(fmt, P.g.H, P.g.I);
          if ((off & 15) || off + bytes > P.pool.base_bytes) code = kErrSlotExtent;
          addr = (uint64_t)P.pool.base + off;
        }
      }
      if (code) {
        set_error(err, BQE_EDEVICE, code);
        n = 0;
        fmt = 0;
      }
    }
    gaddr[gi] = addr;
    gfmt[gi] = fmt;
    gf16[gi] = P.f16 && fmt != BQE_FMT_MXFP4 && fmt != BQE_FMT_NVFP4;  // FP4 values are exact in bf16
    cnt[gi] = n;
  }
  const int padded = (n + kPfRowAlign - 1) / kPfRowAlign * kPfRowAlign;
  const int ntile = (n + kPfTileN - 1) / kPfTileN;
  int rows_total, tiles_total;
  const int row0 = block_excl_scan(padded, s_warp, &rows_total);
  const int tile0 = block_excl_scan(ntile, s_warp, &tiles_total);
  if (gi < G) {
    goff[gi] = row0;
    for (int tt = 0; tt < ntile; ++tt)
      tiles[tile0 + tt] = make_int3(gi, row0 + tt * kPfTileN, min(kPfTileN, n - tt * kPfTileN));
  }
  if (gi == 0) {
    goff[G] = rows_total;
    ctr[0] = tiles_total;
    ctr[1] = rows_total;
  }
}

// ----------------------------------------------------------------------------
// 4. Fill: CTA g lists the (token, choice) pairs of expert g in token order
// (the same order for every run), records each pair's grouped row and the
// padding rows of its range.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_pf_fill(PfParams P) {
  __shared__ int s_warp[32];
  const int g = blockIdx.x, E = P.g.E, K = P.g.K, T = P.g.T;
  const int32_t* cnt = (const int32_t*)(P.ws + P.L.cnt);
  const int32_t* goff = (const int32_t*)(P.ws + P.L.goff);
  const int32_t* gfmt = (const int32_t*)(P.ws + P.L.gfmt);
  const int32_t* idx = (const int32_t*)(P.ws + P.L.idx);
  const float* wsel = (const float*)(P.ws + P.L.w);
  int32_t* prow_tok = (int32_t*)(P.ws + P.L.prow_tok);
  float* prow_w = (float*)(P.ws + P.L.prow_w);
  float* prow_sc = (float*)(P.ws + P.L.prow_sc);
  const float* tok_sc = (const float*)(P.ws + P.L.tok_sc);
  int32_t* pos = (int32_t*)(P.ws + P.L.pos);
  const bool valid = gfmt[g] != 0;
  const int base = goff[g];
  const int n = cnt[g];
  if (g == E) {
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
      pos[(int64_t)t * (K + 1) + K] = valid ? base + t : -1;
      if (valid) {
        prow_tok[base + t] = t;
        prow_w[base + t] = 1.0f;
        prow_sc[base + t] = tok_sc[t];
      }
    }
  } else {
    int running = 0;
    for (int t0 = 0; t0 < T; t0 += blockDim.x) {
      const int t = t0 + threadIdx.x;
      int c = 0;
      if (t < T)
        for (int j = 0; j < K; ++j) c += idx[(int64_t)t * K + j] == g;
      int total;
      const int ex = block_excl_scan(c, s_warp, &total);
      if (c) {
        int r = base + running + ex;
        for (int j = 0; j < K; ++j)
          if (idx[(int64_t)t * K + j] == g) {
            pos[(int64_t)t * (K + 1) + j] = valid ? r : -1;
            if (valid) {
              prow_tok[r] = t;
              prow_w[r] = wsel[(int64_t)t * K + j];
              prow_sc[r] = tok_sc[t];
            }
            ++r;
          }
      }
      running += total;
    }
  }
  if (valid) {
    const int padded = (n + kPfRowAlign - 1) / kPfRowAlign * kPfRowAlign;
    for (int r = n + threadIdx.x; r < padded; r += blockDim.x) {
      prow_tok[base + r] = -1;
      prow_w[base + r] = 0.f;
      prow_sc[base + r] = 1.f;
    }
  }
}

// ----------------------------------------------------------------------------
// 5. Gather, one CTA per tile: grouped row p gets x[prow_tok[p]] 2^s (zeros
// for padding) in the tile's operand type, stored as K-step-major tiles: 64
// columns x 8 rows = one 1024-byte swizzled atom at ((ks R/8) + p/8) 1024, so
// one contiguous copy brings the 64 columns of any run of rows into shared
// memory in the layout the tensor core reads.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_pf_gather(PfParams P) {
  const int tile = blockIdx.x;
  if (tile >= ((const int32_t*)(P.ws + P.L.ctr))[0]) return;
  const int3 tl = ((const int3*)(P.ws + P.L.tile))[tile];
  const bool f16 = ((const int32_t*)(P.ws + P.L.gf16))[tl.x] != 0;
  const int gfmt = ((const int32_t*)(P.ws + P.L.gfmt))[tl.x];
  const int order = f16 && (gfmt == BQE_FMT_Q2_0 || gfmt == BQE_FMT_Q3_K) ? gfmt : 0;
  const int npad = (tl.z + 15) & ~15;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = P.g.H;
  const int64_t R8 = P.g.R / 8;
  uint8_t* xp = P.ws + P.L.xp;
  auto cvt2 = [&](uint32_t lo_bits, uint32_t hi_bits, float scale) -> uint32_t {  // two bf16 -> operand type
    const float lo = __uint_as_float(lo_bits << 16) * scale, hi = __uint_as_float(hi_bits << 16) * scale;
    if (f16) {
      const __half2 h2 = __floats2half2_rn(lo, hi);
      return *reinterpret_cast<const uint32_t*>(&h2);
    }
    return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);  // exact: scaled bf16
  };
  for (int r = warp; r < npad; r += 8) {
    const int p = tl.y + r;
    const int tok = ((const int32_t*)(P.ws + P.L.prow_tok))[p];
    const float scale = 1.0f / ((const float*)(P.ws + P.L.prow_sc))[p];  // 2^s, exact
    const uint16_t* xrow = P.x + (int64_t)(tok < 0 ? 0 : tok) * H;
    for (int i = lane; i < H / 8; i += 32) {  // 16-byte chunk i = K-step i / 8, chunk i % 8
      const int ks = i >> 3, c = i & 7;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (tok >= 0) {
        uint32_t w[4];
        if (order == 0) {
          const uint4 b = reinterpret_cast<const uint4*>(xrow)[i];
          w[0] = b.x; w[1] = b.y; w[2] = b.z; w[3] = b.w;
#pragma unroll
          for (int k = 0; k < 4; ++k) w[k] = cvt2(w[k] & 0xFFFFu, w[k] >> 16, scale);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int p0 = 8 * c + 2 * k;
            w[k] = cvt2(xrow[ks * 64 + paired_col(order, p0)], xrow[ks * 64 + paired_col(order, p0 + 1)], scale);
          }
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(xp + ((int64_t)ks * R8 + (p >> 3)) * 1024 + sw128_offset(p & 7, c)) = v;
    }
  }
}

// ----------------------------------------------------------------------------
// 6/7. Grouped GEMM on the tensor cores.
//
// Work item = (tile, block): tile = up to 256 grouped rows of one expert,
// block = 128 weight rows (phase 0: 64 rows of W1 and the same 64 rows of W3;
// phase 1: 128 rows of W2).  D (128 weight rows x N tokens, fp32) lives in
// tensor memory, two accumulators so the epilogue of one item overlaps the
// main loop of the next.  Per 64-column K-step the A operand (weights) is
// dequantised by warps 0-3 (one 32-row panel each, one row per lane) from a
// ring of raw quantised 256-column groups, and the B operand (tokens) arrives
// by one bulk copy of the pre-swizzled grouped rows.
// ----------------------------------------------------------------------------
// Two fp32 values -> one 32-bit pair of the operand type (round to nearest
// even; the first value in the low half).
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if (F16) {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
}
constexpr float kF16Max = 65504.f;

// Raw 256-column group of one 32-row panel: the pieces of the device tile
// layout that hold these columns, packed as [codes | small fields].
__device__ __forceinline__ void issue_raw_group(int fmt, const uint8_t* tile, int nb, int gi, uint8_t* dst,
                                                uint64_t* bar) {
  switch (fmt) {
    case BQE_FMT_Q2_0:
      bulk_g2s(dst, tile + gi * 2048, 2048, bar);
      bulk_g2s(dst + 2048, tile + nb * 512 + gi * 256, 256, bar);
      break;
    case BQE_FMT_MXFP4:
      bulk_g2s(dst, tile + gi * 4096, 4096, bar);
      bulk_g2s(dst + 4096, tile + nb * 512 + gi * 256, 256, bar);
      break;
    case BQE_FMT_NVFP4:
      bulk_g2s(dst, tile + gi * 4096, 4096, bar);
      bulk_g2s(dst + 4096, tile + nb * 256 + gi * 512, 512, bar);
      break;
    case BQE_FMT_TQ1:
      bulk_g2s(dst, tile + gi * 1536, 1536, bar);
      bulk_g2s(dst + 1536, tile + nb * 1536 + gi * 256, 256, bar);
      break;
    default:  // Q3_K
      bulk_g2s(dst, tile + gi * 2048, 2048, bar);
      bulk_g2s(dst + 2048, tile + nb * 2048 + gi * 1024, 1024, bar);
      bulk_g2s(dst + 3072, tile + nb * 3072 + gi * 384, 384, bar);
      bulk_g2s(dst + 3456, tile + nb * 3456 + gi * 64, 64, bar);
      break;
  }
}
__host__ __device__ constexpr uint32_t raw_group_bytes(int fmt) { return 32u * 256u / fmt_bw(fmt) * fmt_bb(fmt); }

__device__ __forceinline__ void store_chunk(uint8_t* a_stage, int row, int c, uint32_t w0, uint32_t w1, uint32_t w2,
                                            uint32_t w3) {
  *reinterpret_cast<uint4*>(a_stage + sw128_offset(row, c)) = make_uint4(w0, w1, w2, w3);
}

// Q2_0, K-step kq = block kq of the group: w = d (2q - 3) = 8d (1 + q/4) - 11d,
// one exact fp32 fma per weight (1 + q/4 built from the code bits).
template <bool F16>
__device__ __forceinline__ void dq_q2_0(const uint8_t* P, int kq, int lane, uint8_t* A, int row, bool& bad) {
  const uint4 c4 = *reinterpret_cast<const uint4*>(P + kq * 512 + lane * 16);
  const float d = __half2float(*reinterpret_cast<const __half*>(P + 2048 + (kq * 32 + lane) * 2));
  const float a8 = 8.f * d, b11 = -11.f * d;
  if (F16 && !(3.f * fabsf(d) <= kF16Max)) bad = true;
  const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t word = wd[c >> 1];
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = 8 * (c & 1) + 2 * i;
      const float f0 = __uint_as_float(0x3F800000u | (((word >> (2 * j)) & 3u) << 21));
      const float f1 = __uint_as_float(0x3F800000u | (((word >> (2 * j + 2)) & 3u) << 21));
      o[i] = pack2<F16>(fmaf(f0, a8, b11), fmaf(f1, a8, b11));
    }
    store_chunk(A, row, c, o[0], o[1], o[2], o[3]);
  }
}

// MXFP4, K-step kq = blocks 2kq, 2kq+1: w = e2m1(code) * 2^(E-127), exact.
__device__ __forceinline__ void dq_mxfp4(const uint8_t* P, int kq, int lane, uint8_t* A, int row) {  // bf16 only
#pragma unroll
  for (int bi = 0; bi < 2; ++bi) {
    const int b = 2 * kq + bi;
    const uint4 c4 = *reinterpret_cast<const uint4*>(P + b * 512 + lane * 16);
    const float sc = ue8m0_f32(P[4096 + b * 32 + lane]);
    const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {  // one word = 8 weights = one 16-byte chunk
      uint32_t o[4];
#pragma unroll
      for (int by = 0; by < 4; ++by) {
        const float2 v = e2m1x2_f32((wd[w] >> (8 * by)) & 0xFFu);
        o[by] = pack2<false>(v.x * sc, v.y * sc);
      }
      store_chunk(A, row, bi * 4 + w, o[0], o[1], o[2], o[3]);
    }
  }
}

// NVFP4, K-step kq = blocks 4kq .. 4kq + 3 (16 columns each): w = e2m1(code) *
// e4m3(scale), exact in bf16 (at most 6 significant bits).
__device__ __forceinline__ float e4m3_f32(uint32_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  const float mag = e == 0 ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return (b & 0x80) ? -mag : mag;
}
__device__ __forceinline__ void dq_nvfp4(const uint8_t* P, int kq, int lane, uint8_t* A, int row) {  // bf16 only
#pragma unroll
  for (int bi = 0; bi < 4; ++bi) {
    const int b = 4 * kq + bi;
    const uint2 c2 = *reinterpret_cast<const uint2*>(P + b * 256 + lane * 8);
    const float sc = e4m3_f32(P[4096 + b * 32 + lane]);
    const uint32_t wd[2] = {c2.x, c2.y};
#pragma unroll
    for (int w = 0; w < 2; ++w) {  // one word = 8 weights = one 16-byte chunk
      uint32_t o[4];
#pragma unroll
      for (int by = 0; by < 4; ++by) {
        const float2 v = e2m1x2_f32((wd[w] >> (8 * by)) & 0xFFu);
        o[by] = pack2<false>(v.x * sc, v.y * sc);
      }
      store_chunk(A, row, bi * 2 + w, o[0], o[1], o[2], o[3]);
    }
  }
}

// TQ1, K-step KQ = weights 64 KQ .. 64 KQ + 63 of the 256-weight block.  Byte
// i < 51 holds weights 5i .. 5i+4 as base-3 digits (least significant first,
// digit t = w/d + 1), byte 51 holds weight 255.  A weight is one of -d, 0, +d:
// a byte permute picks its 16-bit pattern from a 3-entry table, two weights
// per permute (selector nibbles 2t, 2t + 1 of each).
template <int KQ>
__device__ __forceinline__ void dq_tq1_k(const uint32_t (&W)[14], uint32_t tab_lo, uint32_t tab_hi, uint8_t* A,
                                         int row) {
  constexpr int J0 = 64 * KQ;
  constexpr int B0 = J0 / 5;
  constexpr int B1 = (J0 + 63) / 5 < 51 ? (J0 + 63) / 5 : 51;
  uint32_t t[(B1 - B0 + 1) * 5];
#pragma unroll
  for (int i = B0; i <= B1; ++i) {
    uint32_t v = (W[i >> 2] >> (8 * (i & 3))) & 0xFFu;
    if (i == 51) {
      t[(i - B0) * 5] = v;  // 0..2
    } else {
#pragma unroll
      for (int r = 0; r < 5; ++r) {
        const uint32_t q = (v * 171u) >> 9;  // v / 3 for v <= 255
        t[(i - B0) * 5 + r] = v - 3u * q;
        v = q;
      }
    }
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = J0 + 8 * c + 2 * i - 5 * B0;
      o[i] = __byte_perm(tab_lo, tab_hi, 0x1010u + t[j] * 0x22u + t[j + 1] * 0x2200u);
    }
    store_chunk(A, row, c, o[0], o[1], o[2], o[3]);
  }
}
template <bool F16>
__device__ __forceinline__ void dq_tq1(const uint8_t* P, int kq, int lane, uint8_t* A, int row) {
  uint32_t W[14];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(P + q * 512 + lane * 16);
    W[4 * q] = v.x; W[4 * q + 1] = v.y; W[4 * q + 2] = v.z; W[4 * q + 3] = v.w;
  }
  const uint2 tail = *reinterpret_cast<const uint2*>(P + 1536 + lane * 8);
  W[12] = tail.x;
  W[13] = tail.y;
  // d in the operand type (fp16: exact; bf16: rounded), then the table
  // {-d, 0 | +d, .}: selector values 0, 2, 4 pick bytes of -d, 0, +d
  const uint32_t dbits =
      F16 ? (tail.y & 0xFFFFu)
          : (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__half2float(__ushort_as_half((unsigned short)(tail.y & 0xFFFFu)))));
  const uint32_t tab_lo = dbits ^ 0x8000u, tab_hi = dbits;
  switch (kq) {
    case 0: dq_tq1_k<0>(W, tab_lo, tab_hi, A, row); break;
    case 1: dq_tq1_k<1>(W, tab_lo, tab_hi, A, row); break;
    case 2: dq_tq1_k<2>(W, tab_lo, tab_hi, A, row); break;
    default: dq_tq1_k<3>(W, tab_lo, tab_hi, A, row); break;
  }
}

// fp16 operand paths of Q2_0 and Q3_K in the "paired" K order of a 64-column
// K-step (the grouped x and h are stored in the same order, so the products
// are unchanged): Q2_0 pairs weights j and j + 8 of every 16, Q3_K weights
// j and j + 16 of every 32, which one shift and mask of the packed codes give
// at once.  The codes become exact small integers in both fp16 lanes (bits
// ORed under the exponent of 1024), one fp16x2 subtract removes the offset
// and one fp16x2 multiply applies the scale, rounding once.
__device__ __forceinline__ uint32_t h2sub(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t h2mul(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ void dq_q2_0_paired(const uint8_t* P, int kq, int lane, uint8_t* A, int row, bool& bad) {
  const uint4 c4 = *reinterpret_cast<const uint4*>(P + kq * 512 + lane * 16);
  const uint32_t db = *reinterpret_cast<const uint16_t*>(P + 2048 + (kq * 32 + lane) * 2);
  if (!(3.f * fabsf(__half2float(__ushort_as_half((unsigned short)db))) <= kF16Max)) bad = true;
  const uint32_t d2 = db | (db << 16);
  const uint32_t wd[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = 4 * half + i;
        const uint32_t sh = j == 0 ? (wd[w] << 1) : (wd[w] >> (2 * j - 1));  // 2 q_j, 2 q_{j+8} at bits 1, 17
        const uint32_t x = (sh & 0x00060006u) | 0x64006400u;                  // 1024 + 2q in each lane
        o[i] = h2mul(h2sub(x, 0x64036403u), d2);                              // d (2q - 3)
      }
      store_chunk(A, row, 2 * w + half, o[0], o[1], o[2], o[3]);
    }
  }
}

__device__ __forceinline__ void dq_q3k_paired(const uint8_t* P, int kq, int lane, uint8_t* A, int row, bool& bad) {
  const uint4 lo4 = *reinterpret_cast<const uint4*>(P + kq * 512 + lane * 16);
  const uint2 hi2 = *reinterpret_cast<const uint2*>(P + 2048 + (kq >> 1) * 512 + lane * 16 + (kq & 1) * 8);
  const uint32_t* scw = reinterpret_cast<const uint32_t*>(P + 3072 + lane * 12);
  const uint32_t sc[4] = {scw[0], scw[1], scw[2], 0u};
  const float d = __half2float(*reinterpret_cast<const __half*>(P + 3456 + lane * 2));
  const uint32_t lo[4] = {lo4.x, lo4.y, lo4.z, lo4.w};
#pragma unroll
  for (int mp = 0; mp < 2; ++mp) {  // sub-blocks a = 4 kq + 2 mp and b = a + 1
    float dsv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int bit = 6 * (4 * kq + 2 * mp + e);
      const uint64_t two = (uint64_t)sc[bit >> 5] | ((uint64_t)sc[(bit >> 5) + 1] << 32);
      dsv[e] = d * (float)((uint32_t)(two >> (bit & 31)) & 63u);
      if (!(4.f * fabsf(dsv[e]) <= kF16Max)) bad = true;
    }
    const __half2 ds2h = __floats2half2_rn(dsv[0], dsv[1]);
    const uint32_t ds2 = *reinterpret_cast<const uint32_t*>(&ds2h);
    const uint32_t X = __byte_perm(lo[2 * mp], lo[2 * mp + 1], 0x5410);  // codes 0..7 of a | of b
    const uint32_t Y = __byte_perm(lo[2 * mp], lo[2 * mp + 1], 0x7632);  // codes 8..15 of a | of b
    const uint32_t H = mp == 0 ? hi2.x : hi2.y;                            // high bits of a | of b
#pragma unroll
    for (int cq = 0; cq < 4; ++cq) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = 4 * cq + i;
        const uint32_t src = j < 8 ? X : Y;
        const uint32_t lo2 = (src >> (2 * (j & 7))) & 0x00030003u;
        const uint32_t hb = j < 2 ? (H << (2 - j)) : (H >> (j - 2));  // bits j, 16 + j at 2, 18
        const uint32_t x = (lo2 | (hb & 0x00040004u)) | 0x64006400u;   // 1024 + q in each lane
        o[i] = h2mul(h2sub(x, 0x64046404u), ds2);                      // d s (q - 4)
      }
      store_chunk(A, row, 4 * mp + cq, o[0], o[1], o[2], o[3]);
    }
  }
}

// Q3_K, K-step kq = weights 64 kq .. 64 kq + 63: q = lo2 + 4 hi1, w = d s_j (q - 4)
// with j = weight / 16; as d s (8 (1 + q/8) - 12), one exact fp32 fma.
template <bool F16>
__device__ __forceinline__ void dq_q3k(const uint8_t* P, int kq, int lane, uint8_t* A, int row, bool& bad) {
  const uint4 lo4 = *reinterpret_cast<const uint4*>(P + kq * 512 + lane * 16);
  const uint2 hi2 = *reinterpret_cast<const uint2*>(P + 2048 + (kq >> 1) * 512 + lane * 16 + (kq & 1) * 8);
  const uint32_t* scw = reinterpret_cast<const uint32_t*>(P + 3072 + lane * 12);
  const uint32_t sc[4] = {scw[0], scw[1], scw[2], 0u};
  const float d = __half2float(*reinterpret_cast<const __half*>(P + 3456 + lane * 2));
  const uint32_t lo[4] = {lo4.x, lo4.y, lo4.z, lo4.w};
  const uint32_t hi[2] = {hi2.x, hi2.y};
#pragma unroll
  for (int m = 0; m < 4; ++m) {  // sub-block 4 kq + m: weights 16 m .. 16 m + 15 of this K-step
    const int bit = 6 * (4 * kq + m);
    const uint64_t two = (uint64_t)sc[bit >> 5] | ((uint64_t)sc[(bit >> 5) + 1] << 32);
    const float ds = d * (float)((uint32_t)(two >> (bit & 31)) & 63u);
    const float a8 = 8.f * ds, b12 = -12.f * ds;
    if (F16 && !(4.f * fabsf(ds) <= kF16Max)) bad = true;
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // 8 weights = one chunk
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = 16 * m + 8 * half + 2 * i + e;  // weight within the K-step
          const uint32_t q = ((lo[j >> 4] >> (2 * (j & 15))) & 3u) | (((hi[j >> 5] >> (j & 31)) & 1u) << 2);
          v[e] = fmaf(__uint_as_float(0x3F800000u | (q << 20)), a8, b12);
        }
        o[i] = pack2<F16>(v[0], v[1]);
      }
      store_chunk(A, row, 2 * m + half, o[0], o[1], o[2], o[3]);
    }
  }
}

// One 64-column K-step of the lane's row, as fp16 (f16) or bf16.  `bad` is set
// when an fp16 weight would leave the fp16 range.  fp16 Q2_0 / Q3_K use the
// paired K order.
__device__ __forceinline__ void dequant_kstep(int fmt, bool f16, const uint8_t* P, int kq, int lane, uint8_t* A,
                                              int row, bool& bad) {
  switch (fmt) {
    case BQE_FMT_Q2_0:
      if (f16) dq_q2_0_paired(P, kq, lane, A, row, bad); else dq_q2_0<false>(P, kq, lane, A, row, bad);
      break;
    case BQE_FMT_MXFP4: dq_mxfp4(P, kq, lane, A, row); break;
    case BQE_FMT_NVFP4: dq_nvfp4(P, kq, lane, A, row); break;
    case BQE_FMT_TQ1:
      if (f16) dq_tq1<true>(P, kq, lane, A, row); else dq_tq1<false>(P, kq, lane, A, row);
      break;
    default:
      if (f16) dq_q3k_paired(P, kq, lane, A, row, bad); else dq_q3k<false>(P, kq, lane, A, row, bad);
      break;
  }
}
// K-step order of a group's grouped operands: paired for fp16 Q2_0 / Q3_K.
__device__ __forceinline__ int kstep_order(int fmt, bool f16) {
  return f16 && (fmt == BQE_FMT_Q2_0 || fmt == BQE_FMT_Q3_K) ? fmt : 0;
}

__device__ __forceinline__ long long pf_clk() { return clock64(); }
__device__ __forceinline__ void pf_dbg(const PfParams& P, int ph, int slot, long long v) {
  if (P.diag && blockIdx.x < kPfDbgCtas)
    atomicAdd((unsigned long long*)(P.ws + P.L.dbg) + ((size_t)ph * kPfDbgCtas + blockIdx.x) * kPfDbgSlots + slot,
              (unsigned long long)v);
}

// Stages of the B area for a tile of npad rows: as many as fit, at most kPfBMaxStages.
__device__ __forceinline__ int b_stages(int npad) {
  const int n = (int)(kPfBStages * kPfBStage / ((uint32_t)npad * 128u));
  return n < kPfBMaxStages ? n : kPfBMaxStages;
}

struct PfItem {
  int g, row0, n, npad, blk, fmt;
  bool f16;             // operand type of this expert: fp16 (else bf16)
  const uint8_t* base;  // slot
};

__device__ __forceinline__ PfItem pf_item(const PfParams& P, int item, int nblk) {
  PfItem it;
  const int3 tl = ((const int3*)(P.ws + P.L.tile))[item / nblk];
  it.g = tl.x;
  it.row0 = tl.y;
  it.n = tl.z;
  it.npad = (tl.z + 15) & ~15;
  it.blk = item % nblk;
  it.fmt = ((const int32_t*)(P.ws + P.L.gfmt))[tl.x];
  it.f16 = ((const int32_t*)(P.ws + P.L.gf16))[tl.x] != 0;
  it.base = (const uint8_t*)((const uint64_t*)(P.ws + P.L.gaddr))[tl.x];
  return it;
}

template <int PH>
__global__ void __launch_bounds__(kPfThreads, 1) k_pf_gemm(PfParams P) {
  extern __shared__ uint8_t pf_smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)pf_smem_raw + 1023) & ~(uintptr_t)1023);
  const long long t_cta = clock64();
  uint8_t* sA = sm + kPfOffA;
  uint8_t* sB = sm + kPfOffB;
  uint8_t* sRaw = sm + kPfOffRaw;
  float* sEpi = (float*)(sm + kPfOffEpi);
  uint64_t* bars = (uint64_t*)(sm + kPfOffBar);
  uint64_t* raw_full = bars;                        // [kPfRawStages]
  uint64_t* raw_empty = bars + kPfRawStages;        // [kPfRawStages]
  uint64_t* a_full = bars + 2 * kPfRawStages;       // [kPfAStages]
  uint64_t* a_empty = a_full + kPfAStages;          // [kPfAStages]
  uint64_t* b_full = a_empty + kPfAStages;          // [kPfBMaxStages]
  uint64_t* b_empty = b_full + kPfBMaxStages;       // [kPfBMaxStages]
  uint64_t* acc_full = b_empty + kPfBMaxStages;     // [2]
  uint64_t* acc_empty = acc_full + 2;               // [2]
  uint64_t* fin = acc_empty + 2;
  uint32_t* s_tmem = (uint32_t*)(fin + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PfGeo& g = P.g;
  const int Kc = PH == 0 ? g.H : g.I;  // contraction length
  const int ngrp = Kc / 256;
  const int kc = chunk_cols(Kc), nch = Kc / kc, gpc = kc / 256;
  const int nblk = PH == 0 ? g.nblkA : g.nblkB;
  const int64_t R8 = g.R / 8;
  const int nitems = ((const int32_t*)(P.ws + P.L.ctr))[0] * nblk;
  int32_t* err = (int32_t*)(P.ws + P.L.err);
  const uint64_t lim = P.limit_ns;

  if (tid == 0) {
    for (int i = 0; i < kPfRawStages; ++i) { mbar_init(&raw_full[i], 1); mbar_init(&raw_empty[i], kPfDqWarps); }
    for (int i = 0; i < kPfAStages; ++i) {
      mbar_init(&a_full[i], 4);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kPfBMaxStages; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 4); }
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  // roles: dequant warps, raw-weight load warp, B load warp, MMA warp, epilogue warps
  constexpr int kWRaw = kPfDqWarps, kWB = kPfDqWarps + 1, kWMma = kPfDqWarps + 2, kWEpi = kPfDqWarps + 3;
  if (warp == kWMma) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == kWRaw || warp == kWB) {
    // ---------------- loads: one warp (lane 0) the raw weight groups, the
    // other the B tiles, each as far ahead as its own ring allows (separate
    // warps: a sleeping wait of one never holds the other) ----------------
    if (lane == 0) {
      const uint8_t* bsrc = P.ws + (PH == 0 ? P.L.xp : P.L.hp);
      const bool raw_lane = warp == kWRaw;
      uint32_t nis = 0;  // issues of this lane's ring so far
      uint32_t b_par = 0, b_used = 0;  // B lane: per barrier, uses mod 2 and whether used
      int last_b = -1;
      bool ok = true;
      long long c_wait = 0;
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
        const PfItem it = pf_item(P, item, nblk);
        const int fmt = it.fmt;
        if (raw_lane) {
          const uint64_t m13 = matrix_bytes(fmt, g.I, g.H);
          const uint32_t tb = tile_bytes(fmt, kc);
          const int nb = kc / fmt_bw(fmt);
          const uint8_t* mat[4];
          int panel[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            if (PH == 0) {
              mat[w] = it.base + (w < 2 ? 0 : m13);
              panel[w] = 2 * it.blk + (w & 1);
            } else {
              mat[w] = it.base + 2 * m13;
              panel[w] = 4 * it.blk + w;
            }
          }
          for (int grp = 0; grp < ngrp; ++grp) {
            const int c = grp / gpc, gi = grp % gpc;
            const uint32_t rs = nis % kPfRawStages, rph = (nis / kPfRawStages) & 1;
            const long long tw = pf_clk();
            if (!mbar_wait_sleep_bounded(&raw_empty[rs], rph ^ 1, lim)) { ok = false; break; }
            c_wait += pf_clk() - tw;
            mbar_arrive_expect_tx(&raw_full[rs], 4 * raw_group_bytes(fmt));
#pragma unroll
            for (int w = 0; w < 4; ++w)
              issue_raw_group(fmt, mat[w] + ((uint64_t)panel[w] * nch + c) * tb, nb, gi,
                              sRaw + rs * kPfRawStage + w * kPfRawPanel, &raw_full[rs]);
            ++nis;
          }
        } else {
          // the B area is re-split for this item's row count; every stage of
          // the previous split is released first (per-barrier use parities)
          const uint32_t bbytes = (uint32_t)it.npad * 128u;
          const int nsb = b_stages(it.npad);
          const long long tw = pf_clk();
          for (int i = 0; i < kPfBMaxStages && ok; ++i)
            if ((b_used >> i) & 1u)
              ok = mbar_wait_sleep_bounded(&b_empty[i], ((b_par >> i) & 1u) ^ 1u, lim);
          c_wait += pf_clk() - tw;
          for (int ks = 0; ks < ngrp * 4 && ok; ++ks) {
            const int sb = ks % nsb;
            if (ks >= nsb) {  // stage sb was used earlier in this item: wait for its release
              const long long t2 = pf_clk();
              if (!mbar_wait_sleep_bounded(&b_empty[sb], ((b_par >> sb) & 1u) ^ 1u, lim)) { ok = false; break; }
              c_wait += pf_clk() - t2;
            }
            mbar_arrive_expect_tx(&b_full[sb], bbytes);
            bulk_g2s(sB + (uint32_t)sb * bbytes, bsrc + ((uint64_t)ks * R8 + (it.row0 >> 3)) * 1024, bbytes,
                     &b_full[sb]);
            b_par ^= 1u << sb;  // uses of barrier sb, mod 2
            b_used |= 1u << sb;
            last_b = sb;
            ++nis;
          }
        }
      }
      if (!ok) set_error(err, BQE_ETIMEOUT, kErrPfProducer);
      if (raw_lane) pf_dbg(P, PH, 0, c_wait);
      // every copy this lane started has landed before the CTA may exit
      if (raw_lane) {  // the last (up to ring size) issues are the only ones still in flight
        for (uint32_t i = 0; i < kPfRawStages && i < nis; ++i) {
          const uint32_t n = nis - 1 - i;
          mbar_wait_sleep_bounded(&raw_full[n % kPfRawStages], (n / kPfRawStages) & 1, lim);
        }
      } else {  // the last use of every B barrier
        for (int i = 0; i < kPfBMaxStages; ++i)
          if ((b_used >> i) & 1u) mbar_wait_sleep_bounded(&b_full[i], ((b_par >> i) & 1u) ^ 1u, lim);
      }
      (void)last_b;
    }
  } else if (warp < kPfDqWarps) {
    // ---------------- dequant: panel warp % 4 (A rows 32 (warp % 4) ..), K-steps n % sets == warp / 4
    const int set = warp / 4, pw = warp % 4;
    uint32_t nr = 0, n = 0;  // raw groups and K-steps passed so far (the whole CTA's sequence)
    bool ok = true, bad = false;
    long long c_raw = 0, c_st = 0, c_work = 0;
    const int row = pw * 32 + lane;
    for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x) {
      const PfItem it = pf_item(P, item, nblk);
      for (int grp = 0; grp < ngrp && ok; ++grp) {
        const uint32_t rs = nr % kPfRawStages, rph = (nr / kPfRawStages) & 1;
        long long t0 = pf_clk();
        if (!__all_sync(0xffffffffu, mbar_wait_sleep_bounded(&raw_full[rs], rph, lim))) { ok = false; break; }
        c_raw += pf_clk() - t0;
        const uint8_t* praw = sRaw + rs * kPfRawStage + pw * kPfRawPanel;
        for (int kq = 0; kq < 4; ++kq, ++n) {
          if ((int)(n % kPfDqSets) != set) continue;
          const uint32_t s = n % kPfAStages, sph = (n / kPfAStages) & 1;
          t0 = pf_clk();
          if (!__all_sync(0xffffffffu, mbar_wait_sleep_bounded(&a_empty[s], sph ^ 1, lim))) { ok = false; break; }
          const long long t1 = pf_clk();
          c_st += t1 - t0;
          dequant_kstep(it.fmt, it.f16, praw, kq, lane, sA + s * kPfAStage, row, bad);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[s]);
          c_work += pf_clk() - t1;
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rs]);
        ++nr;
      }
    }
    if (!ok && lane == 0) set_error(err, BQE_ETIMEOUT, kErrPfDequant);
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, BQE_EUNSUPPORTED, kErrPfRange);
    if (lane == 0 && warp == 0) {
      pf_dbg(P, PH, 1, c_raw);
      pf_dbg(P, PH, 2, c_st);
      pf_dbg(P, PH, 3, c_work);
    }
  } else if (warp == kWMma) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0) {
      uint32_t n = 0;  // K-steps consumed so far
      uint32_t bf_par = 0;  // per B barrier: completions consumed, mod 2
      bool ok = true;
      int lc = 0;
      long long c_op = 0, c_iss = 0, c_acc = 0, c_opb = 0;
      for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++lc) {
        const PfItem it = pf_item(P, item, nblk);
        const int ab = lc & 1;
        const uint32_t aph = (lc >> 1) & 1;
        long long t0 = pf_clk();
        if (!mbar_wait_sleep_bounded(&acc_empty[ab], aph ^ 1, lim)) { ok = false; break; }
        c_acc += pf_clk() - t0;
        tc_fence_after();
        const uint32_t d = tmem + ab * 256;
        const uint32_t idesc = umma_idesc_f16(128, it.npad, !it.f16);
        const int nsb = b_stages(it.npad);
        const uint32_t bbytes = (uint32_t)it.npad * 128u;
        for (int ks = 0; ks < ngrp * 4; ++ks, ++n) {
          const uint32_t sa = n % kPfAStages, pa_ = (n / kPfAStages) & 1;
          const uint32_t sb = (uint32_t)(ks % nsb), pb_ = (bf_par >> sb) & 1u;
          t0 = pf_clk();
          if (!mbar_wait_sleep_bounded(&a_full[sa], pa_, lim)) { ok = false; break; }
          const long long tm = pf_clk();
          if (!mbar_wait_sleep_bounded(&b_full[sb], pb_, lim)) { ok = false; break; }
          const long long t1 = pf_clk();
          c_op += tm - t0;
          c_opb += t1 - tm;
          tc_fence_after();
          const uint64_t da = umma_desc_sw128(sA + sa * kPfAStage);
          const uint64_t db = umma_desc_sw128(sB + sb * bbytes);
          bf_par ^= 1u << sb;
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16) umma_f16(d, da + 2 * k16, db + 2 * k16, idesc, (ks | k16) != 0);
          umma_commit(&a_empty[sa]);
          umma_commit(&b_empty[sb]);
          c_iss += pf_clk() - t1;
        }
        if (!ok) break;
        umma_commit(&acc_full[ab]);
      }
      if (!ok) set_error(err, BQE_ETIMEOUT, kErrPfMma);
      pf_dbg(P, PH, 4, c_op);
      pf_dbg(P, PH, 5, c_iss);
      pf_dbg(P, PH, 6, c_acc);
      pf_dbg(P, PH, 10, lc);
      pf_dbg(P, PH, 11, c_opb);
      // all MMAs issued by this thread are complete before tensor memory is freed
      umma_commit(fin);
      mbar_wait_sleep_bounded(fin, 0, lim);
    }
  } else {
    // ---------------- epilogue: warps 6-9, lane quarter warp % 4 ----------------
    const int q = warp & 3;
    const int et = tid - kWEpi * 32;  // 0..127
    bool ok = true;
    int lc = 0;
    long long c_ew = 0, c_ek = 0;
    for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++lc) {
      const PfItem it = pf_item(P, item, nblk);
      const int ab = lc & 1;
      const uint32_t aph = (lc >> 1) & 1;
      const long long t0 = pf_clk();
      const bool got = __all_sync(0xffffffffu, mbar_wait_sleep_bounded(&acc_full[ab], aph, lim));
      if (named_bar_or(1, 128, !got)) { ok = false; break; }
      const long long t1 = pf_clk();
      c_ew += t1 - t0;
      tc_fence_after();
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + ab * 256;
      if (PH == 0) {
        float* ubuf = sEpi;                                       // [64][17] up values
        uint16_t* htile = (uint16_t*)(sEpi + 64 * 17);            // [16 tokens][64 features] 16-bit
        uint8_t* hp = P.ws + P.L.hp;
        const float* prow_sc = (const float*)(P.ws + P.L.prow_sc);
        const int hord = kstep_order(it.fmt, it.f16);
        for (int c0 = 0; c0 < it.npad; c0 += 16) {
          float v[16];
          tmem_ld16(tq + c0, v);
          const float scl = lane < 16 ? prow_sc[it.row0 + c0 + lane] : 1.f;  // 2^-s of the 16 tokens
          if (q >= 2) {
#pragma unroll
            for (int i = 0; i < 16; ++i) ubuf[((q - 2) * 32 + lane) * 17 + i] = v[i];
          }
          named_bar_sync(1, 128);
          if (q < 2) {
            // gate and up come scaled by 2^s (x was): h 2^s = silu(gate 2^s 2^-s) (up 2^s)
            bool big = false;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float u = ubuf[(q * 32 + lane) * 17 + i];
              const float hv = silu_f(v[i] * __shfl_sync(0xffffffffu, scl, i)) * u;
              const int hpos = paired_pos(hord, q * 32 + lane);  // the W2 K-step order of this expert
              if (it.f16) {
                big |= !(fabsf(hv) <= kF16Max);
                htile[i * 64 + hpos] = __half_as_ushort(__float2half_rn(hv));
              } else {
                htile[i * 64 + hpos] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
              }
            }
            if (__any_sync(0xffffffffu, big) && lane == 0) set_error(err, BQE_EUNSUPPORTED, kErrPfRange);
          }
          named_bar_sync(1, 128);
          {
            const int j = et >> 3, c = et & 7;
            const int p = it.row0 + c0 + j;
            const uint4 val = *reinterpret_cast<const uint4*>(htile + j * 64 + c * 8);
            *reinterpret_cast<uint4*>(hp + ((int64_t)it.blk * R8 + (p >> 3)) * 1024 + sw128_offset(p & 7, c)) = val;
          }
          named_bar_sync(1, 128);
        }
      } else {
        float* yb = sEpi + q * (16 * 33);
        const float* prow_w = (const float*)(P.ws + P.L.prow_w);
        const float* prow_sc = (const float*)(P.ws + P.L.prow_sc);
        float* Y = (float*)(P.ws + P.L.y);
        for (int c0 = 0; c0 < it.npad; c0 += 16) {
          float v[16];
          tmem_ld16(tq + c0, v);
          // mixing weight times 2^-s: the accumulator holds 2^s y
          const float wl = lane < 16 ? prow_w[it.row0 + c0 + lane] * prow_sc[it.row0 + c0 + lane] : 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) yb[i * 33 + lane] = v[i] * __shfl_sync(0xffffffffu, wl, i);
          __syncwarp();
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int i = (lane >> 3) + 4 * r, c4 = (lane & 7) * 4;
            if (c0 + i < it.n) {
              const float4 val = make_float4(yb[i * 33 + c4], yb[i * 33 + c4 + 1], yb[i * 33 + c4 + 2],
                                             yb[i * 33 + c4 + 3]);
              *reinterpret_cast<float4*>(Y + (int64_t)(it.row0 + c0 + i) * g.H + it.blk * 128 + q * 32 + c4) = val;
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
      c_ek += pf_clk() - t1;
    }
    if (!ok && et == 0) set_error(err, BQE_ETIMEOUT, kErrPfEpilogue);
    if (et == 0) {
      pf_dbg(P, PH, 7, c_ew);
      pf_dbg(P, PH, 8, c_ek);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) pf_dbg(P, PH, 9, clock64() - t_cta);
  if (warp == kWMma) tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------
// 8. Combine, one CTA per token: out = y_shared + y_0 + ... + y_{K-1} (each y
// already carries its mixing weight), added in this order.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_pf_combine(PfParams P) {
  const int t = blockIdx.x, K = P.g.K, H = P.g.H;
  const int32_t* pos = (const int32_t*)(P.ws + P.L.pos) + (int64_t)t * (K + 1);
  const float* Y = (const float*)(P.ws + P.L.y);
  __shared__ int s_pos[kMaxTopK + 1];
  if (threadIdx.x <= K) s_pos[threadIdx.x] = pos[threadIdx.x == 0 ? K : threadIdx.x - 1];
  __syncthreads();
  float* o = P.out + (int64_t)t * H;
  for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j <= K; ++j) {
      const int p = s_pos[j];
      if (p < 0) continue;
      const float4 v = __ldcs(reinterpret_cast<const float4*>(Y + (int64_t)p * H + c));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (P.accumulate) {
      const float4 prev = *reinterpret_cast<const float4*>(o + c);
      acc.x += prev.x; acc.y += prev.y; acc.z += prev.z; acc.w += prev.w;
    }
    *reinterpret_cast<float4*>(o + c) = acc;
  }
}

// ----------------------------------------------------------------------------
int launch_prefill(const PfParams& P, cudaStream_t st, cudaEvent_t* ev) {
  static int s_attr_done[64] = {};
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BQE_ECUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BQE_ECUDA;
  if (!s_attr_done[dev]) {
    if (cudaFuncSetAttribute(k_pf_gemm<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPfSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_pf_gemm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPfSmemBytes) !=
            cudaSuccess)
      return BQE_ECUDA;
    s_attr_done[dev] = 1;
  }
  const PfGeo& g = P.g;
  auto mark = [&](int i) {
    if (ev) cudaEventRecord(ev[i], st);
  };
  dim3 lg((g.E + kLgBN - 1) / kLgBN, (g.T + kLgBM - 1) / kLgBM);
  mark(0);
  k_pf_logits<<<lg, 256, 0, st>>>(P.x, P.router_w, (float*)(P.ws + P.L.z), g.T, g.E, g.H);
  mark(1);
  k_pf_select<<<(g.T + 7) / 8, 256, 0, st>>>(P);
  mark(2);
  k_pf_plan<<<1, 1024, 0, st>>>(P);
  mark(3);
  k_pf_fill<<<g.E + 1, 256, 0, st>>>(P);
  mark(4);
  k_pf_gather<<<g.maxTiles, 256, 0, st>>>(P);
  mark(5);
  k_pf_gemm<0><<<sms, kPfThreads, kPfSmemBytes, st>>>(P);
  mark(6);
  k_pf_gemm<1><<<sms, kPfThreads, kPfSmemBytes, st>>>(P);
  mark(7);
  k_pf_combine<<<g.T, 256, 0, st>>>(P);
  mark(8);
  return cudaGetLastError() == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

}  // namespace bqe
