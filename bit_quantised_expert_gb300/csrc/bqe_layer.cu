// bqe_layer.cu — the whole decode layer in one persistent kernel.
//
// One CTA per SM, launched cooperatively so every CTA is resident and CTAs
// may wait on one another (every such wait is bounded).  A layer streams only
// ~1 MB per SM, so the fixed costs of separate launches, pipeline fills and
// phase boundaries would dominate; here they overlap:
//
//   * from its first cycle the producer warp streams the shared expert's W1/W3
//     tiles (they do not depend on routing: the shared expert is always used);
//   * meanwhile the consumer warps compute this CTA's share of the router GEMV
//     (z = x Wr^T), publish it, wait until every CTA has, and then select the
//     top-k and build the work list locally (the same result in every CTA);
//   * W1/W3 items (expert u, a group of 32-row panels, one K chunk) leave chunk
//     partial sums; the last chunk of a panel group to finish computes
//     h = silu(g) * u for it and bumps the expert's ready count;
//   * W2 items of expert u start as soon as all of u's h panels are ready; the
//     last (expert, chunk) item of an output panel group adds the weighted
//     expert outputs in a fixed order into out.
//
// The selection and mixing follow the router of the field report (384 routed
// experts, 6 per token) with the selection-only bias of the Strata 4090 post,
// section 5.3; the per-format GEMV groups are those of bqe_gemv.cuh.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bqe_gemv.cuh"
#include "bqe_internal.cuh"

namespace bqe {

constexpr int kMaxEpi = 2;       // epilogue warps
constexpr int kRedF = 4;         // reduction buffers between consumers and epilogue warps
constexpr int kMaxU = kMaxM * kMaxTopK + 1;
constexpr int kMaxEF = 512;      // routed experts supported
constexpr uint32_t kLayerDynBudget = 204 * 1024;

struct FRedMeta {
  int item, u, p0, c, R, phase;
};

// Reduction buffers (kRedF x NW x M x 32 floats), also holding the top-k
// candidates (3 x M x NW x K words) before the first item arrives.
__host__ __device__ inline uint32_t layer_red_bytes(const Geo& g, int NW) {
  uint32_t red = ((uint32_t)kRedF * NW * g.M * 32 * 4 + 127u) & ~127u;
  const uint32_t cand = ((uint32_t)3 * g.M * NW * g.K * 4 + 127u) & ~127u;
  return red > cand ? red : cand;
}

__device__ __forceinline__ float silu_l(float t) { return t / (1.0f + expf(-t)); }

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned int* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *p >= target (another CTA's progress); false on timeout.
__device__ __forceinline__ bool wait_counter(const unsigned int* p, uint32_t target, uint64_t limit_ns,
                                             volatile int* abort_flag) {
  if (ld_acquire_u32(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i) {
      __nanosleep(64);
      if (ld_acquire_u32(p) >= target) return true;
    }
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Generic-proxy writes of one CTA read by another CTA's bulk copies (async
// proxy): a proxy fence on the writing side before the release and on the
// reading side after the acquire.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Diagnostic timeline of the fused kernel: globaltimer stamps per CTA in
// ws.dbg block 0, row = CTA, slot k (0 router done, 1 logits seen, 2 work
// list built, 3 consumers done, 4 epilogue done, 5 producer done, 6 end);
// row 1023 slot 0 = earliest CTA start (atomicMin).
__device__ __forceinline__ void fstamp(const LayerParams& P, int k) {
  if (!P.diag || blockIdx.x >= 1023) return;
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  unsigned long long* p = (unsigned long long*)(P.ws + P.L.dbg);
  atomicMax(p + (size_t)blockIdx.x * 8 + k, (unsigned long long)t);
}

__device__ __forceinline__ uint32_t key_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // order-preserving image
}

// Descriptor of the slot of expert e (e == E: the shared expert), checked
// against the pool; fmt 0 marks an invalid slot (the error is recorded).
__device__ inline void slot_desc(const LayerParams& P, int slot, int32_t* err, int& fmt, uint64_t& addr) {
  fmt = 0;
  addr = 0;
  if (slot < 0 || slot >= P.pool.n_slots) {
    set_error(err, BQE_EDEVICE, kErrSlotRange);
    return;
  }
  const int f = P.pool.slot_fmt[slot];
  const uint64_t off = P.pool.slot_off[slot];
  if (!fmt_ok(f)) {
    set_error(err, BQE_EDEVICE, kErrSlotFmt);
    return;
  }
  const uint64_t bytes = 2 * matrix_bytes(f, P.g.I, P.g.H) + matrix_bytes(f, P.g.H, P.g.I);
  if ((off & 15) || off + bytes > P.pool.base_bytes) {
    set_error(err, BQE_EDEVICE, kErrSlotExtent);
    return;
  }
  fmt = f;
  addr = (uint64_t)P.pool.base + off;
}

__global__ void __launch_bounds__(32 * (1 + kMaxWarps + kMaxEpi), 1) k_layer(LayerParams P) {
  const Geo& g = P.g;
  const int H = g.H, I = g.I, E = g.E, K = g.K, M = g.M;
  const int NW = P.NW, NE = P.NE, G = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* err = (int32_t*)(P.ws + P.L.err);
  unsigned int* fctr = (unsigned int*)(P.ws + P.L.fctr);  // [0] logits + inputs published, [1] CTAs done
  unsigned int* cnt_a = (unsigned int*)(P.ws + P.L.cnt_a);
  unsigned int* h_cnt = (unsigned int*)(P.ws + P.L.h_cnt);
  unsigned int* ctr_out = (unsigned int*)(P.ws + P.L.ctr_out);
  float* z = (float*)(P.ws + P.L.z);
  float* xf = (float*)(P.ws + P.L.xf);
  uint16_t* xh = (uint16_t*)(P.ws + P.L.xh);
  float* pa = (float*)(P.ws + P.L.pa);
  float* pb = (float*)(P.ws + P.L.pb);
  float* hbuf = (float*)(P.ws + P.L.h);

  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ StageHdr hdr[16];
  __shared__ __align__(8) uint64_t full[16], empty[16], rfull[kRedF], rempty[kRedF], route_bar;
  __shared__ FRedMeta rmeta[kRedF];
  __shared__ int32_t s_ufmt[kMaxU], s_unrows[kMaxU];
  __shared__ uint64_t s_uaddr[kMaxU];
  __shared__ int8_t s_urows[kMaxU * kMaxM];
  __shared__ int s_nu, s_bad;
  __shared__ volatile int s_abort;
  __shared__ uint32_t s_mask[kMaxEF];
  __shared__ int s_uof[kMaxEF];
  __shared__ int32_t s_table[kMaxEF + 1];
  __shared__ int s_idx[kMaxM][kMaxTopK];
  __shared__ float s_zsel[kMaxM][kMaxTopK];
  __shared__ int s_list[kMaxM * kMaxTopK];
  __shared__ int s_cu[kMaxM][kMaxTopK], s_cr[kMaxM][kMaxTopK];
  __shared__ float s_cw[kMaxM][kMaxTopK];
  __shared__ float s_inv_rms[kMaxM], s_xsc[kMaxM];
  __shared__ int s_emax[kMaxM];
  __shared__ float s_part[4 * 4][kMaxM];  // (expert of this CTA, quarter) partial dot products
  __shared__ int s_wcnt[kMaxEF / 32];

  const uint32_t red_bytes = layer_red_bytes(g, NW);
  float* red = reinterpret_cast<float*>(dsm);
  const int red_stride = NW * M * 32;
  uint8_t* ring = dsm + red_bytes;
  const int nstages = P.nstages;
  const int nct = NW * 32;  // consumer threads

  // geometry of the two item kinds
  const int kcA = g.kcA, nchA = g.nchA, GA = g.GA, PA = g.PA, npgA = g.npanA / g.PA;
  const int kcB = g.kcB, nchB = g.nchB, GB = g.GB, PB = g.PB, npgB = g.npanB / g.PB;
  const int per_uA = npgA * nchA, per_uB = npgB * nchB;

  if (tid == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    for (int b = 0; b < kRedF; ++b) {
      mbar_init(&rfull[b], NW);
      mbar_init(&rempty[b], 1);
    }
    mbar_init(&route_bar, 1);
    s_abort = 0;
    s_bad = 0;
    s_nu = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (P.diag && tid == 0) dbg_span(P.ws, P.L.dbg, 0, false);
  griddep_wait();  // inputs (x or the residual) may come from the previous kernel

  // =========================== producer (warp 0) ===========================
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int last_issued[16];
      for (int s = 0; s < 16; ++s) last_issued[s] = -1;
      // the shared expert is known before routing
      int sh_fmt;
      uint64_t sh_addr;
      slot_desc(P, P.slot_table[E], err, sh_fmt, sh_addr);
      bool routed = false, inputs_ready = false;
      int nA = per_uA, nTot = per_uA;  // until routing: only the shared expert's W1/W3 items
      int i = 0;
      for (int t = blockIdx.x;; t += G, ++i) {
        if (!routed && t >= per_uA) {
          if (!mbar_wait_bounded(&route_bar, 0, P.limit_ns)) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
            break;
          }
          routed = true;
          nA = s_nu * per_uA;
          nTot = s_nu * (per_uA + per_uB);
        }
        if (t >= nTot || s_abort) break;
        if (sh_fmt == 0) break;  // invalid shared slot: nothing is streamed
        const int s = i % nstages;
        if (i >= nstages && !mbar_wait_bounded(&empty[s], ((i / nstages) - 1) & 1, P.limit_ns)) {
          set_error(err, BQE_ETIMEOUT, kErrWaitEmpty);
          s_abort = 1;
          break;
        }
        if (i == P.drop_item && blockIdx.x == 0) continue;  // test hook: this stage never lands
        const bool isA = t < nA;
        const int tt = isA ? t : t - nA;
        const int u = tt / (isA ? per_uA : per_uB), rem = tt % (isA ? per_uA : per_uB);
        const int nch = isA ? nchA : nchB, kc = isA ? kcA : kcB, Pp = isA ? PA : PB;
        const int pg = rem / nch, c = rem % nch;
        const int fmt = u == 0 ? sh_fmt : s_ufmt[u];
        const uint64_t addr = u == 0 ? sh_addr : s_uaddr[u];
        const int R = u == 0 ? M : s_unrows[u];
        StageHdr& Hd = hdr[s];
        Hd.addr = addr; Hd.u = u; Hd.p0 = pg * Pp; Hd.c = c; Hd.fmt = fmt; Hd.R = R; Hd.pad = isA ? 0 : 1;
        // W2 items wait for the expert's h before anything of the stage is issued
        if (!isA && !wait_counter(&h_cnt[u], (uint32_t)npgA, P.limit_ns, &s_abort)) {
          set_error(err, BQE_ETIMEOUT, kErrWaitFull);
          s_abort = 1;
          break;
        }
        if (!isA) fence_proxy_async_global();
        const uint32_t tb = tile_bytes(fmt, kc);
        const uint32_t wbytes = (uint32_t)(isA ? 2 : 1) * Pp * tb;
        const bool half_act = isA && fmt == BQE_FMT_MXFP4 && P.variant == 1;
        const uint32_t arow = (uint32_t)kc * (half_act ? 2u : 4u);
        uint8_t* dst = ring + (size_t)s * P.slot_bytes;
        mbar_arrive_expect_tx(&full[s], wbytes + (uint32_t)R * arow);
        const uint64_t m13 = matrix_bytes(fmt, I, H);
        for (int j = 0; j < Pp; ++j) {
          if (isA) {
            const uint64_t toff = (uint64_t)((pg * Pp + j) * nch + c) * tb;
            bulk_g2s_hint(dst + j * tb, (const void*)(addr + toff), tb, &full[s], pol);               // W1
            bulk_g2s_hint(dst + (Pp + j) * tb, (const void*)(addr + m13 + toff), tb, &full[s], pol);  // W3
          } else {
            const uint64_t toff = 2 * m13 + (uint64_t)((pg * Pp + j) * nch + c) * tb;
            bulk_g2s_hint(dst + j * tb, (const void*)(addr + toff), tb, &full[s], pol);               // W2
          }
        }
        last_issued[s] = i;
        // activations: the staged layer input (published with the logits), or
        // the expert's h.  The copies are issued even on a timeout (valid
        // addresses, stale data) so the stage completes and nothing stays in flight.
        if (isA && !inputs_ready) {
          if (!wait_counter(&fctr[0], (uint32_t)G, P.limit_ns, &s_abort)) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
          }
          fence_proxy_async_global();
          inputs_ready = true;
        }
        uint8_t* adst = dst + wbytes;
        for (int r = 0; r < R; ++r) {
          const void* src;
          if (isA) {
            const int row = u == 0 ? r : s_urows[u * kMaxM + r];
            src = half_act ? (const void*)(xh + (int64_t)row * H + (int64_t)c * kc)
                           : (const void*)(xf + (int64_t)row * H + (int64_t)c * kc);
          } else {
            src = hbuf + ((int64_t)u * M + r) * I + (int64_t)c * kc;
          }
          bulk_g2s(adst + (size_t)r * arow, src, arow, &full[s]);
        }
        if (s_abort) break;
      }
      // leave no copy of this CTA in flight
      for (int s = 0; s < nstages; ++s)
        if (last_issued[s] >= 0) mbar_wait_bounded(&full[s], (last_issued[s] / nstages) & 1, 2000000000ull);
    }
  }
  // ========================= consumers (warps 1..NW) =========================
  else if (warp <= NW) {
    const int ct = tid - 32;  // 0 .. nct-1
    const int cw = warp - 1;
    const int c = blockIdx.x;
    // ---- layer input: bf16 x, or bf16(rmsnorm(resid)); row scales ------------
    for (int i = ct; i <= E; i += nct) s_table[i] = P.slot_table[i];
    if (ct < M) s_emax[ct] = -1000;
    named_bar_sync(1, nct);
    if (P.resid) {
      // RMS of each residual row (every CTA computes the same value)
      for (int m = 0; m < M; ++m) {
        float ss = 0.f;
        for (int k = ct; k < H; k += nct) {
          const float v = P.resid[(int64_t)m * H + k];
          ss = fmaf(v, v, ss);
        }
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) red[cw * M + m] = ss;  // the reduction buffers are free until items arrive
      }
      named_bar_sync(1, nct);
      if (ct < M) {
        float ss = 0.f;
        for (int w = 0; w < NW; ++w) ss += red[w * M + ct];
        s_inv_rms[ct] = 1.0f / sqrtf(ss / (float)H + 1e-6f);
      }
      named_bar_sync(1, nct);
    }
    auto xval = [&](int m, int k) -> uint16_t {  // bf16 bits of the layer input
      if (P.resid) return __bfloat16_as_ushort(__float2bfloat16_rn(P.resid[(int64_t)m * H + k] * s_inv_rms[m]));
      return P.x[(int64_t)m * H + k];
    };
    for (int m = 0; m < M; ++m) {
      uint32_t mx = 0;
      for (int k = ct; k < H; k += nct) mx = max(mx, (uint32_t)(xval(m, k) & 0x7FFFu));
      for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0 && mx) atomicMax(&s_emax[m], (int)(mx >> 7) - 127);
    }
    named_bar_sync(1, nct);
    if (ct < M) s_xsc[ct] = ldexpf(1.0f, -(s_emax[ct] == -1000 ? 0 : 14 - s_emax[ct]));
    {  // this CTA's slice of the staged input copies
      const int n = M * H, per = (n + G - 1) / G, lo = per * c, hi = min(n, lo + per);
      for (int i = lo + ct; i < hi; i += nct) {
        const int m = i / H, k = i % H;
        const uint16_t b = xval(m, k);
        const float v = __uint_as_float((uint32_t)b << 16);
        const int sh = s_emax[m] == -1000 ? 0 : 14 - s_emax[m];
        xf[i] = v;
        xh[i] = __half_as_ushort(__float2half_rn(ldexpf(v, sh)));
        if (P.t_out) P.t_out[i] = b;
      }
      if (c == 0 && ct < M) ((float*)(P.ws + P.L.xsc))[ct] = ldexpf(1.0f, -(s_emax[ct] == -1000 ? 0 : 14 - s_emax[ct]));
    }
    // ---- router GEMV: this CTA's experts c, c+G, c+2G; task = (expert, quarter)
    {
      const int nexp = (E - c + G - 1) / G;  // experts of this CTA (<= 3 for E <= 3G)
      const int Kq = H / 4, ni = Kq / 128;
      const uint64_t pol = policy_evict_first();
      for (int task = cw; task < nexp * 4; task += NW) {
        const int j = task >> 2, q = task & 3, e = c + j * G;
        const float4* wr = (const float4*)(P.router_w + (int64_t)e * H + (int64_t)q * Kq);
        float4 w4[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < ni) w4[i] = ldg_stream_f4(wr + i * 32 + lane, pol);
        float acc[kMaxM];
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) acc[m] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < ni) {
            const int k = q * Kq + (i * 32 + lane) * 4;
#pragma unroll
            for (int m = 0; m < kMaxM; ++m) {
              if (m < M) {
                uint32_t b0, b1, b2, b3;
                if (P.resid) {
                  b0 = xval(m, k); b1 = xval(m, k + 1); b2 = xval(m, k + 2); b3 = xval(m, k + 3);
                } else {
                  const uint2 xv = *reinterpret_cast<const uint2*>(P.x + (int64_t)m * H + k);  // 4 bf16
                  b0 = xv.x & 0xFFFFu; b1 = xv.x >> 16; b2 = xv.y & 0xFFFFu; b3 = xv.y >> 16;
                }
                acc[m] = fmaf(w4[i].x, __uint_as_float(b0 << 16), acc[m]);
                acc[m] = fmaf(w4[i].y, __uint_as_float(b1 << 16), acc[m]);
                acc[m] = fmaf(w4[i].z, __uint_as_float(b2 << 16), acc[m]);
                acc[m] = fmaf(w4[i].w, __uint_as_float(b3 << 16), acc[m]);
              }
            }
          }
        }
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) {
          float v = acc[m];
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0 && m < M) s_part[task][m] = v;
        }
      }
      named_bar_sync(1, nct);
      if (ct < nexp * M) {
        const int j = ct / M, m = ct % M, e = c + j * G;
        z[(int64_t)m * E + e] = s_part[4 * j][m] + s_part[4 * j + 1][m] + s_part[4 * j + 2][m] + s_part[4 * j + 3][m];
      }
    }
    // publish: logits and input copies of this CTA are written
    named_bar_sync(1, nct);
    if (ct == 0) fstamp(P, 0);
    if (ct == 0) {
      fence_proxy_async_global();
      __threadfence();
      atomicAdd(&fctr[0], 1u);
    }
    // ---- every CTA selects for itself once all logits are in -------------------
    if (ct == 0 && !wait_counter(&fctr[0], (uint32_t)G, P.limit_ns, &s_abort)) {
      set_error(err, BQE_ETIMEOUT, kErrWaitFull);
      s_abort = 1;
    }
    if (ct == 0) fstamp(P, 1);
    for (int i = ct; i < E; i += nct) s_mask[i] = 0u;
    named_bar_sync(1, nct);
    if (!s_abort) {
      // warp w keeps the k best of experts {e : (e / 32) % NW == w}; candidates in red
      uint32_t* cand_k = reinterpret_cast<uint32_t*>(red);                   // [M][NW][K]
      int* cand_i = reinterpret_cast<int*>(red) + M * NW * K;
      float* cand_z = reinterpret_cast<float*>(red) + 2 * M * NW * K;
      if (!P.forced) {
        const int nb = (E + 31) / 32;
        for (int m = 0; m < M; ++m) {
          uint32_t kk[kMaxEF / 32];
          float zz[kMaxEF / 32];
          int nmine = 0;
#pragma unroll
          for (int b = 0; b < kMaxEF / 32; ++b) {
            kk[b] = 0u;
            zz[b] = 0.f;
          }
#pragma unroll
          for (int b = 0; b < kMaxEF / 32; ++b) {
            const int blk = cw + b * NW;
            const int e = blk * 32 + lane;
            if (blk < nb && e < E) {
              zz[b] = __ldcg(z + (int64_t)m * E + e);
              const float sg = 1.0f / (1.0f + expf(-zz[b]));
              kk[b] = key_bits(P.bias ? sg + P.bias[e] : sg);
            }
            if (blk < nb) nmine = b + 1;
          }
          for (int j = 0; j < K; ++j) {
            uint32_t lk = 0u;
            int li = 0x7fffffff;
            float lz = 0.f;
            int lb = -1;
#pragma unroll
            for (int b = 0; b < kMaxEF / 32; ++b) {
              const int e = (cw + b * NW) * 32 + lane;
              if (b < nmine && (kk[b] > lk || (kk[b] == lk && kk[b] != 0u && e < li))) {
                lk = kk[b]; li = e; lz = zz[b]; lb = b;
              }
            }
            const uint32_t wk = __reduce_max_sync(0xffffffffu, lk);
            const int best = (int)__reduce_min_sync(0xffffffffu, (lk == wk && wk != 0u) ? (uint32_t)li : 0x7fffffffu);
            const bool mine = wk != 0u && li == best && lk == wk;
#pragma unroll
            for (int b = 0; b < kMaxEF / 32; ++b)
              if (mine && b == lb) kk[b] = 0u;
            const int q = (m * NW + cw) * K + j;
            if (mine) cand_z[q] = lz;
            if (lane == 0) {
              cand_k[q] = wk;
              cand_i[q] = wk != 0u ? best : 0x7fffffff;
            }
          }
        }
      }
      named_bar_sync(1, nct);
      for (int m = cw; m < M; m += NW) {  // warp cw merges row m
        for (int j = 0; j < K; ++j) {
          int best;
          float zsel;
          if (P.forced) {
            best = P.forced[m * K + j];
            if (best < 0 || best >= E) {
              if (lane == 0) { set_error(err, BQE_EDEVICE, kErrForcedIdx); s_bad = 1; }
              best = 0;
            }
            zsel = __ldcg(z + (int64_t)m * E + best);
          } else {
            uint32_t lk = 0u;
            int li = 0x7fffffff, lq = -1;
            for (int q2 = lane; q2 < NW * K; q2 += 32) {
              const int q = m * NW * K + q2;
              const uint32_t kq = cand_k[q];
              const int iq = cand_i[q];
              if (kq > lk || (kq == lk && iq < li)) { lk = kq; li = iq; lq = q; }
            }
            const uint32_t wk = __reduce_max_sync(0xffffffffu, lk);
            best = (int)__reduce_min_sync(0xffffffffu, lk == wk ? (uint32_t)li : 0x7fffffffu);
            const bool mine = lk == wk && li == best && lq >= 0;
            const uint32_t own = __ballot_sync(0xffffffffu, mine);
            float zc = 0.f;
            if (mine) {
              zc = cand_z[lq];
              cand_k[lq] = 0u;
              cand_i[lq] = 0x7fffffff;
            }
            zsel = __shfl_sync(0xffffffffu, zc, own ? __ffs(own) - 1 : 0);
            __syncwarp();
          }
          if (lane == 0) {
            s_idx[m][j] = best;
            s_zsel[m][j] = zsel;
            atomicOr(&s_mask[best], 1u << m);
          }
        }
        __syncwarp();
        // mixing weights from the unbiased scores, as exp(log s_j - max) / sum
        float ls = -INFINITY;
        if (lane < K) {
          const float zz = s_zsel[m][lane];
          ls = zz < 0.f ? zz - log1pf(expf(zz)) : -log1pf(expf(-zz));
        }
        float mx = ls;
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float ev = lane < K ? expf(ls - mx) : 0.f;
        float tot = ev;
        for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (lane < K) {
          const float w = ev / tot;
          s_cw[m][lane] = w;
          if (c == 0) {
            if (P.topk_idx) P.topk_idx[m * K + lane] = s_idx[m][lane];
            if (P.topk_w) P.topk_w[m * K + lane] = w;
          }
        }
      }
      named_bar_sync(1, nct);
      // ---- work list: chosen experts in ascending id order (u = 1..) ---------
      {
        const int nbw = (E + 31) / 32;
        for (int b = cw; b < nbw; b += NW) {
          const int e = b * 32 + lane;
          const bool on = e < E && s_mask[e] != 0u;
          const uint32_t bal = __ballot_sync(0xffffffffu, on);
          if (lane == 0) s_wcnt[b] = __popc(bal);
        }
        named_bar_sync(1, nct);
        for (int b = cw; b < nbw; b += NW) {
          const int e = b * 32 + lane;
          const bool on = e < E && s_mask[e] != 0u;
          const uint32_t bal = __ballot_sync(0xffffffffu, on);
          if (on) {
            int base = 0;
            for (int b2 = 0; b2 < b; ++b2) base += s_wcnt[b2];
            const int pos = base + __popc(bal & ((1u << lane) - 1u));
            s_list[pos] = e;
            s_uof[e] = 1 + pos;
          }
        }
        if (ct == 0) {
          int tot = 0;
          for (int b2 = 0; b2 < nbw; ++b2) tot += s_wcnt[b2];
          s_nu = 1 + tot;
        }
        named_bar_sync(1, nct);
        const int nU = s_nu;
        for (int u = ct; u < nU; u += nct) {
          const int e = u == 0 ? -1 : s_list[u - 1];
          const uint32_t mask = u == 0 ? ((1u << M) - 1u) : s_mask[e];
          int fmt;
          uint64_t addr;
          slot_desc(P, s_table[u == 0 ? E : e], err, fmt, addr);
          if (fmt == 0) s_bad = 1;
          s_ufmt[u] = fmt;
          s_uaddr[u] = addr;
          int n = 0;
          for (int m = 0; m < M; ++m)
            if (mask & (1u << m)) s_urows[u * kMaxM + n++] = (int8_t)m;
          s_unrows[u] = n;
          if (c == 0) ((int32_t*)(P.ws + P.L.u_fmt))[u] = fmt;
        }
        for (int q = ct; q < M * K; q += nct) {
          const int m = q / K, j = q % K;
          const int e = s_idx[m][j];
          s_cu[m][j] = s_uof[e];
          s_cr[m][j] = __popc(s_mask[e] & ((1u << m) - 1u));
        }
        named_bar_sync(1, nct);
        if (ct == 0) {
          if (s_bad) s_nu = 0;  // invalid slot: stream nothing
          if (c == 0) *(int32_t*)(P.ws + P.L.nu) = s_nu;
        }
      }
    }
    named_bar_sync(1, nct);
    if (ct == 0) fstamp(P, 2);
    if (ct == 0) mbar_arrive(&route_bar);  // work list ready (also on abort: s_nu may be stale)
    if (s_abort) goto consumers_done;
    {
      // ---- consume items --------------------------------------------------
      const int nU = s_nu;
      const int nA = nU * per_uA, nTot = nU * (per_uA + per_uB);
      int i = 0;
      for (int t = c; t < nTot; t += G, ++i) {
        const int s = i % nstages, b = i % kRedF;
        bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (i / nstages) & 1, P.limit_ns));
        if (ok && i >= kRedF)
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&rempty[b], ((i / kRedF) - 1) & 1, P.limit_ns));
        if (!ok) {
          if (lane == 0) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
          }
          break;
        }
        const StageHdr Hd = hdr[s];
        const bool isA = t < nA;
        const int kc = isA ? kcA : kcB, Gg = isA ? GA : GB, Pp = isA ? PA : PB;
        const int nwarps = (isA ? 2 : 1) * Pp * Gg;
        float* rb = red + (size_t)b * red_stride;
        if (cw < nwarps) {
          const int mat = cw / (Pp * Gg), pan = (cw / Gg) % Pp, grp = cw % Gg;
          const uint32_t tb = tile_bytes(Hd.fmt, kc);
          const uint8_t* slot = ring + (size_t)s * P.slot_bytes;
          const uint8_t* tile = slot + (size_t)(mat * Pp + pan) * tb;
          const uint8_t* act = slot + (size_t)(isA ? 2 : 1) * Pp * tb;
          const bool half_act = isA && Hd.fmt == BQE_FMT_MXFP4 && P.variant == 1;
          consume_rows<kRowChunk>(Hd.R, Hd.fmt, tile, kc, kc / fmt_bw(Hd.fmt), grp, act, lane, rb + cw * M * 32,
                                  half_act ? kActF16 : kActF32);
        }
        if (cw == 0 && lane == 0) rmeta[b] = FRedMeta{t, Hd.u, Hd.p0, Hd.c, Hd.R, isA ? 0 : 1};
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[s]);
          mbar_arrive(&rfull[b]);
        }
      }
    }
  consumers_done:;
    if (lane == 0) fstamp(P, 3);
  }
  // ========================= epilogue warps ==================================
  else if (warp <= NW + NE) {
    const int ew = warp - NW - 1;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&route_bar, 0, P.limit_ns))) {
      if (lane == 0) {
        set_error(err, BQE_ETIMEOUT, kErrWaitFull);
        s_abort = 1;
      }
    } else if (!s_abort) {
      const int nU = s_nu;
      const int nTot = nU * (per_uA + per_uB);
      int i = 0;
      for (int t = blockIdx.x; t < nTot; t += G, ++i) {
        if (i % NE != ew) continue;
        const int b = i % kRedF;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&rfull[b], (i / kRedF) & 1, P.limit_ns))) {
          if (lane == 0) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
          }
          break;
        }
        const FRedMeta mt = rmeta[b];
        const float* rb = red + (size_t)b * red_stride;
        if (mt.phase == 0) {
          // W1/W3 chunk partials of PA panels (x scale removed: exact power of two)
          const bool half_act = s_ufmt[mt.u] == BQE_FMT_MXFP4 && P.variant == 1;
          const int pgi = mt.p0 / PA;
          for (int r = 0; r < mt.R; ++r) {
            const int row = mt.u == 0 ? r : s_urows[mt.u * kMaxM + r];
            const float unscale = half_act ? s_xsc[row] : 1.0f;
            for (int pi = 0; pi < PA; ++pi) {
              const int p = mt.p0 + pi;
              const int64_t base = (((int64_t)mt.u * g.npanA + p) * nchA + mt.c) * 2 * M;
              float a0 = 0.f, a1 = 0.f;
              for (int gi = 0; gi < GA; ++gi) {
                a0 += rb[((pi * GA + gi) * M + r) * 32 + lane];
                a1 += rb[(((PA + pi) * GA + gi) * M + r) * 32 + lane];
              }
              pa[(base + r) * 32 + lane] = a0 * unscale;
              pa[(base + M + r) * 32 + lane] = a1 * unscale;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&rempty[b]);
          __threadfence();
          __syncwarp();
          unsigned int old = 0;
          if (lane == 0) old = atomicAdd(&cnt_a[mt.u * g.npanA + pgi], 1u);
          old = __shfl_sync(0xffffffffu, old, 0);
          if (old == (unsigned int)(nchA - 1)) {  // last chunk of this panel group: h = silu(g) * u
            __threadfence();
            for (int pi = 0; pi < PA; ++pi) {
              const int p = mt.p0 + pi;
              for (int r = 0; r < mt.R; ++r) {
                float a0 = 0.f, a1 = 0.f;
                for (int cc = 0; cc < nchA; ++cc) {
                  const int64_t base = (((int64_t)mt.u * g.npanA + p) * nchA + cc) * 2 * M;
                  a0 += __ldcg(pa + (base + r) * 32 + lane);
                  a1 += __ldcg(pa + (base + M + r) * 32 + lane);
                }
                hbuf[((int64_t)mt.u * M + r) * I + p * 32 + lane] = silu_l(a0) * a1;
              }
            }
            fence_proxy_async_global();
            __threadfence();
            __syncwarp();
            if (lane == 0) {
              cnt_a[mt.u * g.npanA + pgi] = 0u;
              atomicAdd(&h_cnt[mt.u], 1u);
            }
          }
        } else {
          // W2 chunk partials of PB output panels
          for (int pi = 0; pi < PB; ++pi) {
            const int n = (mt.p0 + pi) * 32 + lane;
            for (int r = 0; r < mt.R; ++r) {
              float y = 0.f;
              for (int gi = 0; gi < GB; ++gi) y += rb[((pi * GB + gi) * M + r) * 32 + lane];
              pb[(((int64_t)mt.u * nchB + mt.c) * M + r) * H + n] = y;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&rempty[b]);
          __threadfence();
          __syncwarp();
          const int pgi = mt.p0 / PB;
          unsigned int old = 0;
          if (lane == 0) old = atomicAdd(&ctr_out[pgi], 1u);
          old = __shfl_sync(0xffffffffu, old, 0);
          if (old == (unsigned int)(nU * nchB - 1)) {  // last item of this output panel group
            __threadfence();
            for (int pi = 0; pi < PB; ++pi) {
              const int n = (mt.p0 + pi) * 32 + lane;
              for (int m = 0; m < M; ++m) {
                float val = 0.f;
                for (int cc = 0; cc < nchB; ++cc) val += __ldcg(pb + ((int64_t)cc * M + m) * H + n);
                for (int j = 0; j < K; ++j) {
                  const int u = s_cu[m][j], r = s_cr[m][j];
                  float yj = 0.f;
                  for (int cc = 0; cc < nchB; ++cc) yj += __ldcg(pb + (((int64_t)u * nchB + cc) * M + r) * H + n);
                  val = fmaf(s_cw[m][j], yj, val);
                }
                float* o = P.out + (int64_t)m * H + n;
                *o = P.accumulate ? *o + val : val;
              }
            }
            if (lane == 0) ctr_out[pgi] = 0u;
          }
        }
      }
    }
  }

  if (warp > NW && lane == 0) fstamp(P, 4);
  if (warp == 0 && lane == 0) fstamp(P, 5);
  // ===================== end: the last CTA resets counters ====================
  __syncthreads();
  if (tid == 0) fstamp(P, 6);
  if (tid == 0) {
    __threadfence();
    const unsigned int old = atomicAdd(&fctr[1], 1u);
    if (old == (unsigned int)(G - 1)) {
      __threadfence();
      for (int u = 0; u < g.U; ++u) h_cnt[u] = 0u;
      fctr[0] = 0u;
      fctr[1] = 0u;
      __threadfence();
    }
  }
}

uint32_t layer_smem_bytes(const Geo& g, int* nstages_out, int* nw_out, uint32_t* slot_out) {
  const int nwA = 2 * g.PA * g.GA, nwB = g.PB * g.GB;
  const int NW = nwA > nwB ? nwA : nwB;
  uint32_t slot = stage_bytes_for(2, g.PA, g.kcA, g.M);
  const uint32_t sb = stage_bytes_for(1, g.PB, g.kcB, g.M);
  if (sb > slot) slot = sb;
  const uint32_t red = layer_red_bytes(g, NW);
  int ns = (int)((kLayerDynBudget - red) / slot);
  if (ns > 8) ns = 8;
  if (nstages_out) *nstages_out = ns;
  if (nw_out) *nw_out = NW;
  if (slot_out) *slot_out = slot;
  return red + (uint32_t)ns * slot;
}

// Fewer panels per item until two ring stages fit next to the reduction
// buffers (the workspace layout does not depend on the panel counts).
static void fit_layer_geo(Geo& g) {
  int ns = 0;
  layer_smem_bytes(g, &ns, nullptr, nullptr);
  while (ns < 2 && (g.PA > 1 || g.PB > 1)) {
    if (g.PA >= g.PB && g.PA > 1) {
      int p = g.PA - 1;
      while (p > 1 && g.npanA % p) --p;
      g.PA = p;
    } else {
      int p = g.PB - 1;
      while (p > 1 && g.npanB % p) --p;
      g.PB = p;
    }
    layer_smem_bytes(g, &ns, nullptr, nullptr);
  }
}

int launch_layer(const LayerParams& P0, int grid, cudaStream_t st) {
  LayerParams P = P0;
  fit_layer_geo(P.g);
  int ns = 0, nw = 0;
  uint32_t slot = 0;
  const uint32_t smem = layer_smem_bytes(P.g, &ns, &nw, &slot);
  if (ns < 2 || P.g.E > kMaxEF || nw > kMaxWarps) return BQE_EUNSUPPORTED;
  static int limit_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BQE_ECUDA;
  if (limit_set[dev] < (int)smem) {
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, k_layer) != cudaSuccess)
      return BQE_ECUDA;
    const int dyn_max = optin - (int)fa.sharedSizeBytes;
    if (dyn_max < (int)smem) return BQE_EUNSUPPORTED;
    if (cudaFuncSetAttribute(k_layer, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) != cudaSuccess)
      return BQE_ECUDA;
    limit_set[dev] = dyn_max;
  }
  LayerParams Q = P;
  Q.nstages = ns;
  Q.NW = nw;
  Q.NE = kMaxEpi;
  Q.slot_bytes = slot;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * (1 + nw + kMaxEpi));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: CTAs wait on one another
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_layer, Q) == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

}  // namespace bqe
