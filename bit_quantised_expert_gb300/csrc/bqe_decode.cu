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

#include "bqe_gemv.cuh"
#include "bqe_internal.cuh"

namespace bqe {


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
    if (P.diag) dbg_span(P.ws, P.L.dbg, PHASE, false);
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
  griddep_launch_dependents();  // the finalize kernel may be scheduled behind this one

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
      const uint64_t pol = policy_evict_first();
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
        const int amode = act_mode(PHASE, fmt, P.variant);
        const uint32_t arow = (uint32_t)act_row_bytes(amode, fmt, kc);
        const uint32_t abytes = (uint32_t)R * arow;
        uint8_t* dst = ring + (size_t)s * slot_bytes;
        mbar_arrive_expect_tx(&full[s], wbytes + abytes);
        const uint64_t m13 = matrix_bytes(fmt, g.I, g.H);
        if (PHASE == 0) {
          for (int j = 0; j < P_; ++j) {
            const uint64_t toff = (uint64_t)((pg * P_ + j) * nch + c) * tb;
            bulk_g2s_hint(dst + j * tb, (const void*)(addr + toff), tb, &full[s], pol);               // W1
            bulk_g2s_hint(dst + (P_ + j) * tb, (const void*)(addr + m13 + toff), tb, &full[s], pol);  // W3
          }
        } else {
          for (int j = 0; j < P_; ++j) {
            const uint64_t toff = 2 * m13 + (uint64_t)((pg * P_ + j) * nch + c) * tb;
            bulk_g2s_hint(dst + j * tb, (const void*)(addr + toff), tb, &full[s], pol);
          }
        }
        uint8_t* adst = dst + wbytes;
        const uint16_t* xh = (const uint16_t*)(P.ws + P.L.xh);
        for (int r = 0; r < R; ++r) {
          const int64_t row = PHASE == 0 ? s_urows[u * kMaxM + r] : 0;
          if (amode == kActInt) {
            // X_hi and X_lo of this chunk in the format's order, then their 16-column sums:
            // the layer input (W1/W3) or the expert's h (W2)
            const uint32_t xb = (uint32_t)act_x_bytes(fmt, kc), xbl = (uint32_t)act_xl_bytes(fmt, kc);
            const int Kr = PHASE == 0 ? g.H : g.I;
            const int64_t rowi = PHASE == 0 ? row : (int64_t)u * g.M + r;
            const uint8_t* hi0 = P.ws + (PHASE == 0 ? (fmt == BQE_FMT_TQ1 ? P.L.xt : P.L.xq) : P.L.hq);
            const uint8_t* lo0 = P.ws + (PHASE == 0 ? (fmt == BQE_FMT_TQ1 ? P.L.xtl : P.L.xql) : P.L.hql);
            const int64_t cofs_h = (int64_t)c * (fmt == BQE_FMT_TQ1 ? (kc / 256) * kTOrderBlock : kc * 2);
            const int64_t cofs_l = (int64_t)c * (fmt == BQE_FMT_TQ1 ? (kc / 256) * kTOrderBlockL : kc);
            const int64_t so = (rowi * (Kr / 16) + (int64_t)c * (kc / 16)) * 4;
            uint8_t* d0 = adst + (size_t)r * arow;
            const bool tq = fmt == BQE_FMT_TQ1;
            const int64_t roh = PHASE == 0 ? (tq ? rowi * (Kr / 256) * kTOrderBlock : rowi * Kr * 2)
                                           : h_row_off_hi(rowi, Kr);
            const int64_t rol = PHASE == 0 ? (tq ? rowi * (Kr / 256) * kTOrderBlockL : rowi * Kr)
                                           : h_row_off_lo(rowi, Kr);
            bulk_g2s(d0, hi0 + roh + cofs_h, xb, &full[s]);
            bulk_g2s(d0 + xb, lo0 + rol + cofs_l, xbl, &full[s]);
            bulk_g2s(d0 + xb + xbl, P.ws + (PHASE == 0 ? P.L.s16 : P.L.hs16) + so, (uint32_t)kc / 4, &full[s]);
            bulk_g2s(d0 + xb + xbl + kc / 4, P.ws + (PHASE == 0 ? P.L.s16l : P.L.hs16l) + so, (uint32_t)kc / 4,
                     &full[s]);
            bulk_g2s(d0 + xb + xbl + kc / 2, P.ws + (PHASE == 0 ? P.L.xsb : P.L.hsb) + (rowi * nch + c) * 16, 16u,
                     &full[s]);
            continue;
          }
          const void* src;
          if (PHASE == 0)
            src = amode == kActF16 ? (const void*)(xh + row * g.H + (int64_t)c * kc)
                                   : (const void*)(xf + row * g.H + (int64_t)c * kc);
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
      consume_rows(H.R, H.fmt, tile, kc, grp, act, lane, rb + cw * g.M * 32, act_mode(PHASE, H.fmt, P.variant));
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
      const int amode = act_mode(PHASE, s_ufmt[mt.u], P.variant);
      const float* xsc = (const float*)(P.ws + P.L.xsc);
      float* pa = (float*)(P.ws + P.L.pa);
      // W1 warps of panel pi are cw = pi*G + gi, W3 warps cw = (P + pi)*G + gi
      for (int r = 0; r < mt.R; ++r) {
        // f16 rows carry 2^s (removed here, exact); integer rows were unscaled per block
        const float unscale = amode == kActF16 ? xsc[s_urows[mt.u * kMaxM + r]] : 1.0f;
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
    if (P.diag) dbg_span(P.ws, P.L.dbg, PHASE, true);
  }
}

// ---------------------------------------------------------------------------
// finalize: add the chunk partials in chunk order
//   phase A: h[u, r, i] = silu(sum_c g_c) * (sum_c u_c)
//   phase B: out[m, n] (+)= y_shared[m, n] + sum_j w[m, j] y[u(m,j), r(m,j), n]
// ---------------------------------------------------------------------------
// h = silu(g) * u, one CTA per (expert, row, 256 columns), one column per
// thread: the chunk partials of g and u added in a fixed order; h kept in fp32
// and, for the integer W2 paths, as X_hi + X_lo / 128 of h 2^si (max |h| 2^si
// of the 256 columns in [2^13, 2^14)) in the order of the expert's format,
// with the sums of X_hi and X_lo over every 16 columns and 2^-si.
__global__ void __launch_bounds__(256) k_finalize_a(ExpParams P) {
  const Geo& g = P.g;
  griddep_wait();
  griddep_launch_dependents();
  const int nU = *(volatile const int32_t*)(P.ws + P.L.nu);
  const int nbl = g.I / 256;
  const int u = blockIdx.x / (g.M * nbl), r = (blockIdx.x / nbl) % g.M, blk = blockIdx.x % nbl;
  if (u >= nU) return;
  if (r >= ((const int32_t*)(P.ws + P.L.u_nrows))[u]) return;
  const int fmt = ((const int32_t*)(P.ws + P.L.u_fmt))[u];
  const float* pa = (const float*)(P.ws + P.L.pa);
  const int nch = g.nchA, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blk * 256 + tid;
  const int p = i >> 5;
  // every chunk partial is loaded before any is added (independent loads in
  // flight together), then added in chunk order
  constexpr int kMaxCh = 8;  // K chunks of W1/W3 taken this way: hidden / chunk <= 8 (else a plain loop)
  float a0 = 0.f, a1 = 0.f;
  if (nch <= kMaxCh) {
    float pg[kMaxCh], pu[kMaxCh];
#pragma unroll
    for (int c = 0; c < kMaxCh; ++c) {
      if (c < nch) {
        const int64_t base = (((int64_t)u * g.npanA + p) * nch + c) * 2 * g.M;
        pg[c] = pa[(base + r) * 32 + lane];
        pu[c] = pa[(base + g.M + r) * 32 + lane];
      }
    }
#pragma unroll
    for (int c = 0; c < kMaxCh; ++c)
      if (c < nch) {
        a0 += pg[c];
        a1 += pu[c];
      }
  } else {
    for (int c = 0; c < nch; ++c) {
      const int64_t base = (((int64_t)u * g.npanA + p) * nch + c) * 2 * g.M;
      a0 += pa[(base + r) * 32 + lane];
      a1 += pa[(base + g.M + r) * 32 + lane];
    }
  }
  const float hv = silu_f(a0) * a1;
  const int64_t rowi = (int64_t)u * g.M + r;
  ((float*)(P.ws + P.L.h))[rowi * g.I + i] = hv;
  if (act_mode(1, fmt, P.variant) != kActInt) return;
  __shared__ uint32_t s_mx[8];
  const uint32_t mx = __reduce_max_sync(0xffffffffu, __float_as_uint(hv) & 0x7FFFFFFFu);
  if (lane == 0) s_mx[warp] = mx;
  __syncthreads();
  uint32_t bm = 0;
  for (int w = 0; w < 8; ++w) bm = max(bm, s_mx[w]);
  const int ex = (int)(bm >> 23);  // biased exponent of max |h| (0: all zero or subnormal)
  const int si = ex == 0 ? 0 : min(max(13 - (ex - 127), -100), 100);
  if (tid == 0) {
    const int bpc = g.kcB / 256;
    ((float*)(P.ws + P.L.hsb))[(rowi * g.nchB + blk / bpc) * 4 + blk % bpc] = ldexpf(1.0f, -si);
  }
  int16_t* hq = (int16_t*)(P.ws + P.L.hq + h_row_off_hi(rowi, g.I));
  int8_t* hql = (int8_t*)(P.ws + P.L.hql + h_row_off_lo(rowi, g.I));
  const float v = ldexpf(hv, si);
  const int Xh = __float2int_rn(v);
  const int Xl = __float2int_rn((v - (float)Xh) * 128.0f);
  const int j = tid;
  if (fmt == BQE_FMT_TQ1) {
    const int run = j / 20, jr = j % 20, q4 = jr / 5, rd = jr % 5;
    hq[blk * 264 + run * 20 + 4 * rd + 2 * (q4 >> 1) + (q4 & 1)] = (int16_t)Xh;
    hql[blk * 272 + run * 20 + 4 * rd + q4] = (int8_t)Xl;
    if (tid < 16) {  // T-order slots past column 255 and the padding
      const int slot = tid < 4 ? 240 + 4 * (tid + 1) + 3 : 260 + (tid - 4);
      if (tid < 8) hq[blk * 264 + slot] = 0;
      hql[blk * 272 + slot] = 0;
    }
  } else {
    const int jj = j & 15, kq = jj & 3, iq = jj >> 2;
    hq[blk * 256 + (j & ~15) + 4 * kq + 2 * (iq >> 1) + (iq & 1)] = (int16_t)Xh;
    hql[blk * 256 + (j & ~15) + 4 * kq + iq] = (int8_t)Xl;
  }
  int ph = Xh, pl = Xl;
#pragma unroll
  for (int o = 8; o; o >>= 1) {
    ph += __shfl_xor_sync(0xffffffffu, ph, o);
    pl += __shfl_xor_sync(0xffffffffu, pl, o);
  }
  if ((lane & 15) == 0) {
    ((int32_t*)(P.ws + P.L.hs16))[rowi * (g.I / 16) + blk * 16 + (tid >> 4)] = ph;
    ((int32_t*)(P.ws + P.L.hs16l))[rowi * (g.I / 16) + blk * 16 + (tid >> 4)] = pl;
  }
}

__global__ void __launch_bounds__(256) k_finalize_b(ExpParams P) {
  const Geo& g = P.g;
  griddep_wait();
  griddep_launch_dependents();
  const int nU = *(volatile const int32_t*)(P.ws + P.L.nu);
  const float* pb = (const float*)(P.ws + P.L.pb);
  const int nch = g.nchB;
  if (nU == 0) return;  // the router reported an error; out is left untouched
  // every row's (expert slot, row in expert, weight) once in shared memory, so
  // all partial loads of an output element are independent
  __shared__ int s_cu[kMaxM * kMaxTopK], s_cr[kMaxM * kMaxTopK];
  __shared__ float s_cw[kMaxM * kMaxTopK];
  for (int i = threadIdx.x; i < g.M * g.K; i += blockDim.x) {
    s_cu[i] = ((const int32_t*)(P.ws + P.L.comb_u))[i];
    s_cr[i] = ((const int32_t*)(P.ws + P.L.comb_r))[i];
    s_cw[i] = ((const float*)(P.ws + P.L.comb_w))[i];
  }
  __syncthreads();
  const int64_t n = (int64_t)g.M * g.H;
  constexpr int kMaxCh = 4;  // K chunks of W2 taken the fast way: inter / chunk <= 4 (else plain loops)
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int m = (int)(t / g.H), col = (int)(t % g.H);
    if (nch > kMaxCh) {  // many W2 chunks: plain loops, same order
      float val = 0.f;
      for (int c = 0; c < nch; ++c) val += pb[((int64_t)c * g.M + m) * g.H + col];
      for (int j = 0; j < g.K; ++j) {
        const int u = s_cu[m * g.K + j], r = s_cr[m * g.K + j];
        float yj = 0.f;
        for (int c = 0; c < nch; ++c) yj += pb[(((int64_t)u * nch + c) * g.M + r) * g.H + col];
        val = fmaf(s_cw[m * g.K + j], yj, val);
      }
      float* o = P.out + t;
      *o = P.accumulate ? *o + val : val;
      continue;
    }
    // all partials of this element loaded first (independent loads in flight
    // together), then added in a fixed order: shared expert, then j = 0..K-1
    float ps[kMaxCh], py[kMaxTopK][kMaxCh];
#pragma unroll
    for (int c = 0; c < kMaxCh; ++c)
      if (c < nch) ps[c] = pb[((int64_t)c * g.M + m) * g.H + col];  // shared expert, u = 0
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < g.K) {
        const int u = s_cu[m * g.K + j], r = s_cr[m * g.K + j];
#pragma unroll
        for (int c = 0; c < kMaxCh; ++c)
          if (c < nch) py[j][c] = pb[(((int64_t)u * nch + c) * g.M + r) * g.H + col];
      }
    }
    float val = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxCh; ++c)
      if (c < nch) val += ps[c];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < g.K) {
        float yj = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxCh; ++c)
          if (c < nch) yj += py[j][c];
        val = fmaf(s_cw[m * g.K + j], yj, val);
      }
    }
    float* o = P.out + t;
    *o = P.accumulate ? *o + val : val;
  }
}

int launch_finalize(const ExpParams& P, int phase, int sms, cudaStream_t st, bool pdl) {
  int grid;
  if (phase == 0) {
    if (P.g.I % 256) return BQE_EUNSUPPORTED;
    grid = P.g.U * P.g.M * (P.g.I / 256);  // one CTA per (expert, row, 256 columns)
  } else {
    const int64_t n = (int64_t)P.g.M * P.g.H;
    grid = (int)((n + 255) / 256);
    if (grid > 2 * sms) grid = 2 * sms;
    if (grid < 1) grid = 1;
  }
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
