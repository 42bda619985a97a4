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
constexpr int kFinBThreads = 128;  // k_finalize_b CTA size (at most one CTA per SM)
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

// RC: rows decoded together (1 for one-row calls, else kRowChunk)
template <int PHASE, int RC>
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

  // Item t = u * per_u + pg * nch + c (expert u, panel group pg, K chunk c):
  // the quotients by per_u and nch come from a multiply by the rounded-up
  // 2^32 / divisor (up to 2^32 itself for divisor 1), exact for t * divisor < 2^32.
  const uint64_t mag_pu = (0x100000000ull + per_u - 1) / per_u;
  const uint64_t mag_ch = (0x100000000ull + nch - 1) / nch;
  auto split_item = [&](int t, int& u, int& pg, int& c) {
    u = (int)(((uint64_t)t * mag_pu) >> 32);
    const int rem = t - u * per_u;
    pg = (int)(((uint64_t)rem * mag_ch) >> 32);
    c = rem - pg * nch;
  };
  // Stage `s` of item `i`: header and weight tiles.  `pre`: issued before the
  // routing results are visible, so the barrier only learns the byte count now
  // and gets its arrival with the activation rows later.
  auto issue_weights = [&](int s, int u, int pg, int c, int fmt, uint64_t addr, int R, uint32_t tb, bool pre,
                           uint64_t pol) -> uint32_t {
    StageHdr& H = hdr[s];
    H.addr = addr; H.u = u; H.p0 = pg * P_; H.c = (int16_t)c; H.fmt = fmt; H.R = (int16_t)R;
    H.tb = tb; H.nb = (uint16_t)(kc / fmt_bw(fmt)); H.amode = (uint8_t)act_mode(PHASE, fmt, P.variant);
    const uint32_t wbytes = (uint32_t)phase_mats(PHASE) * P_ * tb;
    uint8_t* dst = ring + (size_t)s * slot_bytes;
    if (pre) mbar_expect_tx(&full[s], wbytes);
    const uint64_t src0 = addr + (PHASE == 0 ? 0ull : 2 * matrix_bytes(fmt, g.I, g.H)) +
                          (uint64_t)(pg * P_ * nch + c) * tb;
    const uint64_t m13 = PHASE == 0 ? matrix_bytes(fmt, g.I, g.H) : 0ull;
    for (int j = 0; j < P_; ++j) {
      const uint64_t src = src0 + (uint64_t)j * nch * tb;
      bulk_g2s_hint(dst + j * tb, (const void*)src, tb, &full[s], pol);  // W1 (or W2)
      if (PHASE == 0) bulk_g2s_hint(dst + (P_ + j) * tb, (const void*)(src + m13), tb, &full[s], pol);  // W3
    }
    return wbytes;
  };

  // ---- the shared expert before the routing results --------------------------
  // Its slot comes from the inputs (slot_table[E]), not from the router, so
  // the producer streams the weight tiles of this CTA's first shared-expert
  // items (u = 0 comes first in the item order) into the ring while the
  // previous kernel is still finishing.
  int npre = 0;
  uint64_t pre_addr = 0;
  int pre_fmt = 0;
  if (warp == 0 && lane == 0 && P.slot_table) {
    const int sl = P.slot_table[g.E];
    if (sl >= 0 && sl < P.pool.n_slots) {
      const int fmt = P.pool.slot_fmt[sl];
      const uint64_t off = P.pool.slot_off[sl];
      if (fmt_ok(fmt) && !(off & 15) &&
          off + 2 * matrix_bytes(fmt, g.I, g.H) + matrix_bytes(fmt, g.H, g.I) <= P.pool.base_bytes) {
        pre_addr = (uint64_t)P.pool.base + off;
        pre_fmt = fmt;
        const uint64_t pol = policy_evict_first();
        const uint32_t tb = tile_bytes(fmt, kc);
        for (; npre < nstages && npre < P.max_pre; ++npre) {
          const int t = blockIdx.x + npre * gridDim.x;
          if (t >= per_u) break;
          if (npre == P.drop_item && blockIdx.x == 0) break;  // the test hook's item goes through the main loop
          int u, pg, c;
          split_item(t, u, pg, c);
          issue_weights(npre, u, pg, c, fmt, pre_addr, g.M, tb, true, pol);
        }
      }
    }
  }

  griddep_wait();  // routing / phase A results must be complete and visible
  griddep_launch_dependents();  // the finalize kernel may be scheduled behind this one
  if (P.diag && tid == 0) {
    dbg_time(P.ws, P.L.dbg, PHASE, 2, false);  // first CTA past the wait
    dbg_time(P.ws, P.L.dbg, PHASE, 3, true);   // last CTA past the wait
  }

  // the work list (format, slot address, rows of every distinct expert) and
  // what the producer derives from it, in shared memory, so no item waits on
  // a global load or recomputes a per-expert size
  __shared__ int32_t s_ufmt[kMaxM * kMaxTopK + 1];
  __shared__ int32_t s_unrows[kMaxM * kMaxTopK + 1];
  __shared__ uint64_t s_uaddr[kMaxM * kMaxTopK + 1];
  __shared__ int8_t s_urows[(kMaxM * kMaxTopK + 1) * kMaxM];
  __shared__ uint32_t s_utb[kMaxM * kMaxTopK + 1];   // tile bytes
  __shared__ uint32_t s_uarow[kMaxM * kMaxTopK + 1]; // staged bytes of one activation row
  __shared__ uint64_t s_uact[kMaxM * kMaxTopK + 1];  // workspace offset of the activation rows' chunk 0
  __shared__ uint32_t s_ustr[kMaxM * kMaxTopK + 1];  // ... bytes from one chunk to the next (row stride: chunks * this)
  __shared__ float s_xsc[kMaxM];                     // 2^-s of the f16 rows of x
  // activation rows of expert u: staged bytes of one row, bytes from one chunk
  // to the next, and the workspace offset of its chunk 0
  auto act_table = [&](int u, int fmt, uint32_t& arow, uint32_t& str, uint64_t& act) {
    const int amode = act_mode(PHASE, fmt, P.variant);
    arow = (uint32_t)act_row_bytes(amode, fmt, kc);
    if (amode == kActInt) {
      // one record per (row, chunk): x rows in the format's order, or h rows of this expert
      act = PHASE == 0 ? (fmt == BQE_FMT_TQ1 ? P.L.xrt : P.L.xrq) : P.L.hr + (uint64_t)u * g.M * nch * int_rec_bytes(1, kc);
      str = PHASE == 0 ? arow : int_rec_bytes(1, kc);
    } else {
      act = PHASE == 0 ? (amode == kActF16 ? P.L.xh : P.L.xf) : P.L.h + (uint64_t)u * g.M * g.I * 4;
      str = arow;
    }
  };
  const int nU = *(volatile const int32_t*)(P.ws + P.L.nu);
  const int nItems = nU * per_u;
  if (tid < g.M) s_xsc[tid] = ((const float*)(P.ws + P.L.xsc))[tid];
  for (int u = tid; u < nU; u += blockDim.x) {
    for (int r = 0; r < kMaxM; ++r) s_urows[u * kMaxM + r] = (int8_t)((const int32_t*)(P.ws + P.L.u_rows))[u * kMaxM + r];
    const int fmt = ((const int32_t*)(P.ws + P.L.u_fmt))[u];
    s_ufmt[u] = fmt;
    s_uaddr[u] = ((const uint64_t*)(P.ws + P.L.u_addr))[u];
    s_unrows[u] = ((const int32_t*)(P.ws + P.L.u_nrows))[u];
    if (fmt_ok(fmt)) {
      uint32_t arow, str;
      uint64_t act;
      act_table(u, fmt, arow, str, act);
      s_utb[u] = tile_bytes(fmt, kc);
      s_uarow[u] = arow;
      s_ustr[u] = str;
      s_uact[u] = act;
    }
  }
  __shared__ int s_npre;  // items of this CTA preloaded (shared expert)
  if (tid == 0) s_npre = npre;  // the producer lane is thread 0
  __syncthreads();
  // Preloaded items are processed even when the router reported an error
  // (no items): their stages are armed and must drain.
  const int npre_s = s_npre;

  if (warp == 0) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      int last_issued[16];
      for (int s = 0; s < 16; ++s) last_issued[s] = -1;
      for (int i = 0; i < npre; ++i) last_issued[i] = i;
      long long pw = 0, pi_ = 0;
      const uint64_t pol = policy_evict_first();
      // activation rows of an item into stage s: one bulk copy per row (x rows
      // for W1/W3: the rows that chose the expert; h rows for W2: its own rows)
      auto issue_acts = [&](int s, uint32_t expect_w, uint32_t wbytes, int R, uint32_t arow, uint32_t str,
                            uint64_t act, const int8_t* rows, int c) {
        uint8_t* adst = ring + (size_t)s * slot_bytes + wbytes;
        mbar_arrive_expect_tx(&full[s], expect_w + (uint32_t)R * arow);
        const uint8_t* src0 = P.ws + act + (uint64_t)c * str;
        for (int r = 0; r < R; ++r) {
          const int row = (PHASE == 0 && rows) ? rows[r] : r;
          bulk_g2s(adst + (size_t)r * arow, src0 + (uint64_t)row * nch * str, arow, &full[s]);
        }
      };
      int i = 0;
      if (npre > 0) {
        // the preloaded shared-expert items: their activation rows (all M rows)
        uint32_t arow, str;
        uint64_t act;
        act_table(0, pre_fmt, arow, str, act);
        const uint32_t wb = (uint32_t)phase_mats(PHASE) * P_ * tile_bytes(pre_fmt, kc);
        for (; i < npre; ++i) {
          int u, pg, c;
          split_item(blockIdx.x + i * gridDim.x, u, pg, c);
          const long long t1 = clk();
          issue_acts(i % nstages, 0u, wb, g.M, arow, str, act, nullptr, c);
          pi_ += clk() - t1;
        }
      }
      if (npre > 0 && nItems > 0 && (s_uaddr[0] != pre_addr || s_ufmt[0] != pre_fmt || s_unrows[0] != g.M)) {
        // the work list's shared-expert entry must be the one preloaded
        set_error(err, BQE_EDEVICE, kErrPreload);
        *abort_flag = 1;
      }
      for (int t = blockIdx.x + i * gridDim.x; t < nItems; t += gridDim.x, ++i) {
        const int s = i % nstages;
        if (*abort_flag) break;
        int u, pg, c;
        split_item(t, u, pg, c);
        if (i >= nstages) {
          const long long t0 = clk();
          if (!mbar_wait_sleep_bounded(&empty[s], ((i / nstages) - 1) & 1, P.limit_ns)) {
            set_error(err, BQE_ETIMEOUT, kErrWaitEmpty);
            *abort_flag = 1;
            break;
          }
          pw += clk() - t0;
        }
        const long long t1 = clk();
        if (i == P.drop_item && blockIdx.x == 0) continue;  // test hook: this stage never lands
        const int R = s_unrows[u];
        const uint32_t wbytes = issue_weights(s, u, pg, c, s_ufmt[u], s_uaddr[u], R, s_utb[u], false, pol);
        issue_acts(s, wbytes, wbytes, R, s_uarow[u], s_ustr[u], s_uact[u], &s_urows[u * kMaxM], c);
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
    for (int i = 0;; ++i) {
      const int t = blockIdx.x + i * gridDim.x;
      if (i >= npre_s && t >= nItems) break;
      const int s = i % nstages, b = i % kRed;
      const long long t0 = clk();
      // every lane waits; the warp proceeds only if all lanes saw the stage land
      bool ok = __all_sync(0xffffffffu, mbar_wait_sleep_bounded(&full[s], (i / nstages) & 1, P.limit_ns));
      const long long t1 = clk();
      if (ok && i >= kRed)
        ok = __all_sync(0xffffffffu, mbar_wait_sleep_bounded(&rempty[b], ((i / kRed) - 1) & 1, P.limit_ns));
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
      // the item's sizes come with the header (computed once, by the producer)
      const StageHdr H = hdr[s];
      const uint8_t* slot = ring + (size_t)s * slot_bytes;
      const uint8_t* tile = slot + (size_t)(mat * P_ + pan) * H.tb;
      const uint8_t* act = slot + (size_t)phase_mats(PHASE) * P_ * H.tb;
      float* rb = red + (size_t)b * red_stride;
      consume_rows<RC>(H.R, H.fmt, tile, kc, H.nb, grp, act, lane, rb + cw * g.M * 32, H.amode);
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
  long long ew = 0, eb = 0, tprev = clk();
  const long long tstart = tprev;
  for (int i = 0;; ++i) {
    const int t = blockIdx.x + i * gridDim.x;
    if (i >= npre_s && t >= nItems) break;
    const int b = i % kRed;
    const long long t0 = clk();
    eb += t0 - tprev;
    if (!__all_sync(0xffffffffu, mbar_wait_sleep_bounded(&rfull[b], (i / kRed) & 1, P.limit_ns))) {
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
      float* pa = (float*)(P.ws + P.L.pa);
      // W1 warps of panel pi are cw = pi*G + gi, W3 warps cw = (P + pi)*G + gi
      for (int r = 0; r < mt.R; ++r) {
        // f16 rows carry 2^s (removed here, exact); integer rows were unscaled per block
        const float unscale = amode == kActF16 ? s_xsc[s_urows[mt.u * kMaxM + r]] : 1.0f;
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
// h of 256 columns of row r of expert u (one column per thread)
__device__ __forceinline__ void finalize_a_block(const ExpParams& P, int u, int r, int blk, int fmt) {
  const Geo& g = P.g;
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
  const int tq = fmt == BQE_FMT_TQ1;
  const int bpc = g.kcB / 256, ck = blk / bpc, k = blk % bpc;  // K chunk of W2 holding the block, place in it
  uint8_t* rec = P.ws + P.L.hr + ((size_t)rowi * g.nchB + ck) * int_rec_bytes(1, g.kcB);
  if (tid == 0) rec_put_scale(rec, tq, g.kcB, k, ldexpf(1.0f, -si));
  const float v = ldexpf(hv, si);
  const int Xh = __float2int_rn(v);
  const int Xl = __float2int_rn((v - (float)Xh) * 128.0f);
  rec_put(rec, tq, g.kcB, k, tid, Xh, Xl);
  if (tq && tid < 16) rec_put_pad(rec, g.kcB, k, tid);
  int ph = Xh, pl = Xl;
#pragma unroll
  for (int o = 8; o; o >>= 1) {
    ph += __shfl_xor_sync(0xffffffffu, ph, o);
    pl += __shfl_xor_sync(0xffffffffu, pl, o);
  }
  if ((lane & 15) == 0) rec_put_sums(rec, tq, g.kcB, k, tid >> 4, ph, pl);
}

__global__ void __maxnreg__(32) k_finalize_a(ExpParams P) {  // 32 registers: fits beside a W1/W3 CTA
  const Geo& g = P.g;
  // The W2 kernel may launch now: its CTAs take SMs as the W1/W3 kernel's
  // leave and stream the shared expert's W2 tiles until they may read h.
  griddep_launch_dependents();
  griddep_wait();
  if (P.diag && threadIdx.x == 0) dbg_time(P.ws, P.L.dbg, 2, 4, false);
  const int nbl = g.I / 256;
  // work = (expert, row of the expert, 256 columns).  The expert count, every
  // entry's row count and format come in one round of loads (entries past the
  // count are not used), then the row counts are added up in shared memory.
  __shared__ int s_pre[kMaxM * kMaxTopK + 2];
  __shared__ int s_fmt[kMaxM * kMaxTopK + 1];
  __shared__ int s_nu;
  if (threadIdx.x == 0) s_nu = *(volatile const int32_t*)(P.ws + P.L.nu);
  for (int u = threadIdx.x; u < g.U; u += blockDim.x) {
    s_pre[u + 1] = ((const int32_t*)(P.ws + P.L.u_nrows))[u];
    s_fmt[u] = ((const int32_t*)(P.ws + P.L.u_fmt))[u];
  }
  __syncthreads();
  const int nU = s_nu;
  if (threadIdx.x == 0) {
    s_pre[0] = 0;
    for (int u = 0; u < nU; ++u) s_pre[u + 1] += s_pre[u];
  }
  __syncthreads();
  const int nwork = s_pre[nU] * nbl;
  for (int wk = blockIdx.x; wk < nwork; wk += gridDim.x) {
    const int rowg = wk / nbl, blk = wk % nbl;
    int u = 0;
    while (u + 1 < nU && s_pre[u + 1] <= rowg) ++u;
    const int r = rowg - s_pre[u];
    finalize_a_block(P, u, r, blk, s_fmt[u]);
    __syncthreads();  // shared scratch of the block is reused
  }
  if (P.diag && threadIdx.x == 0) dbg_time(P.ws, P.L.dbg, 2, 5, true);
}

__global__ void __launch_bounds__(kFinBThreads) k_finalize_b(ExpParams P) {
  const Geo& g = P.g;
  griddep_launch_dependents();  // the next layer's router may start loading its weights
  griddep_wait();
  if (P.diag && threadIdx.x == 0) dbg_time(P.ws, P.L.dbg, 2, 6, false);
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
  if (P.diag && threadIdx.x == 0) dbg_time(P.ws, P.L.dbg, 2, 7, true);
}

// The finalize kernels run at most one CTA per SM, each looping over its
// share of the work, so that the whole grid fits beside the expert kernel's
// CTAs (launched early, it waits on the SMs and starts the moment the expert
// kernel completes).
int launch_finalize(const ExpParams& P, int phase, int sms, cudaStream_t st, bool pdl) {
  int grid;
  if (phase == 0) {
    if (P.g.I % 256) return BQE_EUNSUPPORTED;
    grid = P.g.U * P.g.M * (P.g.I / 256);  // (expert, row, 256 columns) work items at most
  } else {
    const int64_t n = (int64_t)P.g.M * P.g.H;
    grid = (int)((n + kFinBThreads - 1) / kFinBThreads);
  }
  if (grid > sms) grid = sms;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(phase == 0 ? 256 : kFinBThreads);
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
  void (*kfns[2][2])(ExpParams) = {{k_experts<0, 1>, k_experts<0, kRowChunk>}, {k_experts<1, 1>, k_experts<1, kRowChunk>}};
  const int rc = P.g.M == 1 ? 0 : 1;
  void (*kfn)(ExpParams) = kfns[phase][rc];
  int ns = 0;
  const uint32_t smem = experts_smem_bytes(P.g, phase, &ns);
  if (ns < 2) return BQE_EUNSUPPORTED;
  // raise the kernel's dynamic shared memory limit once per device (the call is slow)
  static int limit_set[2][2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BQE_ECUDA;
  if (limit_set[phase][rc][dev] < (int)smem) {
    const void* fn = (const void*)kfn;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, fn) != cudaSuccess)
      return BQE_ECUDA;
    const int dyn_max = optin - (int)fa.sharedSizeBytes;  // dynamic + static must fit the opt-in limit
    if (dyn_max < (int)smem) return BQE_EUNSUPPORTED;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) != cudaSuccess)
      return BQE_ECUDA;
    limit_set[phase][rc][dev] = dyn_max;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kfn, P);
  return e == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

}  // namespace bqe
