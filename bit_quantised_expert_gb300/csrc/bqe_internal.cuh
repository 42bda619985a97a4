// bqe_internal.cuh — shared definitions of the CUDA library: block formats,
// the device slot layout, workspace layout, and thin PTX wrappers for
// mbarrier / bulk-copy / grid-dependency control on sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bqe.h"

namespace bqe {

// ----------------------------------------------------------------------------
// Block formats.  Weights per block / bytes per block (bits per weight from
// the Strata 4090 post, section 5.1, and the FP4 per-32 block of the field
// report): TQ1 256/56, Q2_0 64/18, Q3_K 256/110, MXFP4 32/17.
// ----------------------------------------------------------------------------
__host__ __device__ constexpr int fmt_bw(int f) {
  return f == BQE_FMT_TQ1 ? 256 : f == BQE_FMT_Q2_0 ? 64 : f == BQE_FMT_Q3_K ? 256 : f == BQE_FMT_MXFP4 ? 32 : 0;
}
__host__ __device__ constexpr int fmt_bb(int f) {
  return f == BQE_FMT_TQ1 ? 56 : f == BQE_FMT_Q2_0 ? 18 : f == BQE_FMT_Q3_K ? 110 : f == BQE_FMT_MXFP4 ? 17 : 0;
}
__host__ __device__ constexpr bool fmt_ok(int f) { return f >= BQE_FMT_TQ1 && f <= BQE_FMT_MXFP4; }

// ----------------------------------------------------------------------------
// Device layout of one matrix (rows x K) of a slot.
//
//  * rows are grouped in panels of 32 (one row per lane of a warp);
//  * K is cut in chunks of kc columns, kc = the largest of 1024/768/512/256
//    dividing K, so every chunk holds whole blocks of every format;
//  * tile (panel p, chunk c) is contiguous, tiles in order p*nchunks + c;
//  * inside a tile (nb = kc / block_weights blocks per row), every
//    per-(row, block) field is stored field-major, then block, then row, and
//    fields of 16*n bytes are further split into n 16-byte pieces, so that 32
//    lanes reading the same piece of the same block for their own row read
//    512 contiguous bytes:
//      MXFP4: codes16 @ b*512 + r*16           | E   @ nb*512 + b*32 + r
//      Q2_0 : codes16 @ b*512 + r*16           | d   @ nb*512 + (b*32+r)*2
//      TQ1  : bytes0..47 @ (b*3+q)*512 + r*16  | bytes48..55 @ nb*1536 + (b*32+r)*8
//      Q3_K : lo64 @ (b*4+q)*512 + r*16        | hi32 @ nb*2048 + (b*2+q)*512 + r*16
//             | scales12 @ nb*3072 + (b*32+r)*12 | d @ nb*3456 + (b*32+r)*2
//  The bytes of every block are exactly its canonical bytes, rearranged.
// ----------------------------------------------------------------------------
__host__ __device__ constexpr int chunk_cols(int K) {
  return (K % 1024 == 0) ? 1024 : (K % 768 == 0) ? 768 : (K % 512 == 0) ? 512 : 256;
}
__host__ __device__ constexpr uint32_t tile_bytes(int f, int kc) {
  return 32u * (uint32_t)(kc / fmt_bw(f)) * (uint32_t)fmt_bb(f);
}
__host__ __device__ constexpr uint64_t matrix_bytes(int f, int rows, int K) {
  return (uint64_t)rows * (uint64_t)(K / fmt_bw(f)) * (uint64_t)fmt_bb(f);
}

// Destination offset inside a tile of canonical byte `i` of block `b` of row
// `r` (nb blocks per row in the tile).
__host__ __device__ inline uint32_t tile_byte_offset(int f, int nb, int b, int r, int i) {
  switch (f) {
    case BQE_FMT_MXFP4:
      return i < 16 ? (uint32_t)(b * 512 + r * 16 + i) : (uint32_t)(nb * 512 + b * 32 + r);
    case BQE_FMT_Q2_0:
      return i < 16 ? (uint32_t)(b * 512 + r * 16 + i) : (uint32_t)(nb * 512 + (b * 32 + r) * 2 + (i - 16));
    case BQE_FMT_TQ1:
      return i < 48 ? (uint32_t)((b * 3 + i / 16) * 512 + r * 16 + (i % 16))
                    : (uint32_t)(nb * 1536 + (b * 32 + r) * 8 + (i - 48));
    case BQE_FMT_Q3_K:
      if (i < 64) return (uint32_t)((b * 4 + i / 16) * 512 + r * 16 + (i % 16));
      if (i < 96) return (uint32_t)(nb * 2048 + (b * 2 + (i - 64) / 16) * 512 + r * 16 + ((i - 64) % 16));
      if (i < 108) return (uint32_t)(nb * 3072 + (b * 32 + r) * 12 + (i - 96));
      return (uint32_t)(nb * 3456 + (b * 32 + r) * 2 + (i - 108));
  }
  return 0;
}

// ----------------------------------------------------------------------------
// Decode-call geometry shared by host and kernels.
// ----------------------------------------------------------------------------
constexpr int kMaxM = 8;          // rows per decode call
constexpr int kMaxTopK = 16;
constexpr int kRowChunk = 4;      // rows accumulated together by the widest inner loops
constexpr int kMaxU = 64;         // distinct experts of one decode call (M top_k + 1 <= 64)

struct Geo {
  int H, I, E, K, M;
  int U;                          // max distinct experts incl. the shared one = M*K + 1 (<= E+1)
  int kcA, nchA, GA, npanA;       // W1/W3: K = H in chunks of kcA, GA 256-column groups per chunk, I/32 panels
  int kcB, nchB, GB, npanB;       // W2: K = I in chunks of kcB, GB groups per chunk, H/32 panels
};

__host__ __device__ inline Geo make_geo(int H, int I, int E, int K, int M) {
  Geo g;
  g.H = H; g.I = I; g.E = E; g.K = K; g.M = M;
  g.U = M * K + 1;
  if (g.U > E + 1) g.U = E + 1;
  g.kcA = chunk_cols(H); g.nchA = H / g.kcA; g.GA = g.kcA / 256; g.npanA = I / 32;
  g.kcB = chunk_cols(I); g.nchB = I / g.kcB; g.GB = g.kcB / 256; g.npanB = H / 32;
  return g;
}

// Integer staging record of one activation row and one K chunk of kc
// columns (kc a multiple of 256):
//   [X_hi | X_lo | int32 sums of X_hi per 16 columns | the same of X_lo |
//    2^-si of each 256 columns (4 float slots)]
// with X_hi / X_lo in "Q order" (tq = 0: 2 kc + kc bytes) or "T order"
// (tq = 1: 528 + 272 bytes per 256 columns).  One record is exactly one
// staged activation row of a ring stage, so it moves with one bulk copy.
__host__ __device__ constexpr uint32_t int_rec_hi_bytes(int tq, int kc) { return tq ? (kc / 256) * 528 : kc * 2; }
__host__ __device__ constexpr uint32_t int_rec_lo_bytes(int tq, int kc) { return tq ? (kc / 256) * 272 : kc; }
__host__ __device__ constexpr uint32_t int_rec_bytes(int tq, int kc) {
  return int_rec_hi_bytes(tq, kc) + int_rec_lo_bytes(tq, kc) + kc / 2 + 16;
}

// Workspace layout (offsets in bytes, each 256-aligned).
struct WsLayout {
  // the router kernel's arrival counter and the call's work list (distinct
  // experts: slot, format, address, rows), combine indices and weights
  uint64_t err, ctr_route, nu, u_slot, u_fmt, u_addr, u_nrows, u_rows, comb_u, comb_r, comb_w;
  // logits; the layer input in fp32, in f16 x 2^s, 2^-s per row, and as the
  // integer records of the two orders; the diagnostic counters
  uint64_t z, xf, xh, xsc, xrq, xrt, dbg;
  // single-kernel decode layer: (selection key, logit) of every (row, expert)
  uint64_t zk;
  // single-kernel decode layer (k_moe): call epoch, logits arrival counter,
  // per work-list expert the counts of its W1/W3 items done and of its h
  // units written; per "row slot" (an expert's r-th row; M (K + 1) slots at
  // most) the K-chunk partials of g/u, h in fp32 and the integer records of h
  uint64_t epoch, zt, m_ca, m_ch, m_pa, m_h, m_hr;
  uint64_t total;
};
constexpr int kDbgSlots = 8;      // per-CTA counters of the diagnostic mode
constexpr int kDbgMaxCtas = 1024;

__host__ __device__ inline uint64_t al256(uint64_t x) { return (x + 255) & ~(uint64_t)255; }

__host__ __device__ inline WsLayout make_ws(const Geo& g) {
  WsLayout w;
  uint64_t o = 0;
  w.err = o; o = al256(o + 16);
  w.ctr_route = o; o = al256(o + 16);
  w.nu = o; o = al256(o + 16);
  w.u_slot = o; o = al256(o + 4ull * g.U);
  w.u_fmt = o; o = al256(o + 4ull * g.U);
  w.u_addr = o; o = al256(o + 8ull * g.U);
  w.u_nrows = o; o = al256(o + 4ull * g.U);
  w.u_rows = o; o = al256(o + 4ull * g.U * kMaxM);
  w.comb_u = o; o = al256(o + 4ull * g.M * g.K);
  w.comb_r = o; o = al256(o + 4ull * g.M * g.K);
  w.comb_w = o; o = al256(o + 4ull * g.M * g.K);
  w.z = o; o = al256(o + 4ull * g.M * g.E);
  w.xf = o; o = al256(o + 4ull * g.M * g.H);
  w.xh = o; o = al256(o + 2ull * g.M * g.H);   // f16(x * 2^s_m): exact, per-row power-of-two scale
  w.xsc = o; o = al256(o + 4ull * kMaxM);      // 2^-s_m
  // x as X_hi + X_lo / 128 with X_hi = rint(x 2^si) (int16) and X_lo the
  // int8 residual: one record per (row, K chunk) in each of the two orders
  // of the integer GEMV paths (int_rec_bytes)
  w.xrq = o; o = al256(o + (uint64_t)int_rec_bytes(0, g.kcA) * g.M * g.nchA);
  w.xrt = o; o = al256(o + (uint64_t)int_rec_bytes(1, g.kcA) * g.M * g.nchA);
  w.dbg = o; o = al256(o + 8ull * 3 * kDbgMaxCtas * kDbgSlots);
  w.zk = o; o = al256(o + 8ull * g.M * g.E);
  // the call epoch and the counters are contiguous: [epoch, m_pa) clears them
  w.epoch = o; o = al256(o + 16);
  w.zt = o; o = al256(o + 16);                                     // logits arrival counter (64-bit)
  w.m_ca = o; o = al256(o + 4ull * kMaxU);                         // W1/W3 items done, per expert
  w.m_ch = o; o = al256(o + 4ull * kMaxU);                         // h units written, per expert
  const uint64_t nrs = (uint64_t)g.M * (g.K + 1);
  w.m_pa = o; o = al256(o + 4ull * nrs * g.npanA * g.nchA * 2 * 32);
  w.m_h = o; o = al256(o + 4ull * nrs * g.I);
  w.m_hr = o; o = al256(o + (uint64_t)int_rec_bytes(1, g.kcB) * nrs * g.nchB);
  w.total = o;
  return w;
}

// Kernel parameter blocks (passed by value to the kernels).
struct RouteParams {
  Geo g;
  WsLayout L;
  uint8_t* ws;
  const uint16_t* x;          // bf16 M x H, or null when resid is given
  const float* resid;         // fp32 M x H (chained step: normalise first)
  uint16_t* t_out;            // optional bf16 M x H copy of the layer input
  const float* router_w;      // E x H
  const float* bias;          // E or null
  const int32_t* forced;      // M x K or null
  const int32_t* slot_table;  // E + 1
  bqe_pool pool;
  int32_t* topk_idx;          // optional M x K
  float* topk_w;              // optional M x K
  int diag;                   // 1: add cycle counts into ws.dbg
};

// Single-kernel decode layer (bqe_moe.cu).
struct MoeParams {
  Geo g;
  WsLayout L;
  uint8_t* ws;
  const uint16_t* x;          // bf16 M x H, or null when resid is given
  const float* resid;         // fp32 M x H (chained step: normalise first, out += into it)
  uint16_t* t_out;            // optional bf16 M x H copy of the layer input
  const float* router_w;      // E x H
  const float* bias;          // E or null
  const int32_t* forced;      // M x K or null
  const int32_t* slot_table;  // E + 1
  bqe_pool pool;
  float* out;
  int accumulate;
  int32_t* topk_idx;
  float* topk_w;
  uint32_t ring_bytes;        // byte ring for work items
  uint32_t xstage_off;        // ring offset of the bf16 layer input (used until the routing is known)
  uint32_t rt_off;            // ring offset of this CTA's router rows (used until the routing is known)
  uint64_t magA, magA2, magB, magB2;  // ceil(2^32 / d) for the item-index divisors (exact here)
  int PB;                     // W2 output panels per item
  int drop_item, diag;
  uint64_t limit_ns;
};
int launch_moe(const MoeParams& P, int grid, cudaStream_t st);
// Host-side argument checks of a decode-layer call (bqe_api.cu).
int check_layer_args(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* resid, const float* router_w,
                     const bqe_pool* pool, const int32_t* slot_table, const float* out);
// The decode layer on workspace ws (bqe_api.cu); diag = 0 keeps the
// diagnostic counters off whatever the process-wide setting.
int moe_forward(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* router_w, const float* sel_bias,
                const bqe_pool* pool, const int32_t* slot_table, const int32_t* forced_idx, float* out,
                int32_t accumulate, int32_t* topk_idx, float* topk_w, void* ws, uint64_t ws_bytes, cudaStream_t st,
                bool allow_diag);

uint32_t layer_smem_bytes(const Geo& g, int* nstages_out, int* nw_out, uint32_t* slot_out);

// Launchers (one per translation unit that owns the kernel).
int launch_route(const RouteParams& P, cudaStream_t st, bool pdl);

// Error detail codes written to ws.err[1].
enum { kErrSlotRange = 1, kErrSlotFmt = 2, kErrSlotExtent = 3, kErrWaitFull = 4, kErrWaitEmpty = 5,
       kErrForcedIdx = 6 };  // 7..11: the prefill kernels

#ifdef __CUDACC__
// ----------------------------------------------------------------------------
// PTX wrappers (sm_90+ mbarrier / bulk copy; sm_90+ griddepcontrol).
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Raise the transaction count of the current phase without arriving (bulk
// copies issued before the arrival that completes the phase).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_try_wait, but the thread may be suspended until the phase completes
// or about `hint_ns` pass, instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: spins until the phase with `parity` completes or `limit_ns`
// elapses; returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// Bounded wait that lets the thread sleep between checks (for roles that wait
// long, so their spinning takes no issue slots from the working warps).
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes, dst, src
// all multiples of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// L2 policy for data read exactly once per call (expert and router weights):
// evicted first, so the code, work lists and activations stay in L2.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// L2 policy for data fetched ahead of its use in a later kernel of the same
// call: kept while the streams of evict-first data pass through L2.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Bulk prefetch of [src, src + bytes) into L2 (bytes and src multiples of 16;
// no completion to wait for).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// This CTA's share [lo, hi) of n bytes split over `parts` CTAs, on 16-byte
// boundaries.
__device__ __forceinline__ void cta_share16(uint64_t n, int part, int parts, uint64_t& lo, uint64_t& hi) {
  const uint64_t per = ((n + parts - 1) / parts + 15) & ~(uint64_t)15;
  lo = per * part;
  hi = lo + per;
  if (lo > n) lo = n;
  if (hi > n) hi = n;
}
__device__ __forceinline__ float4 ldg_stream_f4(const float4* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
// Writers of the integer staging records (int_rec_bytes): X_hi / X_lo of
// column j (0..255) of the k-th 256-column block of the chunk, in the
// record's order.  Q order: within 16 columns, X_hi word 2q = (x_q, x_{q+4}),
// word 2q + 1 = (x_{q+8}, x_{q+12}), X_lo word q = (x_q, x_{q+4}, x_{q+8},
// x_{q+12}).  T order: in run m of 20 columns, X_hi word 2r = (x_{20m+r},
// x_{20m+5+r}), word 2r + 1 = (x_{20m+10+r}, x_{20m+15+r}), X_lo word r =
// (x_{20m+r}, x_{20m+5+r}, x_{20m+10+r}, x_{20m+15+r}); slots past column
// 255 are zero (rec_put_pad).
__device__ __forceinline__ void rec_put(uint8_t* rec, int tq, int kc, int k, int j, int Xh, int Xl) {
  int16_t* hi = reinterpret_cast<int16_t*>(rec);
  int8_t* lo = reinterpret_cast<int8_t*>(rec + int_rec_hi_bytes(tq, kc));
  if (tq) {
    const int run = j / 20, jr = j % 20, q4 = jr / 5, rd = jr % 5;
    hi[k * 264 + run * 20 + 4 * rd + 2 * (q4 >> 1) + (q4 & 1)] = (int16_t)Xh;
    lo[k * 272 + run * 20 + 4 * rd + q4] = (int8_t)Xl;
  } else {
    const int jj = j & 15, kq = jj & 3, iq = jj >> 2;
    hi[k * 256 + (j & ~15) + 4 * kq + 2 * (iq >> 1) + (iq & 1)] = (int16_t)Xh;
    lo[k * 256 + (j & ~15) + 4 * kq + iq] = (int8_t)Xl;
  }
}
// T order: slot i (0..15) of the padding of block k (run 12's weights 256..259
// and the tail slots), written as zero
__device__ __forceinline__ void rec_put_pad(uint8_t* rec, int kc, int k, int i) {
  int16_t* hi = reinterpret_cast<int16_t*>(rec);
  int8_t* lo = reinterpret_cast<int8_t*>(rec + int_rec_hi_bytes(1, kc));
  const int slot = i < 4 ? 240 + 4 * (i + 1) + 3 : 260 + (i - 4);
  if (i < 8) hi[k * 264 + slot] = 0;
  lo[k * 272 + slot] = 0;
}
// sums of X_hi and X_lo over the 16-column group g16 (0..15) of block k
__device__ __forceinline__ void rec_put_sums(uint8_t* rec, int tq, int kc, int k, int g16, int sh, int sl) {
  int32_t* sp = reinterpret_cast<int32_t*>(rec + int_rec_hi_bytes(tq, kc) + int_rec_lo_bytes(tq, kc));
  sp[k * 16 + g16] = sh;
  sp[kc / 16 + k * 16 + g16] = sl;
}
// 2^-si of block k
__device__ __forceinline__ void rec_put_scale(uint8_t* rec, int tq, int kc, int k, float v) {
  reinterpret_cast<float*>(rec + int_rec_hi_bytes(tq, kc) + int_rec_lo_bytes(tq, kc) + kc / 2)[k] = v;
}

// Selection key of an expert: sigmoid(z) + b as an order-preserving 32-bit
// image (larger key = larger value; 0 is below every real key).
__device__ __forceinline__ uint32_t sel_key(float zv, float b) {
  const float f = 1.0f / (1.0f + expf(-zv)) + b;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads:
// every participant gets the same answer.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %3, 0; bar.red.or.pred q, %1, %2, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// Diagnostic span of a kernel: globaltimer at the first CTA start (atomicMin)
// and at the last CTA end (atomicMax), kept in CTA row 1023 of block `blk`.
__device__ __forceinline__ void dbg_span(uint8_t* ws, uint64_t dbg_off, int blk, bool end) {
  unsigned long long* p = (unsigned long long*)(ws + dbg_off) + ((size_t)blk * 1024 + 1023) * 8;
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  if (end)
    atomicMax(p + 1, (unsigned long long)t);
  else
    atomicMin(p + 0, (unsigned long long)t);
}

// Diagnostic timeline: globaltimer into slot `slot` (2..7) of row 1023 of
// block blk, as a running minimum or maximum over CTAs.
__device__ __forceinline__ void dbg_time(uint8_t* ws, uint64_t dbg_off, int blk, int slot, bool is_max) {
  unsigned long long* p = (unsigned long long*)(ws + dbg_off) + ((size_t)blk * 1024 + 1023) * 8 + slot;
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  if (is_max)
    atomicMax(p, (unsigned long long)t);
  else
    atomicMin(p, (unsigned long long)t);
}

__device__ __forceinline__ void set_error(int32_t* err, int code, int detail) {
  if (atomicCAS(err, 0, code) == 0) err[1] = detail;
}
#endif

}  // namespace bqe
