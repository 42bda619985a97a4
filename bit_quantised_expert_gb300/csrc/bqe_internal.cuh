// bqe_internal.cuh — shared definitions of the CUDA library: block formats,
// the device slot layout, workspace layout, and thin PTX wrappers for
// mbarrier / bulk-copy / grid-dependency control on sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/bqe.h"

namespace bqe {

// ----------------------------------------------------------------------------
// Block formats.  Weights per block / bytes per block (bits per weight from
// the Strata 4090 post, section 5.1, the FP4 per-32 block of the field
// report, and NVIDIA's NVFP4 for the news digest's NVFP4 checkpoint): TQ1
// 256/56, Q2_0 64/18, Q3_K 256/110, MXFP4 32/17, NVFP4 16/9.
// ----------------------------------------------------------------------------
__host__ __device__ constexpr int fmt_bw(int f) {
  return f == BQE_FMT_TQ1 ? 256 : f == BQE_FMT_Q2_0 ? 64 : f == BQE_FMT_Q3_K ? 256 : f == BQE_FMT_MXFP4 ? 32
         : f == BQE_FMT_NVFP4 ? 16 : 0;
}
__host__ __device__ constexpr int fmt_bb(int f) {
  return f == BQE_FMT_TQ1 ? 56 : f == BQE_FMT_Q2_0 ? 18 : f == BQE_FMT_Q3_K ? 110 : f == BQE_FMT_MXFP4 ? 17
         : f == BQE_FMT_NVFP4 ? 9 : 0;
}
__host__ __device__ constexpr bool fmt_ok(int f) { return f >= BQE_FMT_TQ1 && f <= BQE_FMT_NVFP4; }
// Decode-kernel instances by the formats their loops carry: every format
// (kFsAll), MXFP4 only (kFsFp4), or the low-bit formats TQ1 / Q2_0 / Q3_K
// (kFsLowBit); a pool's format mask picks the instance, and an instance
// rejects a slot of any other format like an invalid one.
enum { kFsAll = 0, kFsFp4 = 1, kFsLowBit = 2 };
template <int FS>
__host__ __device__ constexpr bool fs_has(int f) {
  return FS == kFsFp4 ? f == BQE_FMT_MXFP4
         : FS == kFsLowBit ? (f == BQE_FMT_TQ1 || f == BQE_FMT_Q2_0 || f == BQE_FMT_Q3_K)
         : fmt_ok(f);
}
// log2 of the weights per block (every block width is a power of two)
__host__ __device__ constexpr int fmt_lbw(int f) {
  return f == BQE_FMT_TQ1 ? 8 : f == BQE_FMT_Q2_0 ? 6 : f == BQE_FMT_Q3_K ? 8 : f == BQE_FMT_MXFP4 ? 5
         : f == BQE_FMT_NVFP4 ? 4 : 0;
}

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
//      NVFP4: codes8 @ b*256 + r*8             | S   @ nb*256 + b*32 + r
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
    case BQE_FMT_NVFP4:
      return i < 8 ? (uint32_t)(b * 256 + r * 8 + i) : (uint32_t)(nb * 256 + b * 32 + r);
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

// f16 activation rows of the tensor-core loops, in the column order of the
// format (inside every 256 columns):
//   natural (MXFP4): position = column;
//   "P order" (Q2_0, Q3_K): in every 16 columns, position 2p holds column p
//     and 2p + 1 column 8 + p (p = 0..7): the columns of the code pairs that
//     one lop3 lifts out of a 32-bit word of codes;
//   "T order" (TQ1): 288 positions per 256 columns (t16_col), 32 of them zero.
// Halves per 256 columns:
__host__ __device__ constexpr int f16_run(int fmt) { return fmt == BQE_FMT_TQ1 ? 288 : 256; }
// halves of one staged row of kc columns
__host__ __device__ constexpr int f16_len(int fmt, int kc) { return (kc / 256) * f16_run(fmt); }
// Column (0..255) at position pos (0..287) of a T-order run, or -1 (zero).
// The thread tq = (pos / 8) % 4 of a k16 step s = 2 (pos / 32) + (pos / 4) % 2
// holds pair pi = 2 s + (pos / 2) % 2 of its TQ1 codes, half pos % 2; pair pi
// is digit pi % 5 of two code bytes (pi / 5 = 0..5: bytes 2 (pi/5 % 2) + {0, 1}
// of the tq-th 4-byte word of 16-byte piece pi / 10; pi / 5 = 6: code byte
// 48 + tq, in the low half only; pi = 35: none).
__host__ __device__ inline int t16_col(int pos) {
  const int s = 2 * (pos >> 5) + ((pos >> 2) & 1), tq = (pos >> 3) & 3;
  const int pi = 2 * s + ((pos >> 1) & 1), half = pos & 1;
  if (pi >= 35) return -1;
  const int beta = pi / 5, r = pi - 5 * beta;
  int n;
  if (beta == 6) {
    if (half) return -1;
    n = 48 + tq;
    if (n == 51) return r == 0 ? 255 : -1;
  } else {
    n = 16 * (beta >> 1) + 4 * tq + 2 * (beta & 1) + half;
  }
  return 5 * n + r;
}
// P-order position of column c (both within their 16)
__host__ __device__ inline int p16_pos(int c) { return 2 * (c & 7) + (c >> 3); }

// f16 record of h for one row slot and one K chunk of W2 (the tensor-core
// loops): [hi: f16_len halves | 64 bytes | lo: f16_len halves | 2^-s of each
// 256 columns (4 float slots)], h 2^s = hi + lo, in the format's order.
__host__ __device__ constexpr uint32_t h16_rec_bytes(int fmt, int kc) { return 4u * f16_len(fmt, kc) + 80u; }
// workspace stride of the records of h (T order is the longest)
__host__ __device__ constexpr uint32_t hrec_stride(int kc) { return (h16_rec_bytes(BQE_FMT_TQ1, kc) + 15u) & ~15u; }

// Workspace layout (offsets in bytes, each 256-aligned).
struct WsLayout {
  // the router kernel's arrival counter and the call's work list (distinct
  // experts: slot, format, address, rows), combine indices and weights
  uint64_t err, ctr_route, nu, u_slot, u_fmt, u_addr, u_nrows, u_rows, comb_u, comb_r, comb_w;
  // logits; the layer input as f16 x 2^s (per-row s) in the natural, P and T
  // orders; the diagnostic counters
  uint64_t z, xh, xp, xt, dbg;
  // single-kernel decode layer: of every (row, expert) the selection key and
  // the logit, each tagged with the call's epoch (value << 32 | tag)
  uint64_t zk, zl;
  // single-kernel decode layer (k_moe): call epoch, staged-input arrival
  // counter, per work-list expert the counts of its W1/W3 items done and of
  // its h units written; per "row slot" (an expert's r-th row; M (K + 1)
  // slots at most) the K-chunk partials of g/u and the f16 records of h
  // (h16_rec_bytes)
  uint64_t epoch, st, m_ca, m_ch, m_pa, m_hr;
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
  w.xh = o; o = al256(o + 2ull * g.M * g.H);   // f16(x * 2^s_m): exact, per-row power-of-two scale
  w.xp = o; o = al256(o + 2ull * g.M * g.H);   // the same in P order
  w.xt = o; o = al256(o + 2ull * g.M * (g.H / 256) * 288);  // ... and in T order
  w.dbg = o; o = al256(o + 8ull * 3 * kDbgMaxCtas * kDbgSlots);
  // the tagged keys, the logits, the call epoch and the counters are
  // contiguous: [zk, m_pa) clears them
  w.zk = o; o = al256(o + 8ull * g.M * g.E);
  w.zl = o; o = al256(o + 8ull * g.M * g.E);
  w.epoch = o; o = al256(o + 16);
  w.st = o; o = al256(o + 16);                                     // staged-input arrival counter (64-bit)
  w.m_ca = o; o = al256(o + 4ull * kMaxU);                         // W1/W3 items done, per expert
  w.m_ch = o; o = al256(o + 4ull * kMaxU);                         // h units written, per expert
  const uint64_t nrs = (uint64_t)g.M * (g.K + 1);
  w.m_pa = o; o = al256(o + 4ull * nrs * g.npanA * g.nchA * 2 * 32);
  w.m_hr = o; o = al256(o + (uint64_t)hrec_stride(g.kcB) * nrs * g.nchB);
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
// Offsets (from the first slot) of the slots of a pool laid out by
// bqe_pool_init for the formats fmt[0..n-1] (bqe_format.cu); false on a bad format.
bool pool_slot_offsets(const bqe_layer_desc* d, int32_t n, const int32_t* fmt, std::vector<uint64_t>& off);

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
// Non-blocking test of an mbarrier phase (acquire on success).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
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
