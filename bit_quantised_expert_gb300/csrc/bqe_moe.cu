// bqe_moe.cu — the decode layer (M <= 8 token rows) as one persistent kernel.
//
// The layer's cost is the expert bytes each token streams (field report,
// section 2: single-stream speed is set by the bytes each token moves), so
// the kernel is built to keep HBM busy from its first cycle to its last:
//
//   * one CTA per SM, launched cooperatively (every CTA resident, so CTAs may
//     wait on one another; every such wait is bounded by %globaltimer);
//   * warps 0-1 (one lane each) stream work items into a byte ring in shared
//     memory with cp.async.bulk and mbarrier completion; warps 2-17 compute;
//     warp 18 reduces each item (partial sums out, ring bytes freed); warp 19
//     forms h = silu(g) * u;
//   * before the routing is known, the producers stream this CTA's share of
//     the shared expert's W1/W3 (always used), while the compute warps read
//     this CTA's rows of the router (z = x Wr^T, fp32) as soon as they land
//     and publish the selection key and z of those experts, each as a 64-bit
//     word tagged with the call's epoch; warp m reads row m's keys until
//     every tag is this call's and selects its top-k from registers, while
//     the other compute warps stage this CTA's slice of the f16 input copies
//     (published on a counter, for the producers' activation copies); then
//     warp 0 builds the work list, the row slots and the item templates (the
//     same result in every CTA: no serial tail, no second kernel), and the h
//     warp the mixing weights, off the critical path;
//   * work items are (expert, 32-row panel, K chunk) of W1 and W3, then
//     (expert, group of W2 output panels, K chunk) of W2, shared expert first,
//     dealt round-robin over the CTAs, so every expert's W1/W3 is finished by
//     all CTAs together, long before its W2 items come up;
//   * no grid-wide barrier: the reducers count each expert's finished W1/W3
//     items, the h warps form h for an expert once its count is complete, and
//     the producers copy an expert's h rows once its h units are all written;
//   * the W2 reducers add w_j y_j (the shared expert with weight 1) into the
//     output rows with fp32 atomics.
//
// Router, selection and mixing follow the field report (384 routed experts,
// 6 per token, one shared) and the Strata 4090 post, section 5.3 (the bias
// steers the choice; the mixing weights are the unbiased scores).  The
// per-format dequant-GEMV inner loops are those of bqe_gemv.cuh.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "bqe_gemv.cuh"
#include "bqe_internal.cuh"

namespace bqe {

constexpr int kNQ = 16;                    // items in flight per CTA (barrier ring)
constexpr int kCW = 16;                    // compute warps
constexpr int kNP = 2;                     // producer warps
// producers, compute warps, reducer, h warp: 20 warps, 5 per SM
// sub-partition, so each thread may hold 96 registers
constexpr int kMoeThreads = 32 * (kNP + kCW + 2);
constexpr int kRedWarp = kNP + kCW;  // then the h warp (the last)
constexpr int kMaxEM = 512;                // routed experts supported
constexpr int kRouteTasks = 16;            // (expert of this CTA, quarter of hidden) router tasks


// Per-item header (slot i % kNQ): where the item's bytes sit in the ring and
// what they are.
struct ItemHdr {
  uint32_t off;       // ring offset of the item
  uint32_t tb;        // bytes of one weight tile
  uint32_t act;       // offset of the activation rows (from off)
  uint32_t red;       // offset of the partial sums (from off)
  uint32_t arow;      // staged bytes of one activation row (one bulk copy)
  uint32_t astr;      // distance between two staged rows
  int16_t u, p, c, R; // expert (work-list index), panel (W1/W3) or panel group (W2), K chunk, rows
  uint8_t phase, fmt, amode, nb;
};

// Everything about the items of one (phase, expert) but their place: the
// header to copy (off, p, c filled per item), the ring bytes, the weight
// source and the activation rows' addressing in the workspace.
struct ItemTpl {
  ItemHdr h;
  uint32_t size, wbytes;   // ring bytes of an item; bytes of its weight tiles
  uint64_t wsrc;           // W1 (phase 0) or W2 (phase 1) of the expert's slot
  uint32_t m13;            // phase 0: W3 - W1
  uint32_t act_base;       // workspace offset of activation row 0, chunk 0
  uint32_t act_rs, act_cs; // bytes from one row (row slot) to the next, one chunk to the next
};

__device__ __forceinline__ uint32_t al128(uint32_t v) { return (v + 127u) & ~127u; }

__device__ __forceinline__ uint32_t ld_acquire_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const void* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(void* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const void* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(void* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ float silu_m(float t) { return t / (1.0f + expf(-t)); }
// fp32 add into global memory with no value returned
__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Diagnostic timeline of one call: globaltimer stamps kept as minima or
// maxima over CTAs in row 1023 of dbg blocks 0..2 (8 slots each).
__device__ __forceinline__ void mstamp(const MoeParams& P, int k, bool is_max) {
  if (P.diag) dbg_time(P.ws, P.L.dbg, k >> 3, k & 7, is_max);
}
enum {
  kStStart = 0,       // min: first CTA start
  kStZPub = 1,        // max: last CTA published its logits
  kStRouted = 2,      // min / max (+8): CTA knows the routing
  kStRoutedMax = 10,
  kStFirstItem = 3,   // min: first item landed
  kStAEnd = 4,        // max: last W1/W3 item finished
  kStBFirst = 5,      // min: first W2 item landed
  kStEnd = 6,         // max: last CTA end
  kStProdEnd = 7,     // max: last producer done issuing
  kStConsEnd = 9,     // max: last compute warp done
  kStHWaitMax = 11,   // max: a producer's longest h wait (ns, as a value)
};

// Diagnostic per-CTA time accounts (ns) in dbg block 2, row = CTA: 0 producer
// waiting for ring space, 1 producer waiting for h, 2 compute warp 0 waiting
// for items, 3 compute warp 0 computing, 4 reducer waiting, 5 reducer waiting
// for queue space, 6 finishers polling partials, 7 CTA start to end.
// Block 1, row = CTA: 0 producer issuing (outside its waits), 1 items issued,
// 2 CTA start to its logits published, 3 ... to the routing known, 4 ... to
// its router rows landed, 5 reducer working, 6 finishers working.
__device__ __forceinline__ void dacc(const MoeParams& P, int slot, uint64_t ns, int blk = 2) {
  if (P.diag && blockIdx.x < 1023)
    atomicAdd((unsigned long long*)(P.ws + P.L.dbg) + ((size_t)blk * 1024 + blockIdx.x) * 8 + slot,
              (unsigned long long)ns);
}

// Diagnostic: per-CTA time from the CTA's start to routing step k (dbg block
// 0, row 300 + CTA, slot k).
__device__ __forceinline__ void rstamp(const MoeParams& P, int k, uint64_t t0) {
  if (P.diag && blockIdx.x < 700)
    atomicAdd((unsigned long long*)(P.ws + P.L.dbg) + ((size_t)300 + blockIdx.x) * 8 + k,
              (unsigned long long)(globaltimer_ns() - t0));
}

// The CTA's abort flag as lane 0 of the calling warp reads it, the same for
// every lane (a flag set by another warp meanwhile must not split a warp
// before its next warp-wide operation); every lane of the warp calls it.
__device__ __forceinline__ bool warp_abort(volatile int& flag) { return __shfl_sync(0xffffffffu, (int)flag, 0) != 0; }

// Bounded wait on an mbarrier phase, sleeping between checks; also gives up
// when another CTA has already recorded an error.
__device__ __forceinline__ bool mwait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, const int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*(volatile const int32_t*)err) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Bounded wait until *p >= target (other CTAs' progress); false on timeout
// or when an error has been recorded.
__device__ __forceinline__ bool wait_ge(const unsigned int* p, uint32_t target, uint64_t limit_ns,
                                        const int32_t* err) {
  if (ld_acquire_u32(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 16; ++i) {
      __nanosleep(40);
      if (ld_acquire_u32(p) >= target) return true;
    }
    if (*(volatile const int32_t*)err) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Template of the items of (phase ph, expert u) in format fmt at slot address
// addr with R activation rows, the first of them in row slot rb.
__device__ inline void make_tpl(const MoeParams& P, ItemTpl& T, int ph, int u, int fmt, uint64_t addr, int R, int rb) {
  const Geo& g = P.g;
  const int kc = ph ? g.kcB : g.kcA;
  const int amode = act_mode(ph);
  ItemHdr& h = T.h;
  const int lbw = fmt_lbw(fmt);  // blocks by shifts (no division by a format-dependent width)
  h.tb = 32u * (uint32_t)(kc >> lbw) * (uint32_t)fmt_bb(fmt);
  h.arow = (uint32_t)act_row_bytes(amode, fmt, kc);
  h.astr = (uint32_t)act_row_stride(amode, fmt, kc);
  T.wbytes = (uint32_t)(ph ? P.PB : 2) * h.tb;
  h.act = al128(T.wbytes);
  h.red = h.act + al128((uint32_t)R * h.astr);
  h.off = 0;
  h.u = (int16_t)u; h.p = 0; h.c = 0; h.R = (int16_t)R;
  h.phase = (uint8_t)ph; h.fmt = (uint8_t)fmt; h.amode = (uint8_t)amode; h.nb = (uint8_t)(kc >> lbw);
  T.size = h.red + (uint32_t)(ph ? P.PB * g.GB : 2 * g.GA) * R * 32 * 4;
  const uint64_t m13 = (uint64_t)g.I * (uint64_t)(g.H >> lbw) * (uint64_t)fmt_bb(fmt);  // one of W1, W3
  T.m13 = (uint32_t)m13;
  T.wsrc = addr + (ph ? 2 * m13 : 0);
  if (ph == 0) {  // f16 x in the format's order
    T.act_base = (uint32_t)(fmt == BQE_FMT_TQ1 ? P.L.xt : (fmt == BQE_FMT_Q2_0 || fmt == BQE_FMT_Q3_K) ? P.L.xp : P.L.xh);
    T.act_cs = (uint32_t)f16_len(fmt, kc) * 2;
    T.act_rs = (uint32_t)f16_len(fmt, g.H) * 2;
  } else {  // the f16 records of h of the expert's row slots
    const uint32_t rec = hrec_stride(g.kcB);
    T.act_base = (uint32_t)(P.L.m_hr + (uint64_t)rb * g.nchB * rec);
    T.act_cs = rec;
    T.act_rs = rec * g.nchB;
  }
}

// The template of an expert from its format's template (made for expert 0,
// address 0, no rows, row slot 0): the fields that depend on those.
__device__ inline void patch_tpl(const MoeParams& P, ItemTpl& T, const ItemTpl& B, int ph, int u, uint64_t addr,
                                 int R, int rb) {
  const Geo& g = P.g;
  T = B;
  T.h.u = (int16_t)u;
  T.h.R = (int16_t)R;
  T.h.red = B.h.act + al128((uint32_t)R * B.h.astr);
  T.size = T.h.red + (uint32_t)(ph ? P.PB * g.GB : 2 * g.GA) * R * 32 * 4;
  T.wsrc = addr + (ph ? 2 * (uint64_t)B.m13 : 0);
  if (ph) T.act_base = B.act_base + (uint32_t)rb * B.act_rs;
}

template <int RC, int FS>
__global__ void __launch_bounds__(kMoeThreads, 1) k_moe(MoeParams P) {
  const Geo& g = P.g;
  // the one-row instance (RC == 1) runs only calls with M == 1: a constant there
  const int H = g.H, I = g.I, E = g.E, K = g.K, M = RC == 1 ? 1 : g.M;
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* err = (int32_t*)(P.ws + P.L.err);

  extern __shared__ __align__(128) uint8_t dsm[];
  uint8_t* ring = dsm;
  const uint16_t* s_x = reinterpret_cast<const uint16_t*>(ring + P.xstage_off);  // M x H bf16 (startup only)
  const float* s_rw = reinterpret_cast<const float*>(ring + P.rt_off);  // this CTA's router rows (startup only)

  __shared__ ItemHdr hdr[kNQ];
  __shared__ __align__(8) uint64_t full[kNQ], cons[kNQ], freed[kNQ], route_bar, rbar, wbar, xbar;
  __shared__ float s_rsw[kMaxM * (kMaxTopK + 1)];  // mixing weight of each row slot (shared expert: 1)
  __shared__ int s_rbase[kMaxU + 1];   // first row slot of each work-list expert
  __shared__ int s_done[kNQ];
  __shared__ int32_t s_ufmt[kMaxU], s_unrows[kMaxU];
  __shared__ uint64_t s_uaddr[kMaxU];
  __shared__ int8_t s_urows[kMaxU * kMaxM];
  __shared__ float s_cw[kMaxM][kMaxTopK];
  __shared__ int s_idx[kMaxM][kMaxTopK];
  __shared__ float s_zsel[kMaxM][kMaxTopK];
  __shared__ uint32_t s_mask[kMaxEM];
  __shared__ int16_t s_uof[kMaxEM];
  __shared__ int s_fidx[kMaxM][kMaxTopK];  // forced choices
  __shared__ int s_first[kMaxEM];          // first (row, choice) index t = m K + j that chose each expert
  __shared__ float s_part[kRouteTasks][kMaxM];
  __shared__ float s_inv_rms[kMaxM], s_xsc[kMaxM];
  __shared__ int s_emax[kMaxM];
  __shared__ float s_hunit[256];  // h warp: one unit of h (T-order records)
  __shared__ float s_red[kCW][kMaxM];
  __shared__ float s_bias[kMaxEM];
  __shared__ uint64_t s_eaddr[kMaxEM + 1];  // slot address of each expert (E: the shared one)
  __shared__ int16_t s_eslot[kMaxEM + 1];   // its slot
  __shared__ uint8_t s_efmt[kMaxEM + 1];    // its slot's format (0: invalid)
  __shared__ uint8_t s_ebad[kMaxEM + 1];    // error detail of an invalid slot
  __shared__ int s_nu, s_bad;
  __shared__ volatile int s_abort, s_issued[kNP], s_turn;  // s_turn: next item to get ring space
  __shared__ uint32_t s_startq[kNQ];   // ring offset of each item in flight
  __shared__ volatile uint32_t s_head; // end of the newest allocation
  __shared__ volatile int s_oldest;    // oldest item not yet known to be freed
  __shared__ volatile int s_npre;      // items pre-issued before the routing (-1: not yet known)
  __shared__ ItemTpl s_tpl[2][kMaxU];
  __shared__ ItemTpl s_tbase[2][8];  // per (phase, format): the template of expert 0 at address 0, no rows

  const uint32_t tag = *(volatile const uint32_t*)(P.ws + P.L.epoch) + 1u;
  if (tid == 0) {
    for (int s = 0; s < kNQ; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&cons[s], 1);
      mbar_init(&freed[s], 1);
      s_done[s] = 0;
    }
    mbar_init(&route_bar, 1);
    mbar_init(&rbar, 1);
    mbar_init(&wbar, 1);
    mbar_init(&xbar, 1);
    s_abort = 0;
    for (int q = 0; q < kNP; ++q) s_issued[q] = 0;
    s_turn = 0;
    s_npre = -1;
    s_head = 0;
    s_oldest = 0;
    s_bad = 0;
    s_nu = 0;
    fence_mbar_init();
  }
  for (int e = tid; e < E; e += kMoeThreads) {
    s_mask[e] = 0u;
    s_first[e] = 0x7FFF;
  }
  __syncthreads();
  if (tid == 0) mstamp(P, kStStart, false);
  const uint64_t t_cta0 = P.diag ? globaltimer_ns() : 0;

  // geometry of the two item kinds
  const int TA = 2 * g.GA, TB = P.PB * g.GB;             // compute tasks per item
  const int nAper = g.npanA * g.nchA;                    // W1/W3 items per expert
  const int nBper = (g.npanB / P.PB) * g.nchB;           // W2 items per expert
  const int bpcB = g.kcB / 256;                          // 256-column blocks of h per W2 chunk

  if (warp < kNP) {
    // ============================== producers =================================
    // Producer pp (warp pp, one lane) issues items i = pp, pp + kNP, ..., so
    // the bookkeeping of one overlaps the other's bulk-copy issue (a thread
    // waits in cp.async.bulk until the copy engine takes the bytes).  Both
    // share one ring, allocated in item order; items i and i + kNQ share
    // barriers and a producer.
    const int pp = warp;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = -1;  // last own item whose copies went out
      bool ok = true;
      // Ring space [at, at + sz) of [0, end) for item i.  Items get their space
      // in item order (the two producers take turns; the state is shared);
      // waits (bounded) for the turn and for frees when may_wait.  -1: no room
      // (or not this item's turn) without waiting, -2: timeout.
      auto alloc = [&](int i, uint32_t sz, uint32_t end, bool may_wait) -> int64_t {
        if (s_turn != i) {
          if (!may_wait) return -1;
          const uint64_t t0 = globaltimer_ns();
          while (s_turn != i) {
            __nanosleep(32);
            if (s_abort || *(volatile const int32_t*)err || globaltimer_ns() - t0 > P.limit_ns) return -2;
          }
        }
        int oldest = s_oldest;
        uint32_t head = s_head;
        if (i >= kNQ) {
          const int j = i - kNQ;
          if (oldest <= j) {
            if (!may_wait) return -1;
            if (!mwait(&freed[j % kNQ], (j / kNQ) & 1, P.limit_ns, err)) return -2;
            oldest = j + 1;
          }
        }
        int64_t at = -1;
        while (true) {
          if (oldest == i) {
            head = 0;
            at = sz <= end ? 0 : -3;
            break;
          }
          const uint32_t tail = s_startq[oldest % kNQ];
          if (head > tail) {
            if (head + sz <= end) { at = head; break; }
            if (sz <= tail) { at = 0; break; }
          } else if (head < tail) {
            if (head + sz <= tail) { at = head; break; }
          }
          if (!may_wait) break;
          if (!mwait(&freed[oldest % kNQ], (oldest / kNQ) & 1, P.limit_ns, err)) return -2;
          ++oldest;
        }
        s_oldest = oldest;
        if (at >= 0) {
          s_startq[i % kNQ] = (uint32_t)at;
          s_head = (uint32_t)at + sz;
        }
        return at;
      };
      // the copies of item i from template T: weight tiles, then (acts) activation rows
      auto issue = [&](int i, const ItemTpl& T, int p, int c, bool weights, bool acts, bool pre) {
        const uint32_t off = hdr[i % kNQ].off;
        uint8_t* dst = ring + off;
        uint64_t* bar = &full[i % kNQ];
        if (weights) {
          if (pre) mbar_expect_tx(bar, T.wbytes);
          if (T.h.phase == 0) {
            const uint64_t src = T.wsrc + (uint64_t)(p * g.nchA + c) * T.h.tb;
            bulk_g2s_hint(dst, (const void*)src, T.h.tb, bar, pol);                       // W1 tile
            bulk_g2s_hint(dst + T.h.tb, (const void*)(src + T.m13), T.h.tb, bar, pol);   // W3 tile
          } else {
            for (int j = 0; j < P.PB; ++j) {
              const uint64_t src = T.wsrc + (uint64_t)((p * P.PB + j) * g.nchB + c) * T.h.tb;
              bulk_g2s_hint(dst + j * T.h.tb, (const void*)src, T.h.tb, bar, pol);          // W2 tiles
            }
          }
        }
        if (acts) {
          if (pre) mbar_arrive_expect_tx(bar, (uint32_t)T.h.R * T.h.arow);
          const uint8_t* src0 = P.ws + T.act_base + (uint64_t)c * T.act_cs;
          for (int r = 0; r < T.h.R; ++r) {
            const int row = (T.h.phase == 0 && T.h.u != 0) ? s_urows[T.h.u * kMaxM + r] : r;
            bulk_g2s(dst + T.h.act + (size_t)r * T.h.astr, src0 + (uint64_t)row * T.act_rs, T.h.arow, bar);
          }
        }
      };
      // ---- producer 0: this CTA's router rows (experts cta, cta + G, ...)
      if (pp == 0) {
        const int nexp = E > cta ? (E - cta + G - 1) / G : 0;
        const uint32_t rowb = (uint32_t)H * 4;
        mbar_arrive_expect_tx(&rbar, (uint32_t)nexp * rowb);
        for (int j = 0; j < nexp; ++j)
          bulk_g2s_hint(ring + P.rt_off + j * rowb, P.router_w + (int64_t)(cta + j * G) * H, rowb, &rbar, pol);
      }
      // ---- before the routing: own shared-expert W1/W3 items, weights only.
      // The shared expert's slot comes from the inputs, not from the router.
      ItemTpl sh;
      bool sh_ok = false;
      {
        const int sl = P.slot_table[E];
        if (sl >= 0 && sl < P.pool.n_slots) {
          const int f = P.pool.slot_fmt[sl];
          const uint64_t off = P.pool.slot_off[sl];
          if (fs_has<FS>(f) && !(off & 15) && off + 2 * matrix_bytes(f, I, H) + matrix_bytes(f, H, I) <= P.pool.base_bytes) {
            make_tpl(P, sh, 0, 0, f, (uint64_t)P.pool.base + off, M, 0);
            sh_ok = true;
          }
        }
      }
      // producer 0 pre-issues items 0, 1, ... (weights only) while they fit below
      // the startup data; each item's owner (i % kNP) issues its activation rows
      // once the routing is known
      if (!mwait(&rbar, 0, P.limit_ns, err)) sh_ok = false;
      if (pp == 0) {
        int n = 0;
        if (sh_ok) {
          for (int i = 0;; ++i) {
            const int t = cta + i * G;
            if (t >= nAper || i >= kNQ) break;
            if (i == P.drop_item && cta == 0) break;  // the test hook's item goes through the main loop
            const int64_t at = alloc(i, sh.size, P.rt_off, false);
            if (at < 0) break;
            ItemHdr h = sh.h;
            h.off = (uint32_t)at;
            h.p = (int16_t)(t / g.nchA);
            h.c = (int16_t)(t - h.p * g.nchA);
            hdr[i % kNQ] = h;
            s_done[i % kNQ] = 0;
            issue(i, sh, h.p, h.c, true, false, true);
            s_issued[i % kNP] = i + 1;
            s_turn = i + 1;
            ++n;
          }
        }
        s_npre = n;
      } else {
        const uint64_t t0 = globaltimer_ns();  // producer 0's count of pre-issued items
        while (s_npre < 0 && globaltimer_ns() - t0 < P.limit_ns) __nanosleep(32);
      }
      const int npre = max(0, (int)s_npre);
      // ---- the pre-issued items' x rows, once every CTA has published its
      // staged slices of x (well before the routing is known; copied on a
      // failed wait too: the addresses are valid, the stage drains)
      {
        unsigned long long* scnt = (unsigned long long*)(P.ws + P.L.st);
        const unsigned long long target = (unsigned long long)G * tag;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_u64(scnt) < target) {
          __nanosleep(64);
          if (*(volatile const int32_t*)err) {
            ok = false;
            break;
          }
          if (globaltimer_ns() - t0 > P.limit_ns) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            ok = false;
            break;
          }
        }
      }
      fence_proxy_async_global();  // the staged inputs of every CTA are read by bulk copies below
      for (int i = pp; i < npre; i += kNP) {
        issue(i, sh, hdr[i % kNQ].p, hdr[i % kNQ].c, false, true, true);
        issued = i;
      }
      // ---- the routing (work list and item templates built by the compute warps)
      if (!mwait(&route_bar, 0, P.limit_ns, err)) {
        set_error(err, BQE_ETIMEOUT, kErrWaitFull);
        s_abort = 1;
        ok = false;
      }
      const int nU = s_nu;
      const int nTot = nU * (nAper + nBper), nA = nU * nAper;
      long long hwait_max = 0;
      int dropped = -1;
      int h_ready = -1;  // experts below this one have their h written
      long long cyc_loop = P.diag ? clock64() : 0, cyc_bulk = 0, cyc_alloc = 0, cyc_h = 0;
      int first = pp;
      while (first < npre) first += kNP;
      for (int i = first; ok; i += kNP) {
        const int t = cta + i * G;
        if (t >= nTot || s_abort) break;
        // item t: W1/W3 items of experts 0..nU-1 (panel-major, chunk fastest), then W2 items
        int ph, u, p, c;
        if (t < nA) {
          ph = 0;
          u = (int)(((uint64_t)t * P.magA) >> 32);
          const int r = t - u * nAper;
          p = (int)(((uint64_t)r * P.magA2) >> 32);
          c = r - p * g.nchA;
        } else {
          const int tb = t - nA;
          ph = 1;
          u = (int)(((uint64_t)tb * P.magB) >> 32);
          const int r = tb - u * nBper;
          p = (int)(((uint64_t)r * P.magB2) >> 32);
          c = r - p * g.nchB;
        }
        const ItemTpl& T = s_tpl[ph][u];
        const long long ta = P.diag ? clock64() : 0;
        const int64_t at = alloc(i, T.size, P.ring_bytes, true);
        if (P.diag) cyc_alloc += clock64() - ta;
        if (at < 0) {
          set_error(err, at == -2 ? BQE_ETIMEOUT : BQE_EUNSUPPORTED, kErrWaitEmpty);
          s_abort = 1;
          break;
        }
        ItemHdr h = T.h;
        h.off = (uint32_t)at;
        h.p = (int16_t)p;
        h.c = (int16_t)c;
        hdr[i % kNQ] = h;
        s_done[i % kNQ] = 0;
        s_issued[pp] = i + 1;
        s_turn = i + 1;  // the next item may get its ring space
        if (i == P.drop_item && cta == 0) {  // test hook: this item's copies are never issued
          dropped = i;
          continue;
        }
        mbar_arrive_expect_tx(&full[i % kNQ], T.wbytes + (uint32_t)h.R * h.arow);
        const long long tb0 = P.diag ? clock64() : 0;
        issue(i, T, p, c, true, false, false);
        if (P.diag) cyc_bulk += clock64() - tb0;
        issued = i;
        if (ph == 1 && u > h_ready) {
          // every h unit of expert u is written (by the h warps of all CTAs)
          // before its rows are copied; the weights above are already on their way
          const long long w0 = P.diag ? (long long)globaltimer_ns() : 0;
          const long long tc0 = P.diag ? clock64() : 0;
          const uint32_t need = (uint32_t)s_unrows[u] * (uint32_t)(I / 256);
          if (!wait_ge((const unsigned int*)(P.ws + P.L.m_ch) + u, need, P.limit_ns, err)) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
            ok = false;  // the activation copies still go out (valid addresses) so the stage drains
          }
          if (P.diag) {
            hwait_max = max(hwait_max, (long long)globaltimer_ns() - w0);
            dacc(P, 1, globaltimer_ns() - w0);
            cyc_h += clock64() - tc0;
          }
          fence_proxy_async_global();
          h_ready = u;
        }
        const long long tb1 = P.diag ? clock64() : 0;
        issue(i, T, p, c, false, true, false);
        if (P.diag) cyc_bulk += clock64() - tb1;
      }
      if (P.diag) {
        dacc(P, 0, clock64() - cyc_loop, 1);
        dacc(P, 1, (issued + kNP) / kNP, 1);
        dacc(P, 5, cyc_bulk, 1);
        dacc(P, 6, cyc_alloc, 1);
        dacc(P, 7, cyc_h, 1);
        dbg_time(P.ws, P.L.dbg, 0, kStProdEnd, true);
        atomicMax((unsigned long long*)(P.ws + P.L.dbg) + ((size_t)1 * 1024 + 1023) * 8 + (kStHWaitMax & 7),
                  (unsigned long long)hwait_max);
      }
      // leave no copy in flight: every issued own item has landed before the CTA
      // ends (own items older than the last kNQ / kNP were freed, so they landed)
      for (int i = issued; i >= 0 && i > issued - kNQ; i -= kNP)
        if (i != dropped) mbar_wait_bounded(&full[i % kNQ], (i / kNQ) & 1, 2000000000ull);
    }
  } else if (warp < kNP + kCW) {
    // ============================ compute warps ===============================
    const int ct = tid - 32 * kNP, cw = warp - kNP;
    constexpr int NCT = kCW * 32;
    // ---- this CTA's router rows: experts cta + j G, task (j, quarter of hidden)
    const int nexp = E > cta ? (E - cta + G - 1) / G : 0;
    const int Kq = H / 4, ni = Kq / 128;
    const int rj = cw >> 2, rq = cw & 3;
    const bool rtask = cw < nexp * 4;
    // ---- first the loads that nothing computed here feeds (slot table, bias,
    // forced choices): their latency overlaps the input staging below
    const int sl0 = ct <= E ? P.slot_table[ct] : -1;
    const int sl1 = ct + NCT <= E ? P.slot_table[ct + NCT] : -1;
    const float bias0 = (ct < E && P.bias) ? P.bias[ct] : 0.f;
    const int fidx0 = (P.forced && ct < M * K) ? P.forced[ct] : 0;
    // ---- the layer input as bf16 in shared memory: x, or bf16(rmsnorm(resid))
    uint16_t* xs = const_cast<uint16_t*>(s_x);
    if (ct < M) s_emax[ct] = -1000;
    if (P.resid) {
      for (int m = 0; m < M; ++m) {
        float ss = 0.f;
        for (int k = ct; k < H; k += NCT) {
          const float v = P.resid[(int64_t)m * H + k];
          ss = fmaf(v, v, ss);
        }
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_red[cw][m] = ss;
      }
      named_bar_sync(1, NCT);
      if (ct < M) {
        float ss = 0.f;
        for (int w = 0; w < kCW; ++w) ss += s_red[w][ct];
        s_inv_rms[ct] = 1.0f / sqrtf(ss / (float)H + 1e-6f);
      }
      named_bar_sync(1, NCT);
      for (int i = ct; i < M * H; i += NCT)
        xs[i] = __bfloat16_as_ushort(__float2bfloat16_rn(P.resid[i] * s_inv_rms[i / H]));
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(P.x);
      uint4* dst = reinterpret_cast<uint4*>(xs);
      for (int i = ct; i < M * H / 8; i += NCT) dst[i] = src[i];
    }
    // the slot descriptors of the experts (the loads only; checked after the
    // logits are out, so their latency overlaps the router dot products)
    int sf0 = 0, sf1 = 0;
    uint64_t so0 = 0, so1 = 0;
    const bool sv0 = sl0 >= 0 && sl0 < P.pool.n_slots, sv1 = sl1 >= 0 && sl1 < P.pool.n_slots;
    if (sv0) {
      sf0 = P.pool.slot_fmt[sl0];
      so0 = P.pool.slot_off[sl0];
    }
    if (sv1) {
      sf1 = P.pool.slot_fmt[sl1];
      so1 = P.pool.slot_off[sl1];
    }
    // ---- this CTA's slice of the output (zero unless the call accumulates)
    // and, in CTA 0, the per-expert counters of the call: released with this
    // CTA's staged slices of the input, which every CTA acquires before its
    // first item, so before any other CTA adds to them
    if (!P.accumulate) {
      const int n = M * H, per = (n + G - 1) / G, lo = min(n, per * cta), hi = min(n, lo + per);
      for (int i = lo + ct; i < hi; i += NCT) P.out[i] = 0.f;
    }
    if (cta == 0 && ct < kMaxU) {
      ((unsigned int*)(P.ws + P.L.m_ca))[ct] = 0u;
      ((unsigned int*)(P.ws + P.L.m_ch))[ct] = 0u;
    }
    // ---- selection inputs: the bias and the forced choices (validated)
    if (ct < E) s_bias[ct] = bias0;
    if (P.forced && ct < M * K) {
      int f = fidx0;
      if (f < 0 || f >= E) {
        set_error(err, BQE_EDEVICE, kErrForcedIdx);
        s_bad = 1;
        f = 0;
      }
      s_fidx[ct / K][ct % K] = f;
    }
    named_bar_sync(1, NCT);
    if (P.diag && ct == 0) dacc(P, 0, globaltimer_ns() - t_cta0, 0);
    unsigned long long* zk = (unsigned long long*)(P.ws + P.L.zk);
    unsigned long long* zl = (unsigned long long*)(P.ws + P.L.zl);
    // ---- router dot products of this CTA's experts (rows landed in shared memory)
    {
      const bool okr = __all_sync(0xffffffffu, mwait(&rbar, 0, P.limit_ns, err));
      if (!okr && lane == 0) {
        set_error(err, BQE_ETIMEOUT, kErrWaitFull);
        s_abort = 1;
      }
      if (P.diag && ct == 0) dacc(P, 4, globaltimer_ns() - t_cta0, 1);
      float acc[kMaxM];
#pragma unroll
      for (int m = 0; m < kMaxM; ++m) acc[m] = 0.f;
      if (rtask && okr) {
        const float4* wr = reinterpret_cast<const float4*>(s_rw + rj * H + rq * Kq);
#pragma unroll 4
        for (int i = 0; i < ni; ++i) {
          {
            const float4 wv = wr[i * 32 + lane];
            const int k = rq * Kq + (i * 32 + lane) * 4;
#pragma unroll
            for (int m = 0; m < kMaxM; ++m) {
              if (m < M) {
                const uint2 xv = *reinterpret_cast<const uint2*>(xs + m * H + k);
                acc[m] = fmaf(wv.x, __uint_as_float(xv.x << 16), acc[m]);
                acc[m] = fmaf(wv.y, __uint_as_float(xv.x & 0xFFFF0000u), acc[m]);
                acc[m] = fmaf(wv.z, __uint_as_float(xv.y << 16), acc[m]);
                acc[m] = fmaf(wv.w, __uint_as_float(xv.y & 0xFFFF0000u), acc[m]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kMaxM; ++m) {
        if (m < M) {
          float v = acc[m];
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0 && rtask) s_part[cw][m] = v;
        }
      }
    }
    named_bar_sync(1, NCT);  // logits partials of this CTA are in shared memory
    // publish the selection key (the bias only steers the choice) and the
    // logit, each in one 64-bit word with the call's epoch as its tag: a
    // reader that sees the tag has the value, so no fence is needed here
    if (ct < nexp * M) {
      const int j = ct / M, m = ct % M, e = cta + j * G;
      const float zv = (s_part[4 * j][m] + s_part[4 * j + 1][m]) + (s_part[4 * j + 2][m] + s_part[4 * j + 3][m]);
      st_relaxed_u64(zk + (size_t)m * E + e, ((unsigned long long)sel_key(zv, s_bias[e]) << 32) | tag);
      st_relaxed_u64(zl + (size_t)m * E + e, ((unsigned long long)__float_as_uint(zv) << 32) | tag);
    }
    if (ct == 0) {
      mstamp(P, kStZPub, true);
      if (P.diag) dacc(P, 2, globaltimer_ns() - t_cta0, 1);
    }
    // ---- the slot descriptor of every expert (e = E: the shared one), into
    // shared memory, so that no load waits after the routing
    auto slot_desc = [&](int e, int slot, bool valid, int f, uint64_t off) {
      int fmt = 0, bad = 0;
      uint64_t addr = 0;
      if (!valid) {
        bad = kErrSlotRange;
      } else if (!fs_has<FS>(f)) {  // (formats outside this instance's set included)
        bad = kErrSlotFmt;
      } else if ((off & 15) || off + 2 * matrix_bytes(f, I, H) + matrix_bytes(f, H, I) > P.pool.base_bytes) {
        bad = kErrSlotExtent;
      } else {
        fmt = f;
        addr = (uint64_t)P.pool.base + off;
      }
      s_eslot[e] = (int16_t)slot;
      s_efmt[e] = (uint8_t)fmt;
      s_eaddr[e] = addr;
      s_ebad[e] = (uint8_t)bad;
    };
    if (ct <= E) slot_desc(ct, sl0, sv0, sf0, so0);
    if (ct + NCT <= E) slot_desc(ct + NCT, sl1, sv1, sf1, so1);
    // While warps 0 .. M-1 wait for the logits of every CTA and select, the
    // other compute warps write this CTA's slice of the staged copies of the
    // input (read by every CTA's bulk copies) and publish it on a second
    // counter; both groups then meet before the work list is built (which
    // takes the staging warps' per-format templates).
    if (cw >= M) {
      const int sct = ct - 32 * M, NST = NCT - 32 * M;
      // per-row scale: s puts the row's largest |x| in [2^14, 2^15) for the f16
      // copy and in [2^13, 2^14) for the integer records (every CTA derives the same)
      {
        uint32_t mx[kMaxM];
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) mx[m] = 0;
        for (int k = sct; k < H; k += NST)
#pragma unroll
          for (int m = 0; m < kMaxM; ++m)
            if (m < M) mx[m] = max(mx[m], (uint32_t)(xs[m * H + k] & 0x7FFFu));
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) {
          if (m < M) {
            uint32_t v = mx[m];
            for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0 && v) atomicMax(&s_emax[m], (int)(v >> 7) - 127);
          }
        }
      }
      named_bar_sync(3, NST);
      if (sct < M) s_xsc[sct] = ldexpf(1.0f, -(s_emax[sct] == -1000 ? 0 : 14 - s_emax[sct]));
      {
        uint16_t* xh = (uint16_t*)(P.ws + P.L.xh);
        const int n = M * H, per = (n + G - 1) / G, lo = min(n, per * cta), hi = min(n, lo + per);
        uint16_t* xp = (uint16_t*)(P.ws + P.L.xp);
        for (int i = lo + sct; i < hi; i += NST) {
          const int m = i / H;
          const float v = __uint_as_float((uint32_t)xs[i] << 16);
          const int sh = s_emax[m] == -1000 ? 0 : 14 - s_emax[m];
          const uint16_t hv = __half_as_ushort(__float2half_rn(ldexpf(v, sh)));
          xh[i] = hv;
          xp[(i & ~15) + p16_pos(i & 15)] = hv;  // P order
          if (P.t_out) P.t_out[i] = xs[i];
        }
        {  // T order: 288 positions per 256 columns, 32 of them zero
          uint16_t* xt = (uint16_t*)(P.ws + P.L.xt);
          const int nt = M * (H / 256) * 288, pt = (nt + G - 1) / G, tlo = min(nt, pt * cta), thi = min(nt, tlo + pt);
          for (int i = tlo + sct; i < thi; i += NST) {
            const int run = i / 288, pos = i - run * 288, m = run / (H / 256);
            const int col = t16_col(pos);
            uint16_t hv = 0;
            if (col >= 0) {
              const float v = __uint_as_float((uint32_t)xs[run * 256 + col] << 16);
              hv = __half_as_ushort(__float2half_rn(ldexpf(v, s_emax[m] == -1000 ? 0 : 14 - s_emax[m])));
            }
            xt[i] = hv;
          }
        }
      }
      // the item template of every (phase, format), for expert 0 at address 0
      // with no rows (the work list's templates are these with a few fields changed)
      if (sct < 16) {
        const int ph = sct & 1, f = sct >> 1;
        if (fs_has<FS>(f)) make_tpl(P, s_tbase[ph][f], ph, 0, f, 0ull, 0, 0);
      }
      // the slices are read by bulk copies (async proxy) of every CTA; the h
      // warp releases them (and the output slice and counters zeroed above)
      // on the counter, so that the fence waits in no compute warp
      fence_proxy_async_global();
      named_bar_sync(3, NST);
      if (sct == 0) mbar_arrive(&xbar);
    }
    // ---- the routing: per-row selection (warp m takes row m), then warp 0
    // builds the work list, the row slots and the item templates
    const bool forced = P.forced != nullptr;
    int mine = 0;  // row cw's choice (lane) of the selecting warp, also read by warp 0's one-row work list
    if (cw < M) {
      // Expert e's rank value is (key << 32) | ~e: keys descending, ties to
      // the lower id, every value distinct.  Round j takes the largest value
      // below round j - 1's winner (a tree over the lane's values, then the
      // warp), so the values stay in registers.
      const int m = cw;
      constexpr int QN = kMaxEM / 32;
      uint64_t vv[QN];
      {
        // row m's tagged key of every expert, read until each carries this
        // call's tag (bounded): every CTA publishes its own as soon as its
        // logits are out, so the last one arrives one round trip before it
        // is seen here; only the keys not yet seen are read again
        uint32_t need = 0;
#pragma unroll
        for (int q = 0; q < QN; ++q) {
          vv[q] = 0ull;
          if (lane + 32 * q < E) need |= 1u << q;
        }
        const uint64_t t0 = globaltimer_ns();
        bool okz = true;
        for (int spin = 0;; ++spin) {
#pragma unroll
          for (int q = 0; q < QN; ++q)
            if (need & (1u << q)) vv[q] = ld_relaxed_u64(zk + (size_t)m * E + lane + 32 * q);
#pragma unroll
          for (int q = 0; q < QN; ++q)
            if ((need & (1u << q)) && (uint32_t)vv[q] == tag) need &= ~(1u << q);
          if (!__any_sync(0xffffffffu, need != 0u)) break;
          if (__any_sync(0xffffffffu, s_abort || globaltimer_ns() - t0 > P.limit_ns ||
                                          ((spin & 15) == 15 && *(volatile const int32_t*)err))) {
            okz = false;
            break;
          }
          __nanosleep(64);
        }
        okz = __all_sync(0xffffffffu, okz);
        if (!okz && lane == 0) {
          set_error(err, BQE_ETIMEOUT, kErrWaitFull);
          s_abort = 1;
        }
      }
      if (ct == 0) {
        if (P.diag) dacc(P, 2, globaltimer_ns() - t_cta0, 0);
        rstamp(P, 0, t_cta0);
        rstamp(P, 1, t_cta0);
      }
      __syncwarp();
      // (one read of the abort flag for the whole warp: the rounds below use
      // warp-wide reductions)
      if (!warp_abort(s_abort)) {
#pragma unroll
        for (int q = 0; q < QN; ++q) {
          const int e = lane + 32 * q;
          vv[q] = (e < E && !forced) ? ((vv[q] & 0xFFFFFFFF00000000ull) | (uint32_t)~e) : 0ull;
        }
        // lane j keeps round j's winner; the bookkeeping (choice, the
        // expert's row mask and first choice) is done after the rounds, by
        // lanes 0 .. K-1 at once, so no round waits on shared memory
        if (forced) {
          if (lane < K) mine = s_fidx[m][lane];
        } else {
          uint64_t last = ~0ull;
          for (int j = 0; j < K; ++j) {
            uint64_t t[QN / 2];
#pragma unroll
            for (int q = 0; q < QN / 2; ++q) {
              const uint64_t a = vv[2 * q] < last ? vv[2 * q] : 0ull;
              const uint64_t b = vv[2 * q + 1] < last ? vv[2 * q + 1] : 0ull;
              t[q] = a > b ? a : b;
            }
#pragma unroll
            for (int w = QN / 4; w >= 1; w >>= 1)
#pragma unroll
              for (int q = 0; q < w; ++q) t[q] = t[q] > t[q + w] ? t[q] : t[q + w];
            const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(t[0] >> 32));
            const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(t[0] >> 32) == hi ? (uint32_t)t[0] : 0u);
            last = ((uint64_t)hi << 32) | lo;
            if (lane == j) mine = last ? (int)~lo : 0;
          }
        }
        if (lane < K) {
          s_idx[m][lane] = mine;
          atomicOr(&s_mask[mine], 1u << m);
          atomicMin(&s_first[mine], m * K + lane);
        }
        __syncwarp();
        if (ct == 0) rstamp(P, 2, t_cta0);
      }
    }
    // every row's choices, the slot descriptors and the per-row scales are in
    named_bar_sync(1, NCT);
    {
      if (cw == 0) {
        if (lane == 0) {
          mstamp(P, kStRouted, false);
          rstamp(P, 3, t_cta0);
        }
        // work list: the chosen experts in the order of their first choice
        // (row-major over (row, choice)), u = 1..; the shared expert u = 0.
        // One row, selected (not forced): its K choices are distinct, so
        // choice j is entry j + 1 with row slot j + 1; lane j holds it from
        // the selection, lane K takes the shared expert, and the general
        // pass below (and the row-slot scan) is skipped.
        const bool one_row = RC == 1 && !forced;
        if (one_row) {
          const int u = lane < K ? lane + 1 : 0;
          const int e = lane < K ? mine : E;
          const bool act = lane <= K;
          const int my_bad = act ? s_ebad[e] : 0, my_fmt = act ? s_efmt[e] : 0;
          const uint64_t my_addr = act ? s_eaddr[e] : 0ull;
          const uint32_t rbad = __ballot_sync(0xffffffffu, lane < K && my_bad != 0);
          const bool sbad = __shfl_sync(0xffffffffu, my_bad, K) != 0;
          if (act) {
            if (my_bad) set_error(err, BQE_EDEVICE, my_bad);
            if (lane < K) s_uof[e] = (int16_t)u;
            s_ufmt[u] = my_fmt;
            s_uaddr[u] = my_addr;
            s_urows[u * kMaxM] = 0;
            s_unrows[u] = 1;
            s_rbase[u] = u;
            if (lane == K) s_rbase[K + 1] = K + 1;
            if (cta == 0) {  // the call's work list, for bqe_layer_stats
              ((int32_t*)(P.ws + P.L.u_slot))[u] = s_eslot[e];
              ((int32_t*)(P.ws + P.L.u_fmt))[u] = my_fmt;
              ((int32_t*)(P.ws + P.L.u_nrows))[u] = 1;
            }
          }
          if (lane == 0 && (sbad || rbad)) s_bad = sbad ? 2 : 1;
          __syncwarp();
        }
        int base = 1;
        for (int t0 = 0; t0 < (one_row ? 0 : M * K); t0 += 32) {
          const int t = t0 + lane;
          const int e = t < M * K ? s_idx[t / K][t - (t / K) * K] : 0;
          const bool fst = t < M * K && s_first[e] == t;
          const uint32_t bal = __ballot_sync(0xffffffffu, fst);
          if (fst) {
            const int u = base + __popc(bal & ((1u << lane) - 1u));
            const uint32_t mk = s_mask[e];
            s_uof[e] = (int16_t)u;
            const int my_bad = s_ebad[e], my_fmt = s_efmt[e];
            if (my_bad) {
              set_error(err, BQE_EDEVICE, my_bad);
              s_bad = 1;
            }
            s_ufmt[u] = my_fmt;
            s_uaddr[u] = s_eaddr[e];
            int n = 0;
            for (int mm = 0; mm < M; ++mm)
              if (mk & (1u << mm)) s_urows[u * kMaxM + n++] = (int8_t)mm;
            s_unrows[u] = n;
            if (cta == 0) {  // the call's work list, for bqe_layer_stats
              ((int32_t*)(P.ws + P.L.u_slot))[u] = s_eslot[e];
              ((int32_t*)(P.ws + P.L.u_fmt))[u] = my_fmt;
              ((int32_t*)(P.ws + P.L.u_nrows))[u] = n;
            }
          }
          base += __popc(bal);
        }
        const int tot = one_row ? K : base - 1;
        if (lane == 0 && !one_row) {
          // the shared expert (validated like the others)
          const int sh_bad = s_ebad[E], sh_fmt = s_efmt[E];
          if (sh_bad) {
            set_error(err, BQE_EDEVICE, sh_bad);
            s_bad = 2;
          }
          s_ufmt[0] = sh_fmt;
          s_uaddr[0] = s_eaddr[E];
          s_unrows[0] = M;
          if (cta == 0) {
            ((int32_t*)(P.ws + P.L.u_slot))[0] = s_eslot[E];
            ((int32_t*)(P.ws + P.L.u_fmt))[0] = sh_fmt;
            ((int32_t*)(P.ws + P.L.u_nrows))[0] = M;
          }
        }
        if (lane < M && !one_row) s_urows[lane] = (int8_t)lane;
        __syncwarp();
        if (lane == 0) rstamp(P, 4, t_cta0);
        if (!one_row) {
          // row slots: the shared expert's M rows first, then each chosen
          // expert's rows in work-list order (exclusive prefix, two entries a lane)
          const int u0 = 2 * lane, u1 = 2 * lane + 1;
          const int n0 = u0 <= tot ? s_unrows[u0] : 0, n1 = u1 <= tot ? s_unrows[u1] : 0;
          int incl = n0 + n1;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int tv = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += tv;
          }
          const int ex = incl - n0 - n1;
          if (u0 <= tot + 1) s_rbase[u0] = ex;
          if (u1 <= tot + 1) s_rbase[u1] = ex + n0;
        }
        __syncwarp();
        // on an invalid routed slot only the shared expert runs (the call
        // reports the error; its output is undefined); an invalid shared slot
        // or an aborted routing streams nothing
        const int nu = (warp_abort(s_abort) || s_bad == 2) ? 0 : s_bad ? 1 : 1 + tot;
        if (lane == 0) {
          s_nu = nu;
          if (cta == 0) *(int32_t*)(P.ws + P.L.nu) = nu;
        }
        __syncwarp();
        if (lane == 0) rstamp(P, 5, t_cta0);
        // item templates of every (phase, work-list expert): the format's
        // template (made by the staging warps) with the expert's address, rows and
        // first row slot
        for (int t = lane; t < 2 * nu; t += 32) {
          const int ph = t & 1, u = t >> 1, f = s_ufmt[u];
          if (fs_has<FS>(f)) patch_tpl(P, s_tpl[ph][u], s_tbase[ph][f], ph, u, s_uaddr[u], s_unrows[u], s_rbase[u]);
        }
        __syncwarp();
        if (lane == 0) {
          mstamp(P, kStRoutedMax, true);
          rstamp(P, 6, t_cta0);
          if (P.diag) dacc(P, 3, globaltimer_ns() - t_cta0, 1);
          mbar_arrive(&route_bar);
        }
      }
    }
    named_bar_sync(1, NCT);
    // ---- work items: this warp takes tasks cw, cw + 16, ... of the CTA's task sequence
    const int nU = s_nu;
    const int nTot = nU * (nAper + nBper), nA = nU * nAper;
    const int nmine = cta < nTot ? (nTot - cta + G - 1) / G : 0;
    int k = cw, Ki = 0;
    bool first = true, okc = !warp_abort(s_abort);
    auto run_items = [&](int i0, int i1) {
      for (int i = i0; i < i1 && okc; ++i) {
        const bool isA = cta + i * G < nA;
        const int T = isA ? TA : TB;
        if (k >= Ki + T) {  // no task of this warp in item i
          Ki += T;
          continue;
        }
        // Wait until item i is issued: the producer issues it only after item
        // i - kNQ (same barriers) is freed, so the phase parity then names
        // item i's landing and no other; then wait for the landing itself.
        bool ok = true;
        const uint64_t tw = (P.diag && cw == 0) ? globaltimer_ns() : 0;
        if (s_issued[i % kNP] <= i) {
          const uint64_t t0 = globaltimer_ns();
          for (int spin = 0; s_issued[i % kNP] <= i; ++spin) {
            __nanosleep(32);
            if (s_abort || ((spin & 63) == 63 && (*(volatile const int32_t*)err || globaltimer_ns() - t0 > P.limit_ns))) {
              ok = false;
              break;
            }
          }
        }
        ok = __all_sync(0xffffffffu, ok && mwait(&full[i % kNQ], (i / kNQ) & 1, P.limit_ns, err));
        if (!ok || warp_abort(s_abort)) {
          if (lane == 0) {
            if (!ok) set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
          }
          okc = false;
          break;
        }
        if (first && ct == 0) {
          mstamp(P, kStFirstItem, false);
          rstamp(P, 7, t_cta0);
          first = false;
        }
        const uint64_t tc = (P.diag && cw == 0) ? globaltimer_ns() : 0;
        if (P.diag && cw == 0 && lane == 0) dacc(P, 2, tc - tw);
        const ItemHdr h = hdr[i % kNQ];
        const int tau = k - Ki;
        const uint8_t* base = ring + h.off;
        int tile_i, grp;
        if (isA) {
          tile_i = tau / g.GA;
          grp = tau - tile_i * g.GA;
        } else {
          tile_i = tau / g.GB;
          grp = tau - tile_i * g.GB;
        }
        float* red = reinterpret_cast<float*>(const_cast<uint8_t*>(base) + h.red) + tau * h.R * 32;
        consume_mma<RC, FS>(h.R, h.fmt, base + tile_i * h.tb, isA ? g.kcA : g.kcB, h.nb, grp, base + h.act, lane, red,
                        h.amode);
        __syncwarp();
        if (P.diag && cw == 0 && lane == 0) dacc(P, 3, globaltimer_ns() - tc);
        if (lane == 0) {
          __threadfence_block();
          const int old = atomicAdd(&s_done[i % kNQ], 1);
          if (old == T - 1) {
            __threadfence_block();
            mbar_arrive(&cons[i % kNQ]);
          }
        }
        k += kCW;
        Ki += T;
      }
    };
    // ---- every item of this CTA: W1/W3 items, then W2 items (the W2 rows of h
    // wait, in the producers, for the h units of their expert)
    run_items(0, nmine);
    if (lane == 0) mstamp(P, kStConsEnd, true);
  } else if (warp == kRedWarp) {
    // =============================== reducer ==================================
    // Adds each item's task partials in a fixed order, then frees the item's
    // ring bytes.  W1/W3 items: the g/u chunk partials go to the workspace and
    // the expert's count of finished items is released (once per run of items
    // of one expert).  W2 items: w * y is added to the output rows (fp32
    // atomics: the order of these additions, and so the last bits of the
    // output, can differ from call to call).
    const bool ok0 = __all_sync(0xffffffffu, mwait(&route_bar, 0, P.limit_ns, err));
    const int nU = ok0 ? s_nu : 0;
    const int nTot = nU * (nAper + nBper), nA = nU * nAper;
    const int nmine = cta < nTot ? (nTot - cta + G - 1) / G : 0;
    float* pa = (float*)(P.ws + P.L.m_pa);
    unsigned int* ca = (unsigned int*)(P.ws + P.L.m_ca);
    // W1/W3 items reduced but not yet released: expert cur_u (cur_n items)
    // and the one before it (prev_u, prev_n).  The release fence waits for the
    // partials written so far, so it is taken every second change of expert
    // (and after the last W1/W3 item): one fence publishes two experts.
    int cur_u = -1, cur_n = 0, prev_u = -1, prev_n = 0;
    auto release_a = [&]() {
      if ((cur_n > 0 || prev_n > 0) && lane == 0) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");  // the partials (whole warp: __syncwarp above) first
        if (prev_n > 0) atomicAdd(ca + prev_u, (unsigned int)prev_n);
        if (cur_n > 0) atomicAdd(ca + cur_u, (unsigned int)cur_n);
      }
      cur_n = 0;
      prev_n = 0;
    };
    // The reducer's shared-memory reads wait behind the compute warps' (a few
    // hundred cycles each), so the loop keeps them off its critical path: the
    // next item's header is read as soon as its copies have landed (a
    // non-blocking test of its full barrier), the per-expert values (first
    // row slot, rows, scales, mixing weights) only when the expert changes,
    // and all partials of a row are loaded before any is added.
    ItemHdr hn;
    bool have = false, wready = false;
    int eu = -1, eph = -1, erb = 0;
    int erow[kMaxM];
    float esc[kMaxM];
    for (int i = 0; i < nmine; ++i) {
      const uint64_t tr = P.diag ? globaltimer_ns() : 0;
      if (!have) {  // the header of item i is readable once its copies have landed
        if (!__all_sync(0xffffffffu, mwait(&full[i % kNQ], (i / kNQ) & 1, P.limit_ns, err)) || warp_abort(s_abort)) {
          if (lane == 0) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
          }
          break;
        }
        hn = hdr[i % kNQ];
      }
      const ItemHdr h = hn;
      const int u = h.u, R = RC == 1 ? 1 : h.R;
      if (h.phase == 1 && !wready) {  // the mixing weights (h warp) before the first W2 item
        if (!__all_sync(0xffffffffu, mwait(&wbar, 0, P.limit_ns, err)) || warp_abort(s_abort)) {
          if (lane == 0) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
          }
          break;
        }
        wready = true;
      }
      if (u != eu || h.phase != eph) {  // this expert's row slots, rows and scales
        eu = u;
        eph = h.phase;
        erb = s_rbase[u];
#pragma unroll
        for (int r = 0; r < kMaxM; ++r) {
          if (r < R) {
            const int row = u == 0 ? r : s_urows[u * kMaxM + r];
            erow[r] = row;
            esc[r] = h.phase == 0 ? s_xsc[row] : s_rsw[erb + r];
          }
        }
      }
      const bool okc = __all_sync(0xffffffffu, mwait(&cons[i % kNQ], (i / kNQ) & 1, P.limit_ns, err));
      if (P.diag && lane == 0) dacc(P, 4, globaltimer_ns() - tr);
      if (!okc || warp_abort(s_abort)) {
        if (lane == 0) {
          set_error(err, BQE_ETIMEOUT, kErrWaitFull);
          s_abort = 1;
        }
        break;
      }
      // the next item's header, if it has landed already
      have = i + 1 < nmine && mbar_test_wait(&full[(i + 1) % kNQ], ((i + 1) / kNQ) & 1);
      have = __all_sync(0xffffffffu, have);
      if (have) hn = hdr[(i + 1) % kNQ];
      const float* red = reinterpret_cast<const float*>(ring + h.off + h.red);
      if (h.phase == 0) {
        if (u != cur_u) {
          if (prev_n > 0) release_a();  // two experts pending: publish both
          prev_u = cur_u;
          prev_n = cur_n;
          cur_u = u;
          cur_n = 0;
        }
        // chunk partials of g and u for this panel (the f16 input's scale removed: exact power of two)
#pragma unroll
        for (int r = 0; r < (RC == 1 ? 1 : kMaxM); ++r) {
          if (r >= R) break;
          float v0[4], v1[4];
#pragma unroll
          for (int gi = 0; gi < 4; ++gi) {
            v0[gi] = gi < g.GA ? red[(gi * R + r) * 32 + lane] : 0.f;
            v1[gi] = gi < g.GA ? red[((g.GA + gi) * R + r) * 32 + lane] : 0.f;
          }
          const float a0 = ((v0[0] + v0[1]) + v0[2]) + v0[3], a1 = ((v1[0] + v1[1]) + v1[2]) + v1[3];
          const int64_t base = ((((int64_t)(erb + r) * g.npanA + h.p) * g.nchA + h.c) * 2) * 32;
          pa[base + lane] = a0 * esc[r];
          pa[base + 32 + lane] = a1 * esc[r];
        }
        ++cur_n;
        __syncwarp();
        if (cta + (i + 1) * G >= nA) release_a();  // this CTA's last W1/W3 item
      } else {
        for (int pi = 0; pi < P.PB; ++pi) {
          const int n = (h.p * P.PB + pi) * 32 + lane;
#pragma unroll
          for (int r = 0; r < (RC == 1 ? 1 : kMaxM); ++r) {
            if (r >= R) break;
            float v[4];
#pragma unroll
            for (int gi = 0; gi < 4; ++gi) v[gi] = gi < g.GB ? red[((pi * g.GB + gi) * R + r) * 32 + lane] : 0.f;
            const float y = ((v[0] + v[1]) + v[2]) + v[3];
            red_add_f32(P.out + (int64_t)erow[r] * H + n, esc[r] * y);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&freed[i % kNQ]);  // the item's ring bytes may be reused
    }
    __syncwarp();
    release_a();
  } else {
    // ================================ h warp ==================================
    // h = silu(g) * u of this CTA's units (row slot, 256 columns of the
    // intermediate dimension), units dealt round-robin over the CTAs in
    // work-list order: wait (bounded) until every W1/W3 item of the unit's
    // expert is done, add the K-chunk partials in chunk order, and write h in
    // fp32 (MXFP4 W2 loops) or as integer records (X_hi + X_lo / 128 of
    // h 2^si, max |h| 2^si in [2^13, 2^14), in the expert's format order, with
    // the 16-column sums and 2^-si); then release the expert's count of units.
    // ---- first, while the routing runs: the item template of every (phase,
    // format), for expert 0 at address 0 with no rows (the work list's
    // templates are these with a few fields changed)
    // first: this CTA's staged slices of the input, once the staging warps
    // have written them, released on the staged-input counter (one arrival
    // per CTA per call; also releases the zeroed output slice and counters)
    {
      const bool okx = __all_sync(0xffffffffu, mwait(&xbar, 0, P.limit_ns, err));
      if (lane == 0) {
        if (!okx) set_error(err, BQE_ETIMEOUT, kErrWaitFull);
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        atomicAdd((unsigned long long*)(P.ws + P.L.st), 1ull);
        if (P.diag) dacc(P, 1, globaltimer_ns() - t_cta0, 0);
      }
    }
    const bool ok0 = __all_sync(0xffffffffu, mwait(&route_bar, 0, P.limit_ns, err));
    const int nU = ok0 ? s_nu : 0;
    const int nrs = nU > 0 ? s_rbase[nU] : 0;
    const int nblk = I / 256, nunits = nrs * nblk;
    // ---- the mixing weights, off the routing's critical path (the reducer
    // waits for them before its first W2 item): w_j = s_j / sum s over row m's
    // choices as exp(log s_j - max log s) / sum exp(...), finite even when
    // every selected sigmoid underflows in fp32; then each row slot's weight
    // (the sum over the row's choices of that expert; shared expert rows: 1)
    if (ok0 && !warp_abort(s_abort)) {  // (warp-uniform: shuffles below)
      // the selected logits, read until each carries this call's tag
      // (bounded; their keys were seen, so they are normally there)
      const unsigned long long* zl = (const unsigned long long*)(P.ws + P.L.zl);
      bool okl = true;
      for (int t = lane; t < M * K && okl; t += 32) {
        const unsigned long long* a = zl + (size_t)(t / K) * E + s_idx[t / K][t % K];
        const uint64_t t0 = globaltimer_ns();
        unsigned long long v = ld_relaxed_u64(a);
        while ((uint32_t)v != tag) {
          if (globaltimer_ns() - t0 > P.limit_ns || *(volatile const int32_t*)err) {
            okl = false;
            break;
          }
          __nanosleep(64);
          v = ld_relaxed_u64(a);
        }
        s_zsel[t / K][t % K] = __uint_as_float((uint32_t)(v >> 32));
      }
      if (!okl) {
        set_error(err, BQE_ETIMEOUT, kErrWaitFull);
        s_abort = 1;
      }
      __syncwarp();
      for (int m = 0; m < M; ++m) {
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
          if (cta == 0) {
            if (P.topk_idx) P.topk_idx[m * K + lane] = s_idx[m][lane];
            if (P.topk_w) P.topk_w[m * K + lane] = w;
          }
        }
      }
      __syncwarp();
      if (lane < M) s_rsw[lane] = 1.0f;
      if (nU > 1)
        for (int t = lane; t < M * K; t += 32) {
          const int m = t / K, j = t - (t / K) * K;
          const int ee = s_idx[m][j];
          const int rs = s_rbase[s_uof[ee]] + __popc(s_mask[ee] & ((1u << m) - 1u));
          bool fj = true;
          float w = 0.f;
          for (int j2 = 0; j2 < K; ++j2)
            if (s_idx[m][j2] == ee) {
              fj = fj && j2 >= j;
              w += s_cw[m][j2];
            }
          if (fj) s_rsw[rs] = w;
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&wbar);
    const float* pa = (const float*)(P.ws + P.L.m_pa);
    const unsigned int* ca = (const unsigned int*)(P.ws + P.L.m_ca);
    unsigned int* chc = (unsigned int*)(P.ws + P.L.m_ch);
    int u = 0, ready = -1, cur_n = 0;
    bool okh = true;
    auto release_h = [&]() {
      if (cur_n > 0 && lane == 0) {
        fence_proxy_async_global();  // h is read by other CTAs' bulk copies
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        atomicAdd(chc + u, (unsigned int)cur_n);
      }
      cur_n = 0;
    };
    for (int unit = cta; unit < nunits && okh; unit += G) {
      const int rs = unit / nblk, blk = unit - (unit / nblk) * nblk;
      int un = u;
      while (un + 1 < nU && s_rbase[un + 1] <= rs) ++un;
      if (un != u) {
        release_h();
        u = un;
      }
      if (u > ready) {
        bool okw = true;
        if (lane == 0) okw = wait_ge(ca + u, (uint32_t)nAper, P.limit_ns, err);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          if (lane == 0) {
            set_error(err, BQE_ETIMEOUT, kErrWaitFull);
            s_abort = 1;
          }
          okh = false;
          break;
        }
        ready = u;
      }
      // lane: 8 consecutive columns i0 .. i0 + 7 of one 32-column panel, four at
      // a time; the K-chunk partials of g and u added in chunk order, four
      // chunks loaded together
      const int i0 = blk * 256 + lane * 8, p = i0 >> 5, l0 = i0 & 31;
      const float* src = pa + (((int64_t)rs * g.npanA + p) * g.nchA) * 2 * 32 + l0;
      float hv[8];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        for (int c0 = 0; c0 < g.nchA; c0 += 4) {
          float4 gv[4], uv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (c0 + c < g.nchA) {
              gv[c] = __ldcg(reinterpret_cast<const float4*>(src + (c0 + c) * 64 + 4 * q));
              uv[c] = __ldcg(reinterpret_cast<const float4*>(src + (c0 + c) * 64 + 32 + 4 * q));
            }
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (c0 + c < g.nchA) {
              a.x += gv[c].x; a.y += gv[c].y; a.z += gv[c].z; a.w += gv[c].w;
              b.x += uv[c].x; b.y += uv[c].y; b.z += uv[c].z; b.w += uv[c].w;
            }
        }
        hv[4 * q] = silu_m(a.x) * b.x;
        hv[4 * q + 1] = silu_m(a.y) * b.y;
        hv[4 * q + 2] = silu_m(a.z) * b.z;
        hv[4 * q + 3] = silu_m(a.w) * b.w;
      }
      const int fmt = s_ufmt[u];
      {
        // f16 hi + lo of h 2^si, max |h| 2^si in [2^14, 2^15)
        uint32_t mx = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) mx = max(mx, __float_as_uint(hv[k]) & 0x7FFFFFFFu);
        mx = __reduce_max_sync(0xffffffffu, mx);
        const int ex = (int)(mx >> 23);
        const int si = ex == 0 ? 0 : min(max(14 - (ex - 127), -100), 100);
        const int ck = blk / bpcB, kb = blk - ck * bpcB;
        uint8_t* rec = P.ws + P.L.m_hr + ((size_t)rs * g.nchB + ck) * hrec_stride(g.kcB);
        const int flen = f16_len(fmt, g.kcB);
        uint16_t* hdst = reinterpret_cast<uint16_t*>(rec);
        uint16_t* ldst = reinterpret_cast<uint16_t*>(rec + 2 * flen + 64);
        if (lane == 0) reinterpret_cast<float*>(rec + 4 * flen + 64)[kb] = ldexpf(1.0f, -si);
        if (fmt == BQE_FMT_TQ1) {
          // T order: h of the unit through shared memory, 9 positions per lane
          float* sh = s_hunit;
#pragma unroll
          for (int k = 0; k < 8; ++k) sh[lane * 8 + k] = hv[k];
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 9; ++k) {
            const int pos = lane + 32 * k, col = t16_col(pos);
            const float v = col >= 0 ? ldexpf(sh[col], si) : 0.f;
            const __half h0 = __float2half_rn(v);
            hdst[kb * 288 + pos] = __half_as_ushort(h0);
            ldst[kb * 288 + pos] = __half_as_ushort(__float2half_rn(v - __half2float(h0)));
          }
          __syncwarp();
        } else {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float v0 = ldexpf(hv[2 * k], si), v1 = ldexpf(hv[2 * k + 1], si);
            const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
            const __half l0 = __float2half_rn(v0 - __half2float(h0)), l1 = __float2half_rn(v1 - __half2float(h1));
            hw[k] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
            lw[k] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
          }
          if (fmt == BQE_FMT_Q2_0 || fmt == BQE_FMT_Q3_K) {
            // P order: in every 16 columns (lanes 2m, 2m + 1) position 2p holds
            // column p and 2p + 1 column 8 + p: the even lane writes (c0, c8, ..,
            // c3, c11), the odd one (c4, c12, .., c7, c15)
            const bool odd = lane & 1;
            auto p_order = [&](uint32_t& w0, uint32_t& w1, uint32_t& w2, uint32_t& w3) {
              const uint32_t s0 = __shfl_xor_sync(0xffffffffu, odd ? w0 : w2, 1);
              const uint32_t s1 = __shfl_xor_sync(0xffffffffu, odd ? w1 : w3, 1);
              const uint32_t m0 = odd ? s0 : w0, m1 = odd ? s1 : w1;  // columns 0..3 (4..7) of the 16
              const uint32_t n0 = odd ? w2 : s0, n1 = odd ? w3 : s1;  // columns 8..11 (12..15)
              w0 = __byte_perm(m0, n0, 0x5410);
              w1 = __byte_perm(m0, n0, 0x7632);
              w2 = __byte_perm(m1, n1, 0x5410);
              w3 = __byte_perm(m1, n1, 0x7632);
            };
            p_order(hw[0], hw[1], hw[2], hw[3]);
            p_order(lw[0], lw[1], lw[2], lw[3]);
          }
          const int col = kb * 256 + lane * 8;
          *reinterpret_cast<uint4*>(hdst + col) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(ldst + col) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      ++cur_n;
      __syncwarp();
    }
    __syncwarp();
    release_h();
  }

  // ---- end: CTA 0's producers saw every CTA's staged-input arrival (made
  // after that CTA read the tag), so every CTA has read this call's tag: CTA 0
  // advances the epoch for the next call
  __syncthreads();
  if (tid == 0) {
    mstamp(P, kStEnd, true);
    dacc(P, 7, globaltimer_ns() - t_cta0);
    if (cta == 0) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      *(volatile uint32_t*)(P.ws + P.L.epoch) = tag;
    }
  }
}

// W2 output panels per item: the largest count that divides the panels and
// keeps the item at <= 16 compute tasks (one per compute warp).  Fewer, larger
// W2 items cost less per byte in the producers and the reducer.
static int moe_pb(const Geo& g) {
  int best = 1;
  for (int pb = 1; pb * g.GB <= kCW; ++pb)
    if (g.npanB % pb == 0) best = pb;
  return best;
}

// Largest byte size of one item (the largest tile of any format, T-order x
// rows the longest staged rows).
static uint32_t moe_max_item(const Geo& g, int PB) {
  auto a128 = [](uint32_t v) { return (v + 127u) & ~127u; };
  auto max_tile = [](int kc) {
    uint32_t t = 0;
    for (int f = BQE_FMT_TQ1; f <= BQE_FMT_NVFP4; ++f) t = tile_bytes(f, kc) > t ? tile_bytes(f, kc) : t;
    return t;
  };
  const uint32_t actA = (uint32_t)act_row_stride(kActF16, BQE_FMT_TQ1, g.kcA);
  const uint32_t A = a128(2 * max_tile(g.kcA)) + a128(g.M * actA) + 2 * g.GA * g.M * 128;
  const uint32_t actB = hrec_stride(g.kcB);
  const uint32_t B = a128(PB * max_tile(g.kcB)) + a128(g.M * actB) + PB * g.GB * g.M * 128;
  return A > B ? A : B;
}

int launch_moe(const MoeParams& P0, int grid, cudaStream_t st) {
  MoeParams P = P0;
  const Geo& g = P.g;
  if (g.E > kMaxEM || g.E > 4 * grid || g.H / 4 / 128 > 16 || g.H % 512 || g.I % 256 || g.K > kMaxTopK ||
      g.U > kMaxU || 2 * g.nchA > 24 || (uint64_t)g.M * (g.K + 1) * g.nchB * hrec_stride(g.kcB) >= (1ull << 32))
    return BQE_EUNSUPPORTED;
  P.PB = moe_pb(g);
  static int limit_set[2][3][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BQE_ECUDA;
  const int rc = g.M == 1 ? 0 : 1;
  // the instance: one-row calls run one where M is the constant 1 (one B
  // column group per MMA, no wide W2 items); a pool whose format mask names
  // MXFP4 alone, or low-bit formats alone, runs one that carries only those
  // formats' loops (a mask of 0: any format)
  const uint32_t mask = (uint32_t)P.pool.fmt_mask;
  const uint32_t low = (1u << BQE_FMT_TQ1) | (1u << BQE_FMT_Q2_0) | (1u << BQE_FMT_Q3_K);
  const int fs = mask == (1u << BQE_FMT_MXFP4) ? kFsFp4 : (mask != 0 && (mask & ~low) == 0) ? kFsLowBit : kFsAll;
  void (*const kfns[2][3])(MoeParams) = {{k_moe<1, kFsAll>, k_moe<1, kFsFp4>, k_moe<1, kFsLowBit>},
                                         {k_moe<2, kFsAll>, k_moe<2, kFsFp4>, k_moe<2, kFsLowBit>}};
  void (*kfn)(MoeParams) = kfns[rc][fs];
  // the dynamic shared memory an instance may take on this device (queried
  // once per instance and device: the queries cost host time on every call)
  static std::atomic<int> dyn_cache[2][3][64];
  int dyn_max = dyn_cache[rc][fs][dev].load(std::memory_order_relaxed);
  if (dyn_max == 0) {
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, (const void*)kfn) != cudaSuccess)
      return BQE_ECUDA;
    dyn_max = optin - (int)fa.sharedSizeBytes;
    if (dyn_max > 0) dyn_cache[rc][fs][dev].store(dyn_max, std::memory_order_relaxed);
  }
  if (dyn_max <= 0) return BQE_EUNSUPPORTED;
  P.ring_bytes = (uint32_t)dyn_max & ~127u;
  const uint32_t xst = ((uint32_t)g.M * g.H * 2 + 127u) & ~127u;
  const uint32_t rtb = (uint32_t)((g.E + grid - 1) / grid) * g.H * 4;  // router rows of one CTA
  if (P.ring_bytes < moe_max_item(g, P.PB) || P.ring_bytes < xst + rtb + 1024) return BQE_EUNSUPPORTED;
  P.xstage_off = P.ring_bytes - xst;
  P.rt_off = P.xstage_off - rtb;
  // item index t -> (expert, panel, chunk) by multiply-high: exact while t * d < 2^32
  auto mag = [](uint64_t d) { return (0x100000000ull + d - 1) / d; };
  const uint32_t nAper = (uint32_t)g.npanA * g.nchA, nBper = (uint32_t)(g.npanB / P.PB) * g.nchB;
  if ((uint64_t)g.U * (nAper + nBper) * (nAper > nBper ? nAper : nBper) >= (1ull << 32)) return BQE_EUNSUPPORTED;
  P.magA = mag(nAper);
  P.magA2 = mag(g.nchA);
  P.magB = mag(nBper);
  P.magB2 = mag(g.nchB);
  if (limit_set[rc][fs][dev] < dyn_max) {
    if (cudaFuncSetAttribute((const void*)kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) != cudaSuccess)
      return BQE_ECUDA;
    limit_set[rc][fs][dev] = dyn_max;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMoeThreads);
  cfg.dynamicSmemBytes = P.ring_bytes;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: CTAs wait on one another
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kfn, P) == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

}  // namespace bqe
