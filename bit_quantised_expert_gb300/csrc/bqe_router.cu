// bqe_router.cu — router GEMV, sigmoid scores, selection-biased top-k, and the
// per-call expert work list.
//
// Router (field report, section 1: 384 routed experts, 6 per token; Strata
// 4090 post, section 5.3: a routing bias that changes which experts are
// computed while the mixing weights stay exact):
//   z[m,e] = sum_h x[m,h] Wr[e,h]   (fp32 accumulation)
//   s = sigmoid(z), key = s + b, idx = top-k(key) (ties -> lower e),
//   w_j = s[idx_j] / sum_j' s[idx_j'].
// Work list: the distinct experts chosen by the M rows plus the shared
// expert (u = 0), each with the rows that chose it, so every expert's bytes
// are streamed once per call however many rows use it (field report, section
// 4.2: one transfer of an expert's bytes serves every token of a batch).
//
// One kernel: every CTA computes z for two experts (four warps per expert,
// one quarter of hidden each, all loads in flight at once); the last CTA to
// finish (arrival counter, no waiting) selects, weighs and builds the list.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bqe_internal.cuh"

namespace bqe {


constexpr int kRouteThreads = 256;
constexpr int kMaxE = 512;  // routed experts per layer supported by the selection

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

constexpr int kRouteMaxNI = 16;  // float4 router loads per lane: hidden / 512 (hidden <= 8192)

// One instance per row count MR (= M) keeps each instance's code short: a
// decode call runs this kernel once, so every instruction is fetched cold.
template <int MR>
__global__ void __launch_bounds__(kRouteThreads) k_route(RouteParams P) {
  const Geo& g = P.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = g.H, E = g.E, K = g.K;
  constexpr int M = MR;
  const long long t_start = clock64();
  if (P.diag && threadIdx.x == 0) dbg_span(P.ws, P.L.dbg, 2, false);
  int32_t* err = (int32_t*)(P.ws + P.L.err);
  float* z = (float*)(P.ws + P.L.z);
  extern __shared__ __align__(16) uint16_t xs[];  // M x H bf16 layer input

  __shared__ float inv_rms[kMaxM];
  __shared__ float red[8][kMaxM];
  __shared__ int s_last;

  // warp = (expert 2*blockIdx + warp/4, quarter warp%4); every router load of
  // the lane is issued before anything waits
  const int e = blockIdx.x * 2 + (warp >> 2);
  const int q = warp & 3;
  const int Kq = H / 4;
  const int ni = Kq / 128;
  float4 w4[kRouteMaxNI];
  if (e < E) {
    const float4* wr = (const float4*)(P.router_w + (int64_t)e * H + (int64_t)q * Kq);
    const uint64_t pol = policy_evict_first();
#pragma unroll
    for (int i = 0; i < kRouteMaxNI; ++i)
      if (i < ni) w4[i] = ldg_stream_f4(wr + i * 32 + lane, pol);
  }

  // inputs of the selection, read while the previous kernel finishes (no
  // kernel of the layer writes them): the slot of every expert, the slot's
  // format and offset (out-of-range slots are reported when used), the bias
  __shared__ int32_t s_table[kMaxE + 1];
  __shared__ int32_t s_sfmt[kMaxE + 1];
  __shared__ uint64_t s_soff[kMaxE + 1];
  __shared__ float s_bias[kMaxE];
  for (int i = tid; i <= E; i += kRouteThreads) {
    const int sl = P.slot_table[i];
    const bool okr = sl >= 0 && sl < P.pool.n_slots;
    s_table[i] = sl;
    s_sfmt[i] = okr ? P.pool.slot_fmt[sl] : 0;
    s_soff[i] = okr ? P.pool.slot_off[sl] : 0;
    if (i < E) s_bias[i] = P.bias ? P.bias[i] : 0.f;
  }

  griddep_wait();  // the layer input may come from the previous kernels
  griddep_launch_dependents();  // the W1/W3 kernel may start its own prologue now

  // ---- layer input into shared memory: bf16 x, or bf16(rmsnorm(resid)) -------
  if (P.resid) {
    for (int m = 0; m < M; ++m) {
      float ss = 0.f;
      for (int k = tid; k < H; k += kRouteThreads) {
        float v = P.resid[(int64_t)m * H + k];
        ss = fmaf(v, v, ss);
      }
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) red[warp][m] = ss;
    }
    __syncthreads();
    if (tid < M) {
      float ss = 0.f;
      for (int w = 0; w < kRouteThreads / 32; ++w) ss += red[w][tid];
      inv_rms[tid] = 1.0f / sqrtf(ss / (float)H + 1e-6f);
    }
    __syncthreads();
    for (int i = tid; i < M * H; i += kRouteThreads) {
      const int m = i / H;
      const __nv_bfloat16 t = __float2bfloat16_rn(P.resid[i] * inv_rms[m]);
      xs[i] = __bfloat16_as_ushort(t);
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(P.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = tid; i < M * H / 8; i += kRouteThreads) dst[i] = src[i];
  }
  __syncthreads();

  // ---- router GEMV ----------------------------------------------------------
  float acc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) acc[m] = 0.f;
  if (e < E) {
#pragma unroll
    for (int i = 0; i < kRouteMaxNI; ++i) {
      if (i < ni) {
        const int k = q * Kq + (i * 32 + lane) * 4;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const uint2 xv = *reinterpret_cast<const uint2*>(xs + m * H + k);
          acc[m] = fmaf(w4[i].x, __uint_as_float(xv.x << 16), acc[m]);
          acc[m] = fmaf(w4[i].y, __uint_as_float(xv.x & 0xFFFF0000u), acc[m]);
          acc[m] = fmaf(w4[i].z, __uint_as_float(xv.y << 16), acc[m]);
          acc[m] = fmaf(w4[i].w, __uint_as_float(xv.y & 0xFFFF0000u), acc[m]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float v = acc[m];
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    acc[m] = v;
  }
  __syncthreads();  // red[] reuse
  if (lane == 0)
    for (int m = 0; m < M; ++m) red[warp][m] = acc[m];
  __syncthreads();
  if (tid < 2 * M) {
    const int el = tid / M, m = tid % M, ee = blockIdx.x * 2 + el;
    if (ee < E) {
      float sum = red[el * 4 + 0][m] + red[el * 4 + 1][m] + red[el * 4 + 2][m] + red[el * 4 + 3][m];
      z[(int64_t)m * E + ee] = sum;
    }
  }

  if (P.diag && tid == 0 && blockIdx.x < kDbgMaxCtas) {
    atomicAdd((unsigned long long*)(P.ws + P.L.dbg) + ((size_t)2 * kDbgMaxCtas + blockIdx.x) * kDbgSlots + 0,
              (unsigned long long)(clock64() - t_start));
    dbg_span(P.ws, P.L.dbg, 2, true);
  }
  // ---- arrival: the last CTA selects ----------------------------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    unsigned int* ctr = (unsigned int*)(P.ws + P.L.ctr_route);
    s_last = (int)atomicAdd(ctr, 1u);
  }
  __syncthreads();
  const int rank = s_last;
  const bool last = rank == (int)gridDim.x - 1;
  if (!last) return;
  __threadfence();
  auto stamp = [&](int k) {
    if (P.diag && tid == 0)
      atomicAdd((unsigned long long*)(P.ws + P.L.dbg) + ((size_t)2 * kDbgMaxCtas + 1021) * kDbgSlots + k,
                (unsigned long long)(clock64() - t_start));
  };
  stamp(0);


  __shared__ uint32_t s_mask[kMaxE];           // bit m: row m chose expert e
  __shared__ int16_t s_uof[kMaxE];              // work-list index of a chosen expert
  __shared__ int s_idx[kMaxM][kMaxTopK];
  __shared__ float s_zsel[kMaxM][kMaxTopK];
  __shared__ int s_list[kMaxM * kMaxTopK];      // chosen experts, ascending
  __shared__ int s_wcnt[2][kRouteThreads / 32];
  __shared__ int s_bad;
  __shared__ int s_nu;
  if (tid == 0) s_bad = 0;
  for (int i = tid; i < E; i += kRouteThreads) s_mask[i] = 0u;
  __syncthreads();
  stamp(1);

  // ---- top-k: the keys of every row in shared memory (all threads), then
  // warp m selects row m: each lane holds the keys of experts lane, lane + 32,
  // ...; a round takes the lane's largest key (strict compare in ascending
  // expert order keeps the lower id on a tie), then one warp max and one warp
  // min decide the round.  Order: larger key first, ties to the lower id.
  __shared__ uint32_t s_key[kMaxM][kMaxE];
  float* s_zr = reinterpret_cast<float*>(xs);  // logits, row-major M x E (x is no longer needed; E <= H / 2)
  if (!P.forced) {
    for (int i = tid; i < M * E; i += kRouteThreads) {
      const int m = i / E, e = i - m * E;
      const float zv = __ldcg(z + i);
      s_zr[i] = zv;
      s_key[m][e] = sel_key(zv, s_bias[e]);
    }
  }
  __syncthreads();
  stamp(7);
  if (warp < M) {
    const int m = warp;
    constexpr int QN = kMaxE / 32;
    uint32_t kk[QN];
#pragma unroll
    for (int q = 0; q < QN; ++q) {
      const int e = lane + 32 * q;
      kk[q] = (!P.forced && e < E) ? s_key[m][e] : 0u;
    }
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
        uint32_t bk = 0u;
        int bq = 0;
#pragma unroll
        for (int q = 0; q < QN; ++q)
          if (kk[q] > bk) {
            bk = kk[q];
            bq = q;
          }
        const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t eb =
            __reduce_min_sync(0xffffffffu, (bk == wk && wk != 0u) ? (uint32_t)(lane + 32 * bq) : 0xffffffffu);
#pragma unroll
        for (int q = 0; q < QN; ++q)
          if (eb == (uint32_t)(lane + 32 * q)) kk[q] = 0u;
        best = eb == 0xffffffffu ? 0 : (int)eb;
        zsel = s_zr[m * E + best];
      }
      if (lane == 0) {
        s_idx[m][j] = best;
        s_zsel[m][j] = zsel;
        atomicOr(&s_mask[best], 1u << m);
      }
    }
    __syncwarp();
    if (m == 0) stamp(2);
    // mixing weights w_j = s_j / sum s from the unbiased scores, evaluated as
    // exp(log s_j - max log s) / sum exp(...): the same ratio, finite even when
    // every selected sigmoid underflows in fp32.  Lane j takes expert j.
    float ls = -INFINITY;
    if (lane < K) {
      const float zz = s_zsel[m][lane];
      ls = zz < 0.f ? zz - log1pf(expf(zz)) : -log1pf(expf(-zz));  // log sigmoid(z)
    }
    float mx = ls;
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ev = lane < K ? expf(ls - mx) : 0.f;
    float tot = ev;
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane < K) {
      const float w = ev / tot;
      ((float*)(P.ws + P.L.comb_w))[m * K + lane] = w;
      if (P.topk_idx) P.topk_idx[m * K + lane] = s_idx[m][lane];
      if (P.topk_w) P.topk_w[m * K + lane] = w;
    }
  }
  __syncthreads();
  stamp(3);

  int32_t* u_slot = (int32_t*)(P.ws + P.L.u_slot);
  int32_t* u_fmt = (int32_t*)(P.ws + P.L.u_fmt);
  uint64_t* u_addr = (uint64_t*)(P.ws + P.L.u_addr);
  int32_t* u_nrows = (int32_t*)(P.ws + P.L.u_nrows);
  int32_t* u_rows = (int32_t*)(P.ws + P.L.u_rows);

  // compact the chosen experts in ascending id order (u = 1..), shared u = 0:
  // expert e = it*256 + warp*32 + lane, positions from per-warp counts
  bool on[2];
  uint32_t bal[2];
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int ee = it * kRouteThreads + tid;
    on[it] = ee < E && s_mask[ee] != 0u;
    bal[it] = __ballot_sync(0xffffffffu, on[it]);
    if (lane == 0) s_wcnt[it][warp] = __popc(bal[it]);
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    if (on[it]) {
      int base = 0;
      for (int i2 = 0; i2 < it; ++i2)
        for (int w2 = 0; w2 < kRouteThreads / 32; ++w2) base += s_wcnt[i2][w2];
      for (int w2 = 0; w2 < warp; ++w2) base += s_wcnt[it][w2];
      const int pos = base + __popc(bal[it] & ((1u << lane) - 1u));
      const int ee = it * kRouteThreads + tid;
      s_list[pos] = ee;
      s_uof[ee] = 1 + pos;
    }
  }
  if (tid == 0) {
    int tot = 0;
    for (int i2 = 0; i2 < 2; ++i2)
      for (int w2 = 0; w2 < kRouteThreads / 32; ++w2) tot += s_wcnt[i2][w2];
    s_nu = 1 + tot;
  }
  __syncthreads();
  const int nU = s_nu;
  stamp(4);
  // per-u descriptors
  for (int u = tid; u < nU; u += kRouteThreads) {
    const int ee = u == 0 ? -1 : s_list[u - 1];
    const uint32_t mask = u == 0 ? ((M >= 32) ? 0xffffffffu : ((1u << M) - 1u)) : s_mask[ee];
    const int slot = s_table[u == 0 ? E : ee];
    int fmt = 0;
    uint64_t addr = 0;
    if (slot < 0 || slot >= P.pool.n_slots) {
      set_error(err, BQE_EDEVICE, kErrSlotRange);
      s_bad = 1;
    } else {
      fmt = s_sfmt[u == 0 ? E : ee];
      const uint64_t off = s_soff[u == 0 ? E : ee];
      if (!fmt_ok(fmt)) {
        set_error(err, BQE_EDEVICE, kErrSlotFmt);
        s_bad = 1;
      } else {
        const uint64_t bytes = 2 * matrix_bytes(fmt, g.I, g.H) + matrix_bytes(fmt, g.H, g.I);
        if ((off & 15) || off + bytes > P.pool.base_bytes) {
          set_error(err, BQE_EDEVICE, kErrSlotExtent);
          s_bad = 1;
        }
        addr = (uint64_t)P.pool.base + off;
      }
    }
    u_slot[u] = slot;
    u_fmt[u] = fmt;
    u_addr[u] = addr;
    int n = 0;
    for (int m = 0; m < M; ++m)
      if (mask & (1u << m)) u_rows[u * kMaxM + n++] = m;
    u_nrows[u] = n;
  }
  stamp(5);
  if (warp < M && lane < K) {
    const int m = warp, j = lane;
    const int ee = s_idx[m][j];
    ((int32_t*)(P.ws + P.L.comb_u))[m * K + j] = s_uof[ee];
    ((int32_t*)(P.ws + P.L.comb_r))[m * K + j] = __popc(s_mask[ee] & ((1u << m) - 1u));
  }
  __syncthreads();
  stamp(6);
  if (tid == 0) {
    *(int32_t*)(P.ws + P.L.nu) = s_bad ? 0 : nU;
    *(unsigned int*)(P.ws + P.L.ctr_route) = 0u;
    if (P.diag) {
      atomicAdd((unsigned long long*)(P.ws + P.L.dbg) + ((size_t)2 * kDbgMaxCtas + 1022) * kDbgSlots + 1,
                (unsigned long long)(clock64() - t_start));
      dbg_span(P.ws, P.L.dbg, 2, true);
    }
  }
}

int launch_route(const RouteParams& P, cudaStream_t st, bool pdl) {
  const int grid = (P.g.E + 1) / 2;
  const size_t smem = (size_t)P.g.M * P.g.H * 2;
  if (P.g.H / 4 / 128 > kRouteMaxNI || P.g.H % 512 || 2 * P.g.E > P.g.H) return BQE_EUNSUPPORTED;
  static int limit_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BQE_ECUDA;
  void (*fns[kMaxM])(RouteParams) = {k_route<1>, k_route<2>, k_route<3>, k_route<4>,
                                     k_route<5>, k_route<6>, k_route<7>, k_route<8>};
  auto fn = fns[P.g.M - 1];
  if (smem > 48 * 1024 && limit_set[dev] < (int)smem) {
    // dynamic + static shared memory must fit the opt-in limit of a block
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return BQE_ECUDA;
    int lim = 1 << 30;
    for (int m = 0; m < kMaxM; ++m) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, fns[m]) != cudaSuccess) return BQE_ECUDA;
      lim = std::min(lim, optin - (int)fa.sharedSizeBytes);
    }
    if (lim < (int)smem) return BQE_EUNSUPPORTED;
    for (int m = 0; m < kMaxM; ++m)
      if (cudaFuncSetAttribute(fns[m], cudaFuncAttributeMaxDynamicSharedMemorySize, lim) != cudaSuccess)
        return BQE_ECUDA;
    limit_set[dev] = lim;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, P) == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

}  // namespace bqe
