// bqe_api.cu — host entry points of the decode path: argument checks,
// workspace geometry, and the launches (stream-ordered: one persistent kernel
// per layer; the chained step launches one per layer).
#include <cuda_runtime.h>

#include <atomic>

#include "bqe_internal.cuh"
#include "bqe_prefill.cuh"

using namespace bqe;

// Process-wide settings for diagnostics and tests (not part of the operation;
// read at each launch, not synchronised with launches in other threads).
static std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};  // 2 s per wait
static std::atomic<int> g_drop_item{-1};
static std::atomic<int> g_diag{0};
static std::atomic<int> g_pf_f16{1};

extern "C" void bqe_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns; }
extern "C" void bqe_set_test_drop_item(int32_t item) { g_drop_item = item; }
extern "C" void bqe_set_diag(int32_t on) { g_diag = on ? 1 : 0; }
extern "C" void bqe_set_prefill_f16(int32_t on) { g_pf_f16 = on ? 1 : 0; }

static int device_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

static bool desc_ok(const bqe_layer_desc* d) {
  return d && d->hidden > 0 && d->inter > 0 && d->hidden % 256 == 0 && d->inter % 256 == 0 && d->n_experts > 0 &&
         d->n_experts <= 512 && d->top_k > 0 && d->top_k <= kMaxTopK && d->top_k <= d->n_experts &&
         d->n_shared == 1;
}

static Geo geo_of(const bqe_layer_desc* d, int M) { return make_geo(d->hidden, d->inter, d->n_experts, d->top_k, M); }

extern "C" uint64_t bqe_diag_offset(const bqe_layer_desc* d, int32_t M) {
  if (!desc_ok(d) || M < 1 || M > kMaxM) return 0;
  return make_ws(geo_of(d, M)).dbg;
}

extern "C" uint64_t bqe_workspace_bytes(const bqe_layer_desc* d, int32_t M) {
  if (!desc_ok(d) || M < 1 || M > kMaxM) return 0;
  return make_ws(geo_of(d, M)).total;
}

extern "C" int bqe_workspace_init(void* ws, uint64_t ws_bytes, void* stream) {
  if (!ws || ws_bytes == 0) return BQE_EINVAL;
  return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

static int check_pool(const bqe_pool* p) {
  if (!p || !p->base || !p->slot_off || !p->slot_fmt || p->n_slots <= 0 || ((uintptr_t)p->base & 15)) return BQE_EINVAL;
  return BQE_OK;
}

namespace bqe {
// Host-side checks of a decode-layer call (everything but the workspace): the
// same for the workspace and the no-allocation entry points, made before
// anything is enqueued.
int check_layer_args(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* resid, const float* router_w,
                     const bqe_pool* pool, const int32_t* slot_table, const float* out) {
  if (!desc_ok(d) || M < 1 || M > kMaxM || (!x && !resid) || !router_w || !slot_table || !out) return BQE_EINVAL;
  if (((uintptr_t)router_w & 15) || (x && ((uintptr_t)x & 15)) || d->hidden % 512) return BQE_EINVAL;
  return check_pool(pool);
}
}  // namespace bqe

static int route_common(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* router_w,
                        const float* sel_bias, const bqe_pool* pool, const int32_t* slot_table,
                        const int32_t* forced_idx, int32_t* topk_idx, float* topk_w, void* ws, uint64_t ws_bytes,
                        cudaStream_t st) {
  if (!desc_ok(d) || M < 1 || M > kMaxM || !x || !router_w || !slot_table || !ws) return BQE_EINVAL;
  if (((uintptr_t)ws & 255) || ((uintptr_t)router_w & 15)) return BQE_EINVAL;
  int rc = check_pool(pool);
  if (rc) return rc;
  Geo g = geo_of(d, M);
  WsLayout L = make_ws(g);
  if (ws_bytes < L.total) return BQE_ENOSPC;
  RouteParams P;
  P.g = g;
  P.L = L;
  P.ws = (uint8_t*)ws;
  P.x = x;
  P.resid = nullptr;
  P.t_out = nullptr;
  P.router_w = router_w;
  P.bias = sel_bias;
  P.forced = forced_idx;
  P.slot_table = slot_table;
  P.pool = *pool;
  P.topk_idx = topk_idx;
  P.topk_w = topk_w;
  P.diag = 0;
  return launch_route(P, st, false);
}

extern "C" int bqe_route(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* router_w,
                         const float* sel_bias, const bqe_pool* pool, const int32_t* slot_table,
                         const int32_t* forced_idx, int32_t* topk_idx, float* topk_w, void* ws, uint64_t ws_bytes,
                         void* stream) {
  return route_common(d, M, x, router_w, sel_bias, pool, slot_table, forced_idx, topk_idx, topk_w, ws, ws_bytes,
                      (cudaStream_t)stream);
}

// The decode layer as one persistent kernel (bqe_moe.cu).
static int moe_common(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* resid, uint16_t* t_out,
                      const float* router_w, const float* sel_bias, const bqe_pool* pool, const int32_t* slot_table,
                      const int32_t* forced_idx, float* out, int32_t accumulate, int32_t* topk_idx, float* topk_w,
                      void* ws, uint64_t ws_bytes, cudaStream_t st, bool allow_diag = true) {
  int rc = check_layer_args(d, M, x, resid, router_w, pool, slot_table, out);
  if (rc) return rc;
  if (!ws || ((uintptr_t)ws & 255)) return BQE_EINVAL;
  Geo g = geo_of(d, M);
  WsLayout L = make_ws(g);
  if (ws_bytes < L.total) return BQE_ENOSPC;
  const int sms = device_sms();
  if (sms <= 0) return BQE_ECUDA;
  MoeParams P = {};
  P.g = g;
  P.L = L;
  P.ws = (uint8_t*)ws;
  P.x = x;
  P.resid = resid;
  P.t_out = t_out;
  P.router_w = router_w;
  P.bias = sel_bias;
  P.forced = forced_idx;
  P.slot_table = slot_table;
  P.pool = *pool;
  P.out = out;
  P.accumulate = accumulate ? 1 : 0;
  P.topk_idx = topk_idx;
  P.topk_w = topk_w;
  P.drop_item = g_drop_item.load();
  P.diag = allow_diag ? g_diag.load() : 0;
  P.limit_ns = g_wait_limit_ns.load();
  return launch_moe(P, sms, st);
}

namespace bqe {
int moe_forward(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* router_w, const float* sel_bias,
                const bqe_pool* pool, const int32_t* slot_table, const int32_t* forced_idx, float* out,
                int32_t accumulate, int32_t* topk_idx, float* topk_w, void* ws, uint64_t ws_bytes, cudaStream_t st,
                bool allow_diag) {
  if (!x) return BQE_EINVAL;
  return moe_common(d, M, x, nullptr, nullptr, router_w, sel_bias, pool, slot_table, forced_idx, out, accumulate,
                    topk_idx, topk_w, ws, ws_bytes, st, allow_diag);
}
}  // namespace bqe

extern "C" int bqe_moe_layer_forward(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* router_w,
                                     const float* sel_bias, const bqe_pool* pool, const int32_t* slot_table,
                                     const int32_t* forced_idx, float* out, int32_t accumulate, int32_t* topk_idx,
                                     float* topk_w, void* ws, uint64_t ws_bytes, void* stream) {
  if (!x) return BQE_EINVAL;
  return moe_common(d, M, x, nullptr, nullptr, router_w, sel_bias, pool, slot_table, forced_idx, out, accumulate,
                    topk_idx, topk_w, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int bqe_layer_stats(const bqe_layer_desc* d, int32_t M, const void* ws, void* stream, bqe_stats* out) {
  if (!desc_ok(d) || M < 1 || M > kMaxM || !ws || !out) return BQE_EINVAL;
  const Geo g = geo_of(d, M);
  const WsLayout L = make_ws(g);
  cudaStream_t st = (cudaStream_t)stream;
  int32_t nu = 0;
  const uint8_t* w = (const uint8_t*)ws;
  if (cudaStreamSynchronize(st) != cudaSuccess || cudaMemcpy(&nu, w + L.nu, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return BQE_ECUDA;
  if (nu < 0 || nu > g.U) return BQE_EDEVICE;
  int32_t fmt[kMaxM * kMaxTopK + 1] = {}, rows[kMaxM * kMaxTopK + 1] = {};
  if (nu > 0 && (cudaMemcpy(fmt, w + L.u_fmt, 4ull * nu, cudaMemcpyDeviceToHost) != cudaSuccess ||
                 cudaMemcpy(rows, w + L.u_nrows, 4ull * nu, cudaMemcpyDeviceToHost) != cudaSuccess))
    return BQE_ECUDA;
  bqe_stats s = {};
  s.rows = M;
  s.experts_streamed = nu;
  for (int u = 0; u < nu; ++u) {
    if (!fmt_ok(fmt[u])) return BQE_EDEVICE;
    s.per_format[fmt[u]] += 1;
    s.expert_bytes += 2 * matrix_bytes(fmt[u], d->inter, d->hidden) + matrix_bytes(fmt[u], d->hidden, d->inter);
    s.row_uses += rows[u];
  }
  s.router_bytes = 4ull * d->n_experts * d->hidden;
  *out = s;
  return BQE_OK;
}

extern "C" int bqe_moe_step(const bqe_layer_desc* d, int32_t n_layers, int32_t M, float* resid,
                            const float* router_w, const float* sel_bias, const bqe_pool* pool,
                            const int32_t* slot_tables, const int32_t* forced_idx, uint16_t* t_out, void* ws,
                            uint64_t ws_bytes, void* stream) {
  if (!desc_ok(d) || n_layers < 1 || M < 1 || M > kMaxM || !resid || !router_w || !slot_tables) return BQE_EINVAL;
  const int64_t E = d->n_experts, H = d->hidden, K = d->top_k;
  cudaStream_t st = (cudaStream_t)stream;
  for (int l = 0; l < n_layers; ++l) {
    uint16_t* tl = t_out ? t_out + (int64_t)l * M * H : nullptr;
    const float* bl = sel_bias ? sel_bias + l * E : nullptr;
    const int32_t* fl = forced_idx ? forced_idx + (int64_t)l * M * K : nullptr;
    const int rc = moe_common(d, M, nullptr, resid, tl, router_w + l * E * H, bl, pool, slot_tables + l * (E + 1), fl,
                              resid, 1, nullptr, nullptr, ws, ws_bytes, st);
    if (rc) return rc;
  }
  return BQE_OK;
}

// ---------------------------------------------------------------------------
// Prefill
// ---------------------------------------------------------------------------
static constexpr int32_t kPfMaxT = 1 << 20;

// Events of the diagnostic mode, one set per device, created on first use.
static cudaEvent_t* pf_events() {
  static cudaEvent_t ev[64][kPfKernels + 1];
  static bool made[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!made[dev]) {
    for (int i = 0; i <= kPfKernels; ++i)
      if (cudaEventCreate(&ev[dev][i]) != cudaSuccess) return nullptr;
    made[dev] = true;
  }
  return ev[dev];
}

extern "C" uint64_t bqe_prefill_workspace_bytes(const bqe_layer_desc* d, int32_t T) {
  if (!desc_ok(d) || T < 1 || T > kPfMaxT) return 0;
  return make_pf_ws(make_pf_geo(d->hidden, d->inter, d->n_experts, d->top_k, T)).total;
}

extern "C" int bqe_moe_prefill(const bqe_layer_desc* d, int32_t T, const uint16_t* x, const float* router_w,
                               const float* sel_bias, const bqe_pool* pool, const int32_t* slot_table,
                               const int32_t* forced_idx, float* out, int32_t accumulate, int32_t* topk_idx,
                               float* topk_w, void* ws, uint64_t ws_bytes, void* stream) {
  if (!desc_ok(d) || T < 1 || T > kPfMaxT || !x || !router_w || !slot_table || !out || !ws) return BQE_EINVAL;
  if (((uintptr_t)ws & 255) || ((uintptr_t)router_w & 15) || ((uintptr_t)x & 15) || ((uintptr_t)out & 15))
    return BQE_EINVAL;
  int rc = check_pool(pool);
  if (rc) return rc;
  PfParams P;
  P.g = make_pf_geo(d->hidden, d->inter, d->n_experts, d->top_k, T);
  P.L = make_pf_ws(P.g);
  if (ws_bytes < P.L.total) return BQE_ENOSPC;
  P.ws = (uint8_t*)ws;
  P.x = x;
  P.router_w = router_w;
  P.bias = sel_bias;
  P.forced = forced_idx;
  P.slot_table = slot_table;
  P.pool = *pool;
  P.out = out;
  P.accumulate = accumulate ? 1 : 0;
  P.topk_idx = topk_idx;
  P.topk_w = topk_w;
  P.f16 = g_pf_f16.load();
  P.diag = g_diag.load();
  P.limit_ns = g_wait_limit_ns.load();
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(P.ws + P.L.err, 0, 16, st) != cudaSuccess) return BQE_ECUDA;
  if (cudaMemsetAsync(P.ws + P.L.cnt, 0, 4ull * (P.g.E + 1), st) != cudaSuccess) return BQE_ECUDA;
  if (P.diag && cudaMemsetAsync(P.ws + P.L.dbg, 0, P.L.total - P.L.dbg, st) != cudaSuccess) return BQE_ECUDA;
  return launch_prefill(P, st, g_diag.load() ? pf_events() : nullptr);
}

extern "C" uint64_t bqe_prefill_diag_offset(const bqe_layer_desc* d, int32_t T) {
  if (!desc_ok(d) || T < 1 || T > kPfMaxT) return 0;
  return make_pf_ws(make_pf_geo(d->hidden, d->inter, d->n_experts, d->top_k, T)).dbg;
}

extern "C" int bqe_prefill_kernel_ms(float* ms) {
  if (!ms) return BQE_EINVAL;
  cudaEvent_t* ev = pf_events();
  if (!ev) return BQE_ECUDA;
  if (cudaEventSynchronize(ev[kPfKernels]) != cudaSuccess) return BQE_ECUDA;
  for (int i = 0; i < kPfKernels; ++i)
    if (cudaEventElapsedTime(&ms[i], ev[i], ev[i + 1]) != cudaSuccess) return BQE_ECUDA;
  return BQE_OK;
}

extern "C" int bqe_check(void* ws, void* stream, int32_t* detail) {
  if (!ws) return BQE_EINVAL;
  int32_t h[2] = {0, 0};
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return BQE_ECUDA;
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return BQE_ECUDA;
  if (detail) *detail = h[1];
  if (h[0] == 0) return BQE_OK;
  const int32_t z[2] = {0, 0};
  if (cudaMemcpy(ws, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return BQE_ECUDA;
  return h[0];
}
