// bqe_noalloc.cu — a decode-layer entry point that allocates nothing.
//
// bqe_moe_layer_forward needs a workspace that the caller allocates.  Some
// callers cannot allocate device memory at the point where they run a layer:
// a plugin living inside a host framework that owns every byte of device
// memory through its own allocator and exposes none of it, or a service that
// forbids device allocation after start-up so that its memory footprint stays
// fixed.  For them this file keeps the workspace in a file-scope device array
// of a fixed size, and bqe_moe_layer_forward_noalloc runs the same layer with
// it.  The array exists once per device that loads the library and lives
// until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "bqe_internal.cuh"

static constexpr uint64_t kNoAllocBytes = 8ull << 20;  // 8 MiB: every layer whose workspace fits

// The scratch array (device code could name it directly; host code must use
// the address cudaGetSymbolAddress returns, never the symbol itself).
static __device__ __align__(256) uint8_t g_noalloc_ws[kNoAllocBytes];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};  // device address of g_noalloc_ws, per device

// Device address of the array on the current device, found once per device.
// The first call on a device also zeroes the array (cudaMemsetAsync on `st`).
int noalloc_scratch(cudaStream_t st, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BQE_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || !p) return BQE_ECUDA;
    if (cudaMemsetAsync(p, 0, kNoAllocBytes, st) != cudaSuccess) return BQE_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return BQE_OK;
}

}  // namespace

extern "C" int bqe_moe_layer_forward_noalloc(const bqe_layer_desc* d, int32_t M, const uint16_t* x,
                                             const float* router_w, const float* sel_bias, const bqe_pool* pool,
                                             const int32_t* slot_table, const int32_t* forced_idx, float* out,
                                             int32_t accumulate, int32_t* topk_idx, float* topk_w,
                                             int32_t* status_out, void* stream) {
  // every argument check comes before the shared array is touched, so a
  // rejected call leaves a call in flight on another stream undisturbed
  if (!x) return BQE_EINVAL;
  int rc = bqe::check_layer_args(d, M, x, nullptr, router_w, pool, slot_table, out);
  if (rc) return rc;
  const uint64_t need = bqe_workspace_bytes(d, M);
  if (need == 0) return BQE_EINVAL;
  if (need > kNoAllocBytes) return BQE_ENOSPC;  // this layer's workspace is larger than the fixed array
  cudaStream_t st = (cudaStream_t)stream;
  void* ws = nullptr;
  rc = noalloc_scratch(st, &ws);
  if (rc) return rc;
  // the array keeps the previous call's contents: clear the error word and
  // the work list (all in front of the logits), and the epoch-tagged keys
  // with the call epoch and the counters, so a call that failed leaves no
  // trace in the next
  const bqe::WsLayout L = bqe::make_ws(bqe::make_geo(d->hidden, d->inter, d->n_experts, d->top_k, M));
  if (cudaMemsetAsync(ws, 0, L.z, st) != cudaSuccess) return BQE_ECUDA;
  if (cudaMemsetAsync((uint8_t*)ws + L.zk, 0, L.m_pa - L.zk, st) != cudaSuccess) return BQE_ECUDA;
  // diagnostic counters stay off: they would accumulate in the array, where
  // no caller can read them
  rc = bqe::moe_forward(d, M, x, router_w, sel_bias, pool, slot_table, forced_idx, out, accumulate, topk_idx, topk_w,
                        ws, need, st, false);
  if (rc) return rc;
  if (status_out &&
      cudaMemcpyAsync(status_out, (uint8_t*)ws + L.err, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
    return BQE_ECUDA;
  return BQE_OK;
}

extern "C" int bqe_check_noalloc(void* stream, int32_t* detail) {
  void* ws = nullptr;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BQE_ECUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    ws = g_noalloc_ptr[dev];
  }
  if (!ws) {  // no call on this device yet: nothing to report
    if (detail) *detail = 0;
    return BQE_OK;
  }
  return bqe_check(ws, stream, detail);
}
