// bqe_cache.cu — the expert cache: least-recently-used replacement of expert
// slots in a pool smaller than the set of experts, with the uploads of the
// missing experts enqueued on a stream of their own.
//
// The Strata 4090 post (section 5, second paragraph) keeps the hottest
// experts in an LRU set of VRAM slots in front of pinned host memory and a
// disk tier, fetching one layer ahead; the DeepSeek-V4.1-Flash field report
// (section 3B) runs 4288 expert slots and reports per step which tier served
// each expert.  Here the pool in HBM is the cache, caller-owned pinned host
// memory holds every expert's canonical bytes, and the per-layer slot tables
// the decode kernels read are the indirection: a fetch makes a layer's
// requested experts resident and rewrites the tables on an upload stream,
// and the layer's kernels are ordered after those uploads only.
//
// Slot choice (plan c = 0, 1, ...): a requested expert already resident is a
// hit; a missing one takes, among the managed slots of its format that
// neither this plan nor the previous one uses, the one used longest ago
// (never-used first, then the lower slot), evicting its expert.  The previous
// plan's slots stay untouched because its kernels may still be running; a
// slot is overwritten only after the kernels of plan c - 2 (the last that may
// have read it) are complete, an event the caller records with
// bqe_cache_done after each layer's kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "bqe_internal.cuh"

struct bqe_cache {
  bqe_layer_desc d;
  int L = 0, E = 0, S = 0, first = 0;
  uint64_t pair_off = 0;              // staging offset of the table updates (past the largest expert)
  bqe_pool pool;
  int32_t* tables = nullptr;          // device, L x (E + 1)
  std::vector<int32_t> expert_fmt;    // L x E
  std::vector<int32_t> slot_fmt;      // S managed slots
  std::vector<uint64_t> slot_off;     // their offsets from the pool's first slot
  std::vector<int32_t> holder;        // slot -> key (layer E + expert) or -1
  std::vector<int32_t> where;         // key -> slot or -1
  std::vector<int64_t> used;          // slot -> last plan that used it, -1 never
  int64_t c = 0;                      // plans made
  // events (rings of 4, tagged with the plan): the kernels of plan p are
  // complete; the uploads of plan p are complete
  cudaEvent_t done_ev[4] = {};
  int64_t done_plan[4] = {-1, -1, -1, -1};
  cudaEvent_t up_ev[4] = {};
  int64_t up_plan[4] = {-1, -1, -1, -1};
  cudaEvent_t tail_ev = nullptr;
  bool events = false;
  bqe_cache_stats st = {};
};

namespace {

__global__ void k_table_set(int32_t* tables, const int32_t* pairs, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) tables[pairs[2 * i]] = pairs[2 * i + 1];
}

bool make_events(bqe_cache* c) {
  if (c->events) return true;
  for (int i = 0; i < 4; ++i)
    if (cudaEventCreateWithFlags(&c->done_ev[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->up_ev[i], cudaEventDisableTiming) != cudaSuccess)
      return false;
  if (cudaEventCreateWithFlags(&c->tail_ev, cudaEventDisableTiming) != cudaSuccess) return false;
  c->events = true;
  return true;
}

// The slot choice of one plan (see the file comment); false (state unchanged)
// when a miss finds no slot.
bool plan(bqe_cache* c, int layer, int n, const int32_t* experts, int32_t* slot, int32_t* miss, int32_t* evicted) {
  const std::vector<int32_t> holder0 = c->holder;
  const std::vector<int64_t> used0 = c->used;
  std::vector<int32_t> touched;
  const int64_t pc = c->c;
  for (int i = 0; i < n; ++i) {
    const int key = layer * c->E + experts[i];
    int s = c->where[key];
    if (s >= 0) {
      c->used[s] = pc;
      slot[i] = s;
      miss[i] = 0;
      evicted[i] = -1;
      continue;
    }
    const int fmt = c->expert_fmt[key];
    int best = -1;
    for (int t = 0; t < c->S; ++t) {
      if (c->slot_fmt[t] != fmt || (c->used[t] >= 0 && c->used[t] >= pc - 1)) continue;
      if (best < 0 || c->used[t] < c->used[best]) best = t;
    }
    if (best < 0) {  // restore
      for (int k : touched) c->where[k] = -1;
      for (int t = 0; t < c->S; ++t)
        if (holder0[t] >= 0) c->where[holder0[t]] = t;
      c->holder = holder0;
      c->used = used0;
      return false;
    }
    const int old = c->holder[best];
    if (old >= 0) c->where[old] = -1;
    c->holder[best] = key;
    c->where[key] = best;
    touched.push_back(key);
    c->used[best] = pc;
    slot[i] = best;
    miss[i] = 1;
    evicted[i] = old;
  }
  c->c = pc + 1;
  return true;
}

}  // namespace

extern "C" int bqe_cache_create(const bqe_layer_desc* d, int32_t n_layers, const int32_t* expert_fmt,
                                const bqe_pool* pool, const int32_t* pool_slot_fmt, int32_t first_slot,
                                int32_t n_slots, int32_t* slot_tables, bqe_cache** out) {
  if (!out) return BQE_EINVAL;
  *out = nullptr;
  if (!d || n_layers <= 0 || !expert_fmt || !pool || !pool_slot_fmt || n_slots <= 0 || first_slot < 0 ||
      (int64_t)first_slot + n_slots > pool->n_slots || !slot_tables || d->n_experts <= 0)
    return BQE_EINVAL;
  std::vector<uint64_t> off;
  if (!bqe::pool_slot_offsets(d, pool->n_slots, pool_slot_fmt, off)) return BQE_EINVAL;
  bqe_cache* c = new bqe_cache();
  c->d = *d;
  c->L = n_layers;
  c->E = d->n_experts;
  c->S = n_slots;
  c->first = first_slot;
  c->pool = *pool;
  c->tables = slot_tables;
  c->expert_fmt.assign(expert_fmt, expert_fmt + (size_t)n_layers * c->E);
  for (int32_t f : c->expert_fmt)
    if (!bqe::fmt_ok(f)) {
      delete c;
      return BQE_EINVAL;
    }
  c->slot_fmt.assign(pool_slot_fmt + first_slot, pool_slot_fmt + first_slot + n_slots);
  c->slot_off.assign(off.begin() + first_slot, off.begin() + first_slot + n_slots);
  c->holder.assign(n_slots, -1);
  c->where.assign((size_t)n_layers * c->E, -1);
  c->used.assign(n_slots, -1);
  uint64_t eb = 0;
  for (int f = BQE_FMT_TQ1; f <= BQE_FMT_MXFP4; ++f) eb = std::max<uint64_t>(eb, bqe_expert_bytes(d, f));
  c->pair_off = bqe::al256(eb);
  *out = c;
  return BQE_OK;
}

extern "C" void bqe_cache_destroy(bqe_cache* c) {
  if (!c) return;
  if (c->events) {
    for (int i = 0; i < 4; ++i) {
      cudaEventDestroy(c->done_ev[i]);
      cudaEventDestroy(c->up_ev[i]);
    }
    cudaEventDestroy(c->tail_ev);
  }
  delete c;
}

extern "C" int bqe_cache_plan(bqe_cache* c, int32_t layer, int32_t n, const int32_t* experts, int32_t* slots_out,
                              int32_t* miss_out, int32_t* evicted_out) {
  if (!c || layer < 0 || layer >= c->L || n < 0 || (n > 0 && (!experts || !slots_out || !miss_out || !evicted_out)))
    return BQE_EINVAL;
  for (int i = 0; i < n; ++i)
    if (experts[i] < 0 || experts[i] >= c->E) return BQE_EINVAL;
  if (!plan(c, layer, n, experts, slots_out, miss_out, evicted_out)) return BQE_ENOSPC;
  for (int i = 0; i < n; ++i) {
    slots_out[i] += c->first;
    ++c->st.requests;
    if (miss_out[i]) {
      ++c->st.misses;
      c->st.bytes_uploaded += bqe_expert_bytes(&c->d, c->expert_fmt[layer * c->E + experts[i]]);
      if (evicted_out[i] >= 0) ++c->st.evictions;
    } else {
      ++c->st.hits;
    }
  }
  return BQE_OK;
}

extern "C" int bqe_cache_fetch(bqe_cache* c, int32_t layer, int32_t n, const int32_t* experts,
                               const void* const* host_src, void* staging, uint64_t staging_bytes,
                               void* upload_stream, void* compute_stream, int64_t* plan_out,
                               int32_t* n_miss_out) {
  // compute_stream: only read for the fallback wait when plan c - 2 was not recorded
  if (!c || !host_src || !staging || ((uintptr_t)staging & 255) || n < 0 ||
      staging_bytes < c->pair_off + 16ull * (uint64_t)n)
    return BQE_EINVAL;
  if (!make_events(c)) return BQE_ECUDA;
  const int64_t pc = c->c;
  std::vector<int32_t> slot(n > 0 ? n : 1), miss(n > 0 ? n : 1), ev(n > 0 ? n : 1);
  int rc = bqe_cache_plan(c, layer, n, experts, slot.data(), miss.data(), ev.data());
  if (rc) return rc;
  cudaStream_t up = (cudaStream_t)upload_stream, cs = (cudaStream_t)compute_stream;
  int nm = 0;
  std::vector<int32_t> pairs;  // (table index, value)
  for (int i = 0; i < n; ++i) {
    if (!miss[i]) continue;
    const int key = layer * c->E + experts[i];
    const int fmt = c->expert_fmt[key];
    if (!host_src[key]) return BQE_EINVAL;
    if (nm == 0) {
      // a victim was last used by plan pc - 2 or earlier: wait for those kernels
      const int64_t need = pc - 2;
      if (need >= 0) {
        if (c->done_plan[need & 3] == need) {
          if (cudaStreamWaitEvent(up, c->done_ev[need & 3], 0) != cudaSuccess) return BQE_ECUDA;
        } else {  // not recorded: wait for everything enqueued on the compute stream
          if (cudaEventRecord(c->tail_ev, cs) != cudaSuccess || cudaStreamWaitEvent(up, c->tail_ev, 0) != cudaSuccess)
            return BQE_ECUDA;
        }
      }
    }
    ++nm;
    const int s = slot[i] - c->first;
    if (cudaMemcpyAsync(staging, host_src[key], bqe_expert_bytes(&c->d, fmt), cudaMemcpyHostToDevice, up) !=
        cudaSuccess)
      return BQE_ECUDA;
    rc = bqe_pool_pack_slot(&c->d, fmt, staging, (uint8_t*)c->pool.base + c->slot_off[s], up);
    if (rc) return rc;
    pairs.push_back(layer * (c->E + 1) + experts[i]);
    pairs.push_back(slot[i]);
    if (ev[i] >= 0) {
      pairs.push_back((ev[i] / c->E) * (c->E + 1) + ev[i] % c->E);
      pairs.push_back(-1);
    }
  }
  if (nm > 0) {
    // the table updates: pairs staged behind the packed slots (same stream, so
    // the last rewrite has read the staging buffer before this copy lands)
    const uint64_t pb = (uint64_t)pairs.size() * 4;
    uint8_t* pd = (uint8_t*)staging + c->pair_off;
    if (cudaMemcpyAsync(pd, pairs.data(), pb, cudaMemcpyHostToDevice, up) != cudaSuccess) return BQE_ECUDA;
    const int np = (int)(pairs.size() / 2);
    k_table_set<<<(np + 255) / 256, 256, 0, up>>>(c->tables, (const int32_t*)pd, np);
    if (cudaGetLastError() != cudaSuccess) return BQE_ECUDA;
    if (cudaEventRecord(c->up_ev[pc & 3], up) != cudaSuccess) return BQE_ECUDA;
    c->up_plan[pc & 3] = pc;
  }
  if (plan_out) *plan_out = pc;
  if (n_miss_out) *n_miss_out = nm;
  return BQE_OK;
}

extern "C" int bqe_cache_ready(bqe_cache* c, int64_t plan, void* compute_stream) {
  if (!c || plan < 0 || plan >= c->c || plan < c->c - 4) return BQE_EINVAL;
  if (c->up_plan[plan & 3] != plan) return BQE_OK;  // nothing was uploaded for it
  return cudaStreamWaitEvent((cudaStream_t)compute_stream, c->up_ev[plan & 3], 0) == cudaSuccess ? BQE_OK
                                                                                                   : BQE_ECUDA;
}

extern "C" int bqe_cache_done(bqe_cache* c, int64_t plan, void* compute_stream) {
  if (!c || plan < 0 || plan >= c->c || plan < c->c - 4) return BQE_EINVAL;
  if (!make_events(c)) return BQE_ECUDA;
  if (cudaEventRecord(c->done_ev[plan & 3], (cudaStream_t)compute_stream) != cudaSuccess) return BQE_ECUDA;
  c->done_plan[plan & 3] = plan;
  return BQE_OK;
}

extern "C" int bqe_cache_stats_get(const bqe_cache* c, bqe_cache_stats* out) {
  if (!c || !out) return BQE_EINVAL;
  *out = c->st;
  return BQE_OK;
}
