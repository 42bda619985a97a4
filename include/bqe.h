/*
 * bqe.h — block-quantised MoE expert layer for GB300 (sm_103a): C ABI.
 *
 * The operation (DeepSeek-V4.1-Flash on 4xL20 field report, sections 1-2;
 * Strata 4090 post, sections 1, 5.1 and 5.3): one MoE layer of a
 * DeepSeek-V4.1-Flash-shaped model — hidden 5120, expert intermediate 2304,
 * 384 routed experts + 1 shared, 6 experts per token:
 *
 *   z = x Wr^T (fp32 router), s = sigmoid(z), key = s + b (b steers the
 *   choice only), idx = top-k(key) with ties to the lower expert id,
 *   w = s[idx] / sum s[idx],
 *   out = sum_j w_j W2_j (silu(W1_j x) * (W3_j x)) + (same for the shared expert).
 *
 * Expert weights are block-quantised (the pages give bits per weight; the
 * block layouts are this library's specification):
 *   BQE_FMT_TQ1   ternary PTQ1_0, 256 weights / 56 B (1.75 bpw)
 *   BQE_FMT_Q2_0  64 weights / 18 B (2.25 bpw), w = d (2q - 3)
 *   BQE_FMT_Q3_K  256 weights / 110 B (3.4375 bpw), w = d s_j (q - 4)
 *   BQE_FMT_MXFP4 32 weights / 17 B (4.25 bpw), w = e2m1(c) 2^(E-127)
 *   BQE_FMT_NVFP4 16 weights / 9 B (4.5 bpw), w = e2m1(c) e4m3(S): an NVFP4
 *                 checkpoint (news digest) read as NVIDIA's published NVFP4,
 *                 blocks of 16 with an FP8 E4M3 scale, no per-tensor scale
 *
 * Conventions for every entry point:
 *   - Return value: BQE_OK or an error code; nothing throws across the ABI.
 *     Argument errors are detected on the host before anything is enqueued.
 *   - Pointers documented "device" are CUDA device addresses owned by the
 *     caller; the library never allocates, frees or retains them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).  All
 *     GPU work is asynchronous on it.  Errors found by the kernels themselves
 *     (a slot id out of range, a wait that timed out) are recorded in the
 *     workspace's error word and reported by bqe_check().
 *   - Row-major, contiguous layouts throughout.
 */
#ifndef BQE_H
#define BQE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  BQE_OK = 0,
  BQE_EINVAL = 1,       /* bad argument (null pointer, size, alignment, format) */
  BQE_ENOSPC = 2,       /* a caller buffer is too small */
  BQE_ECUDA = 3,        /* a CUDA runtime call failed */
  BQE_EDEVICE = 4,      /* a kernel detected an invalid slot / table entry */
  BQE_ETIMEOUT = 5,     /* a kernel wait exceeded its limit and gave up */
  BQE_EUNSUPPORTED = 6  /* shape or device not supported */
};

enum { BQE_FMT_TQ1 = 1, BQE_FMT_Q2_0 = 2, BQE_FMT_Q3_K = 3, BQE_FMT_MXFP4 = 4, BQE_FMT_NVFP4 = 5 };

/* Shape of one MoE layer.  hidden and inter must be multiples of 256 (every
 * format's block divides 256) and of 32 rows; n_shared must be 1; at most
 * 512 routed experts and top_k <= 16.  The decode router (bqe_route and the
 * layer entry points) also needs hidden a multiple of 512, at most 8192, and
 * n_experts <= hidden / 2 (BQE_EUNSUPPORTED otherwise).
 * DeepSeek-V4.1-Flash: {5120, 2304, 384, 6, 1}. */
typedef struct {
  int32_t hidden;
  int32_t inter;
  int32_t n_experts;
  int32_t top_k;
  int32_t n_shared;
} bqe_layer_desc;

/* A slot pool: one caller-owned device buffer holding expert slots in the
 * device layout (bqe_pool_pack_slot), plus two caller-owned device tables:
 * slot_off[s] = byte offset of slot s in base (multiple of 16), slot_fmt[s]
 * = its format.  The kernels check every slot id they use against n_slots
 * and every slot's extent against base_bytes.  fmt_mask (host value): bit f
 * set when slots of format f may be in the pool, 0 when unknown; the decode
 * call runs a kernel carrying only the inner loops of those formats (MXFP4
 * alone, or TQ1 / Q2_0 / Q3_K alone; any other mask: all formats), and a slot
 * of a format outside them is reported like an invalid slot (BQE_EDEVICE).
 * bqe_pool_init fills it from the slot formats. */
typedef struct {
  const void* base;          /* device */
  uint64_t base_bytes;
  const uint64_t* slot_off;  /* device, n_slots entries */
  const int32_t* slot_fmt;   /* device, n_slots entries */
  int32_t n_slots;
  int32_t fmt_mask;
} bqe_pool;

/* Accounting of one decode call (bqe_layer_stats): what it streamed.  The
 * pages report the same kind of per-step account of where each token's
 * experts came from (field report, section 3B: "experts: N hit, ..."). */
typedef struct {
  int32_t rows;              /* token rows of the call (M) */
  int32_t experts_streamed;  /* distinct experts read, the shared one included */
  int32_t per_format[6];     /* of those, how many in each format (index = BQE_FMT_*) */
  int32_t row_uses;          /* (expert, row) pairs computed: sum over experts of the rows that chose it */
  uint64_t expert_bytes;     /* packed bytes of those experts, each read once */
  uint64_t router_bytes;     /* fp32 router weights read (n_experts x hidden x 4) */
} bqe_stats;

/* ---- formats (host only) ------------------------------------------------ */

/* Weights and bytes of one block of `fmt`; 0 for an unknown format. */
int32_t bqe_block_weights(int32_t fmt);
int32_t bqe_block_bytes(int32_t fmt);

/* Bytes of a rows x cols matrix in `fmt` (canonical and device layouts have
 * the same size); 0 if cols is not a multiple of the block. */
uint64_t bqe_packed_bytes(int32_t fmt, int32_t rows, int32_t cols);

/* Bytes of one expert slot: W1 (inter x hidden) | W3 (inter x hidden) |
 * W2 (hidden x inter). 0 on a bad shape or format. */
uint64_t bqe_expert_bytes(const bqe_layer_desc* d, int32_t fmt);

/* Bytes of the scale field per block that bqe_pack() reads:
 * TQ1 2 (fp16 d), Q2_0 2 (fp16 d), Q3_K 18 (16 six-bit sub-scales as bytes
 * 0..63, then fp16 d), MXFP4 1 (the UE8M0 exponent byte), NVFP4 1 (the E4M3
 * scale byte). */
int32_t bqe_scale_bytes(int32_t fmt);

/* Host: pack a rows x cols matrix into canonical blocks (row-major; each row
 * is cols/block consecutive blocks).  codes: one byte per weight, row-major,
 * in the format's code domain (TQ1: t+1 in 0..2; Q2_0: q in 0..3; Q3_K: q in
 * 0..7; MXFP4, NVFP4: 4-bit code 0..15).  scales: bqe_scale_bytes(fmt) bytes per
 * block, blocks in row-major order.  out: bqe_packed_bytes() bytes.
 * BQE_EINVAL on a code or scale out of its domain (a NaN scale: MXFP4 0xFF,
 * NVFP4 0x7F / 0xFF) (nothing is written then
 * for that block onward). */
int bqe_pack(int32_t fmt, int32_t rows, int32_t cols, const uint8_t* codes,
             const uint8_t* scales, uint8_t* out);

/* Host: the inverse of bqe_pack (a self-check of the format module, not a
 * compute path): canonical blocks back to one code byte per weight and
 * bqe_scale_bytes(fmt) scale bytes per block, in bqe_pack's conventions.
 * BQE_EINVAL on a ternary byte above 242 (never written by bqe_pack). */
int bqe_unpack_host(int32_t fmt, int32_t rows, int32_t cols, const uint8_t* packed, uint8_t* codes,
                    uint8_t* scales);

/* ---- pool --------------------------------------------------------------- */

/* Device: rewrite one expert from canonical bytes (device, bqe_expert_bytes
 * bytes: W1 | W3 | W2 in canonical blocks) into the device layout at
 * slot_dst (device, same size, 16-byte aligned).  The device layout groups
 * 32 rows into a panel and 256..1024 columns into a chunk; each (panel,
 * chunk) tile is contiguous so one bulk copy moves it.  The bytes are the
 * canonical bytes, rearranged. */
int bqe_pool_pack_slot(const bqe_layer_desc* d, int32_t fmt, const void* canon_src,
                       void* slot_dst, void* stream);

/* Bytes of device memory for a slot pool of n_slots experts with formats
 * slot_fmt (host, n_slots entries): the slot-offset table (uint64), the
 * slot-format table (int32), then every slot at a 256-byte-aligned offset,
 * each part 256-byte aligned.  0 on a bad shape, count or format. */
uint64_t bqe_pool_bytes(const bqe_layer_desc* d, int32_t n_slots, const int32_t* slot_fmt);

/* Lay out a slot pool in caller-owned device memory dev_mem (256-byte
 * aligned, dev_bytes >= bqe_pool_bytes): writes the two tables at its front
 * (copies enqueued on `stream`; slot_fmt is host memory and may be released
 * when the call returns) and fills *p (host struct) so that it describes the
 * pool: base = the first slot, slot_off / slot_fmt = the device tables,
 * fmt_mask = the formats of the slots.  The library keeps no reference to
 * dev_mem.  BQE_ENOSPC if dev_bytes is short,
 * BQE_EINVAL on a bad argument. */
int bqe_pool_init(bqe_pool* p, const bqe_layer_desc* d, int32_t n_slots, const int32_t* slot_fmt,
                  void* dev_mem, uint64_t dev_bytes, void* stream);

/* Write one expert into slot `slot` of a pool made by bqe_pool_init: its
 * canonical bytes (device, bqe_expert_bytes(d, fmt of the slot): W1 | W3 |
 * W2) are rewritten into the device layout (as bqe_pool_pack_slot).  The
 * slot's offset and format are read back from the pool's tables, so the call
 * synchronises `stream` once before enqueueing the rewrite.  BQE_EINVAL on a
 * slot out of range or a table entry that does not fit the pool. */
int bqe_pool_upload(const bqe_pool* p, const bqe_layer_desc* d, int32_t slot, const void* canon_dev,
                    void* stream);

/* Device: dequantise one rows x cols matrix stored in the device layout
 * (e.g. W1 of a slot: slot base; W3: + bqe_packed_bytes(fmt, inter, hidden);
 * W2: + 2x that) into fp32 row-major `out` (device, rows*cols floats).
 * Exact: every block value is representable in fp32. */
int bqe_dequant(int32_t fmt, int32_t rows, int32_t cols, const void* src, float* out,
                void* stream);

/* ---- decode layer (M <= 8 token rows) ----------------------------------- */

/* Workspace bytes one decode call with up to M rows needs. */
uint64_t bqe_workspace_bytes(const bqe_layer_desc* d, int32_t M);

/* Zero a workspace before its first use and after any call that reported an
 * error (its counters must start at 0; the kernels leave them at 0 after
 * every successful call). */
int bqe_workspace_init(void* ws, uint64_t ws_bytes, void* stream);

/* One MoE layer for M in 1..8 token rows (the token plus speculative draft
 * rows verified together; each row routes independently).
 *   x          device, M x hidden bf16 (uint16 bit patterns)
 *   router_w   device, n_experts x hidden fp32
 *   sel_bias   device, n_experts fp32, or NULL for no bias
 *   pool       host struct describing the device slot pool
 *   slot_table device, n_experts + 1 int32: slot of each routed expert, then
 *              of the shared expert
 *   forced_idx device, M x top_k int32 or NULL: if given, the selection is
 *              taken from it (the router still computes the scores, and the
 *              mixing weights are the scores of the given experts)
 *   out        device, M x hidden fp32; out = layer(x), or out += layer(x)
 *              when accumulate != 0
 *   topk_idx   device, M x top_k int32 or NULL: selected experts (key order)
 *   topk_w     device, M x top_k fp32 or NULL: their mixing weights
 *   ws         device workspace of ws_bytes >= bqe_workspace_bytes(d, M)
 * Experts chosen by several rows are streamed once and applied to every row
 * that chose them.  Each output element is the sum of the experts' K-chunk
 * contributions added with fp32 atomics: the order of those additions, and so
 * the last bits of out, may differ from call to call (the selection and the
 * mixing weights do not). */
int bqe_moe_layer_forward(const bqe_layer_desc* d, int32_t M, const uint16_t* x,
                          const float* router_w, const float* sel_bias, const bqe_pool* pool,
                          const int32_t* slot_table, const int32_t* forced_idx, float* out,
                          int32_t accumulate, int32_t* topk_idx, float* topk_w, void* ws,
                          uint64_t ws_bytes, void* stream);

/* The routing alone: the router GEMV, the scores, the biased top-k and the
 * mixing weights of M rows (the first stage of bqe_moe_layer_forward, as its
 * own kernel), with the per-call work list left in ws.  topk_idx / topk_w:
 * device, M x top_k, or NULL.  Same argument rules as bqe_moe_layer_forward. */
int bqe_route(const bqe_layer_desc* d, int32_t M, const uint16_t* x, const float* router_w,
              const float* sel_bias, const bqe_pool* pool, const int32_t* slot_table,
              const int32_t* forced_idx, int32_t* topk_idx, float* topk_w, void* ws,
              uint64_t ws_bytes, void* stream);

/* Chained decode step over n_layers layers: r_0 = resid (in place),
 * t_l = bf16(r_l / sqrt(mean(r_l^2) + 1e-6)), r_{l+1} = r_l + MoE_l(t_l).
 *   resid       device, M x hidden fp32, updated in place
 *   router_w    device, n_layers x n_experts x hidden fp32
 *   sel_bias    device, n_layers x n_experts fp32, or NULL
 *   slot_tables device, n_layers x (n_experts + 1) int32
 *   forced_idx  device, n_layers x M x top_k int32, or NULL
 *   t_out       device, n_layers x M x hidden bf16, or NULL: each layer's
 *               normalised input (for per-layer checks)
 * Enqueues one kernel per layer; capture it in a CUDA graph to replay. */
int bqe_moe_step(const bqe_layer_desc* d, int32_t n_layers, int32_t M, float* resid,
                 const float* router_w, const float* sel_bias, const bqe_pool* pool,
                 const int32_t* slot_tables, const int32_t* forced_idx, uint16_t* t_out,
                 void* ws, uint64_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Prefill: one MoE layer over T token rows at once (large T; Strata 4090
 * post, section 4: tensor-core experts for prefill; section 5.3: prefill
 * accelerations must leave the per-token result unchanged).  The result per
 * token is that of bqe_moe_layer_forward: router logits in fp32, the same
 * selection rule and mixing weights, the shared expert on every row.  The
 * tokens are regrouped by expert and each expert's W1/W3 and W2 run as grouped
 * GEMMs on the tensor cores, with the weights dequantised in shared memory to
 * a 16-bit float type and h = silu(W1 x) * (W3 x) rounded to it before W2;
 * products are accumulated in fp32.  The type is fp16 by default (see
 * bqe_set_prefill_f16): x scaled per token by a power of two is exact in it,
 * TQ1 weights are exact, Q2_0 / Q3_K weights keep 11 significant bits, h keeps
 * the token's scale; MXFP4 experts use bf16 (exact for every scale).  A call
 * whose fp16 weights or h would leave the fp16 range reports BQE_EUNSUPPORTED
 * through bqe_check (detail 11).
 *
 * bqe_prefill_workspace_bytes(d, T): bytes of device workspace for T rows
 * (about 4 (K + 1) T hidden x 1.6 bytes: the expert-grouped copies of x, h and
 * the per-expert outputs), 0 if the shape is unsupported (same layer rules as
 * decode; 1 <= T <= 1048576).
 *
 * bqe_moe_prefill: same arguments as bqe_moe_layer_forward with M = T.
 *   x           device, T x hidden bf16 (16-byte aligned)
 *   router_w    device, n_experts x hidden fp32 (16-byte aligned)
 *   sel_bias    device, n_experts fp32 or NULL (selection only)
 *   pool        slot pool; slot_table device, n_experts + 1 int32 (last: shared)
 *   forced_idx  device, T x top_k int32 or NULL (selection given; weights still
 *               from the scores)
 *   out         device, T x hidden fp32 (16-byte aligned); accumulate = 1 adds
 *   topk_idx / topk_w  device, T x top_k, or NULL
 *   ws          device, 256-byte aligned, >= bqe_prefill_workspace_bytes; its
 *               contents need no initialisation (the call clears what it needs)
 * Enqueues 8 kernels on `stream` and returns without waiting.  Device-side
 * problems (bad slot, forced index out of range, a wait past its limit) are
 * reported through bqe_check(ws, ...) like the decode calls; the output of
 * such a call is undefined. */
uint64_t bqe_prefill_workspace_bytes(const bqe_layer_desc* d, int32_t T);
int bqe_moe_prefill(const bqe_layer_desc* d, int32_t T, const uint16_t* x, const float* router_w,
                    const float* sel_bias, const bqe_pool* pool, const int32_t* slot_table,
                    const int32_t* forced_idx, float* out, int32_t accumulate, int32_t* topk_idx,
                    float* topk_w, void* ws, uint64_t ws_bytes, void* stream);

/* The decode layer without a caller-provided workspace.  The pages describe
 * no such call (there is no counterpart in them): it exists for callers that
 * cannot allocate device memory where they run a layer — for instance a
 * plugin inside a host framework whose allocator owns all device memory, or
 * a service that allows no device allocation after start-up.
 * Same arguments and results as bqe_moe_layer_forward, without ws/ws_bytes.
 * The workspace is a fixed 8 MiB array in the library (one per device that
 * loads it, kept until the process exits); a layer whose
 * bqe_workspace_bytes(d, M) exceeds 8 MiB is rejected with BQE_ENOSPC (for
 * the DeepSeek-V4.1-Flash shape that allows M <= 2).  Nothing is allocated:
 * no cudaMalloc, no cudaFree.
 *   - The first call on a device finds the array's address and zeroes it
 *     (enqueued on `stream`); make that first call before any stream capture.
 *   - Every call reuses the same array and clears its counters and error
 *     word first, so calls whose GPU work overlaps (other streams, other
 *     threads) race on it: order them.
 *   - Arguments are checked before the array is touched; a rejected call
 *     enqueues nothing.
 *   - status_out: device, 2 int32 or NULL; receives the call's device error
 *     word and detail (0 = ok, else a BQE_* code as bqe_check reports).  With
 *     NULL, bqe_check_noalloc reads the same word (until the next call).
 *   - The diagnostic counters (bqe_set_diag) stay off for this call. */
int bqe_moe_layer_forward_noalloc(const bqe_layer_desc* d, int32_t M, const uint16_t* x,
                                  const float* router_w, const float* sel_bias,
                                  const bqe_pool* pool, const int32_t* slot_table,
                                  const int32_t* forced_idx, float* out, int32_t accumulate,
                                  int32_t* topk_idx, float* topk_w, int32_t* status_out,
                                  void* stream);

/* Byte-budgeted choice of each routed expert's format (host only; no GPU
 * work).  Strata 4090 post, section 5, first paragraph: ternary (TQ1),
 * Q2_0 or Q3_K per expert under a byte budget (all-Q2_0 bytes makes the
 * mix budget-neutral), by a Lagrangian relaxation with a bisection on the
 * multiplier and a greedy pass over the bytes left; an expert's cost for a
 * format is layer_weight[l] * err / energy[l] (the post counts the first
 * two and last three layers twice); at most floor(tq1_cap_frac * n_experts)
 * ternary experts per layer (the post: half); an expert with fewer than
 * min_tokens held-out tokens stays Q2_0 (the post: 8).
 *   - err: host, n_layers x n_experts x 3 doubles (errors of TQ1, Q2_0,
 *     Q3_K), >= 0; energy: host, n_layers doubles > 0; layer_weight: host,
 *     n_layers doubles >= 0; heldout_tokens: host, n_layers x n_experts or
 *     NULL (nothing locked); fmt_bytes: host, the bytes of one expert in
 *     TQ1, Q2_0, Q3_K (bqe_expert_bytes), strictly increasing.
 *   - fmt_out: host, n_layers x n_experts BQE_FMT_* codes; lambda_out,
 *     bytes_out, cost_out (host, each may be NULL): the multiplier, the
 *     bytes and the summed cost of the result.
 *   - Ties: fewer bytes first; the layer's ternary experts beyond the cap
 *     are those losing least by giving it up (then higher expert index);
 *     100 halvings of the multiplier's range; greedy upgrades by largest
 *     cost decrease per byte (then lower layer, expert, format).
 *   - BQE_EINVAL on a bad argument or a budget below what the guard rails
 *     allow (fmt_out untouched then).  Deterministic: IEEE double in a fixed
 *     order, the same result on every host. */
int bqe_assign_formats(int32_t n_layers, int32_t n_experts, const double* err, const double* energy,
                       const double* layer_weight, const int32_t* heldout_tokens, int32_t min_tokens,
                       double tq1_cap_frac, const uint64_t* fmt_bytes, uint64_t budget, int32_t* fmt_out,
                       double* lambda_out, uint64_t* bytes_out, double* cost_out);

/* ---- expert cache ----------------------------------------------------------
 * Least-recently-used replacement of expert slots when the pool holds fewer
 * slots than there are experts (Strata 4090 post, section 5, second
 * paragraph: an LRU set of VRAM expert slots in front of pinned host memory,
 * fetched one layer ahead; field report, section 3B: 4288 expert slots and a
 * per-step account of where each expert came from).  The cache manages pool
 * slots first_slot .. first_slot + n_slots - 1 (the shared experts and any
 * pinned ones live outside that range) and rewrites the routed entries of
 * the per-layer slot tables (device, n_layers x (n_experts + 1), the layout
 * bqe_moe_step reads; entry -1 = not resident; the caller fills the tables'
 * initial contents and the shared-expert entries).
 *   Plan c (c = 0, 1, ...): a requested expert already resident is a hit; a
 * missing one takes, among the managed slots of its format that neither this
 * plan nor the previous one uses, the one used longest ago (never-used
 * first, then the lower slot), evicting what it held.  No such slot:
 * BQE_ENOSPC and nothing changes. */
typedef struct bqe_cache bqe_cache;  /* opaque, host */

typedef struct {
  uint64_t requests, hits, misses, evictions, bytes_uploaded;
} bqe_cache_stats;

/* Create a cache (host object; no GPU work).  expert_fmt: host, n_layers x
 * d->n_experts formats; pool_slot_fmt: host, pool->n_slots formats (as given
 * to bqe_pool_init); slot_tables: device (not read here).  The caller keeps
 * the pool and the tables alive while the cache is used. */
int bqe_cache_create(const bqe_layer_desc* d, int32_t n_layers, const int32_t* expert_fmt,
                     const bqe_pool* pool, const int32_t* pool_slot_fmt, int32_t first_slot,
                     int32_t n_slots, int32_t* slot_tables, bqe_cache** out);
void bqe_cache_destroy(bqe_cache* c);

/* Host only: the slot choice for `n` requested experts of `layer` (host ids;
 * duplicates allowed).  slots_out: pool slot ids; miss_out: 1 for an expert
 * that was not resident; evicted_out: the key layer * n_experts + expert it
 * displaced, or -1.  Counts the request in the statistics. */
int bqe_cache_plan(bqe_cache* c, int32_t layer, int32_t n, const int32_t* experts, int32_t* slots_out,
                   int32_t* miss_out, int32_t* evicted_out);

/* Plan as above, then make the experts resident: for each miss, copy its
 * canonical bytes (host_src[layer * n_experts + expert], pinned host memory,
 * bqe_expert_bytes of its format) to `staging` and rewrite them into the
 * slot (bqe_pool_pack_slot), then update the tables (the new entries and -1
 * for the evicted experts), all on upload_stream.  Before the first
 * overwrite, upload_stream waits for the kernels of plan c - 2 (recorded by
 * bqe_cache_done; if that was not recorded, for everything enqueued on
 * compute_stream), the last that may have read a victim slot, so the uploads
 * of one layer may run while the previous layer computes.  The layer's own
 * kernels must be ordered after them with bqe_cache_ready.  staging: device, 256-byte aligned, at least
 * (the largest expert of any format, rounded up to 256) + 16 n bytes.
 * plan_out, n_miss_out (host, may be NULL): the plan's number c, the misses. */
int bqe_cache_fetch(bqe_cache* c, int32_t layer, int32_t n, const int32_t* experts,
                    const void* const* host_src, void* staging, uint64_t staging_bytes,
                    void* upload_stream, void* compute_stream, int64_t* plan_out, int32_t* n_miss_out);

/* Make compute_stream wait for the uploads of plan `plan` (fetch's
 * plan_out; one of the last four plans), before the kernels that use its
 * experts; nothing to wait for if the plan had no miss. */
int bqe_cache_ready(bqe_cache* c, int64_t plan, void* compute_stream);

/* After the kernels that use the experts of plan `plan` (fetch's plan_out)
 * are enqueued on compute_stream: record their completion, the point later
 * fetches wait for before overwriting those slots.  One of the last four
 * plans (BQE_EINVAL otherwise).  A plan left unrecorded makes a later fetch
 * wait for everything enqueued on its compute stream instead. */
int bqe_cache_done(bqe_cache* c, int64_t plan, void* compute_stream);

/* The counts since the cache was created (host). */
int bqe_cache_stats_get(const bqe_cache* c, bqe_cache_stats* out);

/* ---- speculative verify pass ---------------------------------------------
 * Bookkeeping around a decode call whose M rows are the last accepted token
 * and M - 1 drafts (the DeepSeek-V4.1-Flash field report, section 3B:
 * draft-and-verify passes, tokens per pass; the 2 x RTX PRO 6000 post:
 * batched verification, the accepted prefix committed, the rejected tail
 * rolled back).  Greedy acceptance: draft i is kept while every draft before
 * it was and it equals target[i], the target's prediction after row i. */
#define BQE_VERIFY_MAX_DRAFT 15

typedef struct {
  uint64_t passes, tokens;                 /* tokens emitted over all passes */
  uint64_t hist[BQE_VERIFY_MAX_DRAFT + 1]; /* passes by accepted draft count */
} bqe_verify_stats;

/* Host.  draft: n_draft tokens (n_draft <= BQE_VERIFY_MAX_DRAFT); target:
 * n_draft + 1 predictions (after rows 0..n_draft).  With a drafts accepted:
 * emitted[0..a] = the a drafts then target[a] (*n_emitted = a + 1), and
 * commit_mask[r] = 1 for the rows r <= a to keep, 0 for those to roll back
 * (n_draft + 1 entries).  stats (host, may be NULL) accumulates the pass.
 * BQE_EINVAL on a bad argument. */
int bqe_verify_pass(int32_t n_draft, const int32_t* draft, const int32_t* target, int32_t* emitted,
                    int32_t* n_emitted, int32_t* commit_mask, bqe_verify_stats* stats);

/* Synchronise `stream` and report the device error word of the last
 * bqe_moe_layer_forward_noalloc call on the current device, then clear it
 * (as bqe_check does for a caller's workspace).  BQE_OK if no call ran. */
int bqe_check_noalloc(void* stream, int32_t* detail);

/* After a decode call (bqe_moe_layer_forward, or the last layer of
 * bqe_moe_step) on `ws`: synchronise `stream` and describe what the call
 * streamed (bqe_stats, host).  BQE_EDEVICE if the workspace holds no valid
 * work list (e.g. the call failed). */
int bqe_layer_stats(const bqe_layer_desc* d, int32_t M, const void* ws, void* stream, bqe_stats* out);

/* Synchronise `stream`, read the workspace error word and clear it.
 * Returns BQE_OK, BQE_EDEVICE or BQE_ETIMEOUT (detail: optional host int,
 * receives the kernel's detail code), or BQE_ECUDA. */
int bqe_check(void* ws, void* stream, int32_t* detail);

/* Human-readable name of a status code. */
const char* bqe_status_str(int status);

/* ---- diagnostics and test hooks ------------------------------------------
 * Process-wide settings, read by each call when it is enqueued; they are not
 * part of the operation and not meant to be changed while other threads
 * enqueue calls (no call reads them twice). */

/* Bound on every in-kernel wait (default 2 s).  A wait that runs out records
 * BQE_ETIMEOUT in the workspace and the kernel returns; the workspace must be
 * re-initialised (bqe_workspace_init) after such an error. */
void bqe_set_wait_limit_ns(uint64_t ns);

/* Test hook for the timeout path, injected from the host: while item >= 0,
 * the first CTA of the decode kernel never issues the copies of its work
 * item number `item`, so the waits for that item run out of their limit and
 * the call reports BQE_ETIMEOUT.  -1 (default) turns it off. */
void bqe_set_test_drop_item(int32_t item);

/* Diagnostic mode (default off): the decode kernel adds per-CTA timings into
 * the workspace at byte offset bqe_diag_offset(d, M): uint64 [3][1024][8],
 * zeroed by bqe_workspace_init.  Row 1023 of blocks 0 and 1 holds globaltimer
 * stamps kept as minima or maxima over CTAs (the caller presets minima to a
 * large value): block 0 [0] first CTA start, [1] last logits published,
 * [2] first selection done, [3] first work item landed, [6] last CTA end,
 * [7] last producer done; block 1 [1] last compute warp done, [2] last
 * routing known, [3] longest producer wait for h (ns).  Rows 0..CTAs-1 (ns
 * unless noted): block 0 [0] input staged, [1] selection inputs stored,
 * [2] all logits seen; block 1 [0] producer loop (cycles), [1] items issued,
 * [2] logits published, [3] routing known, [4] router rows landed, [5] / [6] /
 * [7] producer cycles issuing bulk copies / waiting for ring space / waiting
 * for h; block 2 [1] producer wait for h, [2] / [3] compute warp 0 waiting /
 * computing, [4] reducer waiting, [7] CTA start to end.  Block 0 rows
 * 300 + CTA, ns from the CTA's start: [0] logits seen, [1] keys loaded,
 * [2] top-k, [3] mixing weights, [4] work list, [5] row slots, [6] item
 * templates, [7] first item landed. */
void bqe_set_diag(int32_t on);

/* Operand type of the prefill tensor-core GEMMs: 1 (default) fp16 with the
 * per-token power-of-two scaling described at bqe_moe_prefill, MXFP4 experts
 * in bf16; 0: bf16 for every expert (weights and h rounded to 8 significant
 * bits: relative L2 error about 3e-3 against exact arithmetic, against about
 * 4e-4 for fp16).  Both run at the same tensor-core rate. */
void bqe_set_prefill_f16(int32_t on);

/* Diagnostic (with bqe_set_diag(1)): bqe_moe_prefill records CUDA events on
 * its stream around each of its 8 kernels (router logits, selection, plan,
 * fill, gather, W1/W3 GEMM, W2 GEMM, combine); this waits for the last call's
 * events and writes the 8 durations in milliseconds to ms (host, 8 floats). */
int bqe_prefill_kernel_ms(float* ms);

/* Diagnostic (with bqe_set_diag(1)): byte offset in the prefill workspace of
 * uint64 [2 GEMMs][256 CTAs][12] cycle counters of the last call (load warp
 * waiting; dequant waiting raw data / a free stage / working; MMA waiting
 * operands / issuing / waiting an accumulator; epilogue waiting / working;
 * CTA total; items).  0 for an unsupported shape. */
uint64_t bqe_prefill_diag_offset(const bqe_layer_desc* d, int32_t T);
uint64_t bqe_diag_offset(const bqe_layer_desc* d, int32_t M);

#ifdef __cplusplus
}
#endif

#endif /* BQE_H */
