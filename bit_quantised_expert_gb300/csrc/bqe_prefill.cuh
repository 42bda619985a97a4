// bqe_prefill.cuh — geometry, workspace layout and parameters of the prefill
// path (one MoE layer over many token rows): tokens are routed, regrouped by
// expert, and every expert runs its three matrices as grouped GEMMs on the
// tensor cores after dequantising its weight tiles to a 16-bit float type
// (fp16, or bf16 for MXFP4 experts and on request) in shared memory.
#pragma once

#include "bqe_internal.cuh"

namespace bqe {

constexpr int kPfTileN = 256;       // token rows per GEMM tile (MMA N, multiple of 16)
constexpr int kPfRowAlign = 16;     // every expert's row range starts on a multiple of 16
constexpr int kPfAStages = 5;       // dequantised A ring (one 64-column K-step per stage)
constexpr int kPfBStages = 3;       // B (token rows) area: 3 stages of 256 rows, re-split per item
constexpr int kPfBMaxStages = 16;   // stages of the B area for short tiles (area / (rows * 128 bytes), at most)
constexpr int kPfRawStages = 2;     // quantised-weight ring (one 256-column group per stage)
constexpr uint32_t kPfRawPanel = 4608;                 // 32 rows x 256 columns, largest format (NVFP4)
constexpr uint32_t kPfRawStage = 4 * kPfRawPanel;      // four 32-row panels = one 128-row A tile
constexpr uint32_t kPfAStage = 128 * 128;              // 128 rows x 64 16-bit values
constexpr uint32_t kPfBStage = kPfTileN * 128;         // 256 rows x 64 16-bit values
constexpr uint32_t kPfEpiBytes = 4 * 16 * 33 * 4;      // epilogue staging (largest of the two phases)
constexpr uint32_t kPfOffA = 0;
constexpr uint32_t kPfOffB = kPfOffA + kPfAStages * kPfAStage;
constexpr uint32_t kPfOffRaw = kPfOffB + kPfBStages * kPfBStage;
constexpr uint32_t kPfOffEpi = kPfOffRaw + kPfRawStages * kPfRawStage;
constexpr uint32_t kPfOffBar = kPfOffEpi + kPfEpiBytes;
constexpr uint32_t kPfSmemBytes = kPfOffBar + 256 + 1024;  // + barriers + alignment slack
constexpr int kPfDqSets = 2;       // sets of 4 dequant warps; set j takes the K-steps n with n % sets == j
constexpr int kPfDqWarps = 4 * kPfDqSets;
constexpr int kPfThreads = 32 * (kPfDqWarps + 7);  // dequant warps, then 2 load warps, MMA, 4 epilogue warps
constexpr int kPfMaxE = 1024;

struct PfGeo {
  int H, I, E, K, T;
  int R;          // row capacity of the expert-grouped operands (all groups, each padded to 16)
  int maxTiles;   // upper bound on the GEMM tiles
  int nblkA;      // W1/W3 items per tile: 64 gate + 64 up rows each (I / 64)
  int nblkB;      // W2 items per tile: 128 output rows each (H / 128)
};

__host__ __device__ inline PfGeo make_pf_geo(int H, int I, int E, int K, int T) {
  PfGeo g;
  g.H = H; g.I = I; g.E = E; g.K = K; g.T = T;
  const int64_t pairs = (int64_t)T * (K + 1);
  g.R = (int)(((pairs + (int64_t)(kPfRowAlign - 1) * (E + 1)) + 15) / 16 * 16);
  g.maxTiles = (int)((pairs + kPfTileN - 1) / kPfTileN + (E + 1));
  g.nblkA = I / 64;
  g.nblkB = H / 128;
  return g;
}

constexpr int kPfDbgCtas = 256, kPfDbgSlots = 12;
// diagnostic counters (cycles, summed over the CTA's work): 0 load warp waiting
// for a free raw / B stage, 1 dequant waiting raw data, 2 dequant waiting a free
// A stage, 3 dequant working, 4 MMA waiting operands, 5 MMA issuing, 6 MMA
// waiting a free accumulator, 7 epilogue waiting, 8 epilogue working, 9 CTA
// total, 10 items
struct PfLayout {
  uint64_t err, ctr, z, idx, w, tok_sc, cnt, goff, gaddr, gfmt, gf16, tile, prow_tok, prow_w, prow_sc, pos, xp, hp, y,
      dbg, total;
};

__host__ __device__ inline PfLayout make_pf_ws(const PfGeo& g) {
  PfLayout L;
  uint64_t o = 0;
  L.err = o; o = al256(o + 16);
  L.ctr = o; o = al256(o + 64);                                  // [0] tiles, [1] rows, [2..3] work counters
  L.z = o; o = al256(o + 4ull * g.T * g.E);                      // router logits, fp32
  L.idx = o; o = al256(o + 4ull * g.T * g.K);
  L.w = o; o = al256(o + 4ull * g.T * g.K);
  L.tok_sc = o; o = al256(o + 4ull * g.T);                       // 2^-s_t: x_t 2^s_t has max |.| in [1, 2)
  L.cnt = o; o = al256(o + 4ull * (g.E + 1));                    // rows per group (group E: the shared expert)
  L.goff = o; o = al256(o + 4ull * (g.E + 2));                   // first row of each group
  L.gaddr = o; o = al256(o + 8ull * (g.E + 1));                  // device address of each group's slot
  L.gfmt = o; o = al256(o + 4ull * (g.E + 1));                   // its format (0: invalid, skipped)
  L.gf16 = o; o = al256(o + 4ull * (g.E + 1));                   // 1: its operands are fp16, 0: bf16
  L.tile = o; o = al256(o + 12ull * g.maxTiles);                 // (group, first row, rows) per tile
  L.prow_tok = o; o = al256(o + 4ull * g.R);                     // token of each grouped row (-1: padding)
  L.prow_w = o; o = al256(o + 4ull * g.R);                       // its mixing weight
  L.prow_sc = o; o = al256(o + 4ull * g.R);                      // its token's 2^-s
  L.pos = o; o = al256(o + 4ull * g.T * (g.K + 1));              // grouped row of (token, choice); choice K: shared
  L.xp = o; o = al256(o + 2ull * g.R * g.H);                     // grouped x 2^s, 16-bit, K-step-major swizzled tiles
  L.hp = o; o = al256(o + 2ull * g.R * g.I);                     // grouped h 2^s, same layout
  L.y = o; o = al256(o + 4ull * g.R * g.H);                      // weighted expert outputs, fp32, row-major
  L.dbg = o; o = al256(o + 8ull * 2 * kPfDbgCtas * kPfDbgSlots);  // diagnostic cycle counters [gemm][cta][slot]
  L.total = o;
  return L;
}

struct PfParams {
  PfGeo g;
  PfLayout L;
  uint8_t* ws;
  const uint16_t* x;          // T x H bf16
  const float* router_w;      // E x H
  const float* bias;          // E or null
  const int32_t* forced;      // T x K or null
  const int32_t* slot_table;  // E + 1
  bqe_pool pool;
  float* out;                 // T x H fp32
  int accumulate;
  int32_t* topk_idx;          // optional T x K
  float* topk_w;              // optional T x K
  int f16;                    // 1: fp16 tensor-core operands (MXFP4 experts stay bf16), 0: bf16 everywhere
  int diag;                   // 1: add per-role cycle counts into ws.dbg
  uint64_t limit_ns;
};

constexpr int kPfKernels = 8;
// ev: null, or kPfKernels + 1 events recorded on `st` around the kernels
int launch_prefill(const PfParams& P, cudaStream_t st, cudaEvent_t* ev);

}  // namespace bqe
