// bqe_format.cu — block formats: sizes, host packing into canonical blocks,
// the canonical -> device slot layout rewrite, and an exact dequantiser.
//
// Formats (Strata 4090 post, sections 1 and 5.1: PTQ1_0 ternary at 1.75 bpw
// with 5 trits per byte, Q2_0 at 2.25, Q3_K at 3.44; field report header and
// section 2: FP4 experts in per-32 blocks).  The pages give bits per weight
// only; the block layouts are this library's:
//   TQ1   56 B / 256: bytes 0..50 = sum_r (t_{5i+r}+1) 3^r, byte 51 = t_255+1,
//         52..53 fp16 d, 54..55 zero.  w = d t
//   Q2_0  18 B / 64: weight j's code at bits 2(j%4) of byte j/4, 16..17 fp16 d.
//         w = d (2q - 3)
//   Q3_K  110 B / 256: 0..63 low 2 bits (as Q2_0), 64..95 high bit (weight j:
//         byte 64 + j/8, bit j%8), 96..107 sixteen 6-bit sub-scales packed
//         little-endian, 108..109 fp16 d.  w = d s_{j/16} (q - 4)
//   MXFP4 17 B / 32: byte i = code_{2i} | code_{2i+1} << 4 (E2M1), byte 16 =
//         UE8M0 exponent E.  w = e2m1(code) 2^(E-127)
//   NVFP4 9 B / 16: bytes 0..7 as MXFP4's, byte 8 = FP8 E4M3 scale S (OCP:
//         sign, 4-bit exponent with bias 7, 3-bit mantissa, subnormal at
//         exponent 0, NaN at S = 0x7F / 0xFF).  w = e2m1(code) e4m3(S)
#include <cuda_fp16.h>

#include <cstring>
#include <vector>

#include "bqe_internal.cuh"

using namespace bqe;

extern "C" int32_t bqe_block_weights(int32_t fmt) { return fmt_ok(fmt) ? fmt_bw(fmt) : 0; }
extern "C" int32_t bqe_block_bytes(int32_t fmt) { return fmt_ok(fmt) ? fmt_bb(fmt) : 0; }

extern "C" uint64_t bqe_packed_bytes(int32_t fmt, int32_t rows, int32_t cols) {
  if (!fmt_ok(fmt) || rows < 0 || cols < 0 || cols % fmt_bw(fmt) != 0) return 0;
  return matrix_bytes(fmt, rows, cols);
}

static bool shape_ok(const bqe_layer_desc* d) {
  return d && d->hidden > 0 && d->inter > 0 && d->hidden % 256 == 0 && d->inter % 256 == 0 &&
         d->n_experts > 0 && d->top_k > 0 && d->top_k <= kMaxTopK && d->top_k <= d->n_experts &&
         d->n_shared == 1;
}

extern "C" uint64_t bqe_expert_bytes(const bqe_layer_desc* d, int32_t fmt) {
  if (!shape_ok(d) || !fmt_ok(fmt)) return 0;
  return 2 * matrix_bytes(fmt, d->inter, d->hidden) + matrix_bytes(fmt, d->hidden, d->inter);
}

extern "C" int32_t bqe_scale_bytes(int32_t fmt) {
  switch (fmt) {
    case BQE_FMT_TQ1: return 2;
    case BQE_FMT_Q2_0: return 2;
    case BQE_FMT_Q3_K: return 18;
    case BQE_FMT_MXFP4: return 1;
    case BQE_FMT_NVFP4: return 1;
  }
  return 0;
}

extern "C" int bqe_pack(int32_t fmt, int32_t rows, int32_t cols, const uint8_t* codes, const uint8_t* scales,
                        uint8_t* out) {
  if (!fmt_ok(fmt) || rows <= 0 || cols <= 0 || cols % fmt_bw(fmt) != 0 || !codes || !scales || !out)
    return BQE_EINVAL;
  const int bw = fmt_bw(fmt), bb = fmt_bb(fmt), sb = bqe_scale_bytes(fmt);
  const int64_t nblocks = (int64_t)rows * (cols / bw);
  for (int64_t blk = 0; blk < nblocks; ++blk) {
    const uint8_t* c = codes + blk * bw;
    const uint8_t* s = scales + blk * sb;
    uint8_t* o = out + blk * bb;
    memset(o, 0, bb);
    switch (fmt) {
      case BQE_FMT_MXFP4:
        for (int j = 0; j < 32; ++j) {
          if (c[j] > 15) return BQE_EINVAL;
          o[j >> 1] |= (uint8_t)(c[j] << ((j & 1) * 4));
        }
        if (s[0] == 0xFF) return BQE_EINVAL;  // NaN scale is not a weight
        o[16] = s[0];
        break;
      case BQE_FMT_NVFP4:
        for (int j = 0; j < 16; ++j) {
          if (c[j] > 15) return BQE_EINVAL;
          o[j >> 1] |= (uint8_t)(c[j] << ((j & 1) * 4));
        }
        if ((s[0] & 0x7F) == 0x7F) return BQE_EINVAL;  // NaN scale is not a weight
        o[8] = s[0];
        break;
      case BQE_FMT_Q2_0:
        for (int j = 0; j < 64; ++j) {
          if (c[j] > 3) return BQE_EINVAL;
          o[j >> 2] |= (uint8_t)(c[j] << (2 * (j & 3)));
        }
        o[16] = s[0];
        o[17] = s[1];
        break;
      case BQE_FMT_TQ1:
        for (int i = 0; i < 51; ++i) {
          int v = 0, p = 1;
          for (int r = 0; r < 5; ++r) {
            if (c[5 * i + r] > 2) return BQE_EINVAL;
            v += c[5 * i + r] * p;
            p *= 3;
          }
          o[i] = (uint8_t)v;
        }
        if (c[255] > 2) return BQE_EINVAL;
        o[51] = c[255];
        o[52] = s[0];
        o[53] = s[1];
        break;
      case BQE_FMT_Q3_K: {
        for (int j = 0; j < 256; ++j) {
          if (c[j] > 7) return BQE_EINVAL;
          o[j >> 2] |= (uint8_t)((c[j] & 3) << (2 * (j & 3)));
          o[64 + (j >> 3)] |= (uint8_t)(((c[j] >> 2) & 1) << (j & 7));
        }
        for (int j = 0; j < 16; ++j) {
          if (s[j] > 63) return BQE_EINVAL;
          for (int bit = 0; bit < 6; ++bit) {
            int pos = 6 * j + bit;
            o[96 + (pos >> 3)] |= (uint8_t)(((s[j] >> bit) & 1) << (pos & 7));
          }
        }
        o[108] = s[16];
        o[109] = s[17];
        break;
      }
    }
  }
  return BQE_OK;
}

// ----------------------------------------------------------------------------
// canonical -> device layout (one thread per (row, block) of one matrix)
// ----------------------------------------------------------------------------
__global__ void k_pack_matrix(int fmt, int rows, int K, const uint8_t* __restrict__ src, uint8_t* __restrict__ dst) {
  const int bw = fmt_bw(fmt), bb = fmt_bb(fmt);
  const int nbrow = K / bw;
  const int64_t nblk = (int64_t)rows * nbrow;
  const int kc = chunk_cols(K), nch = K / kc, nb = kc / bw;
  const uint32_t tb = tile_bytes(fmt, kc);
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < nblk; t += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(t / nbrow), blk = (int)(t % nbrow);
    const int p = row >> 5, r = row & 31, c = blk / nb, b = blk % nb;
    const uint8_t* s = src + t * bb;
    uint8_t* tile = dst + (uint64_t)(p * nch + c) * tb;
    for (int i = 0; i < bb; ++i) tile[tile_byte_offset(fmt, nb, b, r, i)] = s[i];
  }
}

static int launch_pack(int fmt, int rows, int K, const uint8_t* src, uint8_t* dst, cudaStream_t st) {
  int64_t nblk = (int64_t)rows * (K / fmt_bw(fmt));
  int grid = (int)((nblk + 255) / 256);
  if (grid > 4096) grid = 4096;
  k_pack_matrix<<<grid, 256, 0, st>>>(fmt, rows, K, src, dst);
  return cudaGetLastError() == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

extern "C" int bqe_pool_pack_slot(const bqe_layer_desc* d, int32_t fmt, const void* canon_src, void* slot_dst,
                                  void* stream) {
  if (!shape_ok(d) || !fmt_ok(fmt) || !canon_src || !slot_dst || ((uintptr_t)slot_dst & 15)) return BQE_EINVAL;
  if (d->hidden % 32 || d->inter % 32) return BQE_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  const uint64_t m13 = matrix_bytes(fmt, d->inter, d->hidden);
  const uint8_t* s = (const uint8_t*)canon_src;
  uint8_t* o = (uint8_t*)slot_dst;
  int rc;
  if ((rc = launch_pack(fmt, d->inter, d->hidden, s, o, st))) return rc;
  if ((rc = launch_pack(fmt, d->inter, d->hidden, s + m13, o + m13, st))) return rc;
  return launch_pack(fmt, d->hidden, d->inter, s + 2 * m13, o + 2 * m13, st);
}

// ----------------------------------------------------------------------------
// slot pool: [slot offsets (uint64) | slot formats (int32) | slots], every
// part 256-byte aligned, in one caller-owned device buffer
// ----------------------------------------------------------------------------
static uint64_t pool_tables_bytes(int32_t n) {
  return al256(8ull * (uint64_t)n) + al256(4ull * (uint64_t)n);
}

// Slot offsets (relative to the first slot) for the formats; false on a bad format.
static bool pool_offsets(const bqe_layer_desc* d, int32_t n, const int32_t* fmt, std::vector<uint64_t>& off,
                         uint64_t& slots_bytes) {
  off.resize(n);
  uint64_t o = 0;
  for (int32_t s = 0; s < n; ++s) {
    if (!fmt_ok(fmt[s])) return false;
    off[s] = o;
    o = al256(o + 2 * matrix_bytes(fmt[s], d->inter, d->hidden) + matrix_bytes(fmt[s], d->hidden, d->inter));
  }
  slots_bytes = o;
  return true;
}

namespace bqe {
bool pool_slot_offsets(const bqe_layer_desc* d, int32_t n, const int32_t* fmt, std::vector<uint64_t>& off) {
  uint64_t sb = 0;
  return pool_offsets(d, n, fmt, off, sb);
}
}  // namespace bqe

extern "C" uint64_t bqe_pool_bytes(const bqe_layer_desc* d, int32_t n_slots, const int32_t* slot_fmt) {
  if (!shape_ok(d) || n_slots <= 0 || !slot_fmt) return 0;
  std::vector<uint64_t> off;
  uint64_t sb = 0;
  if (!pool_offsets(d, n_slots, slot_fmt, off, sb)) return 0;
  return pool_tables_bytes(n_slots) + sb;
}

extern "C" int bqe_pool_init(bqe_pool* p, const bqe_layer_desc* d, int32_t n_slots, const int32_t* slot_fmt,
                             void* dev_mem, uint64_t dev_bytes, void* stream) {
  if (!p || !shape_ok(d) || n_slots <= 0 || !slot_fmt || !dev_mem || ((uintptr_t)dev_mem & 255)) return BQE_EINVAL;
  std::vector<uint64_t> off;
  uint64_t sb = 0;
  if (!pool_offsets(d, n_slots, slot_fmt, off, sb)) return BQE_EINVAL;
  const uint64_t tb = pool_tables_bytes(n_slots);
  if (dev_bytes < tb + sb) return BQE_ENOSPC;
  uint8_t* mem = (uint8_t*)dev_mem;
  cudaStream_t st = (cudaStream_t)stream;
  // from pageable host memory: the call returns once the host arrays are staged
  if (cudaMemcpyAsync(mem, off.data(), 8ull * n_slots, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(mem + al256(8ull * n_slots), slot_fmt, 4ull * n_slots, cudaMemcpyHostToDevice, st) !=
          cudaSuccess)
    return BQE_ECUDA;
  p->base = mem + tb;
  p->base_bytes = sb;
  p->slot_off = (const uint64_t*)mem;
  p->slot_fmt = (const int32_t*)(mem + al256(8ull * n_slots));
  p->n_slots = n_slots;
  int32_t mask = 0;
  for (int32_t s = 0; s < n_slots; ++s) mask |= 1 << slot_fmt[s];
  p->fmt_mask = mask;
  return BQE_OK;
}

extern "C" int bqe_pool_upload(const bqe_pool* p, const bqe_layer_desc* d, int32_t slot, const void* canon_dev,
                               void* stream) {
  if (!p || !p->base || !p->slot_off || !p->slot_fmt || !shape_ok(d) || slot < 0 || slot >= p->n_slots ||
      !canon_dev)
    return BQE_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  uint64_t off = 0;
  int32_t fmt = 0;
  // the slot's place and format, from the pool's own tables (ordered after bqe_pool_init on the stream)
  if (cudaMemcpyAsync(&off, p->slot_off + slot, 8, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(&fmt, p->slot_fmt + slot, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return BQE_ECUDA;
  if (!fmt_ok(fmt) || (off & 15) ||
      off + 2 * matrix_bytes(fmt, d->inter, d->hidden) + matrix_bytes(fmt, d->hidden, d->inter) > p->base_bytes)
    return BQE_EINVAL;
  return bqe_pool_pack_slot(d, fmt, canon_dev, (uint8_t*)p->base + off, stream);
}

extern "C" int bqe_unpack_host(int32_t fmt, int32_t rows, int32_t cols, const uint8_t* packed, uint8_t* codes,
                               uint8_t* scales) {
  if (!fmt_ok(fmt) || rows <= 0 || cols <= 0 || cols % fmt_bw(fmt) != 0 || !packed || !codes || !scales)
    return BQE_EINVAL;
  const int bw = fmt_bw(fmt), bb = fmt_bb(fmt), sb = bqe_scale_bytes(fmt);
  const int64_t nblocks = (int64_t)rows * (cols / bw);
  for (int64_t blk = 0; blk < nblocks; ++blk) {
    const uint8_t* b = packed + blk * bb;
    uint8_t* c = codes + blk * bw;
    uint8_t* s = scales + blk * sb;
    switch (fmt) {
      case BQE_FMT_MXFP4:
        for (int j = 0; j < 32; ++j) c[j] = (uint8_t)((b[j >> 1] >> ((j & 1) * 4)) & 15);
        s[0] = b[16];
        break;
      case BQE_FMT_NVFP4:
        for (int j = 0; j < 16; ++j) c[j] = (uint8_t)((b[j >> 1] >> ((j & 1) * 4)) & 15);
        s[0] = b[8];
        break;
      case BQE_FMT_Q2_0:
        for (int j = 0; j < 64; ++j) c[j] = (uint8_t)((b[j >> 2] >> (2 * (j & 3))) & 3);
        s[0] = b[16];
        s[1] = b[17];
        break;
      case BQE_FMT_TQ1:
        for (int i = 0; i < 51; ++i) {
          if (b[i] > 242) return BQE_EINVAL;
          int v = b[i];
          for (int r = 0; r < 5; ++r) {
            c[5 * i + r] = (uint8_t)(v % 3);
            v /= 3;
          }
        }
        if (b[51] > 2) return BQE_EINVAL;
        c[255] = b[51];
        s[0] = b[52];
        s[1] = b[53];
        break;
      case BQE_FMT_Q3_K:
        for (int j = 0; j < 256; ++j)
          c[j] = (uint8_t)(((b[j >> 2] >> (2 * (j & 3))) & 3) | (((b[64 + (j >> 3)] >> (j & 7)) & 1) << 2));
        for (int j = 0; j < 16; ++j) {
          int v = 0;
          for (int bit = 0; bit < 6; ++bit) {
            const int pos = 6 * j + bit;
            v |= ((b[96 + (pos >> 3)] >> (pos & 7)) & 1) << bit;
          }
          s[j] = (uint8_t)v;
        }
        s[16] = b[108];
        s[17] = b[109];
        break;
    }
  }
  return BQE_OK;
}

// ----------------------------------------------------------------------------
// exact dequantiser (device layout -> fp32 row-major); one thread per block
// ----------------------------------------------------------------------------
__device__ __forceinline__ float fp16_bits_to_f32(uint32_t lo, uint32_t hi) {
  return __half2float(__ushort_as_half((unsigned short)(lo | (hi << 8))));
}

__device__ __forceinline__ float e2m1_value(uint32_t c) {
  // magnitudes of codes 0..7 in OCP E2M1
  const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
  float m = mag[c & 7];
  return (c & 8) ? -m : m;
}

// OCP FP8 E4M3 (sign, exponent bias 7, 3 mantissa bits; exponent 0 subnormal),
// written out from the format's definition: exact in fp32.  NaN is refused
// when packing and never decoded here.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  const float mag = e == 0 ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return (b & 0x80) ? -mag : mag;
}

__device__ __forceinline__ float ue8m0_value(uint32_t e) {
  return e == 0 ? __int_as_float(0x00400000) : __int_as_float((int)(e << 23));  // 2^(E-127)
}

__global__ void k_dequant(int fmt, int rows, int K, const uint8_t* __restrict__ src, float* __restrict__ out) {
  const int bw = fmt_bw(fmt), bb = fmt_bb(fmt);
  const int nbrow = K / bw;
  const int64_t nblk = (int64_t)rows * nbrow;
  const int kc = chunk_cols(K), nch = K / kc, nb = kc / bw;
  const uint32_t tb = tile_bytes(fmt, kc);
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < nblk; t += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(t / nbrow), blk = (int)(t % nbrow);
    const int p = row >> 5, r = row & 31, c = blk / nb, b = blk % nb;
    const uint8_t* tile = src + (uint64_t)(p * nch + c) * tb;
    uint8_t by[112];
    for (int i = 0; i < bb; ++i) by[i] = tile[tile_byte_offset(fmt, nb, b, r, i)];
    float* o = out + (int64_t)row * K + (int64_t)blk * bw;
    if (fmt == BQE_FMT_MXFP4) {
      const float sc = ue8m0_value(by[16]);
      for (int j = 0; j < 32; ++j) o[j] = e2m1_value((by[j >> 1] >> ((j & 1) * 4)) & 15) * sc;
    } else if (fmt == BQE_FMT_NVFP4) {
      const float sc = e4m3_value(by[8]);
      for (int j = 0; j < 16; ++j) o[j] = e2m1_value((by[j >> 1] >> ((j & 1) * 4)) & 15) * sc;
    } else if (fmt == BQE_FMT_Q2_0) {
      const float dd = fp16_bits_to_f32(by[16], by[17]);
      for (int j = 0; j < 64; ++j) o[j] = dd * (float)(2 * ((by[j >> 2] >> (2 * (j & 3))) & 3) - 3);
    } else if (fmt == BQE_FMT_TQ1) {
      const float dd = fp16_bits_to_f32(by[52], by[53]);
      for (int i = 0; i < 51; ++i) {
        int v = by[i];
        for (int r5 = 0; r5 < 5; ++r5) {
          o[5 * i + r5] = dd * (float)(v % 3 - 1);
          v /= 3;
        }
      }
      o[255] = dd * (float)(by[51] % 3 - 1);
    } else {
      const float dd = fp16_bits_to_f32(by[108], by[109]);
      for (int j = 0; j < 256; ++j) {
        const int lo = (by[j >> 2] >> (2 * (j & 3))) & 3;
        const int hi = (by[64 + (j >> 3)] >> (j & 7)) & 1;
        const int sj = j >> 4, bit = 6 * sj;
        const int s = ((by[96 + (bit >> 3)] | ((bit >> 3) + 1 < 12 ? by[97 + (bit >> 3)] << 8 : 0)) >> (bit & 7)) & 63;
        o[j] = (dd * (float)s) * (float)(lo + 4 * hi - 4);
      }
    }
  }
}

extern "C" int bqe_dequant(int32_t fmt, int32_t rows, int32_t cols, const void* src, float* out, void* stream) {
  if (!fmt_ok(fmt) || rows <= 0 || rows % 32 || cols <= 0 || cols % 256 || !src || !out) return BQE_EINVAL;
  int64_t nblk = (int64_t)rows * (cols / fmt_bw(fmt));
  int grid = (int)((nblk + 127) / 128);
  if (grid > 8192) grid = 8192;
  k_dequant<<<grid, 128, 0, (cudaStream_t)stream>>>(fmt, rows, cols, (const uint8_t*)src, out);
  return cudaGetLastError() == cudaSuccess ? BQE_OK : BQE_ECUDA;
}

extern "C" const char* bqe_status_str(int s) {
  switch (s) {
    case BQE_OK: return "ok";
    case BQE_EINVAL: return "invalid argument";
    case BQE_ENOSPC: return "buffer too small";
    case BQE_ECUDA: return "CUDA runtime error";
    case BQE_EDEVICE: return "device-detected error (slot table / pool)";
    case BQE_ETIMEOUT: return "device wait timed out";
    case BQE_EUNSUPPORTED: return "unsupported";
  }
  return "unknown status";
}
