// quantize.cu -- 128x128 block quantization of an FP32 matrix to E4M3 codes and
// one FP32 (or power-of-two) scale per block, after the lpnh.cn DeepGEMM
// walkthrough §4.2 (cut into 128x128 blocks, take max|x|, scale = max_abs/448,
// divide, round to the nearest E4M3 value with ties to even, keep the scales
// in their own array), §3.1 (FP32 scales computed ahead of the GEMM) and §5.4
// (all-zero blocks). The power-of-two variant follows the packed UE8M0 scales of
// pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1.
//
// One CTA of 512 threads owns one 128x128 block: warp w holds rows
// [8w, 8w+8), lane l holds columns [4l, 4l+4), i.e. 8 float4 per thread kept in
// registers between the two passes, so the input is read from HBM once.
// quantize_kernel (below) runs one such CTA per block; at 64-87 registers a
// thread one or two of them are resident per SM.
// Loads are 128-bit and streaming; each warp-wide load covers one 512-byte row
// segment. The block max is a warp-shuffle reduction followed by a 16-entry
// shared-memory reduction (warp-shuffle reduction as in the hotelren.com GEMM
// tuning essay §4.2).
//
// Division: the codes are those of fl32(x / s) (IEEE division) rounded to E4M3.
// With FP32 scales the kernel first multiplies by r = fl32(1/s): q = fl32(x r)
// lies within 1.5 * 2^-23 relative of fl32(x / s), so if the two points
// q (1 - 2^-20) and q (1 + 2^-20) round to the same E4M3 code, every value
// between them -- fl32(x / s) included -- does too (rounding to E4M3 is
// monotone) and that code is exact. Otherwise (an E4M3 rounding boundary within
// 2^-20 of q, about one element in 2^15) the element is divided exactly.
// Power-of-two scales make x * (1/s) itself exact.
//
// Two kernels share that arithmetic:
//  * quantize_stream_kernel (16-byte-aligned input, row stride a multiple of 4
//    floats): one persistent CTA per SM streams 128x128 FP32 blocks (64 KB)
//    through a 3-stage TMA ring in shared memory guarded by mbarriers, two
//    blocks ahead of the one being reduced and encoded (inputs of at most four
//    or three blocks per SM: two or three single-stage CTAs per SM instead).
//    Each block is copied from shared memory to registers once (three CTAs
//    per SM: twice, for the block max and for the encode). Out-of-range rows and columns of
//    edge blocks arrive as zeros (TMA fill), which leaves the block max
//    unchanged.
//  * quantize_kernel (any alignment): one CTA per block, the block held in
//    registers between the two passes.
//
// The row-wise variant (blocks of 1 x 128, per-token activation scales, pzsr.cn
// page §3.1; FP32 or bfloat16 input) runs on quantize_stream_kernel too when
// the input is 16-byte aligned: each warp's eight rows of a tile get one warp
// reduction each, and lane i forms row i's scale and reciprocal for the warp.
// Other inputs take quantize_1x128_kernel, which gives each warp a contiguous
// run of (row, 128-column segment) pairs: lane l holds columns [4l, 4l + 4) of
// a segment, four segments are loaded before any is reduced, the segment max is
// one warp reduction, and the same encode4 arithmetic produces the codes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "dg_device.cuh"
#include "dg_encode.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kBlock = 128;
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kBlock / kWarps;  // 8

template <int kMode, bool kVec>
__device__ __forceinline__ void encode_store(const float4 (&v)[kRowsPerWarp], int64_t r0, int64_t c0,
                                             int64_t rows, int64_t cols, uint8_t* __restrict__ q,
                                             int64_t ld_q, float s, float r) {
  const bool full4 = c0 + 3 < cols;
  if (kVec && full4 && r0 + kRowsPerWarp <= rows) {  // all of this thread's groups are inside
    uint32_t code[kRowsPerWarp];
    encode4_n<kMode>(v, code, s, r);
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
      __stcs(reinterpret_cast<unsigned int*>(q + (r0 + i) * ld_q + c0), code[i]);
    return;
  }
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int64_t row = r0 + i;
    if (row >= rows) continue;
    uint8_t* out = q + row * ld_q + c0;
    if (kVec && full4) {
      __stcs(reinterpret_cast<unsigned int*>(out), encode4<kMode>(v[i], s, r));
    } else {
      const float e[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (c0 + t < cols) out[t] = encode1<kMode>(e[t], s, r);
    }
  }
}

// encode_store for a tile that stays in shared memory (kThreads threads, FP32
// 128 x 128, row-major): this thread's eight rows are read again and encoded
// four at a time, which holds 16 input registers instead of 32.
template <bool kPow2>
__device__ __forceinline__ void encode_store_reread(const uint8_t* tile, int warp, int lane, int64_t r0, int64_t c0,
                                                    int64_t rows, int64_t cols, uint8_t* __restrict__ q,
                                                    int64_t ld_q, float s, float r) {
  const bool inside = r0 + kRowsPerWarp <= rows && c0 + 3 < cols;
#pragma unroll
  for (int h = 0; h < kRowsPerWarp / 4; ++h) {
    float4 w[4];
    uint32_t code[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = reinterpret_cast<const float4*>(tile + (warp * kRowsPerWarp + h * 4 + i) * kBlock * 4)[lane];
    if constexpr (kPow2)
      encode4_n<1>(w, code, s, r);
    else if (s >= 0x1p-126f)
      encode4_n<0>(w, code, s, r);
    else
      encode4_n<2>(w, code, s, r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + h * 4 + i;
      uint8_t* out = q + row * ld_q + c0;
      if (inside) {
        __stcs(reinterpret_cast<unsigned int*>(out), code[i]);
      } else if (row < rows) {
        if (c0 + 3 < cols) {
          __stcs(reinterpret_cast<unsigned int*>(out), code[i]);
        } else {
          for (int t = 0; t < 4; ++t)
            if (c0 + t < cols) out[t] = static_cast<uint8_t>((code[i] >> (8 * t)) & 0xFFu);
        }
      }
    }
  }
}

template <bool kVec, bool kPow2>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const float* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ld_x,
                                                            uint8_t* __restrict__ q, int64_t ld_q,
                                                            float* __restrict__ scales,
                                                            int64_t blocks_per_row) {
  __shared__ float warp_amax[kWarps];
  pdl_wait();
  pdl_trigger();
  const int64_t blk = blockIdx.x;
  const int64_t bi = blk / blocks_per_row;
  const int64_t bj = blk - bi * blocks_per_row;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t r0 = bi * kBlock + warp * kRowsPerWarp;
  const int64_t c0 = bj * kBlock + lane * 4;
  const bool full4 = c0 + 3 < cols;

  // Pass 1: load the block (invalid rows/columns read as 0) and take max|x|.
  float4 v[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t r = r0 + i;
    if (r < rows) {
      const float* p = x + r * ld_x + c0;
      if (kVec && full4) {
        v[i] = __ldcs(reinterpret_cast<const float4*>(p));
      } else {
        if (c0 < cols) v[i].x = p[0];
        if (c0 + 1 < cols) v[i].y = p[1];
        if (c0 + 2 < cols) v[i].z = p[2];
        if (c0 + 3 < cols) v[i].w = p[3];
      }
    }
  }
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  }
  // Non-negative floats order like their bit patterns.
  const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
  if (lane == 0) warp_amax[warp] = __uint_as_float(wmax);
  __syncthreads();
  float amax = warp_amax[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, warp_amax[w]);

  // scale = max_abs / 448 in FP32; an all-zero block (or an underflow to 0) gets 1.
  float s = amax / 448.0f;
  if (s == 0.0f) s = 1.0f;
  if constexpr (kPow2) s = pow2_round_up(s);
  if (threadIdx.x == 0) scales[blk] = s;
  const float r = 1.0f / s;

  // Pass 2: divide by the scale and round to the nearest E4M3 value (RNE, saturating).
  if constexpr (kPow2) {
    encode_store<1, kVec>(v, r0, c0, rows, cols, q, ld_q, s, r);
  } else if (s >= 0x1p-126f) {
    encode_store<0, kVec>(v, r0, c0, rows, cols, q, ld_q, s, r);
  } else {
    encode_store<2, kVec>(v, r0, c0, rows, cols, q, ld_q, s, r);
  }
}

// ------------------------------------------------------------- row-wise --
constexpr int k1xThreads = 256;
constexpr int k1xWarps = k1xThreads / 32;
constexpr int k1xSegs = 4;  // segments in flight per warp

// Four consecutive elements at column c0 of a row, widened to FP32 (exact for
// bfloat16); columns >= cols read as 0.
template <bool kBf16, bool kVec>
__device__ __forceinline__ float4 load_row4(const void* __restrict__ x, int64_t row, int64_t ld_x, int64_t c0,
                                            int64_t cols) {
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if constexpr (kBf16) {
    const uint16_t* p = static_cast<const uint16_t*>(x) + row * ld_x + c0;
    if (kVec && c0 + 3 < cols) {
      const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
      v = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                      __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    } else {
      if (c0 < cols) v.x = __uint_as_float(static_cast<uint32_t>(p[0]) << 16);
      if (c0 + 1 < cols) v.y = __uint_as_float(static_cast<uint32_t>(p[1]) << 16);
      if (c0 + 2 < cols) v.z = __uint_as_float(static_cast<uint32_t>(p[2]) << 16);
      if (c0 + 3 < cols) v.w = __uint_as_float(static_cast<uint32_t>(p[3]) << 16);
    }
  } else {
    const float* p = static_cast<const float*>(x) + row * ld_x + c0;
    if (kVec && c0 + 3 < cols) {
      v = __ldcs(reinterpret_cast<const float4*>(p));
    } else {
      if (c0 < cols) v.x = p[0];
      if (c0 + 1 < cols) v.y = p[1];
      if (c0 + 2 < cols) v.z = p[2];
      if (c0 + 3 < cols) v.w = p[3];
    }
  }
  return v;
}

template <bool kBf16, bool kVec, bool kPow2>
__global__ void __launch_bounds__(k1xThreads) quantize_1x128_kernel(
    const void* __restrict__ x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* __restrict__ q, int64_t ld_q,
    float* __restrict__ scales, int64_t nbc, int64_t per_warp) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * k1xWarps + (threadIdx.x >> 5);
  const int64_t total = rows * nbc;
  int64_t seg = w * per_warp;
  const int64_t end = min(total, seg + per_warp);
  if (seg >= end) return;
  int64_t row = seg / nbc;
  int64_t cb = seg - row * nbc;
  while (seg < end) {
    float4 v[k1xSegs];
    int64_t rr[k1xSegs], cc[k1xSegs];
#pragma unroll
    for (int i = 0; i < k1xSegs; ++i) {
      rr[i] = row;
      cc[i] = cb * kBlock + lane * 4;
      v[i] = (seg + i < end) ? load_row4<kBf16, kVec>(x, row, ld_x, cc[i], cols) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (++cb == nbc) {
        cb = 0;
        ++row;
      }
    }
#pragma unroll
    for (int i = 0; i < k1xSegs; ++i) {
      if (seg + i >= end) break;
      const float m = fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w)));
      // Non-negative floats order like their bit patterns.
      const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m)));
      float s = amax / 448.0f;
      if (s == 0.0f) s = 1.0f;
      if constexpr (kPow2) s = pow2_round_up(s);
      if (lane == 0) scales[rr[i] * nbc + (cc[i] >> 7)] = s;
      const float r = 1.0f / s;
      uint8_t* out = q + rr[i] * ld_q + cc[i];
      uint32_t code;
      if constexpr (kPow2) {
        code = encode4<1>(v[i], s, r);
      } else if (s >= 0x1p-126f) {
        code = encode4<0>(v[i], s, r);
      } else {
        code = encode4<2>(v[i], s, r);
      }
      if (kVec && cc[i] + 3 < cols) {
        __stcs(reinterpret_cast<unsigned int*>(out), code);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (cc[i] + t < cols) out[t] = static_cast<uint8_t>((code >> (8 * t)) & 0xFFu);
      }
    }
    seg += k1xSegs;
  }
}

// Stages of the streaming ring (FP32: 192 KB of shared memory, one CTA per SM).
// A stage is refilled with the block kAhead ahead once its block has been
// copied to registers; with kStages - 1 ahead the refill goes to the stage
// freed an iteration earlier, which keeps two 64 KB FP32 blocks per SM in
// flight (measured on GB300: 16384x7168 FP32 quantized at 6.9 TB/s against
// 6.45 TB/s with three in flight).
// kShort = 2: one stage and two CTAs per SM (64 registers per thread), for
// inputs of at most four blocks per SM. Each SM then encodes two blocks at
// once instead of one after the other once the last loads land (measured:
// 4096x2048 FP32 in 8.2 us against 8.6 us).
// kShort = 3: one stage and three CTAs per SM, for inputs of at most three
// blocks per SM, so that every block is resident from the start and no SM
// takes a second round. Three 64 KB tiles leave 42 registers per thread, too
// few to hold a tile between the block max and the encode, so the encode
// reads the tile from shared memory a second time, four rows at a time
// (measured: 4096x1536 FP32 in 6.68 us against 6.99 us; at 512 blocks the
// two-CTA form stays 1-2 % faster).
// bfloat16 tiles (32 KB) carry half the bytes of FP32 ones for the same
// arithmetic, so that kernel is bound by instruction latency with one CTA's
// 16 warps per SM: it runs two CTAs of three stages per SM (measured:
// 16384x7168 row-wise in 73.5 us against 92.5 us with one CTA of six stages).
template <bool kBf16, int kShort = 0>
struct StreamCfg {
  static_assert(kShort == 0 || ((kShort == 2 || kShort == 3) && !kBf16), "short-input forms: FP32 tiles");
  static constexpr int kElemBytes = kBf16 ? 2 : 4;
  static constexpr uint32_t kTileBytes = kBlock * kBlock * kElemBytes;
  static constexpr int kStages = kShort ? 1 : 3;
  static constexpr int kAhead = kStages > 1 ? kStages - 1 : 1;
  static constexpr int kCtasPerSm = kShort ? kShort : (kBf16 ? 2 : 1);
  static constexpr bool kReread = kShort == 3;  // encode from shared memory, not registers
};

// kRowwise: one scale per row of the tile (1 x 128 blocks) instead of one per
// tile; kBf16: bfloat16 input tiles, widened to FP32 exactly.
template <bool kPow2, bool kRowwise, bool kBf16, int kShort>
__global__ void __launch_bounds__(kThreads, StreamCfg<kBf16, kShort>::kCtasPerSm)
    quantize_stream_kernel(const __grid_constant__ CUtensorMap tmap_x, int64_t rows, int64_t cols,
                           uint8_t* __restrict__ q, int64_t ld_q, float* __restrict__ scales,
                           int64_t blocks_per_row, int64_t nblocks, unsigned int* status,
                           uint64_t limit_ns) {
  using SC = StreamCfg<kBf16, kShort>;
  constexpr int kStages = SC::kStages;
  constexpr int kAhead = SC::kAhead;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stage_data = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * SC::kTileBytes);
  float* warp_amax = reinterpret_cast<float*>(full + kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(warp_amax + kWarps);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    *abort_flag = 0;
    fence_barrier_init();
    // The first stages' blocks start streaming into L2 while the preceding grid finishes.
    for (int j = 0; j < kStages; ++j) {
      const int64_t blk = blockIdx.x + static_cast<int64_t>(j) * gridDim.x;
      if (blk >= nblocks) break;
      const int64_t bi = blk / blocks_per_row, bj = blk - bi * blocks_per_row;
      tma_prefetch_2d(&tmap_x, static_cast<int32_t>(bj * kBlock), static_cast<int32_t>(bi * kBlock));
    }
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  // Block indices fit in 32 bits (the host checks nblocks); 32-bit arithmetic
  // keeps 64-bit division out of the per-block path.
  const int bpr = static_cast<int>(blocks_per_row);
  int issued = 0;  // thread 0: blocks whose load was issued (in order)
  auto issue = [&](int j) {  // load this CTA's j-th block into stage j % kStages
    const int64_t blk = blockIdx.x + static_cast<int64_t>(j) * gridDim.x;
    if (blk >= nblocks) return;
    issued = j + 1;
    const int b32 = static_cast<int>(blk);
    const int bi = b32 / bpr, bj = b32 - bi * bpr;
    const int st = j % kStages;
    const uint32_t fb = smem_u32(&full[st]);
    mbar_arrive_expect_tx(fb, SC::kTileBytes);
    tma_load_2d(smem_u32(stage_data + st * SC::kTileBytes), &tmap_x, fb, bj * kBlock, bi * kBlock);
  };
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmap_x);
    for (int j = 0; j < kAhead; ++j) issue(j);
  }

  // This CTA's block (bi, bj), stage and phase advance as running counters.
  int bi = static_cast<int>(blockIdx.x) / bpr, bj = static_cast<int>(blockIdx.x) - bi * bpr;
  const int gdiv = static_cast<int>(gridDim.x) / bpr, gmod = static_cast<int>(gridDim.x) - gdiv * bpr;
  int st = 0;
  uint32_t ph = 0;
  int j = 0;
  for (int64_t blk = blockIdx.x; blk < nblocks; blk += gridDim.x, ++j) {
    const bool ok = mbar_wait(smem_u32(&full[st]), ph, abort_flag, status, limit_ns);
    if (__syncthreads_or(!ok)) break;
    float4 v[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int tr = warp * kRowsPerWarp + i;
      if constexpr (kBf16) {
        const uint2 u = reinterpret_cast<const uint2*>(stage_data + st * SC::kTileBytes + tr * kBlock * 2)[lane];
        v[i] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
      } else {
        v[i] = reinterpret_cast<const float4*>(stage_data + st * SC::kTileBytes + tr * kBlock * 4)[lane];
      }
    }
    const int64_t r0 = static_cast<int64_t>(bi) * kBlock + warp * kRowsPerWarp;
    const int64_t c0 = static_cast<int64_t>(bj) * kBlock + lane * 4;
    if constexpr (kRowwise) {
      __syncthreads();  // every thread has copied its part of the stage
      if (threadIdx.x == 0) issue(j + kAhead);
      // Row maxima; lane i then computes row i's scale and its reciprocal (one
      // division per warp instead of one per row), which the others read back.
      float my_amax = 0.f;
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const float m =
            fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w)));
        const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m)));
        if (lane == i) my_amax = amax;
      }
      float my_s = my_amax / 448.0f;
      if (my_s == 0.0f) my_s = 1.0f;
      if constexpr (kPow2) my_s = pow2_round_up(my_s);
      const float my_r = 1.0f / my_s;
      if (lane < kRowsPerWarp && r0 + lane < rows) scales[(r0 + lane) * blocks_per_row + bj] = my_s;
      // Rows whose scale is subnormal are always divided (bit i: row i).
      const uint32_t tiny = kPow2 ? 0u : __ballot_sync(0xFFFFFFFFu, lane < kRowsPerWarp && my_s < 0x1p-126f);
      // Every row's codes first (independent work that can interleave), then
      // the rare exact divisions, then the stores.
      uint32_t code[kRowsPerWarp];
      uint32_t bad = tiny;
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const float r = __shfl_sync(0xFFFFFFFFu, my_r, i);
        if constexpr (kPow2) {
          code[i] = encode4<1>(v[i], 1.0f, r);  // power-of-two scale: v * r is exact
        } else {
          bool ok;
          code[i] = encode4_bracketed(v[i], r, ok);
          bad |= (ok ? 0u : 1u) << i;
        }
      }
      if (!kPow2 && __any_sync(0xFFFFFFFFu, bad != 0u)) {
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          const float s = __shfl_sync(0xFFFFFFFFu, my_s, i);
          if ((bad >> i) & 1u) code[i] = encode4<2>(v[i], s, 0.0f);
        }
      }
      if (r0 + kRowsPerWarp <= rows && c0 + 3 < cols) {  // all of this thread's groups are inside
        uint8_t* out = q + r0 * ld_q + c0;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i, out += ld_q) __stcs(reinterpret_cast<unsigned int*>(out), code[i]);
      } else {
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          const int64_t row = r0 + i;
          if (row < rows) {
            uint8_t* out = q + row * ld_q + c0;
            if (c0 + 3 < cols) {
              __stcs(reinterpret_cast<unsigned int*>(out), code[i]);
            } else {
#pragma unroll
              for (int t = 0; t < 4; ++t)
                if (c0 + t < cols) out[t] = static_cast<uint8_t>((code[i] >> (8 * t)) & 0xFFu);
            }
          }
        }
      }
    } else {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
      const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
      if (lane == 0) warp_amax[warp] = __uint_as_float(wmax);
      __syncthreads();  // also: every thread has copied its part of the stage
      // Every thread has copied block j: the stage of block j + kAhead is free
      // (re-reading forms: once the encode below has read it again).
      if (!SC::kReread && threadIdx.x == 0) issue(j + kAhead);
      float amax = warp_amax[0];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, warp_amax[w]);
      float s = amax / 448.0f;
      if (s == 0.0f) s = 1.0f;
      if constexpr (kPow2) s = pow2_round_up(s);
      if (threadIdx.x == 0) scales[blk] = s;
      const float r = 1.0f / s;
      if constexpr (SC::kReread) {
        encode_store_reread<kPow2>(stage_data + st * SC::kTileBytes, warp, lane, r0, c0, rows, cols, q, ld_q, s, r);
      } else if constexpr (kPow2) {
        encode_store<1, true>(v, r0, c0, rows, cols, q, ld_q, s, r);
      } else if (s >= 0x1p-126f) {
        encode_store<0, true>(v, r0, c0, rows, cols, q, ld_q, s, r);
      } else {
        encode_store<2, true>(v, r0, c0, rows, cols, q, ld_q, s, r);
      }
      __syncthreads();  // warp_amax is rewritten by the next block; the stage is read
      if (SC::kReread && threadIdx.x == 0) issue(j + kAhead);
    }
    if (++st == kStages) {
      st = 0;
      ph ^= 1u;
    }
    bi += gdiv;
    bj += gmod;
    if (bj >= bpr) {
      bj -= bpr;
      ++bi;
    }
  }
  // After a timeout, loads still in flight (blocks j .. issued-1) must land
  // before the CTA exits; each gets a bounded wait on its own phase.
  if (threadIdx.x == 0 && *abort_flag) {
    for (int jj = j; jj < issued; ++jj) {
      const uint32_t bar = smem_u32(&full[jj % kStages]);
      const uint32_t par = static_cast<uint32_t>((jj / kStages) & 1);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, par)) {
        if (global_timer_ns() - t0 > 10000000ull) break;
      }
    }
  }
}

// Launch the streaming kernel (16-byte-aligned x, row stride a multiple of 16
// bytes); false if the tensor map cannot be made (the caller falls back).
template <bool kPow2, bool kRowwise, bool kBf16, int kShort = 0>
bool launch_stream(const void* x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* q, int64_t ld_q,
                   float* scales, cudaStream_t stream, cudaError_t& err) {
  using SC = StreamCfg<kBf16, kShort>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return false;
  CUtensorMap tm;
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(ld_x) * SC::kElemBytes};
  const uint32_t box[2] = {kBlock, kBlock};
  if (!encode_tensor_map(&tm, kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x, 2,
                         dims, strides, box, false))
    return false;
  const size_t smem = 1024 + SC::kStages * SC::kTileBytes + SC::kStages * 8 + kWarps * 4 + 16;
  auto kernel = quantize_stream_kernel<kPow2, kRowwise, kBf16, kShort>;
  static std::atomic<uint64_t> attr_set{0};
  if (!(attr_set.load() & (1ull << dev))) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess) {
      err = cudaGetLastError();
      return true;
    }
    attr_set.fetch_or(1ull << dev);
  }
  unsigned int* status = device_status_word();
  if (!status) {
    err = cudaErrorUnknown;
    return true;
  }
  const int64_t nbr = (rows + kBlock - 1) / kBlock;
  const int64_t nbc = (cols + kBlock - 1) / kBlock;
  const int64_t nblocks = nbr * nbc;
  if (nblocks > 0x7FFFFFFFll) return false;  // block indices are 32-bit in the kernel
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(nblocks, SC::kCtasPerSm * sms));
  err = launch_kernel(kernel, dim3(grid), dim3(kThreads), smem, stream, 0, tm, rows, cols, q, ld_q, scales, nbc,
                      nblocks, status, kDefaultWaitLimitNs);
  if (err != cudaSuccess) cudaGetLastError();
  return true;
}

}  // namespace

cudaError_t launch_quantize_1x128(const void* x, bool bf16, int64_t rows, int64_t cols, int64_t ld_x,
                                  uint8_t* q, int64_t ld_q, float* scales, bool pow2_scales,
                                  cudaStream_t stream) {
  const int64_t nbc = (cols + kBlock - 1) / kBlock;
  const int64_t total = rows * nbc;
  const int64_t esize = bf16 ? 2 : 4;
  // TMA streaming when x is 16-byte aligned with a row stride that is a multiple of 16 bytes.
  if (reinterpret_cast<uintptr_t>(x) % 16 == 0 && (ld_x * esize) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(q) % 4 == 0 && ld_q % 4 == 0) {
    cudaError_t err = cudaSuccess;
    bool done;
    if (bf16)
      done = pow2_scales ? launch_stream<true, true, true>(x, rows, cols, ld_x, q, ld_q, scales, stream, err)
                         : launch_stream<false, true, true>(x, rows, cols, ld_x, q, ld_q, scales, stream, err);
    else
      done = pow2_scales ? launch_stream<true, true, false>(x, rows, cols, ld_x, q, ld_q, scales, stream, err)
                         : launch_stream<false, true, false>(x, rows, cols, ld_x, q, ld_q, scales, stream, err);
    if (done) return err;
  }
  const int64_t vbytes = 4 * esize;  // one lane's four elements
  const bool vec = (reinterpret_cast<uintptr_t>(x) % vbytes == 0) && ((ld_x * esize) % vbytes == 0) &&
                   (reinterpret_cast<uintptr_t>(q) % 4 == 0) && (ld_q % 4 == 0);
  int dev = 0;
  int sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) sms = device_sm_count(dev);
  if (sms <= 0) sms = 1;
  // Enough warps to keep every SM's memory pipe busy, each with a contiguous run.
  const int64_t max_blocks = static_cast<int64_t>(sms) * 8;
  int64_t blocks = (total + k1xWarps * k1xSegs - 1) / (k1xWarps * k1xSegs);
  blocks = std::max<int64_t>(1, std::min(blocks, max_blocks));
  const int64_t warps = blocks * k1xWarps;
  int64_t per_warp = (total + warps - 1) / warps;
  per_warp = (per_warp + k1xSegs - 1) / k1xSegs * k1xSegs;
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t err = cudaSuccess;
#define DG_Q1X(BF, VEC, P2)                                                                                \
  err = launch_kernel(quantize_1x128_kernel<BF, VEC, P2>, grid, dim3(k1xThreads), 0, stream, 0, x, rows, cols, \
                      ld_x, q, ld_q, scales, nbc, per_warp)
  if (bf16) {
    if (vec) {
      if (pow2_scales) DG_Q1X(true, true, true); else DG_Q1X(true, true, false);
    } else {
      if (pow2_scales) DG_Q1X(true, false, true); else DG_Q1X(true, false, false);
    }
  } else {
    if (vec) {
      if (pow2_scales) DG_Q1X(false, true, true); else DG_Q1X(false, true, false);
    } else {
      if (pow2_scales) DG_Q1X(false, false, true); else DG_Q1X(false, false, false);
    }
  }
#undef DG_Q1X
  if (err != cudaSuccess) cudaGetLastError();
  return err;
}

cudaError_t launch_quantize(const float* x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* q,
                            int64_t ld_q, float* scales, bool pow2_scales, cudaStream_t stream) {
  const int64_t nbr = (rows + kBlock - 1) / kBlock;
  const int64_t nbc = (cols + kBlock - 1) / kBlock;
  const int64_t nblocks = nbr * nbc;
  if (nblocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
  const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ld_x % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(q) % 4 == 0) && (ld_q % 4 == 0);
  if (vec) {
    int dev = 0;
    const int sms = cudaGetDevice(&dev) == cudaSuccess ? device_sm_count(dev) : 0;
    // Short inputs: every block resident at once with three CTAs per SM, else
    // two per SM while the input has at most four blocks per SM.
    const int64_t per_sm = sms > 0 ? (nblocks + sms - 1) / sms : 0;
    cudaError_t err = cudaSuccess;
    bool done;
    if (sms > 0 && per_sm <= 3)
      done = pow2_scales ? launch_stream<true, false, false, 3>(x, rows, cols, ld_x, q, ld_q, scales, stream, err)
                         : launch_stream<false, false, false, 3>(x, rows, cols, ld_x, q, ld_q, scales, stream, err);
    else if (sms > 0 && per_sm <= 4)
      done = pow2_scales ? launch_stream<true, false, false, 2>(x, rows, cols, ld_x, q, ld_q, scales, stream, err)
                         : launch_stream<false, false, false, 2>(x, rows, cols, ld_x, q, ld_q, scales, stream, err);
    else
      done = pow2_scales ? launch_stream<true, false, false>(x, rows, cols, ld_x, q, ld_q, scales, stream, err)
                         : launch_stream<false, false, false>(x, rows, cols, ld_x, q, ld_q, scales, stream, err);
    if (done) return err;
  }
  const dim3 grid(static_cast<unsigned>(nblocks));
  auto kernel = vec ? (pow2_scales ? quantize_kernel<true, true> : quantize_kernel<true, false>)
                    : (pow2_scales ? quantize_kernel<false, true> : quantize_kernel<false, false>);
  const cudaError_t err = launch_kernel(kernel, grid, dim3(kThreads), 0, stream, 0, x, rows, cols, ld_x, q, ld_q,
                                        scales, nbc);
  if (err != cudaSuccess) cudaGetLastError();
  return err;
}

}  // namespace dg
