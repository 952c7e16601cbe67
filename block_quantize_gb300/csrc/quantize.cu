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
// registers between the two passes, so the input is read from HBM once; small
// CTAs let four blocks stay resident per SM, keeping enough loads in flight.
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
//    through a 3-stage TMA ring in shared memory guarded by mbarriers, so that
//    ~190 KB per SM are in flight while earlier blocks are reduced and encoded
//    from shared memory. Out-of-range rows and columns of edge blocks arrive
//    as zeros (TMA fill), which leaves the block max unchanged.
//  * quantize_kernel (any alignment): one CTA per block, the block held in
//    registers between the two passes.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "dg_device.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kBlock = 128;
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kBlock / kWarps;  // 8

// Smallest power of two >= s (s > 0, finite), not below 2^-127, the smallest
// UE8M0 value. Exponent arithmetic on the binary32 encoding.
__device__ __forceinline__ float pow2_round_up(float s) {
  const uint32_t b = __float_as_uint(s);
  const uint32_t e = b >> 23;
  if (e == 0u) {  // subnormal s < 2^-126
    return (b <= 0x00400000u) ? __uint_as_float(0x00400000u) : __uint_as_float(0x00800000u);
  }
  return __uint_as_float((e + ((b & 0x007FFFFFu) != 0u ? 1u : 0u)) << 23);
}

__device__ __forceinline__ uint32_t cvt2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// E4M3 codes of fl32(v / s) for the four values of v, packed little-endian.
// kMode 0: exact division with the r = 1/s fast path (valid for normal s);
// kMode 1: power-of-two s, v * r exact; kMode 2: plain division (tiny s).
template <int kMode>
__device__ __forceinline__ uint32_t encode4(const float4 v, float s, float r) {
  if constexpr (kMode == 2) {
    return cvt2(v.x / s, v.y / s) | (cvt2(v.z / s, v.w / s) << 16);
  } else {
    const float q0 = v.x * r, q1 = v.y * r, q2 = v.z * r, q3 = v.w * r;
    const uint32_t c = cvt2(q0, q1) | (cvt2(q2, q3) << 16);
    if constexpr (kMode == 1) {
      return c;
    } else {
      constexpr float kLo = 1.0f - 0x1p-20f, kHi = 1.0f + 0x1p-20f;
      const uint32_t lo = cvt2(q0 * kLo, q1 * kLo) | (cvt2(q2 * kLo, q3 * kLo) << 16);
      const uint32_t hi = cvt2(q0 * kHi, q1 * kHi) | (cvt2(q2 * kHi, q3 * kHi) << 16);
      if (lo == hi) return lo;  // no E4M3 rounding boundary near q: exact
      return cvt2(v.x / s, v.y / s) | (cvt2(v.z / s, v.w / s) << 16);
    }
  }
}

template <int kMode>
__device__ __forceinline__ uint8_t encode1(float v, float s, float r) {
  const uint32_t c = encode4<kMode>(make_float4(v, 0.f, 0.f, 0.f), s, r);
  return static_cast<uint8_t>(c & 0xFFu);
}

template <int kMode, bool kVec>
__device__ __forceinline__ void encode_store(const float4 (&v)[kRowsPerWarp], int64_t r0, int64_t c0,
                                             int64_t rows, int64_t cols, uint8_t* __restrict__ q,
                                             int64_t ld_q, float s, float r) {
  const bool full4 = c0 + 3 < cols;
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

template <bool kVec, bool kPow2>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const float* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ld_x,
                                                            uint8_t* __restrict__ q, int64_t ld_q,
                                                            float* __restrict__ scales,
                                                            int64_t blocks_per_row) {
  __shared__ float warp_amax[kWarps];
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

constexpr int kStreamStages = 3;
constexpr uint32_t kBlockBytes = kBlock * kBlock * 4;

template <bool kPow2>
__global__ void __launch_bounds__(kThreads, 1)
    quantize_stream_kernel(const __grid_constant__ CUtensorMap tmap_x, int64_t rows, int64_t cols,
                           uint8_t* __restrict__ q, int64_t ld_q, float* __restrict__ scales,
                           int64_t blocks_per_row, int64_t nblocks, unsigned int* status,
                           uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* stage_data = reinterpret_cast<float*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStreamStages * kBlockBytes);
  float* warp_amax = reinterpret_cast<float*>(full + kStreamStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(warp_amax + kWarps);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStreamStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  int64_t issued = 0;  // thread 0: blocks whose load was issued (in order)
  auto issue = [&](int64_t j) {  // load this CTA's j-th block into stage j % kStreamStages
    const int64_t blk = blockIdx.x + j * gridDim.x;
    if (blk >= nblocks) return;
    issued = j + 1;
    const int64_t bi = blk / blocks_per_row, bj = blk - bi * blocks_per_row;
    const int st = static_cast<int>(j % kStreamStages);
    const uint32_t fb = smem_u32(&full[st]);
    mbar_arrive_expect_tx(fb, kBlockBytes);
    tma_load_2d(smem_u32(stage_data + st * (kBlock * kBlock)), &tmap_x, fb,
                static_cast<int32_t>(bj * kBlock), static_cast<int32_t>(bi * kBlock));
  };
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmap_x);
    for (int j = 0; j < kStreamStages; ++j) issue(j);
  }

  int64_t j = 0;
  for (int64_t blk = blockIdx.x; blk < nblocks; blk += gridDim.x, ++j) {
    const int st = static_cast<int>(j % kStreamStages);
    const bool ok = mbar_wait(smem_u32(&full[st]), static_cast<uint32_t>((j / kStreamStages) & 1),
                              abort_flag, status, limit_ns);
    if (__syncthreads_or(!ok)) break;
    const int64_t bi = blk / blocks_per_row, bj = blk - bi * blocks_per_row;
    const float* tile = stage_data + st * (kBlock * kBlock);
    float4 v[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
      v[i] = reinterpret_cast<const float4*>(tile + (warp * kRowsPerWarp + i) * kBlock)[lane];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
    if (lane == 0) warp_amax[warp] = __uint_as_float(wmax);
    __syncthreads();  // also: every thread has copied its part of the stage
    // The stage is free again: refill it with the block kStreamStages ahead.
    if (threadIdx.x == 0) issue(j + kStreamStages);
    float amax = warp_amax[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, warp_amax[w]);
    float s = amax / 448.0f;
    if (s == 0.0f) s = 1.0f;
    if constexpr (kPow2) s = pow2_round_up(s);
    if (threadIdx.x == 0) scales[blk] = s;
    const float r = 1.0f / s;
    const int64_t r0 = bi * kBlock + warp * kRowsPerWarp;
    const int64_t c0 = bj * kBlock + lane * 4;
    if constexpr (kPow2) {
      encode_store<1, true>(v, r0, c0, rows, cols, q, ld_q, s, r);
    } else if (s >= 0x1p-126f) {
      encode_store<0, true>(v, r0, c0, rows, cols, q, ld_q, s, r);
    } else {
      encode_store<2, true>(v, r0, c0, rows, cols, q, ld_q, s, r);
    }
    __syncthreads();  // warp_amax is rewritten by the next block
  }
  // After a timeout, loads still in flight (blocks j .. issued-1) must land
  // before the CTA exits; each gets a bounded wait on its own phase.
  if (threadIdx.x == 0 && *abort_flag) {
    for (int64_t jj = j; jj < issued; ++jj) {
      const uint32_t bar = smem_u32(&full[jj % kStreamStages]);
      const uint32_t par = static_cast<uint32_t>((jj / kStreamStages) & 1);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, par)) {
        if (global_timer_ns() - t0 > 10000000ull) break;
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize(const float* x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* q,
                            int64_t ld_q, float* scales, bool pow2_scales, cudaStream_t stream) {
  const int64_t nbr = (rows + kBlock - 1) / kBlock;
  const int64_t nbc = (cols + kBlock - 1) / kBlock;
  const int64_t nblocks = nbr * nbc;
  if (nblocks > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
  const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ld_x % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(q) % 4 == 0) && (ld_q % 4 == 0);
  int dev = 0;
  if (vec && cudaGetDevice(&dev) == cudaSuccess) {
    const int sms = device_sm_count(dev);
    CUtensorMap tm;
    const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(ld_x) * 4};
    const uint32_t box[2] = {kBlock, kBlock};
    if (sms > 0 && encode_tensor_map(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x, 2, dims, strides, box, false)) {
      const size_t smem = 1024 + kStreamStages * kBlockBytes + kStreamStages * 8 + kWarps * 4 + 16;
      static std::atomic<uint64_t> attr_set{0};
      if (dev < 64 && !(attr_set.load() & (1ull << dev))) {
        if (cudaFuncSetAttribute(quantize_stream_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess ||
            cudaFuncSetAttribute(quantize_stream_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
          return cudaGetLastError();
        attr_set.fetch_or(1ull << dev);
      }
      unsigned int* status = device_status_word();
      if (!status) return cudaGetLastError();
      const unsigned grid = static_cast<unsigned>(std::min<int64_t>(nblocks, sms));
      if (pow2_scales)
        quantize_stream_kernel<true><<<grid, kThreads, smem, stream>>>(tm, rows, cols, q, ld_q, scales, nbc,
                                                                        nblocks, status, kDefaultWaitLimitNs);
      else
        quantize_stream_kernel<false><<<grid, kThreads, smem, stream>>>(tm, rows, cols, q, ld_q, scales, nbc,
                                                                         nblocks, status, kDefaultWaitLimitNs);
      return cudaGetLastError();
    }
  }
  const dim3 grid(static_cast<unsigned>(nblocks));
  if (vec) {
    if (pow2_scales)
      quantize_kernel<true, true><<<grid, kThreads, 0, stream>>>(x, rows, cols, ld_x, q, ld_q, scales, nbc);
    else
      quantize_kernel<true, false><<<grid, kThreads, 0, stream>>>(x, rows, cols, ld_x, q, ld_q, scales, nbc);
  } else {
    if (pow2_scales)
      quantize_kernel<false, true><<<grid, kThreads, 0, stream>>>(x, rows, cols, ld_x, q, ld_q, scales, nbc);
    else
      quantize_kernel<false, false><<<grid, kThreads, 0, stream>>>(x, rows, cols, ld_x, q, ld_q, scales, nbc);
  }
  return cudaGetLastError();
}

}  // namespace dg
