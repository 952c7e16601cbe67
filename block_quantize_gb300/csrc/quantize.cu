// quantize.cu -- 128x128 block quantization of an FP32 matrix to E4M3 codes and
// one FP32 (or power-of-two) scale per block, after the lpnh.cn DeepGEMM
// walkthrough §4.2 (cut into 128x128 blocks, take max|x|, scale = max_abs/448,
// divide, round to the nearest E4M3 value with ties to even, keep the scales
// in their own array), §3.1 (FP32 scales computed ahead of the GEMM) and §5.4
// (all-zero blocks). The power-of-two variant follows the packed UE8M0 scales of
// pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1.
//
// One CTA of 256 threads owns one 128x128 block: warp w holds rows
// [16w, 16w+16), lane l holds columns [4l, 4l+4), i.e. 16 float4 per thread kept
// in registers between the two passes, so the input is read from HBM once.
// Loads are 128-bit and streaming; each warp-wide load covers one 512-byte row
// segment. The block max is a warp-shuffle reduction followed by an 8-entry
// shared-memory reduction (warp-shuffle reduction as in the hotelren.com GEMM
// tuning essay §4.2).
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kBlock = 128;
constexpr int kThreads = 256;
constexpr int kRowsPerWarp = kBlock / (kThreads / 32);  // 16

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

// fl32(v / s), exactly. With a power-of-two scale, v * (1/s) is the same
// correctly rounded quotient because 1/s is exact.
template <bool kPow2>
__device__ __forceinline__ float divide(float v, float s, float inv) {
  if constexpr (kPow2) return v * inv;
  else return v / s;
}

template <bool kPow2>
__device__ __forceinline__ uint32_t encode4(const float4 v, float s, float inv) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
      make_float2(divide<kPow2>(v.x, s, inv), divide<kPow2>(v.y, s, inv)), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
      make_float2(divide<kPow2>(v.z, s, inv), divide<kPow2>(v.w, s, inv)), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

template <bool kVec, bool kPow2>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const float* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ld_x,
                                                            uint8_t* __restrict__ q, int64_t ld_q,
                                                            float* __restrict__ scales,
                                                            int64_t blocks_per_row) {
  __shared__ float warp_amax[kThreads / 32];
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
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, warp_amax[w]);

  // scale = max_abs / 448 in FP32; an all-zero block (or an underflow to 0) gets 1.
  float s = amax / 448.0f;
  if (s == 0.0f) s = 1.0f;
  if constexpr (kPow2) s = pow2_round_up(s);
  if (threadIdx.x == 0) scales[blk] = s;
  const float inv = kPow2 ? 1.0f / s : 0.0f;

  // Pass 2: divide by the scale and round to the nearest E4M3 value (RNE, saturating).
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int64_t r = r0 + i;
    if (r >= rows) continue;
    uint8_t* out = q + r * ld_q + c0;
    if (kVec && full4) {
      __stcs(reinterpret_cast<unsigned int*>(out), encode4<kPow2>(v[i], s, inv));
    } else {
      const float e[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (c0 + t < cols) {
          out[t] = __nv_cvt_float_to_fp8(divide<kPow2>(e[t], s, inv), __NV_SATFINITE, __NV_E4M3);
        }
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
