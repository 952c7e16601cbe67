// gemv.cu -- the block-scaled NT GEMM for a single row of A (M = 1, one-token
// decode), B stored K-major ([N][ld_b]).
//
// The arithmetic of the other GEMM kernels (lpnh.cn DeepGEMM walkthrough §2.2,
// §3.2; pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1, §4.1): the products
// of every 128-wide K block carry the factor sa[kb] * sb[n/128][kb], and the
// sum runs in FP32. With one row of A the GEMM reads each byte of B once and
// does two FLOPs per byte, so the HBM stream alone sets its time. Tensor-core
// tiles would only add what a split-K schedule costs at this size: 128-byte
// TMA rows, whole waves of tiles and a reduction between CTAs. Instead:
//   * a CTA owns kRows consecutive rows of B (kRows outputs), all in one
//     128-row scale block, and adds nothing across CTAs. kRows is 4 for
//     K <= 4096 and 8 above (measured: more, smaller CTAs suit short rows);
//   * thread t owns the 16-byte K segments t, t + T, t + 2T, ... of those rows
//     (T threads). It loads the segment's 16 A values once, multiplies them by
//     the segment's K-block factor, then reads the segment in each of the
//     kRows B rows and accumulates 16 products per row with FP32 FMAs. Lanes read
//     consecutive segments, so every warp load is 512 contiguous bytes;
//   * the CTA adds its threads' sums in a fixed order (warp shuffles, then
//     shared memory) and rounds them to bf16.
// Each product is formed as (s a) b, not s (a b): the factor is applied before
// the FP32 sum, not after. The two are FP32 evaluations of the same sum, within
// the GEMM tolerance. With power-of-two factors and small-integer codes every
// step is exact, so such inputs give the same bits as the other kernels.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/dgfp8.h"
#include "dg_device.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kMaxThreads = 256;  // 16-byte K segments in flight per row per CTA

struct GemvArgs {
  __nv_bfloat16* c;   // row 0 of C
  const uint8_t* a;   // A's row: element k at a + k * a_step
  int64_t a_step;     // 1 (K-major A) or ld_a (A stored [K][ld_a])
  const uint8_t* b;   // B [N][ld_b], K-major
  int64_t ld_b;
  const float* sa;    // row 0 of A's scales: sa[kb]
  const float* sb;    // sb[nb * ld_sb + kb]
  int64_t ld_sb;
  int64_t N;
  int segs;           // K / 16
};

// The 16 E4M3 codes of v (little-endian, element 0 in the lowest byte) as FP32.
// E4M3 -> FP16 is exact (every E4M3 value is an FP16 value), and so is FP16 -> FP32.
__device__ __forceinline__ void decode16(const uint4 v, float (&x)[16]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
    const float2 f0 = __half22float2(__half2(lo));
    const float2 f1 = __half22float2(__half2(hi));
    x[4 * i] = f0.x;
    x[4 * i + 1] = f0.y;
    x[4 * i + 2] = f1.x;
    x[4 * i + 3] = f1.y;
  }
}

// kRows rows of B (outputs) per CTA; divides 128.
template <int kRows>
__global__ void __launch_bounds__(kMaxThreads, kRows <= 4 ? 4 : 3) fp8_gemv_kernel(const GemvArgs args) {
  __shared__ float red[kMaxThreads / 32][kRows];
  const int T = static_cast<int>(blockDim.x);  // a multiple of 32
  const int t = static_cast<int>(threadIdx.x);
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kRows;
  const int rows = static_cast<int>(min(static_cast<int64_t>(kRows), args.N - n0));  // >= 1
  const float* sb_row = args.sb + (n0 / 128) * args.ld_sb;
  const uint8_t* b0 = args.b + n0 * args.ld_b;
  // The first pass over this CTA's B rows starts streaming into L2 while the
  // preceding grid finishes (whole rows of a long K would crowd L2).
  if (t < rows) bulk_prefetch_l2(b0 + t * args.ld_b, static_cast<uint32_t>(min(args.segs, T)) * 16u);
  pdl_wait();
  pdl_trigger();

  float acc[kRows];
#pragma unroll
  for (int j = 0; j < kRows; ++j) acc[j] = 0.f;

  for (int u = t; u < args.segs; u += T) {
    // The B segment of every row first (kRows loads in flight), then A and the factor.
    uint4 bv[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j)
      bv[j] = (j < rows) ? __ldcs(reinterpret_cast<const uint4*>(b0 + j * args.ld_b) + u) : make_uint4(0, 0, 0, 0);
    uint4 av;
    if (args.a_step == 1) {
      av = __ldg(reinterpret_cast<const uint4*>(args.a) + u);
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i >> 2] |= static_cast<uint32_t>(__ldg(args.a + (static_cast<int64_t>(u) * 16 + i) * args.a_step))
                     << (8 * (i & 3));
      av = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const int kb = u >> 3;  // 8 segments per 128-wide K block
    const float s = __ldg(args.sa + kb) * __ldg(sb_row + kb);
    float x[16];
    decode16(av, x);
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] *= s;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      float y[16];
      decode16(bv[j], y);
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[j] = fmaf(x[i], y[i], acc[j]);
    }
  }

  const int warp = t >> 5, lane = t & 31;
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    float v = acc[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    if (lane == 0) red[warp][j] = v;
  }
  __syncthreads();
  if (t < rows) {
    float sum = 0.f;
    for (int w = 0; w < T / 32; ++w) sum += red[w][t];
    args.c[n0 + t] = __float2bfloat16_rn(sum);
  }
}

}  // namespace

bool gemv_supported(const GemmProblem& p) {
  return p.M == 1 && p.m_indices == nullptr && !p.b_mn && p.rq.q == nullptr && p.num_sms_cap == 0 && p.K > 0;
}

int launch_gemv(const GemmProblem& p, cudaStream_t stream) {
  GemvArgs args{};
  args.c = static_cast<__nv_bfloat16*>(p.c);
  args.a = p.a;
  args.a_step = p.a_mn ? p.ld_a : 1;
  args.b = p.b;
  args.ld_b = p.ld_b;
  args.sa = p.sa;
  args.sb = p.sb;
  args.ld_sb = p.ld_sb;
  args.N = p.N;
  args.segs = static_cast<int>(p.K / 16);
  const int threads = std::min(kMaxThreads, (args.segs + 31) / 32 * 32);
  const bool short_k = p.K <= 4096;
  const int rows = short_k ? 4 : 8;
  const int64_t grid = (p.N + rows - 1) / rows;
  const cudaError_t e =
      short_k ? launch_kernel(fp8_gemv_kernel<4>, dim3(static_cast<unsigned>(grid)), dim3(threads), 0, stream, 0, args)
              : launch_kernel(fp8_gemv_kernel<8>, dim3(static_cast<unsigned>(grid)), dim3(threads), 0, stream, 0, args);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  return DG_OK;
}

}  // namespace dg
