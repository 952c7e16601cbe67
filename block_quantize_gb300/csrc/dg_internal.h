// dg_internal.h -- host-side launchers shared by the C ABI (api.cpp) and the
// CUDA translation units. Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

namespace dg {

// Bits of the per-device status word: kernels OR one in when a bounded wait
// runs out, or when an M-grouped call meets an expert id outside [0, num_groups).
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned int kStatusBadGroup = 2u;

// Launch a kernel with programmatic dependent launch allowed (and a cluster
// of cluster_x CTAs when cluster_x > 0). The kernel may then begin while the
// previous work on the stream finishes, so it must execute griddepcontrol.wait
// (pdl_wait) before it touches global memory; our kernels do that right after
// their set-up (barriers, TMEM, tensor-map prefetch) and then let the next
// launch begin (pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// 128x128 block quantizer launch (sizes already validated, rows, cols > 0).
cudaError_t launch_quantize(const float* x, int64_t rows, int64_t cols, int64_t ld_x,
                            uint8_t* q, int64_t ld_q, float* scales, bool pow2_scales,
                            cudaStream_t stream);

// Row-wise 1x128 quantizer launch (sizes already validated, rows, cols > 0).
cudaError_t launch_quantize_1x128(const void* x, bool bf16, int64_t rows, int64_t cols, int64_t ld_x,
                                  uint8_t* q, int64_t ld_q, float* scales, bool pow2_scales,
                                  cudaStream_t stream);

// E4M3 output of a requantizing GEMM: the FP32 accumulators are encoded with
// one scale per block of block_rows x 128 output elements.
struct RequantOut {
  uint8_t* q;       // [M][ld_q] E4M3 codes (nullptr: bf16 output instead)
  int64_t ld_q;     // multiple of 16; q 16-byte aligned
  float* s;         // [M or ceil(M/128)][ld_s] scales
  int64_t ld_s;     // ceil(N / 128)
  int block_rows;   // 1 (one scale per row and 128 columns) or 128 (128 x 128 blocks)
  int pow2;         // scales rounded up to powers of two
};

// One dense or M-grouped GEMM problem (sizes already validated).
struct GemmProblem {
  void* c;
  int64_t ld_c;
  const uint8_t* a;
  int64_t ld_a;
  const float* sa;
  const uint8_t* b;
  int64_t ld_b;            // dense: row stride of B; grouped: K
  const float* sb;
  const int32_t* m_indices;  // nullptr for the dense GEMM
  int num_groups;            // 1 for the dense GEMM
  int64_t M, N, K;
  int num_sms_cap;           // 0 = every SM
  bool pow2_scales;          // every scale is a power of two (DG_SCALE_UE8M0)
  bool sa_per_row;           // sa is [M][K/128] (one A scale per row and K block)
  RequantOut rq;             // rq.q != nullptr: E4M3 output instead of bf16 c
  bool a_mn;                 // A stored [K][ld_a] (M contiguous) instead of [M][ld_a]
  bool b_mn;                 // B stored [K][ld_b] (N contiguous) instead of [N][ld_b]
  int64_t ld_sa, ld_sb;      // row strides of sa and sb in floats (normally K/128)
};

// Returns a dg_status value.
int launch_gemm(const GemmProblem& p, cudaStream_t stream);

// DG_GEMM_BLOCK_N set: every GEMM takes the 1-SM kernel with that tile width.
bool tile_width_forced();

// Writes v into n consecutive floats of device memory.
cudaError_t launch_fill_f32(float* dst, int64_t n, float v, cudaStream_t stream);

// Dense GEMMs with M > 128 on CTA pairs (gemm_pair.cu); DG_ERR_UNSUPPORTED_SHAPE
// when the problem or the launch limits do not allow a pair kernel.
int launch_gemm_pair(const GemmProblem& p, cudaStream_t stream);

// K-grouped TN GEMM with FP32 scales on CTA pairs, every non-empty K range in
// one launch: C_g [M][ld_c] at c + g * M * ld_c is A^T B over the K rows of
// range g (k_sizes[g] rows each, in order, multiples of 128; p.K is their
// sum). Ranges with K = 0 are left untouched (the caller zero-fills them).
// DG_ERR_UNSUPPORTED_SHAPE when the call needs the per-range path.
int launch_gemm_pair_k_grouped(const GemmProblem& p, const int64_t* k_sizes, int num_groups, cudaStream_t stream);

// Dense GEMMs with M <= 128 use the cluster split-K kernel (gemm_smallm.cu).
bool small_m_supported(int64_t M, const void* m_indices);
int launch_gemm_small_m(const GemmProblem& p, cudaStream_t stream);

// M = 1 with K-major B and bf16 output, all SMs allowed: the streaming kernel
// of gemv.cu.
bool gemv_supported(const GemmProblem& p);
int launch_gemv(const GemmProblem& p, cudaStream_t stream);

// Takes and clears the current device's status word (kStatusTimeout,
// kStatusBadGroup bits) in one atomic step on `stream`, then waits for the
// stream. Returns the CUDA error of the launch or the copy.
cudaError_t read_and_clear_status(unsigned int* out, cudaStream_t stream);

// Launches one block that waits on a barrier nothing arrives at, so that its
// bounded wait runs out after limit_ns.
cudaError_t launch_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (128-byte
// swizzle or none); false if the driver call is unavailable or rejects the map.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                       const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                       bool swizzle128);

// Same with an explicit swizzle mode.
bool encode_tensor_map_swizzle(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                               const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                               CUtensorMapSwizzle swizzle);

// Device address of the current device's status word (resolved once per device
// with cudaGetSymbolAddress); nullptr on failure.
unsigned int* device_status_word();

// Number of SMs of device `dev` (0 if unknown).
int device_sm_count(int dev);

// Default limit of every in-kernel wait (1 second).
constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;

}  // namespace dg
