// api.cpp -- the extern "C" boundary declared in include/dgfp8.h: argument
// validation (before any CUDA call, so that bad arguments launch nothing and
// are reported without a GPU), device checks, and dispatch to the kernels.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/dgfp8.h"
#include "dg_internal.h"

namespace {

std::atomic<int> g_num_sms_cap{0};

constexpr int64_t kDimLimit = int64_t(1) << 31;  // TMA and index arithmetic bound

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// The library is built for sm_103a only; every compute entry point checks the
// current device once per device.
int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_NO_DEVICE;
  }
  static std::atomic<int> ok_mask[2] = {{0}, {0}};  // bit per device: checked, supported
  if (dev >= 0 && dev < 31 && (ok_mask[0].load() & (1 << dev)))
    return (ok_mask[1].load() & (1 << dev)) ? DG_OK : DG_ERR_NO_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_NO_DEVICE;
  }
  const bool supported = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 31) {
    if (supported) ok_mask[1].fetch_or(1 << dev);
    ok_mask[0].fetch_or(1 << dev);
  }
  return supported ? DG_OK : DG_ERR_NO_DEVICE;
}

// Validates a GEMM call. Returns DG_OK to proceed, kEmpty when there is
// nothing to do (M or N is 0: every pointer may then be NULL), else an error.
constexpr int kEmpty = -1;

// a_row / b_row: the row length the operand's storage needs (K for K-major
// operands, M or N for MN-major ones).
int validate_gemm_rows(const void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a, const float* sa,
                       const uint8_t* b, int64_t ld_b, const float* sb, int64_t M, int64_t N, int64_t K,
                       int scale_mode, int64_t a_row, int64_t b_row) {
  if (M < 0 || N < 0 || K < 0) return DG_ERR_INVALID_ARG;
  if (scale_mode != DG_SCALE_FP32 && scale_mode != DG_SCALE_UE8M0) return DG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return kEmpty;
  if (!c || ld_c < N) return DG_ERR_INVALID_ARG;
  if (K % 128 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
  if (M >= kDimLimit || N >= kDimLimit || K >= kDimLimit || ld_c >= kDimLimit)
    return DG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(c, 16) || ld_c % 8 != 0) return DG_ERR_MISALIGNED;
  if (K == 0) return DG_OK;  // C = 0; the operands are not read
  if (!a || !b || !sa || !sb) return DG_ERR_INVALID_ARG;
  if (ld_a < a_row || ld_b < b_row) return DG_ERR_INVALID_ARG;
  if (ld_a >= kDimLimit || ld_b >= kDimLimit) return DG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(sa, 4) || !aligned(sb, 4))
    return DG_ERR_MISALIGNED;
  if (ld_a % 16 != 0 || ld_b % 16 != 0) return DG_ERR_MISALIGNED;
  return DG_OK;
}

int validate_gemm_common(const void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a, const float* sa,
                         const uint8_t* b, int64_t ld_b, const float* sb, int64_t M, int64_t N,
                         int64_t K, int scale_mode) {
  return validate_gemm_rows(c, ld_c, a, ld_a, sa, b, ld_b, sb, M, N, K, scale_mode, K, K);
}

// C = 0 when the K extent is empty.
int zero_output(void* c, int64_t ld_c, int64_t M, int64_t N, cudaStream_t st) {
  if (cudaMemset2DAsync(c, static_cast<size_t>(ld_c) * 2, 0, static_cast<size_t>(N) * 2,
                        static_cast<size_t>(M), st) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  return DG_OK;
}

// Checks the E4M3 output arguments of a requantizing GEMM (after the common
// checks, which have already applied the bf16 rules to q and ld_q).
int validate_requant_out(const uint8_t* q, int64_t ld_q, const float* s, int out_block_rows,
                         int out_scale_mode, int a_scale_rows) {
  if (out_block_rows != 1 && out_block_rows != 128) return DG_ERR_INVALID_ARG;
  if (a_scale_rows != 1 && a_scale_rows != 128) return DG_ERR_INVALID_ARG;
  if (out_scale_mode != DG_SCALE_FP32 && out_scale_mode != DG_SCALE_UE8M0) return DG_ERR_INVALID_ARG;
  if (!q || !s) return DG_ERR_INVALID_ARG;
  if (!aligned(s, 4)) return DG_ERR_MISALIGNED;
  if (!aligned(q, 16) || ld_q % 16 != 0) return DG_ERR_MISALIGNED;
  return DG_OK;
}

// Requantized C = 0 when the K extent is empty: codes 0, every scale 1.
int zero_requant_output(const dg::RequantOut& o, int64_t M, int64_t N, cudaStream_t st) {
  if (cudaMemset2DAsync(o.q, static_cast<size_t>(o.ld_q), 0, static_cast<size_t>(N), static_cast<size_t>(M),
                        st) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  const int64_t rows = o.block_rows == 1 ? M : (M + 127) / 128;
  if (dg::launch_fill_f32(o.s, rows * o.ld_s, 1.0f, st) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  return DG_OK;
}

dg::RequantOut make_requant(uint8_t* q, int64_t ld_q, float* s, int out_block_rows, int out_scale_mode,
                            int64_t N) {
  dg::RequantOut o{};
  o.q = q;
  o.ld_q = ld_q;
  o.s = s;
  o.ld_s = (N + 127) / 128;
  o.block_rows = out_block_rows;
  o.pow2 = out_scale_mode == DG_SCALE_UE8M0 ? 1 : 0;
  return o;
}

}  // namespace

extern "C" {

DG_API uint32_t dg_get_abi_version(void) { return DG_ABI_VERSION; }

DG_API const char* dg_status_string(int status) {
  switch (status) {
    case DG_OK: return "ok";
    case DG_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size, bad mode or stride)";
    case DG_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (K or M_tot not a multiple of 128, or a dimension >= 2^31)";
    case DG_ERR_MISALIGNED: return "misaligned pointer or stride (16-byte TMA rules)";
    case DG_ERR_CUDA: return "CUDA runtime error or failed launch";
    case DG_ERR_NO_DEVICE: return "no usable CUDA device (sm_103 required)";
    case DG_ERR_TIMEOUT: return "a bounded in-kernel wait ran out";
    case DG_ERR_BAD_GROUP: return "an M-grouped call met an expert id >= num_groups (those blocks were written as zeros)";
    default: return "unknown status";
  }
}

DG_API int dg_get_mk_alignment_for_contiguous_layout(void) { return 128; }

DG_API int dg_set_num_sms(int n) {
  if (n < 0) return DG_ERR_INVALID_ARG;
  g_num_sms_cap.store(n);
  return DG_OK;
}

DG_API int dg_get_num_sms(void) { return g_num_sms_cap.load(); }

DG_API int dg_quantize_fp8_block(const float* x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t* q,
                                 int64_t ld_q, float* scales, int scale_mode, void* stream) {
  if (rows < 0 || cols < 0) return DG_ERR_INVALID_ARG;
  if (scale_mode != DG_SCALE_FP32 && scale_mode != DG_SCALE_UE8M0) return DG_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return DG_OK;  // nothing to do; pointers may be NULL
  if (!x || !q || !scales) return DG_ERR_INVALID_ARG;
  if (ld_x < cols || ld_q < cols) return DG_ERR_INVALID_ARG;
  if (!aligned(x, 4) || !aligned(scales, 4)) return DG_ERR_MISALIGNED;
  const int64_t blocks = ((rows + 127) / 128) * ((cols + 127) / 128);
  if (blocks >= kDimLimit) return DG_ERR_UNSUPPORTED_SHAPE;
  const int dev_st = check_device();
  if (dev_st != DG_OK) return dev_st;
  const cudaError_t e = dg::launch_quantize(x, rows, cols, ld_x, q, ld_q, scales,
                                            scale_mode == DG_SCALE_UE8M0,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

DG_API int dg_quantize_fp8_1x128(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x,
                                 uint8_t* q, int64_t ld_q, float* scales, int scale_mode, void* stream) {
  if (rows < 0 || cols < 0) return DG_ERR_INVALID_ARG;
  if (scale_mode != DG_SCALE_FP32 && scale_mode != DG_SCALE_UE8M0) return DG_ERR_INVALID_ARG;
  if (x_dtype != DG_INPUT_FP32 && x_dtype != DG_INPUT_BF16) return DG_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return DG_OK;  // nothing to do; pointers may be NULL
  if (!x || !q || !scales) return DG_ERR_INVALID_ARG;
  if (ld_x < cols || ld_q < cols) return DG_ERR_INVALID_ARG;
  if (!aligned(x, x_dtype == DG_INPUT_BF16 ? 2 : 4) || !aligned(scales, 4)) return DG_ERR_MISALIGNED;
  if (rows * ((cols + 127) / 128) >= (int64_t(1) << 40)) return DG_ERR_UNSUPPORTED_SHAPE;
  const int dev_st = check_device();
  if (dev_st != DG_OK) return dev_st;
  const cudaError_t e = dg::launch_quantize_1x128(x, x_dtype == DG_INPUT_BF16, rows, cols, ld_x, q, ld_q,
                                                  scales, scale_mode == DG_SCALE_UE8M0,
                                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

// Argument checks of a requantized output; with M or N zero only the block shape is checked.
static int check_requant_args(const uint8_t* cq, int64_t ld_cq, const float* cs, int out_block_rows,
                              int out_scale_mode, int a_scale_rows, int64_t M, int64_t N) {
  if (M > 0 && N > 0) return validate_requant_out(cq, ld_cq, cs, out_block_rows, out_scale_mode, a_scale_rows);
  return (out_block_rows != 1 && out_block_rows != 128) ? DG_ERR_INVALID_ARG : DG_OK;
}

// One dense GEMM in any layout. rq.q != nullptr: E4M3 output (c and ld_c then describe the codes).
static int gemm_dense(void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a, const float* sa,
                      const uint8_t* b, int64_t ld_b, const float* sb, int64_t M, int64_t N, int64_t K,
                      int layout, int scale_mode, void* stream, bool a_1x128, const dg::RequantOut& rq) {
  const bool a_mn = layout == DG_LAYOUT_TN || layout == DG_LAYOUT_TT;
  const bool b_mn = layout == DG_LAYOUT_TN || layout == DG_LAYOUT_NN;
  const int v = validate_gemm_rows(c, ld_c, a, ld_a, sa, b, ld_b, sb, M, N, K, scale_mode, a_mn ? M : K,
                                   b_mn ? N : K);
  if (v == kEmpty) return DG_OK;
  if (v != DG_OK) return v;
  const int dev_st = check_device();
  if (dev_st != DG_OK) return dev_st;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return rq.q ? zero_requant_output(rq, M, N, st) : zero_output(c, ld_c, M, N, st);
  dg::GemmProblem p{};
  p.rq = rq;
  p.c = c;
  p.ld_c = ld_c;
  p.a = a;
  p.ld_a = ld_a;
  p.sa = sa;
  p.b = b;
  p.ld_b = ld_b;
  p.sb = sb;
  p.m_indices = nullptr;
  p.num_groups = 1;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_sms_cap = g_num_sms_cap.load();
  p.pow2_scales = scale_mode == DG_SCALE_UE8M0;
  p.sa_per_row = a_1x128;
  p.a_mn = a_mn;
  p.b_mn = b_mn;
  p.ld_sa = p.ld_sb = K / 128;
  return dg::launch_gemm(p, st);
}

DG_API int dg_fp8_gemm_nt(void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a, const float* sa,
                          const uint8_t* b, int64_t ld_b, const float* sb, int64_t M, int64_t N,
                          int64_t K, int scale_mode, void* stream) {
  return gemm_dense(c, ld_c, a, ld_a, sa, b, ld_b, sb, M, N, K, DG_LAYOUT_NT, scale_mode, stream, false,
                    dg::RequantOut{});
}

DG_API int dg_fp8_gemm_nt_1x128(void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a, const float* sa,
                                const uint8_t* b, int64_t ld_b, const float* sb, int64_t M, int64_t N,
                                int64_t K, int scale_mode, void* stream) {
  return gemm_dense(c, ld_c, a, ld_a, sa, b, ld_b, sb, M, N, K, DG_LAYOUT_NT, scale_mode, stream, true,
                    dg::RequantOut{});
}

DG_API int dg_fp8_gemm_nt_requant(uint8_t* cq, int64_t ld_cq, float* cs, int out_block_rows, int out_scale_mode,
                                  const uint8_t* a, int64_t ld_a, const float* sa, int a_scale_rows,
                                  const uint8_t* b, int64_t ld_b, const float* sb, int64_t M, int64_t N,
                                  int64_t K, int scale_mode, void* stream) {
  const int v = check_requant_args(cq, ld_cq, cs, out_block_rows, out_scale_mode, a_scale_rows, M, N);
  if (v != DG_OK) return v;
  return gemm_dense(cq, ld_cq, a, ld_a, sa, b, ld_b, sb, M, N, K, DG_LAYOUT_NT, scale_mode, stream,
                    a_scale_rows == 1, make_requant(cq, ld_cq, cs, out_block_rows, out_scale_mode, N));
}

static int gemm_grouped(void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a, const float* sa,
                        const uint8_t* b, const float* sb, int num_groups, const int32_t* m_indices,
                        int64_t M_tot, int64_t N, int64_t K, int scale_mode, void* stream, bool a_1x128,
                        const dg::RequantOut& rq) {
  const int v = validate_gemm_common(c, ld_c, a, ld_a, sa, b, K, sb, M_tot, N, K, scale_mode);
  if (v == kEmpty) return (num_groups < 1 || M_tot % 128 != 0) ? DG_ERR_INVALID_ARG : DG_OK;
  if (v != DG_OK) return v;
  if (!m_indices || num_groups < 1) return DG_ERR_INVALID_ARG;
  if (M_tot % 128 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
  if (N * K >= (int64_t(1) << 40)) return DG_ERR_UNSUPPORTED_SHAPE;  // one expert's B: TMA stride limit
  if (!aligned(m_indices, 16)) return DG_ERR_MISALIGNED;
  const int dev_st = check_device();
  if (dev_st != DG_OK) return dev_st;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0) return rq.q ? zero_requant_output(rq, M_tot, N, st) : zero_output(c, ld_c, M_tot, N, st);
  dg::GemmProblem p{};
  p.rq = rq;
  p.c = c;
  p.ld_c = ld_c;
  p.a = a;
  p.ld_a = ld_a;
  p.sa = sa;
  p.b = b;
  p.ld_b = K;
  p.sb = sb;
  p.m_indices = m_indices;
  p.num_groups = num_groups;
  p.M = M_tot;
  p.N = N;
  p.K = K;
  p.num_sms_cap = g_num_sms_cap.load();
  p.pow2_scales = scale_mode == DG_SCALE_UE8M0;
  p.sa_per_row = a_1x128;
  p.ld_sa = p.ld_sb = K / 128;
  return dg::launch_gemm(p, st);
}

DG_API int dg_fp8_grouped_gemm_contiguous(void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a,
                                          const float* sa, const uint8_t* b, const float* sb,
                                          int num_groups, const int32_t* m_indices, int64_t M_tot,
                                          int64_t N, int64_t K, int scale_mode, void* stream) {
  return gemm_grouped(c, ld_c, a, ld_a, sa, b, sb, num_groups, m_indices, M_tot, N, K, scale_mode, stream,
                      false, dg::RequantOut{});
}

DG_API int dg_fp8_grouped_gemm_contiguous_1x128(void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a,
                                                const float* sa, const uint8_t* b, const float* sb,
                                                int num_groups, const int32_t* m_indices, int64_t M_tot,
                                                int64_t N, int64_t K, int scale_mode, void* stream) {
  return gemm_grouped(c, ld_c, a, ld_a, sa, b, sb, num_groups, m_indices, M_tot, N, K, scale_mode, stream,
                      true, dg::RequantOut{});
}

DG_API int dg_fp8_grouped_gemm_contiguous_requant(uint8_t* cq, int64_t ld_cq, float* cs, int out_block_rows,
                                                  int out_scale_mode, const uint8_t* a, int64_t ld_a,
                                                  const float* sa, int a_scale_rows, const uint8_t* b,
                                                  const float* sb, int num_groups, const int32_t* m_indices,
                                                  int64_t M_tot, int64_t N, int64_t K, int scale_mode,
                                                  void* stream) {
  const int v = check_requant_args(cq, ld_cq, cs, out_block_rows, out_scale_mode, a_scale_rows, M_tot, N);
  if (v != DG_OK) return v;
  return gemm_grouped(cq, ld_cq, a, ld_a, sa, b, sb, num_groups, m_indices, M_tot, N, K, scale_mode, stream,
                      a_scale_rows == 1, make_requant(cq, ld_cq, cs, out_block_rows, out_scale_mode, N));
}

DG_API int dg_fp8_gemm(void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a, const float* sa,
                       const uint8_t* b, int64_t ld_b, const float* sb, int64_t M, int64_t N, int64_t K,
                       int layout, int scale_mode, void* stream) {
  if (layout < DG_LAYOUT_NT || layout > DG_LAYOUT_TT) return DG_ERR_INVALID_ARG;
  return gemm_dense(c, ld_c, a, ld_a, sa, b, ld_b, sb, M, N, K, layout, scale_mode, stream, false,
                    dg::RequantOut{});
}

DG_API int dg_fp8_gemm_requant(uint8_t* cq, int64_t ld_cq, float* cs, int out_block_rows, int out_scale_mode,
                               const uint8_t* a, int64_t ld_a, const float* sa, int a_scale_rows, const uint8_t* b,
                               int64_t ld_b, const float* sb, int64_t M, int64_t N, int64_t K, int layout,
                               int scale_mode, void* stream) {
  if (layout < DG_LAYOUT_NT || layout > DG_LAYOUT_TT) return DG_ERR_INVALID_ARG;
  const int v = check_requant_args(cq, ld_cq, cs, out_block_rows, out_scale_mode, a_scale_rows, M, N);
  if (v != DG_OK) return v;
  return gemm_dense(cq, ld_cq, a, ld_a, sa, b, ld_b, sb, M, N, K, layout, scale_mode, stream,
                    a_scale_rows == 1, make_requant(cq, ld_cq, cs, out_block_rows, out_scale_mode, N));
}

DG_API int dg_fp8_k_grouped_gemm_tn(void* c, int64_t ld_c, const uint8_t* a, int64_t ld_a, const float* sa,
                                    const uint8_t* b, int64_t ld_b, const float* sb, int num_groups,
                                    const int64_t* k_sizes, int64_t M, int64_t N, int scale_mode,
                                    void* stream) {
  if (num_groups < 1 || !k_sizes) return DG_ERR_INVALID_ARG;
  int64_t k_tot = 0;
  for (int g = 0; g < num_groups; ++g) {
    if (k_sizes[g] < 0) return DG_ERR_INVALID_ARG;
    if (k_sizes[g] % 128 != 0) return DG_ERR_UNSUPPORTED_SHAPE;
    k_tot += k_sizes[g];
    if (k_tot >= kDimLimit) return DG_ERR_UNSUPPORTED_SHAPE;
  }
  const int v = validate_gemm_rows(c, ld_c, a, ld_a, sa, b, ld_b, sb, M, N, k_tot, scale_mode, M, N);
  if (v == kEmpty) return DG_OK;
  if (v != DG_OK) return v;
  if (static_cast<int64_t>(num_groups) * M >= kDimLimit) return DG_ERR_UNSUPPORTED_SHAPE;
  const int dev_st = check_device();
  if (dev_st != DG_OK) return dev_st;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t* c16 = static_cast<uint16_t*>(c);
  if (!dg::tile_width_forced()) {
    // Every non-empty range in one launch on CTA pairs (FP32 scales, M > 128).
    dg::GemmProblem p{};
    p.c = c;
    p.ld_c = ld_c;
    p.a = a;
    p.ld_a = ld_a;
    p.sa = sa;
    p.b = b;
    p.ld_b = ld_b;
    p.sb = sb;
    p.num_groups = 1;
    p.M = M;
    p.N = N;
    p.K = k_tot;
    p.num_sms_cap = g_num_sms_cap.load();
    p.pow2_scales = scale_mode == DG_SCALE_UE8M0;
    p.a_mn = true;
    p.b_mn = true;
    p.ld_sa = p.ld_sb = k_tot / 128;
    int r = dg::launch_gemm_pair_k_grouped(p, k_sizes, num_groups, st);
    if (r != DG_ERR_UNSUPPORTED_SHAPE) {
      for (int g = 0; g < num_groups && r == DG_OK; ++g)
        if (k_sizes[g] == 0) r = zero_output(c16 + static_cast<int64_t>(g) * M * ld_c, ld_c, M, N, st);
      return r;
    }
  }
  int64_t k_off = 0;
  for (int g = 0; g < num_groups; ++g) {
    void* cg = c16 + static_cast<int64_t>(g) * M * ld_c;
    const int64_t kg = k_sizes[g];
    int r;
    if (kg == 0) {
      r = zero_output(cg, ld_c, M, N, st);
    } else {
      // Group g: C_g = A[k_off : k_off + kg]^T B[k_off : k_off + kg] with its K blocks' scales.
      dg::GemmProblem p{};
      p.c = cg;
      p.ld_c = ld_c;
      p.a = a + k_off * ld_a;
      p.ld_a = ld_a;
      p.sa = sa + k_off / 128;
      p.b = b + k_off * ld_b;
      p.ld_b = ld_b;
      p.sb = sb + k_off / 128;
      p.num_groups = 1;
      p.M = M;
      p.N = N;
      p.K = kg;
      p.num_sms_cap = g_num_sms_cap.load();
      p.pow2_scales = scale_mode == DG_SCALE_UE8M0;
      p.a_mn = true;
      p.b_mn = true;
      p.ld_sa = p.ld_sb = k_tot / 128;
      r = dg::launch_gemm(p, st);
    }
    if (r != DG_OK) return r;
    k_off += kg;
  }
  return DG_OK;
}

DG_API int dg_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  unsigned int word = 0;
  if (dg::read_and_clear_status(&word, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  if (word & dg::kStatusTimeout) return DG_ERR_TIMEOUT;
  return (word & dg::kStatusBadGroup) ? DG_ERR_BAD_GROUP : DG_OK;
}

DG_API int dg_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  const int dev_st = check_device();
  if (dev_st != DG_OK) return dev_st;
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 1000000000) limit_ns = 1000000000;
  return dg::launch_timeout_selftest(static_cast<uint64_t>(limit_ns),
                                     static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DG_OK
             : DG_ERR_CUDA;
}

}  // extern "C"
