/*
 * dgfp8.h -- C ABI of the GB300 (sm_103a) FP8 E4M3 block-scaled GEMM library.
 *
 * The library computes, on one GPU:
 *   1. 128x128 block quantization of an FP32 matrix to E4M3 codes plus one
 *      scale per block (scale = block max|x| / 448, FP32, or rounded up to a
 *      power of two), as the lpnh.cn DeepGEMM walkthrough describes in §3.1 and
 *      §4.2 (steps 1-5, round to nearest even) and §5.4 (all-zero blocks);
 *   2. the NT GEMM  C[M,N] (bf16) = sum over 128-wide K blocks kb of
 *      sa[m/128,kb] * sb[n/128,kb] * (A_kb . B_kb^T), with A[M,K] and B[N,K]
 *      E4M3 codes stored K-contiguous, FP32 accumulation (walkthrough §2.2 and
 *      §3.2; pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1 NT layout and
 *      §4.1 fp8_gemm_nt(c, a, b, a_sf, b_sf));
 *   3. the M-grouped contiguous variant for MoE experts, where each 128-row
 *      block of A belongs to one expert whose B and scales it uses (pzsr.cn
 *      page §2.3, §3.2, §3.3);
 *   4. both GEMMs with their FP32 accumulators requantized to E4M3 codes plus
 *      block scales in the epilogue instead of rounded to bf16 (walkthrough
 *      §2.2: quantize on demand at write-back; §6: fuse the scale computation
 *      into the kernel to save a round trip through memory);
 *   5. the dense GEMM in all four operand layouts NT, TN, NN, TT, and the
 *      K-grouped GEMM (pzsr.cn page §3.1: from SM100 on all four layouts;
 *      §3.2: grouping along M or along K for MoE).
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is a DEVICE pointer that the caller allocated and owns;
 *     the library allocates no device memory per call and keeps no pointer.
 *   - Matrices are row-major. `ld_*` is the row stride in ELEMENTS.
 *   - Scale arrays are row-major FP32, one value per 128x128 block, with
 *     ceil-division at ragged edges: sa is [ceil(M/128)][K/128],
 *     sb is [ceil(N/128)][K/128], quantizer scales are
 *     [ceil(rows/128)][ceil(cols/128)]. Their row stride is their width.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Every compute
 *     call is asynchronous on it; argument errors are reported synchronously
 *     and launch nothing.
 *   - Return value: a dg_status. No C++ exception crosses this boundary.
 *   - Timeouts: every wait inside a kernel is bounded; a wait that runs out sets
 *     a per-device status word and makes the kernel return early (its output is
 *     then undefined). dg_get_device_status() reads and clears that word. The
 *     compute calls return before their kernels run, so they cannot report
 *     this: a caller that must know whether a result is valid calls
 *     dg_get_device_status() after it (the tests and the benchmark do so after
 *     each check and each timed region).
 */
#ifndef DGFP8_H_
#define DGFP8_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define DG_API __declspec(dllexport)
#else
#define DG_API __attribute__((visibility("default")))
#endif

#define DG_ABI_VERSION 6u

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad mode or stride */
    DG_ERR_UNSUPPORTED_SHAPE = 2,  /* K not a multiple of 128, M_tot not a multiple of 128, dim >= 2^31 */
    DG_ERR_MISALIGNED = 3,         /* pointer or stride breaks a 16-byte (TMA) rule */
    DG_ERR_CUDA = 4,               /* a CUDA runtime call or a launch failed */
    DG_ERR_NO_DEVICE = 5,          /* no CUDA device, or the device is not sm_103 */
    DG_ERR_TIMEOUT = 6,            /* a bounded in-kernel wait ran out (see above) */
    DG_ERR_BAD_GROUP = 7           /* an M-grouped call met an expert id >= num_groups */
} dg_status;

typedef enum {
    DG_SCALE_FP32 = 0,   /* scale = fl32(max|x| / 448); 1.0 for an all-zero block */
    DG_SCALE_UE8M0 = 1   /* the FP32 scale rounded up to a power of two, >= 2^-127 */
} dg_scale_mode;

/* Operand layouts of dg_fp8_gemm, named as op(A) op(B) in C = op(A) . op(B):
 * N = stored as the product uses it, T = stored transposed. With logical
 * A (M x K) and B (K x N):
 *   NT: a [M][ld_a] (K contiguous), b [N][ld_b] (K contiguous)  -- C = A . B^T, the default layout
 *   TN: a [K][ld_a] (M contiguous), b [K][ld_b] (N contiguous)
 *   NN: a [M][ld_a] (K contiguous), b [K][ld_b] (N contiguous)
 *   TT: a [K][ld_a] (M contiguous), b [N][ld_b] (K contiguous) */
typedef enum {
    DG_LAYOUT_NT = 0,
    DG_LAYOUT_TN = 1,
    DG_LAYOUT_NN = 2,
    DG_LAYOUT_TT = 3
} dg_layout;

/* Element type of a matrix handed to the row-wise quantizer. */
typedef enum {
    DG_INPUT_FP32 = 0,
    DG_INPUT_BF16 = 1   /* raw 16-bit bfloat16 storage */
} dg_input_dtype;

/* ABI version of the loaded library (DG_ABI_VERSION at build time). */
DG_API uint32_t dg_get_abi_version(void);

/* Static English text for a status code (never NULL). */
DG_API const char *dg_status_string(int status);

/* Row alignment that the M-grouped contiguous layout needs: every expert's
 * rows start on a multiple of this (128). pzsr.cn page §3.3 names the query
 * get_mk_alignment_for_contiguous_layout(). */
DG_API int dg_get_mk_alignment_for_contiguous_layout(void);

/* Cap the number of SMs the GEMM's persistent grid uses (0 = all SMs), the
 * DG_SET_NUM_SMS knob of pzsr.cn page §3.3. Applies to later calls from every
 * thread. Single-row GEMMs (M = 1) stream B over every SM when no cap is set
 * and run on the capped persistent kernels when one is. Returns
 * DG_ERR_INVALID_ARG for n < 0. */
DG_API int dg_set_num_sms(int n);

/* The current cap (0 = all SMs). */
DG_API int dg_get_num_sms(void);

/* Block quantizer (walkthrough §4.2 steps 1-5, §3.1, §5.4).
 *   x       [rows][ld_x] FP32, finite values (NaN/Inf give unspecified codes)
 *   q       [rows][ld_q] E4M3 codes out: RNE of fl32(x / s), saturated to +-448,
 *           the sign of zero kept
 *   scales  [ceil(rows/128)][ceil(cols/128)] FP32 out
 *   scale_mode  a dg_scale_mode
 * rows == 0 or cols == 0 is a no-op. Needs ld_x >= cols and ld_q >= cols.
 * Any alignment works; 16-byte aligned x with ld_x % 4 == 0, and q with
 * ld_q % 4 == 0, take the vectorized path. */
DG_API int dg_quantize_fp8_block(const float *x, int64_t rows, int64_t cols, int64_t ld_x,
                                 uint8_t *q, int64_t ld_q, float *scales,
                                 int scale_mode, void *stream);

/* Row-wise quantizer: one scale per row and 128-column block, the per-token
 * activation scaling that sits beside 128x128 weight scales (walkthrough §2.3:
 * the block shape trades accuracy against overhead; pzsr.cn page §3.1). The
 * steps are those of dg_quantize_fp8_block with blocks of 1 x 128.
 *   x       [rows][ld_x] elements of x_dtype (a dg_input_dtype), finite values;
 *           bfloat16 inputs are widened to FP32 exactly
 *   q       [rows][ld_q] E4M3 codes out
 *   scales  [rows][ceil(cols/128)] FP32 out
 *   scale_mode  a dg_scale_mode
 * rows == 0 or cols == 0 is a no-op. Needs ld_x >= cols and ld_q >= cols.
 * Any alignment works; x 16-byte aligned with ld_x * element size a multiple
 * of 16 bytes, and q 4-byte aligned with ld_q % 4 == 0, take the vectorized
 * path. */
DG_API int dg_quantize_fp8_1x128(const void *x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x,
                                 uint8_t *q, int64_t ld_q, float *scales,
                                 int scale_mode, void *stream);

/* Dense NT GEMM (walkthrough §2.2, §3.2; pzsr.cn page §3.1, §4.1).
 *   c   [M][ld_c] bf16 out (raw 16-bit storage), rounded to nearest even
 *   a   [M][ld_a] E4M3 codes, K contiguous;  sa [ceil(M/128)][K/128] FP32
 *   b   [N][ld_b] E4M3 codes, K contiguous;  sb [ceil(N/128)][K/128] FP32
 *   scale_mode  DG_SCALE_UE8M0 promises that every scale is a power of two
 *               >= 2^-127 (it is not checked): for M > 128 the tensor core then
 *               applies each scale's exponent itself (block-scaled MMA), so a
 *               scale that is not a power of two acts as its power-of-two
 *               floor. DG_SCALE_FP32 accepts any finite scale.
 * Needs K % 128 == 0, ld_a >= K, ld_b >= K, ld_c >= N; a, b and c 16-byte
 * aligned, ld_a and ld_b multiples of 16, ld_c a multiple of 8; sa, sb 4-byte
 * aligned. M == 0 or N == 0 is a no-op; K == 0 writes zeros. */
DG_API int dg_fp8_gemm_nt(void *c, int64_t ld_c,
                          const uint8_t *a, int64_t ld_a, const float *sa,
                          const uint8_t *b, int64_t ld_b, const float *sb,
                          int64_t M, int64_t N, int64_t K,
                          int scale_mode, void *stream);

/* Dense NT GEMM with one A scale per row and K block (row-wise activation
 * scales from dg_quantize_fp8_1x128; pzsr.cn page §3.1): as dg_fp8_gemm_nt
 * with
 *   sa  [M][K/128] FP32: the scale of A[m, 128 kb .. 128 kb + 127]
 * so that C[m, n] = bf16( sum_kb sa[m, kb] * sb[n/128, kb] * sum_{k in kb} A[m,k] B[n,k] ).
 * Same size, stride and alignment rules as dg_fp8_gemm_nt. */
DG_API int dg_fp8_gemm_nt_1x128(void *c, int64_t ld_c,
                                const uint8_t *a, int64_t ld_a, const float *sa,
                                const uint8_t *b, int64_t ld_b, const float *sb,
                                int64_t M, int64_t N, int64_t K,
                                int scale_mode, void *stream);

/* M-grouped contiguous GEMM for MoE experts (pzsr.cn page §2.3, §3.2, §3.3).
 *   c          [M_tot][ld_c] bf16 out
 *   a          [M_tot][ld_a] E4M3 codes; sa [M_tot/128][K/128] FP32
 *   b          [num_groups][N][K] E4M3 codes, packed (row stride K)
 *   sb         [num_groups][ceil(N/128)][K/128] FP32
 *   m_indices  [M_tot] int32 on the device: the expert of each row, or -1 for a
 *              padding row. Rows of one 128-row block carry one expert id or -1
 *              (each expert's rows start on a multiple of 128). Output rows with
 *              -1 are written as zeros; a block made only of -1 rows is zero.
 *              A block whose id is >= num_groups reads no B or sb, is written
 *              as zeros, and sets the status that dg_get_device_status()
 *              then reports as DG_ERR_BAD_GROUP.
 * Needs M_tot % 128 == 0 and the alignment rules of dg_fp8_gemm_nt (with
 * ld_b = K). */
DG_API int dg_fp8_grouped_gemm_contiguous(void *c, int64_t ld_c,
                                          const uint8_t *a, int64_t ld_a, const float *sa,
                                          const uint8_t *b, const float *sb, int num_groups,
                                          const int32_t *m_indices,
                                          int64_t M_tot, int64_t N, int64_t K,
                                          int scale_mode, void *stream);

/* M-grouped contiguous GEMM with one A scale per row and K block:
 * as dg_fp8_grouped_gemm_contiguous with sa [M_tot][K/128] FP32. */
DG_API int dg_fp8_grouped_gemm_contiguous_1x128(void *c, int64_t ld_c,
                                                const uint8_t *a, int64_t ld_a, const float *sa,
                                                const uint8_t *b, const float *sb, int num_groups,
                                                const int32_t *m_indices,
                                                int64_t M_tot, int64_t N, int64_t K,
                                                int scale_mode, void *stream);

/* Dense NT GEMM with the output requantized in the epilogue (walkthrough §2.2
 * "quantize on demand at write-back", §6 fusing the scale computation): the
 * FP32 accumulator value v[m, n] of dg_fp8_gemm_nt (before any bf16 rounding)
 * is quantized by the steps of dg_quantize_fp8_block with blocks of
 * out_block_rows x 128 elements of C:
 *   cq  [M][ld_cq] E4M3 codes out: RNE of fl32(v / s), saturated to +-448
 *   cs  scales out, FP32, s = fl32(max|v| / 448) over the block (1.0 for an
 *       all-zero block; rounded up to a power of two with out_scale_mode =
 *       DG_SCALE_UE8M0):
 *         out_block_rows = 1:   [M][ceil(N/128)]  (per-row activation scales,
 *                               the sa layout of dg_fp8_gemm_nt_1x128)
 *         out_block_rows = 128: [ceil(M/128)][ceil(N/128)]
 *   a_scale_rows  128: sa is [ceil(M/128)][K/128] (dg_fp8_gemm_nt);
 *                 1:   sa is [M][K/128] (dg_fp8_gemm_nt_1x128)
 * The operands, scale_mode and their rules are those of dg_fp8_gemm_nt. cq
 * must be 16-byte aligned with ld_cq >= N a multiple of 16; cs 4-byte aligned.
 * Bad out_block_rows, a_scale_rows or out_scale_mode give DG_ERR_INVALID_ARG.
 * M == 0 or N == 0 is a no-op; K == 0 writes codes 0 and scales 1. */
DG_API int dg_fp8_gemm_nt_requant(uint8_t *cq, int64_t ld_cq, float *cs, int out_block_rows,
                                  int out_scale_mode,
                                  const uint8_t *a, int64_t ld_a, const float *sa, int a_scale_rows,
                                  const uint8_t *b, int64_t ld_b, const float *sb,
                                  int64_t M, int64_t N, int64_t K,
                                  int scale_mode, void *stream);

/* M-grouped contiguous GEMM with the output requantized as in
 * dg_fp8_gemm_nt_requant. Padding rows (m_indices -1) get codes 0 and, with
 * out_block_rows = 1, scale 1; they count as zeros in a 128 x 128 block.
 * sa is [M_tot / a_scale_rows][K/128]; the other arguments and rules are those
 * of dg_fp8_grouped_gemm_contiguous. */
DG_API int dg_fp8_grouped_gemm_contiguous_requant(uint8_t *cq, int64_t ld_cq, float *cs,
                                                  int out_block_rows, int out_scale_mode,
                                                  const uint8_t *a, int64_t ld_a, const float *sa,
                                                  int a_scale_rows,
                                                  const uint8_t *b, const float *sb, int num_groups,
                                                  const int32_t *m_indices,
                                                  int64_t M_tot, int64_t N, int64_t K,
                                                  int scale_mode, void *stream);

/* Dense GEMM in any of the four layouts (pzsr.cn page §3.1; see dg_layout):
 *   C[m, n] = bf16( sum_kb sa[m/128, kb] * sb[n/128, kb] * sum_{k in kb} A(m, k) B(k, n) )
 * where A(m, k) and B(k, n) are the logical elements wherever the layout
 * stores them. The scales are per 128 x 128 block of the logical operands
 * whatever the layout: sa [ceil(M/128)][K/128], sb [ceil(N/128)][K/128].
 * ld_a >= K (A stored N) or >= M (A stored T); ld_b >= K (B stored T) or
 * >= N (B stored N); every other rule is that of dg_fp8_gemm_nt, which equals
 * this call with layout DG_LAYOUT_NT. A bad layout gives DG_ERR_INVALID_ARG. */
DG_API int dg_fp8_gemm(void *c, int64_t ld_c,
                       const uint8_t *a, int64_t ld_a, const float *sa,
                       const uint8_t *b, int64_t ld_b, const float *sb,
                       int64_t M, int64_t N, int64_t K,
                       int layout, int scale_mode, void *stream);

/* Dense GEMM in any layout with the output requantized in the epilogue: the
 * layouts, strides and scales of dg_fp8_gemm, the output arguments
 * (cq, ld_cq, cs, out_block_rows, out_scale_mode) and a_scale_rows of
 * dg_fp8_gemm_nt_requant, which equals this call with layout DG_LAYOUT_NT.
 * Row-wise A scales (a_scale_rows = 1) are [M][K/128] in every layout. */
DG_API int dg_fp8_gemm_requant(uint8_t *cq, int64_t ld_cq, float *cs, int out_block_rows,
                               int out_scale_mode,
                               const uint8_t *a, int64_t ld_a, const float *sa, int a_scale_rows,
                               const uint8_t *b, int64_t ld_b, const float *sb,
                               int64_t M, int64_t N, int64_t K,
                               int layout, int scale_mode, void *stream);

/* K-grouped GEMM in the TN layout (pzsr.cn page §3.2: grouping along K, the
 * shape of MoE weight gradients): the K extent is cut into num_groups
 * consecutive ranges, and group g gets its own output
 *   C_g[m, n] = bf16( sum over the K blocks kb of range g of
 *                     sa[m/128, kb] * sb[n/128, kb] * sum_{k in kb} A[k][m] B[k][n] )
 *   c        [num_groups][M][ld_c] bf16 out (group g at c + g * M * ld_c)
 *   a        [K_tot][ld_a] E4M3, M contiguous (ld_a >= M); sa [ceil(M/128)][K_tot/128]
 *   b        [K_tot][ld_b] E4M3, N contiguous (ld_b >= N); sb [ceil(N/128)][K_tot/128]
 *   k_sizes  HOST array of num_groups sizes, each >= 0 and a multiple of 128
 *            (DG_ERR_UNSUPPORTED_SHAPE otherwise); K_tot is their sum. A group
 *            of size 0 gets C_g = 0.
 * Alignment rules as dg_fp8_gemm_nt. With M > 128 every non-empty group runs
 * in one launch on CTA pairs (at most 256 non-empty groups; more take the
 * per-group path): FP32 scales on the promotion kernel, power-of-two scales on
 * the block-scaled one. Otherwise the groups run one after another on
 * `stream`. */
DG_API int dg_fp8_k_grouped_gemm_tn(void *c, int64_t ld_c,
                                    const uint8_t *a, int64_t ld_a, const float *sa,
                                    const uint8_t *b, int64_t ld_b, const float *sb,
                                    int num_groups, const int64_t *k_sizes,
                                    int64_t M, int64_t N, int scale_mode, void *stream);

/* Synchronize `stream`, then take and clear the current device's status word
 * in one atomic step (a kernel on another stream that sets it meanwhile is
 * reported by this call or the next, never lost). Returns DG_ERR_TIMEOUT if a
 * kernel's bounded wait ran out since the last call, else DG_ERR_BAD_GROUP if
 * an M-grouped call met an expert id >= num_groups, DG_ERR_CUDA if the stream
 * reports an error, else DG_OK. The word is one per device, shared by all
 * streams: it does not say which call set it. */
DG_API int dg_get_device_status(void *stream);

/* Self-test of the timeout path: launches one block whose wait on a barrier
 * that nothing arrives at runs out after `limit_ns` nanoseconds (clamped to
 * [1e3, 1e9]); the block then records the timeout and returns. Follow with
 * dg_get_device_status(), which must report DG_ERR_TIMEOUT. */
DG_API int dg_selftest_wait_timeout(int64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DGFP8_H_ */
