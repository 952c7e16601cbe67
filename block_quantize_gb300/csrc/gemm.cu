// gemm.cu -- persistent FP8 (E4M3) block-scaled NT GEMM for sm_103a, dense and
// M-grouped contiguous.
//
//   C[m, n] = bf16( sum_kb sa[m/128, kb] * sb[n/128, kb] * sum_{k in kb} A[m,k] B[n,k] )
//
// The method: E4M3 operands with one FP32 scale per 128x128 block, partial
// products restored with scale_a * scale_b and accumulated in FP32 (lpnh.cn
// DeepGEMM walkthrough §2.2, §3.1, §3.2); NT layout and the
// fp8_gemm_nt(c, a, b, a_sf, b_sf) call (pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库
// 解析" §3.1, §4.1); grouped GEMM over MoE experts (same page §2.3, §3.2).
//
// Blackwell design (not the pages' Hopper pipeline):
//   * one CTA per SM, persistent over 128 x BN output tiles in a grouped
//     raster (16 M-blocks at a time) so the tiles in flight share A and B in L2;
//   * warp 0 issues TMA loads of 128x128-byte A and BNx128-byte B tiles
//     (128-byte swizzle, out-of-bounds rows zero-filled) into a ring of stages
//     guarded by full/empty mbarriers;
//   * warps 1..kIssuers take turns, one K block each, issuing the four
//     tcgen05.mma kind::f8f6f4 (K = 32 each) of a K block into its own TMEM
//     buffer, then committing to the stage's empty barrier and the buffer's
//     full barrier. One issuing thread needs ~70 cycles per MMA and ~150 per
//     mbarrier wait (measured on GB300), more than a K block's MMA time, so the
//     issue work is spread over several warps;
//   * the epilogue warpgroups (one per column slice) read each K block's
//     partial sums from TMEM (tcgen05.ld), release the buffer and promote them
//     in FP32 registers: acc += (sa * sb) * partial. After the last K block each
//     warp rounds its 32 x 64 box to bf16 into 128-byte-swizzled shared memory
//     and writes it with a TMA store (clipped at the M and N edges).
// Every mbarrier wait is bounded; on a timeout the CTA raises an abort flag,
// records it in the device status word, drains its in-flight copies and MMAs,
// frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "dg_device.cuh"
#include "dg_encode.cuh"
#include "dg_internal.h"
#include "../../include/dgfp8.h"

namespace dg {

__device__ unsigned int g_status_word;
__device__ unsigned int g_status_taken;  // the word's value at the last read-and-clear

namespace {

constexpr int kBM = 128;          // tile rows (tcgen05 M)
constexpr int kBK = 128;          // K block = scale block = one 128-byte swizzle row
constexpr int kMaxStages = 32;
constexpr int kGroupM = 16;       // raster group height in M-blocks
constexpr uint32_t kATileBytes = kBM * kBK;    // what one MMA reads for A
constexpr size_t kMinSmemPerCta = 120 * 1024;  // > half the SM's shared memory
constexpr size_t kMaxDynSmem = 227 * 1024;
constexpr uint32_t kWarpOutBytes = 32 * 32 * 2;  // one warp's 32 x 32 bf16 output box

struct GemmArgs {
  __nv_bfloat16* c;
  int sa_per_row;  // sa is [M][K/128] instead of [ceil(M/128)][K/128]
  int64_t ld_c;
  const float* sa;
  const float* sb;
  const int32_t* m_indices;
  int M, N;
  int num_kb;      // K / 128
  int ld_sa, ld_sb;  // row strides of sa and sb (floats)
  uint32_t idesc;  // MMA instruction descriptor (shape and operand majorness)
  int a_mn, b_mn;  // MN-major A ([K][M]) / B ([K][N]) tiles
  int num_mb;      // ceil(M / 128)
  int num_nb;      // ceil(N / BN)
  int nbs;         // ceil(N / 128): rows of one expert's sb
  int num_groups;  // experts of an M-grouped call (ids outside [0, num_groups) are skipped)
  int num_stages;
  uint32_t a_stage_bytes;  // smem bytes of one A stage (>= the A box, 1024-aligned)
  uint32_t a_box_bytes;    // bytes one A TMA box delivers
  uint64_t wait_limit_ns;
};

// Arguments of the requantizing kernels. A separate type: with the extra
// fields in the common struct the grouped bf16 kernel ran ~7 % slower (measured).
struct GemmArgsQ : GemmArgs {
  RequantOut rq;   // E4M3 output
};
template <bool kQ>
using GemmArgsT = std::conditional_t<kQ, GemmArgsQ, GemmArgs>;

template <int BN>
struct Cfg {
  // Wide tiles: four epilogue warpgroups, 64 columns and accumulators each.
  static constexpr int kEpiWG = (BN == 256) ? 4 : 2;
  // Warps 1 and 2 take turns issuing the MMAs of successive K blocks. With an
  // even number of TMEM buffers and of stages, issuer i only ever touches the
  // buffers and stages with index parity i, so each barrier has one waiter
  // that sees its phases in order (a parity wait cannot tell phase n from n-2).
  static constexpr int kIssuers = 2;
  static constexpr int kFirstEpiWarp = 1 + kIssuers;  // warp 0 produces
  static constexpr int kEpiWarps = 4 * kEpiWG;
  static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
  static constexpr uint32_t kBTileBytes = BN * kBK;
  static constexpr int kNumPBuf = (512 / BN) < 8 ? (512 / BN) : 8;
  static constexpr uint32_t kTmemCols = kNumPBuf * BN;  // power of two in [32, 512]
  static constexpr int kCols = BN / kEpiWG;             // columns per epilogue thread
  // Columns per tcgen05.ld: 16 on wide tiles, whose 19 warps leave 96 registers a thread.
  static constexpr int kChunk = (BN == 256) ? 16 : (kCols < 32 ? kCols : 32);
  static constexpr int kBatch = (BN == 256) ? 1 : (kCols / kChunk);  // loads per wait
  static constexpr int kUnroll =
      (32 / kCols) > 1 ? ((32 / kCols) < kNumPBuf / 2 ? 32 / kCols : kNumPBuf / 2) : 1;
  // 64-column slices leave through shared memory and TMA (each warp stages its
  // 32 x 64 slice as two 32 x 32 boxes in turn); narrow tiles (small M) store
  // straight from registers.
  static constexpr bool kTmaStore = (kCols == 64);
  static constexpr uint32_t kOutBytes = kTmaStore ? kEpiWarps * kWarpOutBytes : 0;
  static constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, BN);
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 N for M=128");
  static_assert(kCols % (kChunk * kBatch) == 0, "epilogue batching");
  static_assert(kThreads <= 1024, "CTA size");
  static_assert(kNumPBuf % kIssuers == 0, "buffer ownership by issuer");
};

// Shared memory behind the operand ring for the output: bf16 staging boxes, or
// with requantization (64-column slices only) the slices' maxima exchange.
template <int BN, bool kQ>
__host__ __device__ constexpr uint32_t out_bytes() {
  static_assert(!kQ || Cfg<BN>::kCols == 64, "the requantizing epilogue takes 64-column slices");
  return kQ ? requant_smem_bytes(Cfg<BN>::kEpiWarps) : Cfg<BN>::kOutBytes;
}

// Output tile of persistent iteration t: grouped raster, M fastest inside a
// group of kGroupM M-blocks.
__device__ __forceinline__ void tile_coords(int t, int num_mb, int num_nb, int& mb, int& nb) {
  const int per_group = kGroupM * num_nb;
  const int grp = t / per_group;
  const int first = grp * kGroupM;
  const int gm = min(kGroupM, num_mb - first);
  const int r = t - grp * per_group;
  mb = first + r % gm;
  nb = r / gm;
}


// Bounded wait that ignores the abort flag (used while draining).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) break;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int BN, bool kGrouped, bool kQ>
__global__ void __launch_bounds__(Cfg<BN>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_c, const GemmArgsT<kQ> args) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = args.num_stages;
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + static_cast<size_t>(S) * args.a_stage_bytes;
  // An MMA always reads a full 128-row A tile (16 KB) from its stage's start;
  // rows past a short A box are junk that only feeds output rows >= M. Keep the
  // read of the last stage inside the allocation.
  size_t tail_off = static_cast<size_t>(S) * (args.a_stage_bytes + C::kBTileBytes);
  const size_t a_read_end = static_cast<size_t>(S - 1) * args.a_stage_bytes + kATileBytes;
  if (a_read_end > tail_off) tail_off = a_read_end;
  uint8_t* smem_out = smem + tail_off;  // kEpiWarps boxes of kWarpOutBytes (kTmaStore)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_out + out_bytes<BN, kQ>());
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + kMaxStages;
  uint64_t* tfull_bar = bars + 2 * kMaxStages;
  uint64_t* tempty_bar = tfull_bar + C::kNumPBuf;
  uint64_t* drain_bar = tempty_bar + C::kNumPBuf;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = args.wait_limit_ns;
  unsigned int* status = &g_status_word;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < C::kNumPBuf; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), C::kEpiWarps);
    }
    mbar_init(smem_u32(drain_bar), C::kIssuers);
    if constexpr (kQ) requant_xchg_init(smem_out, C::kEpiWarps);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    if (C::kTmaStore) tma_prefetch_desc(&tmap_c);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  const int num_tiles = args.num_mb * args.num_nb;
  uint32_t loads_issued = 0;  // producer: K-block loads issued

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, args.num_mb, args.num_nb, mb, nb);
      int g = 0;
      if constexpr (kGrouped) {
        g = m_block_group(args.m_indices, mb, lane);
        if (g < 0 || g >= args.num_groups) continue;
      }
      for (int kb = 0; kb < args.num_kb; ++kb, ++it) {
        const uint32_t stage = it % S;
        const uint32_t par = (it / S) & 1u;
        if (lane == 0) {
          ok = mbar_wait(smem_u32(&empty_bar[stage]), par ^ 1u, abort_flag, status, limit);
          if (ok) {
            const uint32_t fb = smem_u32(&full_bar[stage]);
            mbar_arrive_expect_tx(fb, args.a_box_bytes + C::kBTileBytes);
            // Grouped operands are K-major: no layout branches in that instantiation.
            tma_load_operand(smem_u32(smem_a + stage * args.a_stage_bytes), &tmap_a, fb, kb * kBK, mb * kBM,
                             kGrouped ? 0u : static_cast<uint32_t>(args.a_mn));
            const uint32_t bdst = smem_u32(smem_b + stage * C::kBTileBytes);
            if constexpr (kGrouped) {
              tma_load_3d(bdst, &tmap_b, fb, kb * kBK, nb * BN, g);
            } else if (args.b_mn) {
              // MN-major B: 128-column boxes (one 128-byte swizzle atom column each), 16 KB apart.
#pragma unroll
              for (int h = 0; h < (BN >= 128 ? BN / 128 : 1); ++h)
                tma_load_2d(bdst + h * 16384u, &tmap_b, fb, nb * BN + h * 128, kb * kBK);
            } else {
              tma_load_2d(bdst, &tmap_b, fb, kb * kBK, nb * BN);
            }
            ++loads_issued;
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp <= C::kIssuers) {
    // ----------------------------------------------------------- MMA issue --
    // This warp issues K blocks it with it % kIssuers == warp - 1; K block it
    // accumulates into TMEM buffer it % kNumPBuf.
    const uint32_t me = static_cast<uint32_t>(warp - 1);
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, args.num_mb, args.num_nb, mb, nb);
      if constexpr (kGrouped) {
        const int g = m_block_group(args.m_indices, mb, lane);
        if (g < 0 || g >= args.num_groups) continue;
      }
      for (int kb = 0; kb < args.num_kb; ++kb, ++it) {
        if (it % C::kIssuers != me) continue;
        const uint32_t stage = it % S;
        const uint32_t par = (it / S) & 1u;
        const uint32_t buf = it % C::kNumPBuf;
        const uint32_t bpar = (it / C::kNumPBuf) & 1u;
        if (lane == 0) {
          // The buffer's previous use has been read by every epilogue warp, and
          // the stage's operands have landed.
          ok = mbar_wait(smem_u32(&tempty_bar[buf]), bpar ^ 1u, abort_flag, status, limit) &&
               mbar_wait(smem_u32(&full_bar[stage]), par, abort_flag, status, limit);
          if (ok) {
            tc_fence_after();
            const uint32_t d = tmem_base + buf * BN;
            if constexpr (kGrouped) {
              // K-major operands: 32 E4M3 values = 32 bytes further along the swizzled row.
              const uint64_t adesc = sw128_kmajor_desc(smem_u32(smem_a + stage * args.a_stage_bytes));
              const uint64_t bdesc = sw128_kmajor_desc(smem_u32(smem_b + stage * C::kBTileBytes));
#pragma unroll
              for (int k = 0; k < kBK / 32; ++k) mma_e4m3(d, adesc + 2u * k, bdesc + 2u * k, C::kIdesc, k > 0 ? 1u : 0u);
            } else {
              // MN-major tiles advance by four 8-row groups per MMA.
              const OperandTile at{static_cast<uint32_t>(args.a_mn), 128u}, bt{static_cast<uint32_t>(args.b_mn), 128u};
              const uint64_t adesc = at.desc(smem_u32(smem_a + stage * args.a_stage_bytes));
              const uint64_t bdesc = bt.desc(smem_u32(smem_b + stage * C::kBTileBytes));
#pragma unroll
              for (int k = 0; k < kBK / 32; ++k)
                mma_e4m3(d, adesc + at.kstep() * k, bdesc + bt.kstep() * k, args.idesc, k > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&empty_bar[stage]));
            mma_commit(smem_u32(&tfull_bar[buf]));
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - C::kFirstEpiWarp;
    const int part = ew / 4;               // which slice of the tile's columns
    const int lg = warp & 3;               // TMEM lane quadrant this warp may access
    const int row_in_tile = lg * 32 + lane;
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(lg * 32) << 16);
    constexpr int kCols = C::kCols;
    constexpr int kU = C::kUnroll;
    constexpr int kPer = C::kChunk * C::kBatch;  // columns per load-wait round
    uint8_t* out_box = smem_out + ew * kWarpOutBytes;  // this warp's 32 x 64 bf16 box
    bool stores_issued = false;
    uint32_t it = 0;
    bool ok = true;
    bool ready = false;  // the full barrier of K block `it` is known complete
    uint32_t tl = 0;     // tiles done by this CTA
    for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tl) {
      int mb, nb;
      tile_coords(t, args.num_mb, args.num_nb, mb, nb);
      int g = 0;
      if constexpr (kGrouped) {
        g = m_block_group(args.m_indices, mb, lane);
        // An id past the last expert: the block is written as zeros, no B or sb
        // of that id is read, and the status word records it.
        if (g >= args.num_groups && ew == 0 && lane == 0) atomicOr(status, kStatusBadGroup);
      }
      const bool skip = kGrouped && (g < 0 || g >= args.num_groups);
      const int col0 = nb * BN + part * kCols;
      const bool part_valid = col0 < args.N;
      const int sb_block = min(col0 / kBK, args.nbs - 1);
      // This thread's row's scales (rows past M read the last row's).
      const float* sa_row =
          args.sa + static_cast<int64_t>(args.sa_per_row ? min(mb * kBM + row_in_tile, args.M - 1) : mb) * args.ld_sa;
      const float* sb_row =
          args.sb + (static_cast<int64_t>(g) * args.nbs + sb_block) * args.ld_sb;

      // FP32 accumulators, two columns per 64-bit register (f32x2 FMA).
      uint64_t acc[kCols / 2];
#pragma unroll
      for (int j = 0; j < kCols / 2; ++j) acc[j] = 0ull;

      if (!skip) {
        for (int kb = 0; kb < args.num_kb && ok; kb += kU) {
          const int cnt = min(kU, args.num_kb - kb);
          float s[kU];
#pragma unroll
          for (int u = 0; u < kU; ++u)
            s[u] = (u < cnt && part_valid) ? __ldg(sa_row + kb + u) * __ldg(sb_row + kb + u) : 0.f;
          bool w = true;
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            if (u < cnt && !(u == 0 && ready)) {
              const uint32_t buf = (it + u) % C::kNumPBuf;
              const uint32_t bpar = ((it + u) / C::kNumPBuf) & 1u;
              w = w && mbar_wait(smem_u32(&tfull_bar[buf]), bpar, abort_flag, status, limit);
            }
          }
          ok = __all_sync(0xFFFFFFFFu, w);
          if (!ok) break;
          tc_fence_after();
          if constexpr (kU > 1) {
            // Narrow tiles: the partials of kU K blocks at once.
            uint32_t r[kU][kCols];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              if (u < cnt) {
                const uint32_t col = ((it + u) % C::kNumPBuf) * BN + part * kCols;
                tmem_ld<kCols>(tmem_row + col, &r[u][0]);
              }
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int u = 0; u < kU; ++u)
                if (u < cnt) mbar_arrive(smem_u32(&tempty_bar[(it + u) % C::kNumPBuf]));
            }
            ready = false;
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              if (u < cnt) {
                const uint64_t s2 = f32x2(__float_as_uint(s[u]), __float_as_uint(s[u]));
#pragma unroll
                for (int j = 0; j < kCols / 2; ++j) ffma2(acc[j], s2, f32x2(r[u][2 * j], r[u][2 * j + 1]));
              }
            }
          } else {
            // kPer columns per round (one wait::ld per round) to bound registers.
            const uint32_t col = (it % C::kNumPBuf) * BN + part * kCols;
#pragma unroll
            for (int rd = 0; rd < kCols / kPer; ++rd) {
              uint32_t r[kPer];
#pragma unroll
              for (int b2 = 0; b2 < C::kBatch; ++b2)
                tmem_ld<C::kChunk>(tmem_row + col + rd * kPer + b2 * C::kChunk, &r[b2 * C::kChunk]);
              tmem_wait_ld();
              if (rd == kCols / kPer - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[it % C::kNumPBuf]));
                // Test the next K block's buffer now: the test's latency hides
                // behind the multiply-adds below.
                const uint32_t nx = it + 1;
                ready = mbar_test(smem_u32(&tfull_bar[nx % C::kNumPBuf]), (nx / C::kNumPBuf) & 1u);
              }
              const uint64_t s2 = f32x2(__float_as_uint(s[0]), __float_as_uint(s[0]));
#pragma unroll
              for (int j = 0; j < kPer / 2; ++j)
                ffma2(acc[(rd * kPer) / 2 + j], s2, f32x2(r[2 * j], r[2 * j + 1]));
            }
          }
          it += cnt;
        }
        if (!ok) break;
      }

      const int row = mb * kBM + row_in_tile;
      bool zero_row = skip;
      if constexpr (kGrouped) zero_row = zero_row || (row < args.M && __ldg(args.m_indices + row) < 0);
      if constexpr (kQ) {
        // Padding rows of the grouped layout are written as zeros (scale 1).
        if (!requant_store_slice<C::kEpiWarps>(acc, row < args.M && !zero_row, kGrouped, mb * kBM + lg * 32, args.M,
                                               args.N, col0, ew, lane, tl, smem_out, args.rq, &tmap_c,
                                               requant_box(smem_out, C::kEpiWarps, ew), stores_issued, abort_flag,
                                               status, limit)) {
          ok = false;
          break;
        }
      } else if constexpr (C::kTmaStore) {
        // bf16 row segment -> this warp's 64-byte-swizzled 32 x 32 box (16-byte
        // chunk c of row r at chunk c ^ ((r / 2) % 4)) -> TMA store at
        // (col0 + 32 h, mb*128 + lg*32), clipped at M and N; the two halves
        // of the slice share the box in turn. Only this warp touches it.
        // A box that crosses column N is written element by element instead:
        // the swizzled store clips N only to whole 16-byte chunks.
        const int row0 = mb * kBM + lg * 32;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int bcol = col0 + 32 * h;
          if (bcol + 32 > args.N) {
            if (row < args.M && bcol < args.N) {
              __nv_bfloat16* crow = args.c + static_cast<int64_t>(row) * args.ld_c;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float2 v = zero_row ? make_float2(0.f, 0.f) : f32x2_split(acc[h * 16 + j]);
                if (bcol + 2 * j < args.N) crow[bcol + 2 * j] = __float2bfloat16_rn(v.x);
                if (bcol + 2 * j + 1 < args.N) crow[bcol + 2 * j + 1] = __float2bfloat16_rn(v.y);
              }
            }
            continue;
          }
          if (lane == 0 && stores_issued) bulk_wait_read_all();  // the last store has read the box
          __syncwarp();
          uint8_t* my_row = out_box + lane * 64;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 pk;
            const uint64_t* a2 = &acc[h * 16 + c * 4];
            const float2 v0 = f32x2_split(a2[0]), v1 = f32x2_split(a2[1]);
            const float2 v2 = f32x2_split(a2[2]), v3 = f32x2_split(a2[3]);
            pk.x = zero_row ? 0u : pack_bf16x2(v0.x, v0.y);
            pk.y = zero_row ? 0u : pack_bf16x2(v1.x, v1.y);
            pk.z = zero_row ? 0u : pack_bf16x2(v2.x, v2.y);
            pk.w = zero_row ? 0u : pack_bf16x2(v3.x, v3.y);
            *reinterpret_cast<uint4*>(my_row + ((c ^ ((lane >> 1) & 3)) << 4)) = pk;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && part_valid && row0 < args.M) {
            tma_store_2d(&tmap_c, smem_u32(out_box), bcol, row0);
            bulk_commit();
            stores_issued = true;
          }
        }
      } else {
        // Narrow tiles: store this thread's row segment directly.
        if (row < args.M && part_valid) {
          __nv_bfloat16* crow = args.c + static_cast<int64_t>(row) * args.ld_c + col0;
#pragma unroll
          for (int j = 0; j < kCols; j += 8) {
            float v[8];
#pragma unroll
            for (int t2 = 0; t2 < 8; t2 += 2) {
              const float2 pr = f32x2_split(acc[(j + t2) / 2]);
              v[t2] = zero_row ? 0.f : pr.x;
              v[t2 + 1] = zero_row ? 0.f : pr.y;
            }
            if (col0 + j + 8 <= args.N) {
              uint4 pk;
              pk.x = pack_bf16x2(v[0], v[1]);
              pk.y = pack_bf16x2(v[2], v[3]);
              pk.z = pack_bf16x2(v[4], v[5]);
              pk.w = pack_bf16x2(v[6], v[7]);
              *reinterpret_cast<uint4*>(crow + j) = pk;
            } else {
#pragma unroll
              for (int t2 = 0; t2 < 8; ++t2)
                if (col0 + j + t2 < args.N) crow[j + t2] = __float2bfloat16_rn(v[t2]);
            }
          }
        }
      }
    }
    if (C::kTmaStore && lane == 0 && stores_issued) bulk_wait_all();
    __syncwarp();
  }

  // ------------------------------------------------------------- teardown --
  __syncthreads();
  if (*abort_flag) {
    const uint64_t drain_ns = 10000000ull;  // 10 ms per outstanding operation
    if (warp == 0 && lane == 0) {
      const uint32_t n = loads_issued < static_cast<uint32_t>(S) ? loads_issued : S;
      for (uint32_t j = loads_issued - n; j < loads_issued; ++j)
        drain_wait(smem_u32(&full_bar[j % S]), (j / S) & 1u, drain_ns);
    }
    // Every issuer commits once: the barrier completes when all their MMAs are done.
    if (warp >= 1 && warp <= C::kIssuers && lane == 0) mma_commit(smem_u32(drain_bar));
    if (warp == 1 && lane == 0) drain_wait(smem_u32(drain_bar), 0, drain_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Takes the status word and clears it in one atomic step, so that a bit another
// stream's kernel sets at the same time lands either in this read or the next.
__global__ void status_take_kernel() { g_status_taken = atomicExch(&g_status_word, 0u); }

// dst[i] = v for i < n (grid-stride).
__global__ void fill_f32_kernel(float* dst, int64_t n, float v) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = v;
}

// A block whose only wait is on a barrier that nothing arrives at.
__global__ void timeout_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, &g_status_word, limit_ns);
  }
  __syncthreads();
}

// --------------------------------------------------------------- host side --
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct DeviceInfo {
  int num_sms = 0;
};

DeviceInfo device_info(int dev) {
  static DeviceInfo cache[64];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return DeviceInfo{};
  if (cache[dev].num_sms == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev].num_sms = n;
  }
  return cache[dev];
}

// Fraction of SM slots busy over the waves of a persistent launch.
double wave_efficiency(int64_t tiles, int sms) {
  const int64_t waves = (tiles + sms - 1) / sms;
  return static_cast<double>(tiles) / static_cast<double>(waves * sms);
}

// Tile width override for tuning: DG_GEMM_BLOCK_N in {16, 32, 64, 128, 256}.
int block_n_override() {
  static const int v = [] {
    const char* e = std::getenv("DG_GEMM_BLOCK_N");
    const int n = e ? std::atoi(e) : 0;
    return (n == 16 || n == 32 || n == 64 || n == 128 || n == 256) ? n : 0;
  }();
  return v;
}

int pick_bn(int64_t M, int64_t N, int sms) {
  if (block_n_override()) return block_n_override();
  if (M > 256) return 256;
  // Small M streams B from HBM: pick the widest tile that keeps the SMs evenly loaded.
  const int cands[4] = {128, 64, 32, 16};
  int best = 16;
  double best_eff = -1.0;
  for (int bn : cands) {
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
    const double eff = wave_efficiency(tiles, sms);
    if (eff >= 0.85 && tiles >= sms) return bn;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = bn;
    }
  }
  return best;
}

template <int BN, bool kGrouped, bool kQ>
int run_gemm(const GemmProblem& p, cudaStream_t stream, int dev, int sms) {
  using Cf = Cfg<BN>;
  constexpr uint32_t kOut = out_bytes<BN, kQ>();
  GemmArgsT<kQ> args{};
  args.c = static_cast<__nv_bfloat16*>(p.c);
  if constexpr (kQ) args.rq = p.rq;
  args.ld_c = p.ld_c;
  args.sa = p.sa;
  args.sa_per_row = p.sa_per_row ? 1 : 0;
  args.sb = p.sb;
  args.m_indices = p.m_indices;
  args.M = static_cast<int>(p.M);
  args.N = static_cast<int>(p.N);
  args.num_kb = static_cast<int>(p.K / kBK);
  args.ld_sa = static_cast<int>(p.ld_sa);
  args.ld_sb = static_cast<int>(p.ld_sb);
  args.a_mn = p.a_mn ? 1 : 0;
  args.b_mn = p.b_mn ? 1 : 0;
  args.idesc = Cf::kIdesc | idesc_majors(p.a_mn, p.b_mn);
  if (p.b_mn && (BN < 128 || kGrouped)) return DG_ERR_UNSUPPORTED_SHAPE;
  args.num_mb = static_cast<int>((p.M + kBM - 1) / kBM);
  args.num_nb = static_cast<int>((p.N + BN - 1) / BN);
  args.nbs = static_cast<int>((p.N + kBK - 1) / kBK);
  args.num_groups = p.num_groups;
  args.wait_limit_ns = kDefaultWaitLimitNs;

  // A box: all 128 rows, or the valid rows (multiple of 8) when M is small.
  const uint32_t a_rows = (p.M >= kBM || p.a_mn) ? kBM : static_cast<uint32_t>((p.M + 7) / 8 * 8);
  args.a_box_bytes = a_rows * kBK;
  args.a_stage_bytes = (args.a_box_bytes + 1023u) / 1024u * 1024u;
  const uint32_t stage_bytes = args.a_stage_bytes + Cf::kBTileBytes;
  const size_t bar_bytes = (2 * kMaxStages + 2 * Cf::kNumPBuf + 1) * sizeof(uint64_t) + 16;
  const size_t budget = kMaxDynSmem - 1024 - kOut - bar_bytes;
  // The operand ring, including the padding a short A box needs (see the kernel).
  auto ring_bytes = [&](int st) {
    return std::max<size_t>(static_cast<size_t>(st) * stage_bytes,
                            static_cast<size_t>(st - 1) * args.a_stage_bytes + kATileBytes);
  };
  int stages = std::min<int>(kMaxStages, static_cast<int>(budget / stage_bytes));
  stages = std::min<int64_t>(stages, std::max<int64_t>(6, args.num_kb * 2));
  while (stages > 2 && ring_bytes(stages) > budget) --stages;
  // Stage s must only ever be waited on by issuer s % kIssuers (see Cfg):
  // a multiple of kIssuers stages.
  stages = stages / Cf::kIssuers * Cf::kIssuers;
  if (stages < Cf::kIssuers || ring_bytes(stages) > budget) return DG_ERR_UNSUPPORTED_SHAPE;
  args.num_stages = stages;
  size_t smem = 1024 + ring_bytes(stages) + kOut + bar_bytes;
  // One CTA per SM: the grid is persistent and each CTA owns its SM's TMEM.
  smem = std::max<size_t>(smem, kMinSmemPerCta);
  if (smem > kMaxDynSmem) return DG_ERR_UNSUPPORTED_SHAPE;

  CUtensorMap ta, tb, tc;
  if (p.a_mn) {
    // A as [K][ld_a]: 128 (M) x 128 (K) boxes.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(p.K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.ld_a)};
    const cuuint32_t box[2] = {kBM, kBK};
    if (!encode_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 2, dims, strides, box)) return DG_ERR_CUDA;
  } else {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.ld_a)};
    const cuuint32_t box[2] = {kBK, a_rows};
    if (!encode_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 2, dims, strides, box)) return DG_ERR_CUDA;
  }
  if (kGrouped) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.N),
                                static_cast<cuuint64_t>(p.num_groups)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.K),
                                   static_cast<cuuint64_t>(p.K) * static_cast<cuuint64_t>(p.N)};
    const cuuint32_t box[3] = {kBK, static_cast<cuuint32_t>(BN), 1};
    if (!encode_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 3, dims, strides, box)) return DG_ERR_CUDA;
  } else if (p.b_mn) {
    // B as [K][ld_b]: 128 (N) x 128 (K) boxes.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.ld_b)};
    const cuuint32_t box[2] = {128, kBK};
    if (!encode_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 2, dims, strides, box)) return DG_ERR_CUDA;
  } else {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.ld_b)};
    const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(BN)};
    if (!encode_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 2, dims, strides, box)) return DG_ERR_CUDA;
  }
  if (kQ) {
    // E4M3 codes [M][ld_q]: 64 x 32 boxes, 64-byte swizzle.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.rq.ld_q)};
    const cuuint32_t box[2] = {64, 32};
    if (!encode_map(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.rq.q, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
      return DG_ERR_CUDA;
  } else if (Cf::kTmaStore) {
    // C as bf16 [M][ld_c]: 32 x 32 boxes, 64-byte swizzle.
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.ld_c) * 2};
    const cuuint32_t box[2] = {32, 32};
    if (!encode_map(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.c, 2, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_64B))
      return DG_ERR_CUDA;
  } else {
    tc = ta;  // not read by narrow tiles
  }

  auto kernel = fp8_gemm_kernel<BN, kGrouped, kQ>;
  static std::atomic<uint64_t> attr_set{0};
  if (dev < 64 && !(attr_set.load() & (1ull << dev))) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMaxDynSmem)) != cudaSuccess)
      return DG_ERR_CUDA;
    attr_set.fetch_or(1ull << dev);
  }
  const int64_t tiles = static_cast<int64_t>(args.num_mb) * args.num_nb;
  int grid = static_cast<int>(std::min<int64_t>(tiles, sms));
  if (p.num_sms_cap > 0) grid = std::min(grid, p.num_sms_cap);
  grid = std::max(grid, 1);
  if (launch_kernel(kernel, dim3(grid), dim3(Cf::kThreads), smem, stream, 0, ta, tb, tc, args) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  return DG_OK;
}

}  // namespace

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                       const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                       bool swizzle128) {
  return encode_tensor_map_swizzle(map, dtype, base, rank, dims, strides, box,
                                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool encode_tensor_map_swizzle(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                               const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                               CUtensorMapSwizzle swizzle) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  const CUresult r = fn(map, dtype, rank, const_cast<void*>(base), d, st, b, e,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_sm_count(int dev) { return device_info(dev).num_sms; }

bool tile_width_forced() { return block_n_override() != 0; }

unsigned int* device_status_word() {
  static unsigned int* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

int launch_gemm(const GemmProblem& p, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DG_ERR_NO_DEVICE;
  const int sms = device_info(dev).num_sms;
  if (sms <= 0) return DG_ERR_NO_DEVICE;
  // Decode shapes: one row streams B (gemv.cu); M <= 128, cluster split-K.
  if (!block_n_override() && gemv_supported(p)) return launch_gemv(p, stream);
  // Small problems with 64-128 rows (B up to 12 MB, bf16 output, K-major B):
  // one CTA per narrow tile over all of K starts faster than a cluster that
  // splits K and reduces (single launches on GB300: 128x256x512 8.1 against
  // 13.2 us, 128x2048x2048 12.7 against 18.3 us; at 16 rows, or from 16 MB of
  // B, the split kernel is as fast or faster).
  if (!block_n_override() && p.m_indices == nullptr && p.M >= 64 && p.M <= kBM && !p.rq.q && !p.b_mn &&
      p.N * p.K <= (12ll << 20)) {
    if ((p.N + 31) / 32 <= sms) return run_gemm<32, false, false>(p, stream, dev, sms);
    return run_gemm<64, false, false>(p, stream, dev, sms);
  }
  if (!block_n_override() && small_m_supported(p.M, p.m_indices)) return launch_gemm_small_m(p, stream);
  // Dense M > 128 and M-grouped calls with power-of-two scales: CTA pairs (the
  // grouped calls fall back to the 1-SM kernel below when fewer than two SMs
  // are allowed).
  if (!block_n_override() && (p.m_indices != nullptr || p.M > kBM)) {
    const int r = launch_gemm_pair(p, stream);
    if (r != DG_ERR_UNSUPPORTED_SHAPE) return r;
  }
  const bool grouped = p.m_indices != nullptr;
  if (p.rq.q != nullptr) {
    // The requantizing epilogue needs whole 128-column output blocks per tile.
    const int bn = (block_n_override() == 128 || (!block_n_override() && p.M <= 2 * kBM)) ? 128 : 256;
    if (bn == 128)
      return grouped ? run_gemm<128, true, true>(p, stream, dev, sms) : run_gemm<128, false, true>(p, stream, dev, sms);
    return grouped ? run_gemm<256, true, true>(p, stream, dev, sms) : run_gemm<256, false, true>(p, stream, dev, sms);
  }
  int bn = pick_bn(p.M, p.N, sms);
  if (p.b_mn && bn < 128) bn = 128;  // MN-major B tiles are whole 128-column swizzle atoms
  switch (bn) {
    case 16: return grouped ? run_gemm<16, true, false>(p, stream, dev, sms) : run_gemm<16, false, false>(p, stream, dev, sms);
    case 32: return grouped ? run_gemm<32, true, false>(p, stream, dev, sms) : run_gemm<32, false, false>(p, stream, dev, sms);
    case 64: return grouped ? run_gemm<64, true, false>(p, stream, dev, sms) : run_gemm<64, false, false>(p, stream, dev, sms);
    case 128:
      return grouped ? run_gemm<128, true, false>(p, stream, dev, sms) : run_gemm<128, false, false>(p, stream, dev, sms);
    default:
      return grouped ? run_gemm<256, true, false>(p, stream, dev, sms) : run_gemm<256, false, false>(p, stream, dev, sms);
  }
}

cudaError_t read_and_clear_status(unsigned int* out, cudaStream_t stream) {
  static std::mutex mu;  // one snapshot slot per device: one reader at a time
  std::lock_guard<std::mutex> lock(mu);
  status_take_kernel<<<1, 1, 0, stream>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(out, g_status_taken, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

cudaError_t launch_fill_f32(float* dst, int64_t n, float v, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
  fill_f32_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(dst, n, v);
  return cudaGetLastError();
}

cudaError_t launch_timeout_selftest(uint64_t limit_ns, cudaStream_t stream) {
  timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

}  // namespace dg
