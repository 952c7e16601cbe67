// gemm_pair.cu -- dense FP8 (E4M3) block-scaled NT GEMM on CTA pairs (sm_103a).
//
//   C[m, n] = bf16( sum_kb sa[m/128, kb] * sb[n/128, kb] * sum_{k in kb} A[m,k] B[n,k] )
//
// Same arithmetic as gemm.cu (lpnh.cn DeepGEMM walkthrough §2.2, §3.1, §3.2;
// pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1, §4.1): the tensor core
// forms each 128-deep K block's partial sums, which are then multiplied by
// sa * sb and added to FP32 accumulators held in registers.
//
// Why pairs: the promotion reads every K block's partial tile out of TMEM, so
// the tensor core can only run ahead of the epilogue by as many K blocks as
// TMEM holds partial tiles. A 128x256 tile per SM leaves room for two; here a
// thread-block cluster of two CTAs computes a 256x128 tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 128), so each SM accumulates a
// 128x128 partial and TMEM holds four of them. Each CTA also holds half as
// many FP32 accumulators in registers, and each SM stages only its half of B.
//
//   * CTA r of a pair loads A rows [256 pm + 128 r, +128) (warp 0) and B rows
//     [128 nb + 64 r, +64) (the last warp; warp 0 too in the requantizing
//     instantiation) of every K block with TMA; all loads count on the even
//     CTA's `full` barrier, which the even CTA arms for both CTAs' bytes;
//   * warps 1 and 2 of the even CTA take turns issuing the four MMAs (K = 32)
//     of a K block into TMEM buffer it % 4 of both CTAs; each commit arrives on
//     the stage's `empty` barrier and the buffer's `tfull` barrier in both
//     CTAs. Issuer i owns the stages and buffers of index parity i, so each
//     barrier it waits on sees its phases in order;
//   * the epilogue warps of each CTA read their 32 TMEM lanes of the partial,
//     release the buffer by arriving on the even CTA's `tempty` barrier, and
//     promote it in registers (two FP32 FMAs per f32x2 instruction, each
//     rounded like fmaf). After the last K block each warp rounds its 32 x 64
//     slice to bf16 and writes it with one TMA store (128-byte swizzle) clipped
//     at M; a slice that crosses N is written element by element;
//   * pairs are persistent over the 256x128 tiles in a grouped raster.
// K-grouped calls (one output per range of K, pzsr.cn page §3.2) run this
// kernel (FP32 scales; see KUnit) or the block-scaled kernel below
// (power-of-two scales; see ScaledUnit) over every range's tiles in one launch.
// M-grouped calls (MoE experts, pzsr.cn page §2.3, §3.2) with power-of-two
// scales run on the block-scaled kernel below (with FP32 scales, on the 1-SM
// kernel of gemm.cu): both 128-row halves of a pair tile multiply one B, so a pair row
// whose two blocks belong to one expert is one unit, and a pair row whose
// blocks belong to different experts (or to an expert and padding) becomes
// two units, each with one CTA keeping its rows and the other discarding its
// (see pair_unit). Blocks of padding rows only, or of an id past the last
// expert, run no MMAs and are written as zeros.
// Every mbarrier wait is bounded; on a timeout the CTA raises its abort flag,
// records it in the device status word, drains what it has in flight, frees
// TMEM and leaves through the final cluster barrier.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "../../include/dgfp8.h"
#include "dg_device.cuh"
#include "dg_encode.cuh"
#include "dg_internal.h"
#include "dg_pair.cuh"

namespace dg {
namespace {

constexpr int kMaxStages = 16;
constexpr int kNumBuf = 4;             // TMEM partial buffers of 128 columns
constexpr int kIssuers = 2;
constexpr uint32_t kBHalfBytes = (kBN / 2) * kBK;  // 8 KB
constexpr uint32_t kStageBytes = kABytes + kBHalfBytes;
constexpr uint32_t kIdesc = idesc_e4m3_f32(2 * kBM, kBN);

template <int kEpiCols, bool kQ>
struct PCfg {
  static constexpr int kEpiPerQuad = kBN / kEpiCols;  // warps per TMEM lane quadrant
  static constexpr int kEpiWarps = 4 * kEpiPerQuad;
  static constexpr int kFirstEpiWarp = 1 + kIssuers;
  // bf16 output: the last warp loads B. The requantizing epilogue keeps one
  // producer for both operands (measured 3-7 % faster there).
  static constexpr int kBProducer = kFirstEpiWarp + kEpiWarps;
  static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps + (kQ ? 0 : 1));
  // bf16 output: staging boxes for the TMA stores; E4M3 output: the slices'
  // maxima exchange (codes are stored straight from registers).
  static constexpr uint32_t kOutBytes =
      kQ ? requant_smem_bytes(kEpiWarps) : kEpiWarps * kBoxBytes * (kEpiCols / 32);
  static_assert(!kQ || kEpiCols == 64, "the requantizing epilogue takes 64-column slices");
  static_assert(kEpiCols == 32 || kEpiCols == 64, "epilogue slice");
  static_assert(kThreads <= 1024, "CTA size");
};
constexpr int kEpiCols = 64;

// One unit of the FP32-promotion kernel: pair tile (pm, nb) over K blocks
// [kb0, kb0 + nkb), written to output matrix g (K-grouped calls; else g = 0
// and the whole K).
struct KUnit {
  int pm, nb, kb0, nkb, g;
};
template <bool kKG, class Args>
__device__ __forceinline__ int pair_units(const Args& a) {
  if constexpr (kKG)
    return a.num_kg * a.num_pm * a.num_nb;
  else
    return a.num_pm * a.num_nb;
}
template <bool kKG, class Args>
__device__ __forceinline__ KUnit pair_kunit(int t, const Args& a) {
  KUnit u;
  if constexpr (kKG) {
    const int per = a.num_pm * a.num_nb;
    const int i = t / per;
    pair_tile_coords(t - i * per, a.num_pm, a.num_nb, a.group_pm, u.pm, u.nb);
    u.kb0 = a.kb_lo[i];
    u.nkb = a.kb_n[i];
    u.g = a.g_out[i];
  } else {
    pair_tile_coords(t, a.num_pm, a.num_nb, a.group_pm, u.pm, u.nb);
    u.kb0 = 0;
    u.nkb = a.num_kb;
    u.g = 0;
  }
  return u;
}

// TMA producer of the FP32-promotion pair kernel. CTA r loads A rows
// [256 pm + 128 r, +128) and B rows [128 nb + 64 r, +64) of each K block into
// ring stage it % S; both CTAs' bytes count on the even CTA's `full` barrier,
// which the even CTA's A producer arms for the pair (a B load that lands
// before the arm only takes the barrier's byte count below zero for the
// phase). Each TMA issue blocks its thread for a few hundred cycles, about
// what the tensor core spends on a K block, so one thread per operand issues
// (kPart 1: A and the arm, kPart 2: B). Stage and phase are running counters.
// Returns the number of stages it filled.
template <bool kNT, bool kKG = false, int kPart = 0, class Args>
__device__ __forceinline__ uint32_t pair_producer(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                                  const Args& args, uint32_t ring0, uint64_t* full_bar,
                                                  uint64_t* empty_bar, uint32_t rank, int pair, int num_pairs,
                                                  volatile int* abort_flag, unsigned int* status) {
  const int S = args.num_stages;
  const bool leader = rank == 0;
  const uint32_t leader_full = mapa_shared(smem_u32(full_bar), 0);
  const uint32_t empty0 = smem_u32(empty_bar);
  const int num_units = pair_units<kKG>(args);
  uint32_t stage = 0, phase = 0, issued = 0;
  for (int t = pair; t < num_units; t += num_pairs) {
    const KUnit u = pair_kunit<kKG>(t, args);
    const int arow = u.pm * (2 * kBM) + static_cast<int>(rank) * kBM;
    const int brow = u.nb * kBN + static_cast<int>(rank) * (kBN / 2);
    for (int kb = u.kb0; kb < u.kb0 + u.nkb; ++kb) {
      if (!mbar_wait(empty0 + stage * 8u, phase ^ 1u, abort_flag, status, args.wait_limit_ns)) return issued;
      if (leader && kPart != 2) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), 2u * kStageBytes);
      const uint32_t fb = leader_full + stage * 8u;
      const uint32_t dst = ring0 + stage * kStageBytes;
      // K-major maps are {K, rows}; MN-major maps {rows, K} (the tile's K rows hold 128 or 64 bytes).
      if (kPart != 2) {
        if (!kNT && args.a_mn)
          tma_load_2d_pair(dst, &tmap_a, fb, arow, kb * kBK);
        else
          tma_load_2d_pair(dst, &tmap_a, fb, kb * kBK, arow);
      }
      if (kPart != 1) {
        if (!kNT && args.b_mn)
          tma_load_2d_pair(dst + kABytes, &tmap_b, fb, brow, kb * kBK);
        else
          tma_load_2d_pair(dst + kABytes, &tmap_b, fb, kb * kBK, brow);
      }
      ++issued;
      if (++stage == static_cast<uint32_t>(S)) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  return issued;
}

// kNT: both operands K-major (the NT layout). Its instantiation keeps layout
// handling out of the TMA and MMA issue loops, where runtime branches on the
// layout and runtime descriptors cost ~10 % (measured); other layouts take
// the runtime path. kKG: a K-grouped call (bf16 output, any layout), its units
// spread over all ranges' tiles in one launch.
template <int EC, bool kQ, bool kNT, bool kKG = false>
__global__ void __launch_bounds__(PCfg<EC, kQ>::kThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ PairArgsF<kQ, kKG> args) {
  static_assert(!(kKG && kQ), "K-grouped calls write bf16");
  using C = PCfg<EC, kQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = args.num_stages;
  uint8_t* ring = smem;  // stage s: A tile, then this CTA's half of the B tile
  uint8_t* smem_out = smem + static_cast<size_t>(S) * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_out + C::kOutBytes);
  uint64_t* full_bar = bars;                      // even CTA: both CTAs' stage bytes landed
  uint64_t* empty_bar = bars + kMaxStages;        // the stage's MMAs are done
  uint64_t* tfull_bar = bars + 2 * kMaxStages;    // the buffer holds a finished partial
  uint64_t* tempty_bar = tfull_bar + kNumBuf;     // even CTA: both epilogues read the buffer
  uint64_t* drain_bar = tempty_bar + kNumBuf;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);
  const uint64_t limit = args.wait_limit_ns;
  unsigned int* status = args.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < kNumBuf; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), 2 * C::kEpiWarps);
    }
    mbar_init(smem_u32(drain_bar), kIssuers);
    if constexpr (kQ) requant_xchg_init(smem_out, C::kEpiWarps);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_c);
    // The first stages' B half-tiles of this CTA's first tile start streaming
    // into L2 while the preceding grid finishes.
    if (pair < pair_units<kKG>(args)) {
      const KUnit u = pair_kunit<kKG>(pair, args);
      const int brow = u.nb * kBN + static_cast<int>(rank) * (kBN / 2);
      const int n_pre = min(S, u.nkb);
      for (int kb = u.kb0; kb < u.kb0 + n_pre; ++kb) {
        if (!kNT && args.b_mn)
          tma_prefetch_2d(&tmap_b, brow, kb * kBK);
        else
          tma_prefetch_2d(&tmap_b, kb * kBK, brow);
      }
    }
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kNumBuf * kBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or load
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  const int num_tiles = pair_units<kKG>(args);
  uint32_t loads_issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0)
      loads_issued = pair_producer<kNT, kKG, kQ ? 0 : 1>(tmap_a, tmap_b, args, smem_u32(ring), full_bar, empty_bar,
                                                         rank, pair, num_pairs, abort_flag, status);
    __syncwarp();
  } else if (!kQ && warp == C::kBProducer) {
    // ---------------------------------------------------------- B producer --
    if (lane == 0)
      pair_producer<kNT, kKG, 2>(tmap_a, tmap_b, args, smem_u32(ring), full_bar, empty_bar, rank, pair, num_pairs,
                                 abort_flag, status);
    __syncwarp();
  } else if (warp <= kIssuers) {
    // ----------------------------------------------------------- MMA issue --
    // Issuer i takes K blocks i, i + 2, i + 4, ... of this pair's sequence, so
    // its stages and buffers advance by two (S is even, four buffers).
    if (leader && lane == 0) {
      const uint32_t me = static_cast<uint32_t>(warp - 1);
      uint32_t total;
      if constexpr (kKG) {
        total = 0;
        for (int t = pair; t < num_tiles; t += num_pairs) total += static_cast<uint32_t>(pair_kunit<true>(t, args).nkb);
      } else {
        const int my_tiles = num_tiles > pair ? (num_tiles - 1 - pair) / num_pairs + 1 : 0;
        total = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(args.num_kb);
      }
      const uint32_t full0 = smem_u32(full_bar), empty0 = smem_u32(empty_bar);
      const uint32_t tfull0 = smem_u32(tfull_bar), tempty0 = smem_u32(tempty_bar);
      const uint32_t ring0 = smem_u32(ring);
      // A tiles: 128 rows; B tiles: this CTA's 64 of the pair's 128 columns.
      const OperandTile at{static_cast<uint32_t>(args.a_mn), 128u}, bt{static_cast<uint32_t>(args.b_mn), 64u};
      const uint64_t afields = at.desc_fields(), bfields = bt.desc_fields();
      const uint32_t astep = at.kstep(), bstep = bt.kstep();
      const uint32_t idesc = args.idesc;
      uint32_t stage = me, sphase = 0, buf = me, bphase = 0;
      for (uint32_t it = me; it < total; it += kIssuers) {
        if (!mbar_wait(tempty0 + buf * 8u, bphase ^ 1u, abort_flag, status, limit)) break;
        if (!mbar_wait(full0 + stage * 8u, sphase, abort_flag, status, limit)) break;
        tc_fence_after();
        const uint32_t base = ring0 + stage * kStageBytes;
        const uint32_t d = tmem_base + buf * kBN;
        if constexpr (kNT) {
          const uint64_t adesc = sw128_kmajor_desc(base);
          const uint64_t bdesc = sw128_kmajor_desc(base + kABytes);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k)
            mma_e4m3_pair(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, k > 0 ? 1u : 0u);
        } else {
          const uint64_t adesc = desc_at(afields, base);
          const uint64_t bdesc = desc_at(bfields, base + kABytes);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k)
            mma_e4m3_pair(d, adesc + astep * k, bdesc + bstep * k, idesc, k > 0 ? 1u : 0u);
        }
        mma_commit_pair_mc(empty0 + stage * 8u, 0x3);
        mma_commit_pair_mc(tfull0 + buf * 8u, 0x3);
        stage += kIssuers;
        if (stage >= static_cast<uint32_t>(S)) {
          stage -= S;
          sphase ^= 1u;
        }
        buf += kIssuers;
        if (buf >= static_cast<uint32_t>(kNumBuf)) {
          buf -= kNumBuf;
          bphase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - C::kFirstEpiWarp;
    const int part = ew >> 2;   // columns [EC part, EC part + EC) of the tile
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + part * EC;
    const uint32_t leader_tempty = mapa_shared(smem_u32(tempty_bar), 0);
    uint8_t* out_box = smem_out + ew * kBoxBytes * (EC / 32);
    bool stores_issued = false;
    uint32_t it = 0;
    uint32_t tl = 0;  // tiles done by this pair
    bool ok = true;
    bool ready = false;  // the full barrier of slot `it` is known to be complete
    for (int t = pair; t < num_tiles && ok; t += num_pairs, ++tl) {
      const KUnit u = pair_kunit<kKG>(t, args);
      const int pm = u.pm, nb = u.nb;
      const int mb = min(pm * 2 + static_cast<int>(rank), args.num_mb - 1);
      // This thread's row's scales (rows past M read the last row's).
      const int arow = min(pm * (2 * kBM) + static_cast<int>(rank) * kBM + quad * 32 + lane, args.M - 1);
      const float* sa_p = args.sa + static_cast<int64_t>(args.sa_per_row ? arow : mb) * args.ld_sa + u.kb0;
      const float* sb_p = args.sb + static_cast<int64_t>(nb) * args.ld_sb + u.kb0;
      uint64_t acc[EC / 2];  // FP32 accumulators, two columns per register pair
#pragma unroll
      for (int j = 0; j < EC / 2; ++j) acc[j] = 0ull;
      // Scales of K blocks kb + 1 (a1, b1) and kb + 2 (a2, b2) are loaded ahead
      // and multiplied only when used: a product right after its loads would
      // stall every K block on the load latency (measured: ~200 cycles).
      const int num_kb = u.nkb;
      float s = __ldg(sa_p) * __ldg(sb_p);
      float a1 = num_kb > 1 ? __ldg(sa_p + 1) : 0.f, b1 = num_kb > 1 ? __ldg(sb_p + 1) : 0.f;
      float a2 = num_kb > 2 ? __ldg(sa_p + 2) : 0.f, b2 = num_kb > 2 ? __ldg(sb_p + 2) : 0.f;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const uint32_t buf = it % kNumBuf;
        if (!ready) {
          const bool w = mbar_wait(smem_u32(&tfull_bar[buf]), (it / kNumBuf) & 1u, abort_flag, status, limit);
          if (!__all_sync(0xFFFFFFFFu, w)) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        uint32_t r[EC];
        if constexpr (kQ) {
          // The requantizing instantiation reads the slice in 32-column loads:
          // one 64-column load made it ~20 % slower (168 registers, spills).
#pragma unroll
          for (int q = 0; q < EC / 32; ++q) tmem_ld<32>(tmem_row + buf * kBN + q * 32, &r[q * 32]);
        } else {
          tmem_ld<EC>(tmem_row + buf * kBN, r);  // one load of the whole slice (measured 1-3 % faster than two)
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_addr(leader_tempty + buf * 8u);
        // Look ahead: test the next slot's barrier now, so that the test's
        // latency hides behind the multiply-adds below.
        const uint32_t nx = it + 1;
        const bool next_done = mbar_test(smem_u32(&tfull_bar[nx % kNumBuf]), (nx / kNumBuf) & 1u);
        const uint64_t s2 = f32x2(__float_as_uint(s), __float_as_uint(s));
#pragma unroll
        for (int j = 0; j < EC / 2; ++j) ffma2(acc[j], s2, f32x2(r[2 * j], r[2 * j + 1]));
        ready = __all_sync(0xFFFFFFFFu, next_done);
        s = a1 * b1;
        a1 = a2;
        b1 = b2;
        a2 = kb + 3 < num_kb ? __ldg(sa_p + kb + 3) : 0.f;
        b2 = kb + 3 < num_kb ? __ldg(sb_p + kb + 3) : 0.f;
      }
      if (!ok) break;

      const int row0 = pm * (2 * kBM) + static_cast<int>(rank) * kBM + quad * 32;
      if constexpr (kQ) {
        if (!requant_store_slice<C::kEpiWarps>(acc, row0 + lane < args.M, false, row0, args.M, args.N,
                                               nb * kBN + part * EC, ew, lane, tl, smem_out, args.rq, &tmap_c,
                                               requant_box(smem_out, C::kEpiWarps, ew), stores_issued, abort_flag,
                                               status, limit)) {
          ok = false;
          break;
        }
      } else {
        store_tile_rows64<kKG>(acc, tmap_c, args, out_box, row0, nb * kBN + part * EC, lane, stores_issued, u.g);
      }
    }
    if (lane == 0 && stores_issued) bulk_wait_all();
    __syncwarp();
  }

  // ------------------------------------------------------------- teardown --
  __syncthreads();
  if (*abort_flag) {
    const uint64_t drain_ns = 10000000ull;  // 10 ms per outstanding operation
    if (warp == 0 && lane == 0) {
      if (leader) {
        const uint32_t n = loads_issued < static_cast<uint32_t>(S) ? loads_issued : S;
        for (uint32_t j = loads_issued - n; j < loads_issued; ++j)
          drain_wait(smem_u32(&full_bar[j % S]), (j / S) & 1u, drain_ns);
      } else {
        // This CTA's loads count on the even CTA's barrier; give them time to land.
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 200000ull) {
        }
      }
    }
    if (leader && warp >= 1 && warp <= kIssuers && lane == 0) mma_commit_pair(smem_u32(drain_bar));
    if (leader && warp == 1 && lane == 0) drain_wait(smem_u32(drain_bar), 0, drain_ns);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA frees TMEM or leaves while its peer may still use it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kNumBuf * kBN);
  }
}

// ---------------------------------------------------------------------------
// Power-of-two scales: the tensor core applies them (block-scaled MMA).
//
// With every scale a power of two, sa * sb * sum(a b) equals the sum of the
// products (a 2^ea)(b 2^eb) exactly, which is what tcgen05.mma
// kind::mxf8f6f4.block_scale computes from UE8M0 scale factors (one per 32 K
// elements of each row of A and column of B). A 128x128 scale block gives all
// 128 rows (columns) and all four 32-element K slices of a K block the same
// factor, so each K block needs one exponent byte for A and one for B, written
// into every lane and byte of a few TMEM columns. The tile's partial sums then
// stay in TMEM across all K blocks and the epilogue reads them once per tile.
// Without the per-K-block promotion the limits are the issuing threads: each
// TMA issue and each MMA issue blocks its thread (the MMA until the tensor pipe
// takes it), so
//   * warps 0 and 3: TMA producers, alternating ring stages; a stage holds two
//     K blocks (one 3-D box of A and one of B per CTA), counted on the even
//     CTA's `full` barrier;
//   * warps 1-2 of the even CTA: MMA issue, alternating stages. Per valid K
//     block four block-scaled MMAs go into the tile's accumulator (two
//     accumulators alternate between tiles); each stage's MMAs are committed to
//     its `empty` barrier and each issuer commits the accumulator after its
//     last stage of the tile. The first MMA of a tile overwrites the
//     accumulator, so the MMAs must reach the pipe in K-block order: the
//     issuers pass a turn counter in shared memory (deterministic results);
//   * warps 4-7 (one per TMEM lane quadrant): write each stage's exponents
//     (this CTA's A block, the tile's B block) into the stage's TMEM scale
//     columns; they wait on the stage's `empty` barrier like the producers and
//     arrive on its `full` barrier, which thus completes when both CTAs'
//     operands and scales are in place;
//   * warps 8 on: per tile, read the accumulator, release it, round to bf16
//     and store.
// A stage past an odd number of K blocks holds a zero-filled K block that gets
// no MMA and no scale. K-grouped calls (kKG) give each unit its own K range:
// its stages start at the range's first K block, a last stage past an odd
// count holds the next range's first K block (again no MMA, no scale), and a
// one-stage unit's issuer commits the accumulator twice, once for each
// issuer the barrier counts.
//
// Two tile widths. 256x128 pair tiles (N = 128 MMAs, two accumulators of 128
// columns alternating between tiles) serve every layout and the requantizing
// epilogue. 256x256 pair tiles (N = 256 MMAs) serve bf16 output in the NT
// layout: each MMA does twice the work per instruction and per byte of A read
// from shared memory (per SM and K block 48 KB of operand reads and 32 KB of
// TMA writes for 512 tensor cycles, against 32 + 24 KB for 256 cycles), at
// the price of one 256-column accumulator, which the epilogue must read before
// the next tile's first MMA.
// Where the MMA reads the scale factors (probed on the GPU with exponents that
// encode their TMEM position): every TMEM lane quadrant holds its own copy;
// the factor of B column n (of A row m) sits in lane 32 q + n % 32 of column
// n / 32 of the B (A) scale area. A 128-row scale block therefore fills four
// columns uniformly: four B columns for 128-column tiles, eight (the tile's two
// B blocks, both CTAs writing both) for 256-column tiles.
// ---------------------------------------------------------------------------
constexpr int kNatMaxStages = 8;
constexpr int kNatFirstEpiWarp = 8;

template <int kBNs>
struct NatCfg {
  static_assert(kBNs == 128 || kBNs == 256, "pair tile width");
  static constexpr int kNumAcc = kBNs == 256 ? 1 : 2;                   // tile accumulators in TMEM
  static constexpr uint32_t kAccCols = kNumAcc * kBNs;
  static constexpr uint32_t kBHalf = (kBNs / 2) * kBK;                   // this CTA's B rows per K block
  // K blocks per stage: two (one 3-D box of each operand carries both), or one
  // for the 256-column tiles, whose 64 KB double stages would leave room for
  // only two of them next to the output staging (the count must be even).
  static constexpr int kKbPerStage = kBNs == 256 ? 1 : 2;
  static constexpr uint32_t kAStage = kKbPerStage * kABytes;
  static constexpr uint32_t kStageBytes = kAStage + kKbPerStage * kBHalf;
  static constexpr int kEpiWarps = kBNs / 16;                            // 4 quadrants x BN/64 slices of 64
  static constexpr int kThreads = 32 * (kNatFirstEpiWarp + kEpiWarps);
  static constexpr int kBoxes = kBNs == 256 ? 1 : 2;                     // bf16 staging boxes per warp
  static constexpr uint32_t kIdesc = idesc_e4m3_block_scaled(2 * kBM, kBNs);
  // Scale columns per K block: 4 for A, then 4 (or 8) for B; rounded to whole
  // 8-column stores.
  static constexpr uint32_t kSfCols = kBNs == 256 ? 16 : 8;
  static_assert(kAccCols + kNatMaxStages * kKbPerStage * kSfCols <= 512, "TMEM");
};
template <int kBNs>
__host__ __device__ constexpr uint32_t nat_out_bytes(bool requant) {
  return requant ? requant_smem_bytes(NatCfg<kBNs>::kEpiWarps)
                 : NatCfg<kBNs>::kEpiWarps * kBoxBytes * NatCfg<kBNs>::kBoxes;
}

// Biased exponent of a power-of-two FP32 scale = its UE8M0 code (2^-127,
// stored as an FP32 subnormal, has code 0), replicated into four bytes.
__device__ __forceinline__ uint32_t ue8m0_word(float s) {
  return 0x01010101u * ((__float_as_uint(s) >> 23) & 0xFFu);
}

// A unit of the block-scaled kernel: the pair unit, its K blocks
// [kb0, kb0 + nkb) and its output matrix. K-grouped calls: unit t is tile
// t % T of range t / T (T = num_pm * num_nb tiles per range); otherwise all
// of K and matrix 0.
struct ScaledUnit {
  PairUnit u;
  int kb0, nkb, gout;
};
template <bool kKG, class Args>
__device__ __forceinline__ int scaled_num_units(const Args& a) {
  if constexpr (kKG)
    return a.num_kg * a.num_pm * a.num_nb;
  else
    return pair_num_units(a);
}
template <bool kGrouped, bool kKG, class Args>
__device__ __forceinline__ ScaledUnit scaled_unit(int t, const Args& a, const UnitIds& ids) {
  ScaledUnit s;
  if constexpr (kKG) {
    const int per = a.num_pm * a.num_nb;
    const int i = t / per;
    s.u = pair_unit<false>(t - i * per, a, ids);
    s.kb0 = a.kb_lo[i];
    s.nkb = a.kb_n[i];
    s.gout = a.g_out[i];
  } else {
    s.u = pair_unit<kGrouped>(t, a, ids);
    s.kb0 = 0;
    s.nkb = a.num_kb;
    s.gout = 0;
  }
  return s;
}

template <bool kQ, bool kNT, bool kGrouped, int kBNs, bool kKG = false>
__global__ void __launch_bounds__(NatCfg<kBNs>::kThreads, 1)
    fp8_gemm_pair_scaled_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                const __grid_constant__ CUtensorMap tmap_b,
                                const __grid_constant__ CUtensorMap tmap_c,
                                const std::conditional_t<kKG, PairArgsKG, PairArgsT<kQ, kGrouped>> args) {
  using NC = NatCfg<kBNs>;
  static_assert(kBNs == 128 || (!kQ && kNT), "256-column pair tiles: bf16 output, NT layout");
  static_assert(!kKG || (!kQ && !kGrouped && kBNs == 128), "K-grouped calls: bf16 output, 128-column tiles");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = args.num_stages;
  uint8_t* ring = smem;
  uint8_t* smem_out = smem + static_cast<size_t>(S) * NC::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_out + nat_out_bytes<kBNs>(kQ));
  uint64_t* full_bar = bars;                       // even CTA: operands and scales of both CTAs
  uint64_t* empty_bar = bars + kNatMaxStages;      // the stage's MMAs are done
  uint64_t* tfull_bar = bars + 2 * kNatMaxStages;  // [kNumAcc] the tile's accumulator is final
  uint64_t* tempty_bar = tfull_bar + 2;            // [kNumAcc] even CTA: both epilogues read it
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* issue_turn = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);
  const uint64_t limit = args.wait_limit_ns;
  unsigned int* status = args.status;
  const int nst = (args.num_kb + NC::kKbPerStage - 1) / NC::kKbPerStage;  // stages per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1 + 2 * 4);  // producer (with bytes) + 4 scale writers per CTA
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < NC::kNumAcc; ++b) {
      // One commit per issuer with stages in the tile (K-grouped units of one
      // stage: its issuer commits twice).
      mbar_init(smem_u32(&tfull_bar[b]), (kKG || nst >= 2) ? 2 : 1);
      mbar_init(smem_u32(&tempty_bar[b]), 2 * NC::kEpiWarps);
    }
    mbar_init(smem_u32(drain_bar), 2);
    if constexpr (kQ) requant_xchg_init(smem_out, NC::kEpiWarps);
    *abort_flag = 0;
    *issue_turn = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_c);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  const int num_units = scaled_num_units<kKG>(args);
  uint32_t loads_issued = 0;

  if (warp == 0 || warp == 3) {
    // ----------------------------------------------------------- producers --
    // Dense calls: lane 0 alone; M-grouped calls: the whole warp (warp-
    // collective unit reads) with lane 0 issuing.
    if (kGrouped || lane == 0) {
      const uint32_t me = warp == 0 ? 0u : 1u;
      const uint32_t leader_full = mapa_shared(smem_u32(full_bar), 0);
      const uint32_t empty0 = smem_u32(empty_bar), ring0 = smem_u32(ring);
      uint32_t g = 0, stage = me, phase = 0;  // g: stages of this pair's MMA units so far
      bool ok = true;
      UnitIds nxt = pair_unit_ids<kGrouped>(pair, args, lane);
      for (int t = pair; t < num_units && ok; t += num_pairs) {
        const UnitIds cur = nxt;
        nxt = pair_unit_ids<kGrouped>(t + num_pairs, args, lane);
        const ScaledUnit su = scaled_unit<kGrouped, kKG>(t, args, cur);
        const PairUnit& u = su.u;
        const int unst = kKG ? (su.nkb + NC::kKbPerStage - 1) / NC::kKbPerStage : nst;  // stages of the unit
        for (int slot = 0; slot < u.nslots && ok; ++slot) {
        const PairSlot ps = pair_slot<kGrouped>(u, slot, args);
        if (!ps.mma) continue;
        const int arow = u.pm * (2 * kBM) + static_cast<int>(rank) * kBM;
        const int brow = u.nb * kBNs + static_cast<int>(rank) * (kBNs / 2);
        for (int sl = 0; sl < unst; ++sl, ++g) {
          if ((g & 1u) != me) continue;
          if (!kGrouped || lane == 0) {
            ok = mbar_wait(empty0 + stage * 8u, phase ^ 1u, abort_flag, status, limit);
            if (ok) {
              if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), 2u * NC::kStageBytes);
              const uint32_t fb = leader_full + stage * 8u;
              const uint32_t dst = ring0 + stage * NC::kStageBytes;
              // K-major: 3-D maps {128, rows, K/128} (M-grouped B: 4-D with the
              // expert last); MN-major: 2-D maps {rows, K} whose 256-row boxes
              // stack the stage's two K blocks.
              const int kbs = su.kb0 + sl * NC::kKbPerStage;  // first K block of the stage
              if (!kNT && args.a_mn)
                tma_load_2d_pair(dst, &tmap_a, fb, arow, kbs * kBK);
              else
                tma_load_3d_pair(dst, &tmap_a, fb, 0, arow, kbs);
              if constexpr (kGrouped)
                tma_load_4d_pair(dst + NC::kAStage, &tmap_b, fb, 0, brow, kbs, ps.g);
              else if (!kNT && args.b_mn)
                tma_load_2d_pair(dst + NC::kAStage, &tmap_b, fb, brow, kbs * kBK);
              else
                tma_load_3d_pair(dst + NC::kAStage, &tmap_b, fb, 0, brow, kbs);
              ++loads_issued;
            }
          }
          if constexpr (kGrouped) ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          stage += 2;
          if (stage >= static_cast<uint32_t>(S)) {
            stage -= S;
            phase ^= 1u;
          }
        }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ----------------------------------------------------------- MMA issue --
    if (leader && (kGrouped || lane == 0)) {
      const uint32_t me = static_cast<uint32_t>(warp - 1);
      const uint32_t full0 = smem_u32(full_bar), empty0 = smem_u32(empty_bar);
      const uint32_t ring0 = smem_u32(ring);
      // g: stages of this pair's MMA units so far (this issuer's: index parity
      // me); tl: MMA units so far (the accumulator alternates with it).
      uint32_t g = 0, stage = me, sphase = 0, tl = 0;
      const OperandTile at{static_cast<uint32_t>(args.a_mn), 128u}, bt{static_cast<uint32_t>(args.b_mn), 64u};
      const uint64_t afields = at.desc_fields(), bfields = bt.desc_fields();
      const uint32_t astep = at.kstep(), bstep = bt.kstep();
      const uint32_t idesc = args.idesc;
      bool ok = true;
      UnitIds nxt = pair_unit_ids<kGrouped>(pair, args, lane);
      for (int t = pair; t < num_units && ok; t += num_pairs) {
        const UnitIds cur = nxt;
        nxt = pair_unit_ids<kGrouped>(t + num_pairs, args, lane);
        const ScaledUnit su = scaled_unit<kGrouped, kKG>(t, args, cur);
        const PairUnit& u = su.u;
        const int unst = kKG ? (su.nkb + NC::kKbPerStage - 1) / NC::kKbPerStage : nst;  // stages of the unit
        for (int slot = 0; slot < u.nslots && ok; ++slot) {
        if (!pair_slot<kGrouped>(u, slot, args).mma) continue;
        const uint32_t abuf = tl % NC::kNumAcc;
        const uint32_t d = tmem_base + abuf * kBNs;
        for (int sl = 0; sl < unst; ++sl, ++g) {
          if ((g & 1u) != me) continue;
          if (!kGrouped || lane == 0) {
            ok = mbar_wait(full0 + stage * 8u, sphase, abort_flag, status, limit);
            if (ok && sl == 0)
              ok = mbar_wait(smem_u32(&tempty_bar[abuf]), ((tl / NC::kNumAcc) & 1u) ^ 1u, abort_flag, status,
                             limit);
            // Wait for the other issuer to have handed the tensor pipe stage g - 1.
            if (ok && *issue_turn != g) {
              const uint64_t t0 = global_timer_ns();
              for (uint32_t i = 0; *issue_turn != g; ++i) {
                if ((i & 63u) == 63u && (*abort_flag || global_timer_ns() - t0 > limit)) {
                  if (!*abort_flag) {
                    *abort_flag = 1;
                    atomicOr(status, kStatusTimeout);
                  }
                  ok = false;
                  break;
                }
              }
            }
          }
          if constexpr (kGrouped) ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (!kGrouped || lane == 0) {
            tc_fence_after();
            const uint32_t base = ring0 + stage * NC::kStageBytes;
#pragma unroll
            for (int j = 0; j < NC::kKbPerStage; ++j) {
              const int kb = sl * NC::kKbPerStage + j;
              if (kb < su.nkb) {
                const uint32_t sfa = tmem_base + NC::kAccCols + (stage * NC::kKbPerStage + j) * NC::kSfCols;
                if constexpr (kNT) {
                  const uint64_t adesc = sw128_kmajor_desc(base + j * kABytes);
                  const uint64_t bdesc = sw128_kmajor_desc(base + NC::kAStage + j * NC::kBHalf);
#pragma unroll
                  for (int k = 0; k < kBK / 32; ++k)
                    mma_e4m3_pair_scaled(d, adesc + 2u * k, bdesc + 2u * k, NC::kIdesc, sfa, sfa + 4,
                                         (kb > 0 || k > 0) ? 1u : 0u);
                } else {
                  const uint64_t adesc = desc_at(afields, base + j * kABytes);
                  const uint64_t bdesc = desc_at(bfields, base + NC::kAStage + j * NC::kBHalf);
#pragma unroll
                  for (int k = 0; k < kBK / 32; ++k)
                    mma_e4m3_pair_scaled(d, adesc + astep * k, bdesc + bstep * k, idesc, sfa, sfa + 4,
                                         (kb > 0 || k > 0) ? 1u : 0u);
                }
              }
            }
            mma_commit_pair_mc(empty0 + stage * 8u, 0x3);
            if (sl + 2 >= unst) {
              mma_commit_pair_mc(smem_u32(&tfull_bar[abuf]), 0x3);
              if (kKG && unst == 1) mma_commit_pair_mc(smem_u32(&tfull_bar[abuf]), 0x3);
            }
            *issue_turn = g + 1;
          }
          stage += 2;
          if (stage >= static_cast<uint32_t>(S)) {
            stage -= S;
            sphase ^= 1u;
          }
        }
        ++tl;
        }
      }
    }
    __syncwarp();
  } else if (warp < kNatFirstEpiWarp) {
    // ------------------------------------------------------- scale writers --
    const uint32_t quad = warp & 3;
    const uint32_t sf_row = tmem_base + ((quad * 32) << 16) + NC::kAccCols;
    const uint32_t leader_full = mapa_shared(smem_u32(full_bar), 0);
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    UnitIds nxt = pair_unit_ids<kGrouped>(pair, args, lane);
    for (int t = pair; t < num_units && ok; t += num_pairs) {
      const UnitIds cur = nxt;
      nxt = pair_unit_ids<kGrouped>(t + num_pairs, args, lane);
      const ScaledUnit su = scaled_unit<kGrouped, kKG>(t, args, cur);
      const PairUnit& u = su.u;
      const int unst = kKG ? (su.nkb + NC::kKbPerStage - 1) / NC::kKbPerStage : nst;  // stages of the unit
      for (int slot = 0; slot < u.nslots && ok; ++slot) {
      const PairSlot ps = pair_slot<kGrouped>(u, slot, args);
      if (!ps.mma) continue;
      const int mb = min(u.pm * 2 + static_cast<int>(rank), args.num_mb - 1);
      // The tile's B scale blocks: one for 128-column tiles, two (lo, hi) for
      // 256-column tiles; a block past N repeats the last one (no output there).
      const int sbb = kBNs == 256 ? u.nb * 2 : u.nb;
      const float* sa_p = args.sa + static_cast<int64_t>(mb) * args.ld_sa;
      const int nbs = (args.N + kBK - 1) / kBK;  // 128-row scale blocks of B (per expert)
      const float* sb_p = args.sb + (static_cast<int64_t>(ps.g) * nbs + sbb) * args.ld_sb;
      const float* sb_hi = sb_p + (sbb + 1 < nbs ? args.ld_sb : 0);
      for (int sl = 0; sl < unst; ++sl) {
        const int kb0 = su.kb0 + sl * NC::kKbPerStage;
        const bool two = NC::kKbPerStage == 2 && sl * NC::kKbPerStage + 1 < su.nkb;
        const uint32_t ea0 = ue8m0_word(__ldg(sa_p + kb0)), eb0 = ue8m0_word(__ldg(sb_p + kb0));
        const uint32_t ea1 = two ? ue8m0_word(__ldg(sa_p + kb0 + 1)) : ea0;
        const uint32_t eb1 = two ? ue8m0_word(__ldg(sb_p + kb0 + 1)) : eb0;
        const bool w = mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag, status, limit);
        if (!__all_sync(0xFFFFFFFFu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = sf_row + stage * NC::kKbPerStage * NC::kSfCols;
        tmem_st8(col, ea0, ea0, ea0, ea0, eb0, eb0, eb0, eb0);
        if constexpr (kBNs == 256) {
          const uint32_t eh = ue8m0_word(__ldg(sb_hi + kb0));
          tmem_st8(col + 8, eh, eh, eh, eh, eh, eh, eh, eh);
        }
        if constexpr (NC::kKbPerStage == 2) tmem_st8(col + NC::kSfCols, ea1, ea1, ea1, ea1, eb1, eb1, eb1, eb1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_addr(leader_full + stage * 8u);
        if (++stage == static_cast<uint32_t>(S)) {
          stage = 0;
          phase ^= 1u;
        }
      }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - kNatFirstEpiWarp;
    const int part = ew >> 2;   // columns [64 part, 64 part + 64) of the tile
    const int quad = warp & 3;
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + part * 64;
    const uint32_t leader_tempty = mapa_shared(smem_u32(tempty_bar), 0);
    uint8_t* out_box = smem_out + ew * kBoxBytes * NC::kBoxes;
    bool stores_issued = false;
    uint32_t tl = 0;  // MMA units read so far (the accumulator alternates with it)
    uint32_t xl = 0;  // tiles this CTA stored (the requantizing exchange's sequence)
    bool ok = true;
    for (int t = pair; t < num_units && ok; t += num_pairs) {
      // No look-ahead here: the epilogue waits a whole tile for its accumulator,
      // and the prefetched ids would cost registers that its loads need.
      const ScaledUnit su = scaled_unit<kGrouped, kKG>(t, args, pair_unit_ids<kGrouped>(t, args, lane));
      const PairUnit& u = su.u;
      for (int slot = 0; slot < u.nslots; ++slot) {
      const PairSlot ps = pair_slot<kGrouped>(u, slot, args);
      const bool mine = ((ps.keep >> rank) & 1) != 0;
      if constexpr (kBNs == 256) {
        // bf16 output: round each 32-column load to bf16 before the next one,
        // so that 32 registers, not 64, hold the slice.
        uint32_t pk[32];
        if (kGrouped && !ps.mma) {
          if (ps.bad && mine && ew == 0 && lane == 0) atomicOr(status, kStatusBadGroup);
#pragma unroll
          for (int j = 0; j < 32; ++j) pk[j] = 0u;
        } else {
          const uint32_t abuf = tl % NC::kNumAcc;
          const bool w = mbar_wait(smem_u32(&tfull_bar[abuf]), (tl / NC::kNumAcc) & 1u, abort_flag, status, limit);
          if (!__all_sync(0xFFFFFFFFu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t r[32];
            tmem_ld<32>(tmem_row + abuf * kBNs + q * 32, r);
            tmem_wait_ld();
            if (q == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster_addr(leader_tempty + abuf * 8u);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[q * 16 + j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
          }
          ++tl;
        }
        if (!mine) continue;
        const int row0 = u.pm * (2 * kBM) + static_cast<int>(rank) * kBM + quad * 32;
        if constexpr (kGrouped) {
          if (!ps.mma || __ldg(args.m_indices + row0 + lane) < 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) pk[j] = 0u;
          }
        }
        store_packed_rows(pk, tmap_c, args, out_box, row0, u.nb * kBNs + part * 64, lane, stores_issued);
        continue;
      }
      uint64_t acc[32];
      if (kGrouped && !ps.mma) {
        // No MMAs: the kept rows are written as zeros; an id past the last
        // expert is reported in the status word.
        if (ps.bad && mine && ew == 0 && lane == 0) atomicOr(status, kStatusBadGroup);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0ull;
      } else {
        const uint32_t abuf = tl % NC::kNumAcc;
        const bool w = mbar_wait(smem_u32(&tfull_bar[abuf]), (tl / NC::kNumAcc) & 1u, abort_flag, status, limit);
        if (!__all_sync(0xFFFFFFFFu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r[64];
        tmem_ld<32>(tmem_row + abuf * kBNs, &r[0]);
        tmem_ld<32>(tmem_row + abuf * kBNs + 32, &r[32]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_addr(leader_tempty + abuf * 8u);
        ++tl;
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = f32x2(r[2 * j], r[2 * j + 1]);
      }
      if (!mine) continue;
      const int row0 = u.pm * (2 * kBM) + static_cast<int>(rank) * kBM + quad * 32;
      // M-grouped: rows of padding (id -1) are zeros.
      bool zero_row = false;
      if constexpr (kGrouped) {
        zero_row = !ps.mma || __ldg(args.m_indices + row0 + lane) < 0;
        if (zero_row) {
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] = 0ull;
        }
      }
      if constexpr (kQ) {
        if (!requant_store_slice<NC::kEpiWarps>(acc, row0 + lane < args.M && !zero_row, kGrouped, row0, args.M,
                                                args.N, u.nb * kBNs + part * 64, ew, lane, xl, smem_out, args.rq,
                                                &tmap_c, requant_box(smem_out, NC::kEpiWarps, ew), stores_issued,
                                                abort_flag, status, limit)) {
          ok = false;
          break;
        }
        ++xl;
      } else {
        store_tile_rows<64, NC::kBoxes, kKG>(acc, tmap_c, args, out_box, row0, u.nb * kBNs + part * 64, lane,
                                              stores_issued, su.gout);
      }
      }
    }
    if (lane == 0 && stores_issued) bulk_wait_all();
    __syncwarp();
  }

  // ------------------------------------------------------------- teardown --
  __syncthreads();
  if (*abort_flag) {
    const uint64_t drain_ns = 10000000ull;
    if ((warp == 0 || warp == 3) && lane == 0) {
      if (leader) {
        // The last stages this producer filled: g = me + 2k.
        const uint32_t me = warp == 0 ? 0u : 1u;
        const uint32_t per = static_cast<uint32_t>(S) / 2;
        const uint32_t n = loads_issued < per ? loads_issued : per;
        for (uint32_t k = loads_issued - n; k < loads_issued; ++k) {
          const uint32_t g = me + 2 * k;
          drain_wait(smem_u32(&full_bar[g % S]), (g / S) & 1u, drain_ns);
        }
      } else {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 200000ull) {
        }
      }
    }
    if (leader && (warp == 1 || warp == 2) && lane == 0) mma_commit_pair(smem_u32(drain_bar));
    if (leader && warp == 1 && lane == 0) drain_wait(smem_u32(drain_bar), 0, drain_ns);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// The two pair kernels: FP32 scales promoted in registers, or power-of-two
// scales applied by the tensor core.
struct PairKind {
  const void* kernel;
  int threads;
  size_t fixed_smem;    // output staging + barriers
  uint32_t stage_bytes;
  int max_stages;
  int kb_per_stage;
};
template <bool kQ, bool kNT, bool kGrouped, int kBNs>
PairKind nat_kind_t() {
  using NC = NatCfg<kBNs>;
  return {reinterpret_cast<const void*>(&fp8_gemm_pair_scaled_kernel<kQ, kNT, kGrouped, kBNs>), NC::kThreads,
          nat_out_bytes<kBNs>(kQ) + (2 * kNatMaxStages + 4 + 1) * sizeof(uint64_t) + 16, NC::kStageBytes,
          kNatMaxStages, NC::kKbPerStage};
}
// The FP32-promotion pair kernel serves dense calls only (M-grouped calls with
// FP32 scales take the kernels of gemm.cu): kGrouped kinds are block-scaled.
template <bool kQ, bool kNT, bool kGrouped>
PairKind pair_kind_t(bool scaled, bool wide) {
  using C = PCfg<kEpiCols, kQ>;
  if (kGrouped || scaled) {
    if constexpr (!kQ && kNT) {
      if (wide) return nat_kind_t<kQ, kNT, kGrouped, 256>();
    }
    return nat_kind_t<kQ, kNT, kGrouped, 128>();
  }
  return {reinterpret_cast<const void*>(&fp8_gemm_pair_kernel<kEpiCols, kQ, kNT>), C::kThreads,
          C::kOutBytes + (2 * kMaxStages + 2 * kNumBuf + 1) * sizeof(uint64_t) + 16, kStageBytes, kMaxStages, 1};
}
// variant = scaled + 2 * requant + 4 * NT layout + 8 * M-grouped (always NT)
//           + 16 * 256-column block-scaled tiles (bf16 output, NT);
// kKGroupedVariant: the FP32-promotion kernel over K ranges (bf16 output);
// kKGroupedScaledVariant: the block-scaled kernel over K ranges.
constexpr int kKGroupedVariant = 32;
constexpr int kKGroupedScaledVariant = 33;
constexpr int kNumVariants = 34;
PairKind pair_kind(int variant) {
  if (variant == kKGroupedVariant) {
    using C = PCfg<kEpiCols, false>;
    return {reinterpret_cast<const void*>(&fp8_gemm_pair_kernel<kEpiCols, false, false, true>), C::kThreads,
            C::kOutBytes + (2 * kMaxStages + 2 * kNumBuf + 1) * sizeof(uint64_t) + 16, kStageBytes, kMaxStages, 1};
  }
  if (variant == kKGroupedScaledVariant) {
    using NC = NatCfg<128>;
    return {reinterpret_cast<const void*>(&fp8_gemm_pair_scaled_kernel<false, false, false, 128, true>),
            NC::kThreads, nat_out_bytes<128>(false) + (2 * kNatMaxStages + 4 + 1) * sizeof(uint64_t) + 16,
            NC::kStageBytes, kNatMaxStages, NC::kKbPerStage};
  }
  const bool scaled = (variant & 1) != 0, wide = (variant & 16) != 0;
  if (variant & 8)
    return (variant & 2) ? pair_kind_t<true, true, true>(scaled, wide) : pair_kind_t<false, true, true>(scaled, wide);
  if (variant & 4)
    return (variant & 2) ? pair_kind_t<true, true, false>(scaled, wide)
                         : pair_kind_t<false, true, false>(scaled, wide);
  return (variant & 2) ? pair_kind_t<true, false, false>(scaled, wide) : pair_kind_t<false, false, false>(scaled, wide);
}

// Largest number of co-resident CTA pairs of a kernel (cached per device).
int max_active_pairs(int variant, size_t smem) {
  static std::mutex mu;
  static int cache[64][kNumVariants] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][variant];
  if (c == 0) {
    const PairKind k = pair_kind(variant);
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * 512, 1, 1);
    cfg.blockDim = dim3(k.threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k.kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = -1;
    }
    c = n;
  }
  return c;
}

bool set_pair_smem_attribute(int variant) {
  static std::atomic<uint64_t> done[kNumVariants] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::atomic<uint64_t>& d = done[variant];
  if (d.load() & (1ull << dev)) return true;
  if (cudaFuncSetAttribute(pair_kind(variant).kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kMaxDynSmem)) != cudaSuccess)
    return false;
  d.fetch_or(1ull << dev);
  return true;
}

template <bool kQ, bool kNT, bool kGrouped>
cudaError_t launch_pair(bool scaled, bool wide, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                        const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        const PairArgsT<kQ, kGrouped>& a) {
  if (kGrouped || scaled) {
    if constexpr (!kQ && kNT) {
      if (wide)
        return launch_kernel(fp8_gemm_pair_scaled_kernel<kQ, kNT, kGrouped, 256>, grid, block, smem, stream, 2u, ta,
                             tb, tc, a);
    }
    return launch_kernel(fp8_gemm_pair_scaled_kernel<kQ, kNT, kGrouped, 128>, grid, block, smem, stream, 2u, ta, tb,
                         tc, a);
  } else {
    return launch_kernel(fp8_gemm_pair_kernel<kEpiCols, kQ, kNT>, grid, block, smem, stream, 2u, ta, tb, tc, a);
  }
}

// The argument struct of an instantiation: the dense fields, plus the requant
// output and/or the M-grouped fields.
template <bool kQ, bool kG>
PairArgsT<kQ, kG> make_args(const PairArgs& base, const GemmProblem& p) {
  PairArgsT<kQ, kG> a{};
  static_cast<PairArgs&>(a) = base;
  if constexpr (kQ) a.rq = p.rq;
  if constexpr (kG) {
    a.m_indices = p.m_indices;
    a.num_groups = p.num_groups;
  }
  return a;
}

}  // namespace

int launch_gemm_pair(const GemmProblem& p, cudaStream_t stream) {
  const bool grouped = p.m_indices != nullptr;
  if (grouped ? (p.a_mn || p.b_mn) : p.M <= kBM) return DG_ERR_UNSUPPORTED_SHAPE;
  // The block-scaled kernel fills its scale columns uniformly, which needs one
  // A scale per 128 rows; per-row A scales take the FP32 promotion (exact too).
  const bool scaled = p.pow2_scales && !p.sa_per_row;
  if (grouped && !scaled) return DG_ERR_UNSUPPORTED_SHAPE;
  unsigned int* status = device_status_word();
  if (!status) return DG_ERR_CUDA;
  const bool requant = p.rq.q != nullptr;
  const bool nt = !p.a_mn && !p.b_mn;
  // 256-column block-scaled tiles for bf16 output in the NT layout once N spans them.
  const bool wide = scaled && !requant && nt && p.N > kBN;
  const int bn = wide ? 2 * kBN : kBN;
  const int variant = (scaled ? 1 : 0) + (requant ? 2 : 0) + (nt ? 4 : 0) + (grouped ? 8 : 0) + (wide ? 16 : 0);
  const PairKind kind = pair_kind(variant);
  PairArgs args{};
  args.c = static_cast<__nv_bfloat16*>(p.c);
  args.ld_c = p.ld_c;
  args.sa = p.sa;
  args.sa_per_row = p.sa_per_row ? 1 : 0;
  args.sb = p.sb;
  args.status = status;
  args.M = static_cast<int>(p.M);
  args.N = static_cast<int>(p.N);
  args.num_kb = static_cast<int>(p.K / kBK);
  args.ld_sa = static_cast<int>(p.ld_sa);
  args.ld_sb = static_cast<int>(p.ld_sb);
  args.a_mn = p.a_mn ? 1 : 0;
  args.b_mn = p.b_mn ? 1 : 0;
  args.idesc = (scaled ? (wide ? NatCfg<256>::kIdesc : NatCfg<128>::kIdesc) : kIdesc) | idesc_majors(p.a_mn, p.b_mn);
  args.num_mb = static_cast<int>((p.M + kBM - 1) / kBM);
  args.num_pm = static_cast<int>((p.M + 2 * kBM - 1) / (2 * kBM));
  args.num_nb = static_cast<int>((p.N + bn - 1) / bn);
  // All of M in one raster group when A fits comfortably in L2 (B is then
  // read once), else groups of kGroupPM pair rows.
  args.group_pm = (p.M * p.K <= kRasterABytes) ? std::max(args.num_pm, 1) : kGroupPM;
  args.wait_limit_ns = kDefaultWaitLimitNs;

  const size_t budget = kMaxDynSmem - 1024 - kind.fixed_smem;
  int stages = std::min<int>(kind.max_stages, static_cast<int>(budget / kind.stage_bytes));
  stages = stages / 2 * 2;  // issuer (and producer) i owns the stages of index parity i
  if (stages < 4) return DG_ERR_UNSUPPORTED_SHAPE;
  args.num_stages = stages;
  const size_t smem = 1024 + static_cast<size_t>(stages) * kind.stage_bytes + kind.fixed_smem;
  if (!set_pair_smem_attribute(variant)) return DG_ERR_CUDA;

  const int64_t tiles = static_cast<int64_t>(args.num_pm) * args.num_nb * (grouped ? 2 : 1);
  int pairs = max_active_pairs(variant, smem);
  if (pairs <= 0) return DG_ERR_UNSUPPORTED_SHAPE;
  if (p.num_sms_cap > 0) pairs = std::min(pairs, p.num_sms_cap / 2);
  pairs = static_cast<int>(std::min<int64_t>(pairs, tiles));
  if (pairs < 1) return DG_ERR_UNSUPPORTED_SHAPE;

  CUtensorMap ta, tb, tc;
  const uint32_t kbs = static_cast<uint32_t>(kind.kb_per_stage);
  if (p.a_mn) {
    // A as [K][ld_a]: 128 (M) x 128 kb_per_stage (K) boxes, 128-byte swizzle.
    const uint64_t dims[2] = {static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.K)};
    const uint64_t str[1] = {static_cast<uint64_t>(p.ld_a)};
    const uint32_t box[2] = {kBM, kBK * kbs};
    if (!encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 2, dims, str, box, true)) return DG_ERR_CUDA;
  }
  if (p.b_mn) {
    // B as [K][ld_b]: 64 (N) x 128 kb_per_stage (K) boxes, 64-byte swizzle.
    const uint64_t dims[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.K)};
    const uint64_t str[1] = {static_cast<uint64_t>(p.ld_b)};
    const uint32_t box[2] = {kBN / 2, kBK * kbs};
    if (!encode_tensor_map_swizzle(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 2, dims, str, box,
                                   CU_TENSOR_MAP_SWIZZLE_64B))
      return DG_ERR_CUDA;
  }
  if (grouped) {
    // B as [G][N][K] (row stride K): the FP32-promotion kernel loads 2-D
    // {K, N, G} boxes of 128 x 64 x 1; the block-scaled kernel {128, N, K/128,
    // G} boxes of 128 x BN/2 x (K blocks per stage) x 1.
    const uint64_t K = static_cast<uint64_t>(p.K), N = static_cast<uint64_t>(p.N);
    const uint64_t G = static_cast<uint64_t>(p.num_groups);
    if (!scaled) {
      const uint64_t bdims[3] = {K, N, G};
      const uint64_t bstr[2] = {K, K * N};
      const uint32_t bbox[3] = {kBK, kBN / 2, 1};
      if (!encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 3, bdims, bstr, bbox, true)) return DG_ERR_CUDA;
    } else {
      const uint64_t bdims[4] = {kBK, N, K / kBK, G};
      const uint64_t bstr[3] = {K, kBK, K * N};
      const uint32_t bbox[4] = {kBK, static_cast<uint32_t>(bn / 2), kbs, 1};
      if (!encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 4, bdims, bstr, bbox, true)) return DG_ERR_CUDA;
    }
  }
  if (!scaled) {
    // The FP32-promotion kernel: 2-D maps {K, rows}, one K block per box.
    const uint64_t adims[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.M)};
    const uint64_t astr[1] = {static_cast<uint64_t>(p.ld_a)};
    const uint32_t abox[2] = {kBK, kBM};
    const uint64_t bdims[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.N)};
    const uint64_t bstr[1] = {static_cast<uint64_t>(p.ld_b)};
    const uint32_t bbox[2] = {kBK, kBN / 2};
    if ((!p.a_mn && !encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 2, adims, astr, abox, true)) ||
        (!p.b_mn && !grouped && !encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 2, bdims, bstr, bbox, true)))
      return DG_ERR_CUDA;
  } else {
    // The block-scaled kernel: 3-D maps [K/128][rows][128 bytes], one box
    // carries the stage's K blocks (B: BN/2 rows per CTA).
    const uint64_t adims[3] = {kBK, static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.K / kBK)};
    const uint64_t astr[2] = {static_cast<uint64_t>(p.ld_a), kBK};
    const uint32_t abox[3] = {kBK, kBM, kbs};
    const uint64_t bdims[3] = {kBK, static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.K / kBK)};
    const uint64_t bstr[2] = {static_cast<uint64_t>(p.ld_b), kBK};
    const uint32_t bbox[3] = {kBK, static_cast<uint32_t>(bn / 2), kbs};
    if ((!p.a_mn && !encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 3, adims, astr, abox, true)) ||
        (!p.b_mn && !grouped && !encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 3, bdims, bstr, bbox, true)))
      return DG_ERR_CUDA;
  }
  if (requant) {
    // E4M3 codes [M][ld_q]: 64 x 32 boxes, 64-byte swizzle.
    const uint64_t dims[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.rq.ld_q)};
    const uint32_t box[2] = {64, 32};
    if (!encode_tensor_map_swizzle(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.rq.q, 2, dims, strides, box,
                                   CU_TENSOR_MAP_SWIZZLE_64B))
      return DG_ERR_CUDA;
  } else {
    // C as bf16 [M][ld_c]: 32 x 32 boxes, 64-byte swizzle (the FP32-promotion
    // kernel: 32 x 64 boxes, 128-byte swizzle).
    const uint64_t dims[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.ld_c) * 2};
    const uint32_t box[2] = {scaled ? 32u : 64u, 32};
    if (!encode_tensor_map_swizzle(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.c, 2, dims, strides, box,
                                   scaled ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
      return DG_ERR_CUDA;
  }

  cudaError_t e;
  const dim3 grid(2 * pairs), block(kind.threads);
  if (requant) {
    e = grouped ? launch_pair<true, true, true>(scaled, wide, grid, block, smem, stream, ta, tb, tc,
                                                make_args<true, true>(args, p))
        : nt    ? launch_pair<true, true, false>(scaled, wide, grid, block, smem, stream, ta, tb, tc,
                                                 make_args<true, false>(args, p))
                : launch_pair<true, false, false>(scaled, wide, grid, block, smem, stream, ta, tb, tc,
                                                  make_args<true, false>(args, p));
  } else {
    e = grouped ? launch_pair<false, true, true>(scaled, wide, grid, block, smem, stream, ta, tb, tc,
                                                 make_args<false, true>(args, p))
        : nt    ? launch_pair<false, true, false>(scaled, wide, grid, block, smem, stream, ta, tb, tc, args)
                : launch_pair<false, false, false>(scaled, wide, grid, block, smem, stream, ta, tb, tc, args);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  return DG_OK;
}

int launch_gemm_pair_k_grouped(const GemmProblem& p, const int64_t* k_sizes, int num_groups, cudaStream_t stream) {
  if (p.rq.q || p.m_indices || p.sa_per_row || !p.a_mn || !p.b_mn || p.M <= kBM) return DG_ERR_UNSUPPORTED_SHAPE;
  // Power-of-two scales: the block-scaled kernel (accumulators stay in TMEM
  // across each range's K blocks); FP32 scales: the promotion kernel.
  const bool scaled = p.pow2_scales;
  const int variant = scaled ? kKGroupedScaledVariant : kKGroupedVariant;
  PairArgsKG args{};
  int nkg = 0;
  int64_t kb = 0, max_k = 0;
  for (int g = 0; g < num_groups; ++g) {
    if (k_sizes[g] > 0) {
      if (nkg == kMaxKGroups) return DG_ERR_UNSUPPORTED_SHAPE;
      args.kb_lo[nkg] = static_cast<int>(kb);
      args.kb_n[nkg] = static_cast<int>(k_sizes[g] / kBK);
      args.g_out[nkg] = g;
      ++nkg;
      max_k = std::max(max_k, k_sizes[g]);
    }
    kb += k_sizes[g] / kBK;
  }
  if (nkg == 0) return DG_OK;
  args.num_kg = nkg;
  unsigned int* status = device_status_word();
  if (!status) return DG_ERR_CUDA;
  args.c = static_cast<__nv_bfloat16*>(p.c);
  args.ld_c = p.ld_c;
  args.sa = p.sa;
  args.sa_per_row = 0;
  args.sb = p.sb;
  args.status = status;
  args.M = static_cast<int>(p.M);
  args.N = static_cast<int>(p.N);
  args.num_kb = static_cast<int>(kb);
  args.ld_sa = static_cast<int>(p.ld_sa);
  args.ld_sb = static_cast<int>(p.ld_sb);
  args.a_mn = 1;
  args.b_mn = 1;
  args.idesc = (scaled ? NatCfg<128>::kIdesc : kIdesc) | idesc_majors(true, true);
  args.num_mb = static_cast<int>((p.M + kBM - 1) / kBM);
  args.num_pm = static_cast<int>((p.M + 2 * kBM - 1) / (2 * kBM));
  args.num_nb = static_cast<int>((p.N + kBN - 1) / kBN);
  args.group_pm = (p.M * max_k <= kRasterABytes) ? std::max(args.num_pm, 1) : kGroupPM;
  args.wait_limit_ns = kDefaultWaitLimitNs;

  const PairKind kind = pair_kind(variant);
  const size_t budget = kMaxDynSmem - 1024 - kind.fixed_smem;
  int stages = std::min<int>(kind.max_stages, static_cast<int>(budget / kind.stage_bytes));
  stages = stages / 2 * 2;
  if (stages < 4) return DG_ERR_UNSUPPORTED_SHAPE;
  args.num_stages = stages;
  const size_t smem = 1024 + static_cast<size_t>(stages) * kind.stage_bytes + kind.fixed_smem;
  if (!set_pair_smem_attribute(variant)) return DG_ERR_CUDA;
  const int64_t units = static_cast<int64_t>(args.num_pm) * args.num_nb * nkg;
  int pairs = max_active_pairs(variant, smem);
  if (pairs <= 0) return DG_ERR_UNSUPPORTED_SHAPE;
  if (p.num_sms_cap > 0) pairs = std::min(pairs, p.num_sms_cap / 2);
  pairs = static_cast<int>(std::min<int64_t>(pairs, units));
  if (pairs < 1) return DG_ERR_UNSUPPORTED_SHAPE;

  CUtensorMap ta, tb, tc;
  const uint32_t kbs = static_cast<uint32_t>(kind.kb_per_stage);
  {
    // A as [K_tot][ld_a]: 128 (M) x 128 kb_per_stage (K) boxes, 128-byte swizzle.
    const uint64_t dims[2] = {static_cast<uint64_t>(p.M), static_cast<uint64_t>(kb * kBK)};
    const uint64_t str[1] = {static_cast<uint64_t>(p.ld_a)};
    const uint32_t box[2] = {kBM, kBK * kbs};
    if (!encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 2, dims, str, box, true)) return DG_ERR_CUDA;
  }
  {
    // B as [K_tot][ld_b]: 64 (N) x 128 kb_per_stage (K) boxes, 64-byte swizzle.
    const uint64_t dims[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(kb * kBK)};
    const uint64_t str[1] = {static_cast<uint64_t>(p.ld_b)};
    const uint32_t box[2] = {kBN / 2, kBK * kbs};
    if (!encode_tensor_map_swizzle(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 2, dims, str, box,
                                   CU_TENSOR_MAP_SWIZZLE_64B))
      return DG_ERR_CUDA;
  }
  {
    // C as bf16 [G][M][ld_c]: 64 x 32 x 1 boxes, 128-byte swizzle (the
    // block-scaled kernel: 32 x 32 x 1, 64-byte swizzle); rows past M of one
    // matrix are clipped instead of reaching the next.
    const uint64_t dims[3] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.M),
                              static_cast<uint64_t>(num_groups)};
    const uint64_t str[2] = {static_cast<uint64_t>(p.ld_c) * 2, static_cast<uint64_t>(p.ld_c) * 2 * p.M};
    const uint32_t box[3] = {scaled ? 32u : 64u, 32, 1};
    if (!encode_tensor_map_swizzle(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.c, 3, dims, str, box,
                                   scaled ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
      return DG_ERR_CUDA;
  }
  const cudaError_t e =
      scaled ? launch_kernel(fp8_gemm_pair_scaled_kernel<false, false, false, 128, true>, dim3(2 * pairs),
                             dim3(kind.threads), smem, stream, 2u, ta, tb, tc, args)
             : launch_kernel(fp8_gemm_pair_kernel<kEpiCols, false, false, true>, dim3(2 * pairs),
                             dim3(kind.threads), smem, stream, 2u, ta, tb, tc, args);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  return DG_OK;
}

}  // namespace dg
