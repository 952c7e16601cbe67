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
//   * CTA r of a pair loads A rows [256 pm + 128 r, +128) and B rows
//     [128 nb + 64 r, +64) of every K block with TMA; both loads count on the
//     even CTA's `full` barrier, which the even CTA arms for both CTAs' bytes;
//   * warps 1 and 2 of the even CTA take turns issuing the four MMAs (K = 32)
//     of a K block into TMEM buffer it % 4 of both CTAs; each commit arrives on
//     the stage's `empty` barrier and the buffer's `tfull` barrier in both
//     CTAs. Issuer i owns the stages and buffers of index parity i, so each
//     barrier it waits on sees its phases in order;
//   * the epilogue warps of each CTA read their 32 TMEM lanes of the partial,
//     release the buffer by arriving on the even CTA's `tempty` barrier, and
//     promote it in registers (two FP32 FMAs per f32x2 instruction, each
//     rounded like fmaf). After the last K block each warp rounds its 32 x 32
//     boxes to bf16 and writes them with TMA stores clipped at the M and N edges;
//   * pairs are persistent over the 256x128 tiles in a grouped raster.
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

#include "../../include/dgfp8.h"
#include "dg_device.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kBM = 128;               // rows per CTA (256 per pair)
constexpr int kBN = 128;               // columns per pair tile
constexpr int kBK = 128;               // K block = scale block
constexpr int kMaxStages = 16;
constexpr int kNumBuf = 4;             // TMEM partial buffers of 128 columns
constexpr int kIssuers = 2;
constexpr int kGroupPM = 8;            // raster group height in pair rows
constexpr uint32_t kABytes = kBM * kBK;            // 16 KB
constexpr uint32_t kBHalfBytes = (kBN / 2) * kBK;  // 8 KB
constexpr uint32_t kStageBytes = kABytes + kBHalfBytes;
constexpr uint32_t kBoxBytes = 32 * 32 * 2;        // one warp's 32 x 32 bf16 output box
constexpr size_t kMaxDynSmem = 227 * 1024;
constexpr uint32_t kIdesc = idesc_e4m3_f32(2 * kBM, kBN);

template <int kEpiCols>
struct PCfg {
  static constexpr int kEpiPerQuad = kBN / kEpiCols;  // warps per TMEM lane quadrant
  static constexpr int kEpiWarps = 4 * kEpiPerQuad;
  static constexpr int kFirstEpiWarp = 1 + kIssuers;
  static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
  static constexpr uint32_t kOutBytes = kEpiWarps * kBoxBytes;
  static_assert(kEpiCols == 32 || kEpiCols == 64, "epilogue slice");
  static_assert(kThreads <= 1024, "CTA size");
};
constexpr int kEpiCols = 64;

struct PairArgs {
  __nv_bfloat16* c;
  int64_t ld_c;
  const float* sa;
  const float* sb;
  unsigned int* status;
  int M, N;
  int num_kb;   // K / 128
  int num_mb;   // ceil(M / 128)
  int num_pm;   // ceil(M / 256)
  int num_nb;   // ceil(N / 128)
  int num_stages;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void pair_tile_coords(int t, int num_pm, int num_nb, int& pm, int& nb) {
  const int per_group = kGroupPM * num_nb;
  const int grp = t / per_group;
  const int first = grp * kGroupPM;
  const int gm = min(kGroupPM, num_pm - first);
  const int r = t - grp * per_group;
  pm = first + r % gm;
  nb = r / gm;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) break;
  }
}

template <int EC>
__global__ void __launch_bounds__(PCfg<EC>::kThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_c, const PairArgs args) {
  using C = PCfg<EC>;
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
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_c);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kNumBuf * kBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or load
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = args.num_pm * args.num_nb;
  uint32_t loads_issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    // Lane 0 works; the warp shares its SM sub-partition with busy epilogue
    // warps, so the loop keeps its stage and phase in running counters.
    if (lane == 0) {
      const uint32_t leader_full = mapa_shared(smem_u32(full_bar), 0);
      const uint32_t empty0 = smem_u32(empty_bar);
      const uint32_t ring0 = smem_u32(ring);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += num_pairs) {
        int pm, nb;
        pair_tile_coords(t, args.num_pm, args.num_nb, pm, nb);
        const int arow = pm * (2 * kBM) + static_cast<int>(rank) * kBM;
        const int brow = nb * kBN + static_cast<int>(rank) * (kBN / 2);
        for (int kb = 0; kb < args.num_kb; ++kb) {
          ok = mbar_wait(empty0 + stage * 8u, phase ^ 1u, abort_flag, status, limit);
          if (!ok) break;
          if (leader) mbar_arrive_expect_tx(smem_u32(&full_bar[stage]), 2u * kStageBytes);
          const uint32_t fb = leader_full + stage * 8u;
          const uint32_t dst = ring0 + stage * kStageBytes;
          tma_load_2d_pair(dst, &tmap_a, fb, kb * kBK, arow);
          tma_load_2d_pair(dst + kABytes, &tmap_b, fb, kb * kBK, brow);
          ++loads_issued;
          if (++stage == static_cast<uint32_t>(S)) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp <= kIssuers) {
    // ----------------------------------------------------------- MMA issue --
    // Issuer i takes K blocks i, i + 2, i + 4, ... of this pair's sequence, so
    // its stages and buffers advance by two (S is even, four buffers).
    if (leader && lane == 0) {
      const uint32_t me = static_cast<uint32_t>(warp - 1);
      const int my_tiles = num_tiles > pair ? (num_tiles - 1 - pair) / num_pairs + 1 : 0;
      const uint32_t total = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(args.num_kb);
      const uint32_t full0 = smem_u32(full_bar), empty0 = smem_u32(empty_bar);
      const uint32_t tfull0 = smem_u32(tfull_bar), tempty0 = smem_u32(tempty_bar);
      const uint32_t ring0 = smem_u32(ring);
      uint32_t stage = me, sphase = 0, buf = me, bphase = 0;
      for (uint32_t it = me; it < total; it += kIssuers) {
        if (!mbar_wait(tempty0 + buf * 8u, bphase ^ 1u, abort_flag, status, limit)) break;
        if (!mbar_wait(full0 + stage * 8u, sphase, abort_flag, status, limit)) break;
        tc_fence_after();
        const uint32_t base = ring0 + stage * kStageBytes;
        const uint64_t adesc = sw128_kmajor_desc(base);
        const uint64_t bdesc = sw128_kmajor_desc(base + kABytes);
        const uint32_t d = tmem_base + buf * kBN;
#pragma unroll
        for (int k = 0; k < kBK / 32; ++k)
          mma_e4m3_pair(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, k > 0 ? 1u : 0u);
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
    uint8_t* out_box = smem_out + ew * kBoxBytes;
    bool stores_issued = false;
    uint32_t it = 0;
    bool ok = true;
    bool ready = false;  // the full barrier of slot `it` is known to be complete
    for (int t = pair; t < num_tiles && ok; t += num_pairs) {
      int pm, nb;
      pair_tile_coords(t, args.num_pm, args.num_nb, pm, nb);
      const int mb = min(pm * 2 + static_cast<int>(rank), args.num_mb - 1);
      const float* sa_p = args.sa + static_cast<int64_t>(mb) * args.num_kb;
      const float* sb_p = args.sb + static_cast<int64_t>(nb) * args.num_kb;
      uint64_t acc[EC / 2];  // FP32 accumulators, two columns per register pair
#pragma unroll
      for (int j = 0; j < EC / 2; ++j) acc[j] = 0ull;
      float s = __ldg(sa_p) * __ldg(sb_p);
      for (int kb = 0; kb < args.num_kb; ++kb, ++it) {
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
#pragma unroll
        for (int q = 0; q < EC / 32; ++q) tmem_ld<32>(tmem_row + buf * kBN + q * 32, &r[q * 32]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_addr(leader_tempty + buf * 8u);
        // Look ahead: test the next slot's barrier and fetch its scales now, so
        // that their latency hides behind the multiply-adds below.
        const uint32_t nx = it + 1;
        const bool next_done = mbar_test(smem_u32(&tfull_bar[nx % kNumBuf]), (nx / kNumBuf) & 1u);
        const float s_next = kb + 1 < args.num_kb ? __ldg(sa_p + kb + 1) * __ldg(sb_p + kb + 1) : 0.f;
        const uint64_t s2 = f32x2(__float_as_uint(s), __float_as_uint(s));
#pragma unroll
        for (int j = 0; j < EC / 2; ++j) ffma2(acc[j], s2, f32x2(r[2 * j], r[2 * j + 1]));
        ready = __all_sync(0xFFFFFFFFu, next_done);
        s = s_next;
      }
      if (!ok) break;

      // bf16 row segment -> this warp's 64-byte-swizzled 32 x 32 box (16-byte
      // chunk c of row r at chunk c ^ ((r / 2) % 4)) -> TMA store, clipped at M.
      // A box that crosses column N is written element by element instead: the
      // swizzled store clips N only to whole 16-byte chunks.
      const int row0 = pm * (2 * kBM) + static_cast<int>(rank) * kBM + quad * 32;
      const int col0 = nb * kBN + part * EC;
#pragma unroll
      for (int h = 0; h < EC / 32; ++h) {
        const int bcol = col0 + 32 * h;
        if (bcol + 32 > args.N) {
          const int row = row0 + lane;
          if (row < args.M && bcol < args.N) {
            __nv_bfloat16* crow = args.c + static_cast<int64_t>(row) * args.ld_c;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float2 v = f32x2_split(acc[h * 16 + j]);
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
          const float2 v0 = f32x2_split(acc[h * 16 + c * 4]), v1 = f32x2_split(acc[h * 16 + c * 4 + 1]);
          const float2 v2 = f32x2_split(acc[h * 16 + c * 4 + 2]), v3 = f32x2_split(acc[h * 16 + c * 4 + 3]);
          uint4 pk;
          pk.x = pack_bf16(v0.x, v0.y);
          pk.y = pack_bf16(v1.x, v1.y);
          pk.z = pack_bf16(v2.x, v2.y);
          pk.w = pack_bf16(v3.x, v3.y);
          *reinterpret_cast<uint4*>(my_row + ((c ^ ((lane >> 1) & 3)) << 4)) = pk;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < args.M) {
          tma_store_2d(&tmap_c, smem_u32(out_box), bcol, row0);
          bulk_commit();
          stores_issued = true;
        }
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

// Largest number of co-resident CTA pairs (cached per device).
int max_active_pairs(size_t smem) {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * 512, 1, 1);
    cfg.blockDim = dim3(PCfg<kEpiCols>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_pair_kernel<kEpiCols>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = -1;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

bool set_pair_smem_attribute() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (done.load() & (1ull << dev)) return true;
  if (cudaFuncSetAttribute(fp8_gemm_pair_kernel<kEpiCols>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kMaxDynSmem)) != cudaSuccess)
    return false;
  done.fetch_or(1ull << dev);
  return true;
}

}  // namespace

int launch_gemm_pair(const GemmProblem& p, cudaStream_t stream) {
  using Cf = PCfg<kEpiCols>;
  if (p.m_indices != nullptr || p.M <= kBM) return DG_ERR_UNSUPPORTED_SHAPE;
  unsigned int* status = device_status_word();
  if (!status) return DG_ERR_CUDA;
  PairArgs args{};
  args.c = static_cast<__nv_bfloat16*>(p.c);
  args.ld_c = p.ld_c;
  args.sa = p.sa;
  args.sb = p.sb;
  args.status = status;
  args.M = static_cast<int>(p.M);
  args.N = static_cast<int>(p.N);
  args.num_kb = static_cast<int>(p.K / kBK);
  args.num_mb = static_cast<int>((p.M + kBM - 1) / kBM);
  args.num_pm = static_cast<int>((p.M + 2 * kBM - 1) / (2 * kBM));
  args.num_nb = static_cast<int>((p.N + kBN - 1) / kBN);
  args.wait_limit_ns = kDefaultWaitLimitNs;

  const size_t bar_bytes = (2 * kMaxStages + 2 * kNumBuf + 1) * sizeof(uint64_t) + 16;
  const size_t budget = kMaxDynSmem - 1024 - Cf::kOutBytes - bar_bytes;
  int stages = std::min<int>(kMaxStages, static_cast<int>(budget / kStageBytes));
  stages = stages / kIssuers * kIssuers;  // issuer i owns the stages of index parity i
  if (stages < 2 * kIssuers) return DG_ERR_UNSUPPORTED_SHAPE;
  args.num_stages = stages;
  const size_t smem = 1024 + static_cast<size_t>(stages) * kStageBytes + Cf::kOutBytes + bar_bytes;
  if (!set_pair_smem_attribute()) return DG_ERR_CUDA;

  const int64_t tiles = static_cast<int64_t>(args.num_pm) * args.num_nb;
  int pairs = max_active_pairs(smem);
  if (pairs <= 0) return DG_ERR_UNSUPPORTED_SHAPE;
  if (p.num_sms_cap > 0) pairs = std::min(pairs, p.num_sms_cap / 2);
  pairs = static_cast<int>(std::min<int64_t>(pairs, tiles));
  if (pairs < 1) return DG_ERR_UNSUPPORTED_SHAPE;

  CUtensorMap ta, tb, tc;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.ld_a)};
    const uint32_t box[2] = {kBK, kBM};
    if (!encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 2, dims, strides, box, true))
      return DG_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.N)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.ld_b)};
    const uint32_t box[2] = {kBK, kBN / 2};
    if (!encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 2, dims, strides, box, true))
      return DG_ERR_CUDA;
  }
  {
    // C as bf16 [M][ld_c]: 32 x 32 boxes, 64-byte swizzle.
    const uint64_t dims[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.ld_c) * 2};
    const uint32_t box[2] = {32, 32};
    if (!encode_tensor_map_swizzle(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.c, 2, dims, strides, box,
                                   CU_TENSOR_MAP_SWIZZLE_64B))
      return DG_ERR_CUDA;
  }

  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(Cf::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fp8_gemm_pair_kernel<kEpiCols>, ta, tb, tc, args) != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  return DG_OK;
}

}  // namespace dg
