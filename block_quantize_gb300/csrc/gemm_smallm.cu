// gemm_smallm.cu -- block-scaled NT GEMM for small M (M <= 128, decode shapes).
//
// Same arithmetic as gemm.cu (lpnh.cn DeepGEMM walkthrough §2.2, §3.2; pzsr.cn
// "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1, §4.1): per 128-wide K block the
// partial products are restored with sa*sb and accumulated in FP32. With few
// rows the work is streaming B from HBM, so the kernel is shaped for bytes in
// flight on as many SMs as possible:
//   * a thread-block cluster of `split` CTAs shares one BN-column tile of C
//     (BN = 128, 192 or 256, see plan_and_run); CTA r of the cluster streams B over
//     its own contiguous K range through a deep TMA ring, issues the MMAs and
//     promotes the partials in registers exactly like the large-M kernel.
//     TMA boxes of 128-byte rows stream at ~40 GB/s per SM and, over all SMs,
//     at ~4.8 TB/s with 128-row boxes and ~5.4 TB/s with 256-row boxes
//     (measured on GB300), hence wide tiles and a split of K over the SMs;
//   * the cluster then reduces its `split` FP32 partial tiles through
//     distributed shared memory: CTA r owns a share of the tile's columns;
//     every CTA stores each column unit of its partial into slot `rank` of
//     the owner's buffer (remote stores) and signals every peer's `ready`
//     mbarrier; CTA r sums the slots of its share in rank order
//     (deterministic), rounds to bf16 and stores; then it signals every peer's
//     `consumed` mbarrier so the buffers can be refilled for the next tile;
//   * clusters are persistent over the N tiles.
// All waits are bounded (see dg_device.cuh). The only unbounded synchronisation
// is the cluster-wide barrier at kernel start (peers' barriers initialised
// before any remote arrive) and at kernel end (no CTA leaves while a peer may
// still read its shared memory), both executed unconditionally by every thread.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "../../include/dgfp8.h"
#include "dg_device.cuh"
#include "dg_encode.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kMaxStages = 32;
constexpr uint32_t kATileBytes = kBM * kBK;
constexpr size_t kMaxDynSmem = 227 * 1024;
constexpr size_t kMinSmemPerCta = 120 * 1024;
constexpr int kMaxSplit = 8;
constexpr int kMaxSplitC = kMaxSplit;

template <int BN, bool kQ = false>
struct SCfg {
  // TMEM: 512 columns of buffers. Issuer i owns the buffers and the stages
  // congruent to i modulo the issuer count, so every mbarrier has one
  // in-order waiter.
  static constexpr int kNumPBuf = 512 / BN;
  // The requantizing 128-column kernel takes two issuers (two buffers each):
  // with 13 warps the compiler holds every thread to 128 registers, and the
  // tile-end code spilled; 11 warps give it 168 (16x7168x16384: 39.2 -> 29.9 us).
  static constexpr int kIssuers = (kQ && BN == 128) ? 2 : kNumPBuf;
  static constexpr int kFirstEpiWarp = 1 + kIssuers;
  static constexpr int kGroups = BN / 64;           // 64-column groups per tile
  static constexpr int kEpiWarps = 4 * kGroups;     // x 4 lane quadrants
  static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
  static constexpr uint32_t kBTileBytes = BN * kBK;
  static constexpr int kUnits = BN / 8;             // 8-column units of a tile (column shares)
  // Columns per tcgen05.ld: 16 when 19 warps leave 96 registers per thread.
  static constexpr int kChunk = (kThreads > 512) ? 16 : 32;
  static constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, BN);
  static_assert(kThreads <= 1024, "CTA size");
  // Requantized output: 128-column blocks per tile, and the shared memory of
  // the block-max exchange (per tile parity: the epilogue slices' exchange of
  // a CTA that reduces alone, this CTA's partial maxima and every rank's copy
  // of them, and two pairs of barriers).
  static constexpr int kNBlk = BN / 128;
  static constexpr uint32_t kRqXchg = (requant_xchg_bytes(kEpiWarps) + 15u) / 16u * 16u;
  static constexpr uint32_t kRqPmaxWords = 2 * kBM * kNBlk;
  static constexpr uint32_t kRqXmaxWords = 2 * kMaxSplitC * kBM * kNBlk;
  static constexpr uint32_t kRqBytes = kRqXchg + 4 * (kRqPmaxWords + kRqXmaxWords) + 4 * 8;
};

struct SmallArgs {
  __nv_bfloat16* c;
  int sa_per_row;  // sa is [M][K/128] instead of [1][K/128]
  int64_t ld_c;
  const float* sa;
  const float* sb;
  unsigned int* status;
  int M, N;
  int num_kb, num_nb, nbs;
  int ld_sa, ld_sb;   // row strides of sa and sb (floats)
  uint32_t idesc;     // MMA instruction descriptor (shape and operand majorness)
  int a_mn, b_mn;     // MN-major A ([K][M]) / B ([K][N]) tiles
  int split;          // cluster size = number of K ranges
  int num_clusters;   // persistent clusters (grid = num_clusters * split)
  int num_stages;
  int part_stride;    // floats per row of a reduction slot (split >= 2)
  uint32_t a_stage_bytes, a_box_bytes;
  uint64_t wait_limit_ns;
};

// Arguments of the requantizing kernels. A separate type: with the extra
// fields in the common struct the bf16 kernel with 256-column tiles spilled
// more registers and lost ~1 us per decode call (measured).
struct SmallArgsQ : SmallArgs {
  RequantOut rq;      // E4M3 output
};
template <bool kQ>
using SmallArgsT = std::conditional_t<kQ, SmallArgsQ, SmallArgs>;

// Column shares of a cluster of `split` CTAs over a tile of `units` 8-column
// units: rank r reduces and stores units [floor(r units / split),
// floor((r + 1) units / split)).
__host__ __device__ constexpr int share_lo(int r, int units, int split) { return r * units / split; }
// Rank whose share holds unit u: the largest r with share_lo(r) <= u.
__host__ __device__ constexpr int share_owner(int u, int units, int split) {
  return ((u + 1) * split + units - 1) / units - 1;
}
// Widest share, in columns.
__host__ __device__ constexpr int share_cols_max(int units, int split) { return (units + split - 1) / split * 8; }

__device__ __forceinline__ void st_dsmem_f4(uint32_t cluster_addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// Eight consecutive outputs at column gcol as bf16 (a 16-byte store when all
// eight are inside the matrix, else element by element up to N).
__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* dst, int gcol, int N, float2 a, float2 b,
                                             float2 c, float2 d) {
  if (gcol + 8 <= N) {
    uint4 pk;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(b.x, b.y);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(c.x, c.y);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(d.x, d.y);
    pk.x = *reinterpret_cast<uint32_t*>(&h0);
    pk.y = *reinterpret_cast<uint32_t*>(&h1);
    pk.z = *reinterpret_cast<uint32_t*>(&h2);
    pk.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(dst) = pk;
  } else {
    const float v[8] = {a.x, a.y, b.x, b.y, c.x, c.y, d.x, d.y};
    for (int q = 0; q < 8; ++q)
      if (gcol + q < N) dst[q] = __float2bfloat16_rn(v[q]);
  }
}

// Requantizing end of a tile for a cluster of split >= 2 CTAs. This CTA has
// the sums of its column share; the block maxima span the cluster:
//   1. sum this thread's items (row, 8 columns) over the ranks' slots of this
//      CTA's buffer in rank order and keep them in registers (at most 4 items:
//      work <= M * ceil(BN/8/split) <= 8 BN items over 2 BN threads), then
//      tell every peer that the buffer is read (`consumed`);
//   2. fold each item's max|v| into this CTA's maxima (shared atomicMax on the
//      bit patterns of non-negative floats), per (row, 128-column block) or
//      per block; wait until every epilogue warp of the CTA has folded;
//   3. write the CTA's maxima into slot `rank` of every peer and arrive on the
//      peer's exchange barrier (lane s -> peer s); wait on this CTA's;
//   4. the block max is the max over the ranks' slots: scale, encode the
//      items and store their 8 codes; rank 0 stores the scales.
// Two parities alternate between tiles. A parity's maxima are cleared after
// its exchange wait (every local warp has sent them by then); a peer writes a
// parity's slot again only after the next tile's exchange, which comes after
// this CTA's reads. Returns false if a wait failed.
template <int BN>
__device__ __forceinline__ bool requant_cluster_tile(const SmallArgsQ& args, const float* part, uint32_t rank,
                                                     int split, int nb, int col_lo, int groups8, int work, int ew,
                                                     int lane, uint32_t tile_seq, uint32_t* rq_pmax,
                                                     uint32_t* rq_xmax, uint64_t* rq_bar, uint64_t* consumed_bar,
                                                     volatile int* abort_flag, unsigned int* status,
                                                     uint64_t limit) {
  using C = SCfg<BN, true>;
  constexpr int kNB = C::kNBlk;
  constexpr int kT = C::kEpiWarps * 32;
  const RequantOut& o = args.rq;
  const bool per_row = o.block_rows == 1;
  const uint32_t p = tile_seq & 1u;
  const uint32_t ph = (tile_seq >> 1) & 1u;
  uint32_t* pm = rq_pmax + p * (kBM * kNB);
  uint32_t* xm = rq_xmax + p * (kMaxSplit * kBM * kNB);
  const int tid = ew * 32 + lane;

  float v[4][8];
  int rr[4], col[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int g = tid + i * kT;
    rr[i] = -1;
    col[i] = 0;
    if (g < work) {
      rr[i] = g / groups8;
      col[i] = col_lo + (g % groups8) * 8;
#pragma unroll
      for (int q = 0; q < 8; ++q) v[i][q] = 0.f;
      const float* src = part + rr[i] * args.part_stride + (col[i] - col_lo);
      for (int s = 0; s < split; ++s) {
        const float* q = src + s * args.M * args.part_stride;
        const float4 x0 = *reinterpret_cast<const float4*>(q), x1 = *reinterpret_cast<const float4*>(q + 4);
        v[i][0] += x0.x; v[i][1] += x0.y; v[i][2] += x0.z; v[i][3] += x0.w;
        v[i][4] += x1.x; v[i][5] += x1.y; v[i][6] += x1.z; v[i][7] += x1.w;
      }
    }
  }
  __syncwarp();
  if (lane < split) mbar_arrive_remote(mapa_shared(smem_u32(consumed_bar), lane));

  // 2. this CTA's maxima
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (rr[i] < 0) continue;
    float m = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(v[i][q]));
    atomicMax(&pm[(per_row ? rr[i] : 0) * kNB + col[i] / 128], __float_as_uint(m));
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&rq_bar[2 + p]));
  if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&rq_bar[2 + p]), ph, abort_flag, status, limit))) return false;

  // 3. send them to every rank (this one included)
  const int entries = (per_row ? args.M : 1) * kNB;
  for (int e = tid; e < entries * split; e += kT) {
    const int s = e % split, ent = e / split;
    st_dsmem_u32(mapa_shared(smem_u32(xm + static_cast<int>(rank) * (kBM * kNB) + ent), s), pm[ent]);
  }
  __syncwarp();
  if (lane < split) mbar_arrive_remote(mapa_shared(smem_u32(&rq_bar[p]), lane));
  if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(smem_u32(&rq_bar[p]), ph, abort_flag, status, limit)))
    return false;
  for (int e = tid; e < entries; e += kT) pm[e] = 0u;  // ready for tile + 2

  // 4. scales, codes
  const bool pow2 = o.pow2 != 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (rr[i] < 0) continue;
    const int ent = (per_row ? rr[i] : 0) * kNB + col[i] / 128;
    uint32_t am = 0u;
    for (int s = 0; s < split; ++s) am = max(am, xm[s * (kBM * kNB) + ent]);
    const float sc = block_scale(__uint_as_float(am), pow2);
    const float r = 1.0f / sc;
    const uint64_t r2 = f32x2(__float_as_uint(r), __float_as_uint(r));
    const uint32_t c0 = encode4_pairs(f32x2(__float_as_uint(v[i][0]), __float_as_uint(v[i][1])),
                                      f32x2(__float_as_uint(v[i][2]), __float_as_uint(v[i][3])), sc, r2, pow2);
    const uint32_t c1 = encode4_pairs(f32x2(__float_as_uint(v[i][4]), __float_as_uint(v[i][5])),
                                      f32x2(__float_as_uint(v[i][6]), __float_as_uint(v[i][7])), sc, r2, pow2);
    const int gcol = nb * BN + col[i];
    uint8_t* dst = o.q + static_cast<int64_t>(rr[i]) * o.ld_q + gcol;
    if (gcol + 8 <= args.N) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(c0, c1);  // 8-byte aligned: gcol % 8 == 0, ld_q % 16 == 0
    } else {
      const uint64_t cc = (static_cast<uint64_t>(c1) << 32) | c0;
      for (int q = 0; q < 8; ++q)
        if (gcol + q < args.N) dst[q] = static_cast<uint8_t>(cc >> (8 * q));
    }
  }
  if (rank == 0) {
    for (int e = tid; e < entries; e += kT) {
      const int gblk = nb * kNB + e % kNB;
      if (gblk * 128 >= args.N) continue;
      uint32_t am = 0u;
      for (int s = 0; s < split; ++s) am = max(am, xm[s * (kBM * kNB) + e]);
      o.s[static_cast<int64_t>(per_row ? e / kNB : 0) * o.ld_s + gblk] = block_scale(__uint_as_float(am), pow2);
    }
  }
  __syncwarp();
  return true;
}

// kRed: the plan splits K (split >= 2) and the cluster reduces. The
// instantiations without it carry no reduction code, which kept the compiler's
// register allocation of their K loop as lean as before the reduction grew.
template <int BN, bool kQ, bool kRed>
__global__ void __launch_bounds__(SCfg<BN, kQ>::kThreads, 1)
    fp8_gemm_splitk_kernel(const __grid_constant__ CUtensorMap tmap_a,
                           const __grid_constant__ CUtensorMap tmap_b, const SmallArgsT<kQ> args) {
  using C = SCfg<BN, kQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = args.num_stages;
  uint8_t* smem_a = smem;
  uint8_t* smem_b = smem + static_cast<size_t>(S) * args.a_stage_bytes;
  size_t off = static_cast<size_t>(S) * (args.a_stage_bytes + C::kBTileBytes);
  const size_t a_read_end = static_cast<size_t>(S - 1) * args.a_stage_bytes + kATileBytes;
  if (a_read_end > off) off = a_read_end;  // an MMA reads 128 A rows from its stage
  // The partial tile parked for the cluster's reduction (split >= 2 only: a
  // CTA that reduces alone stores from registers and gets no buffer).
  float* part = reinterpret_cast<float*>(smem + off);
  if constexpr (kRed) off += static_cast<size_t>(args.split) * args.M * args.part_stride * sizeof(float);
  // Requantized output (kQ): the block-max exchange.
  uint8_t* rq_xchg = nullptr;
  uint32_t* rq_pmax = nullptr;  // [2][128][kNBlk]
  uint32_t* rq_xmax = nullptr;  // [2][kMaxSplit][128][kNBlk]
  uint64_t* rq_bar = nullptr;   // amax[2], lmax[2]
  if constexpr (kQ) {
    off = (off + 15) & ~static_cast<size_t>(15);
    rq_xchg = smem + off;
    rq_pmax = reinterpret_cast<uint32_t*>(rq_xchg + C::kRqXchg);
    rq_xmax = rq_pmax + C::kRqPmaxWords;
    rq_bar = reinterpret_cast<uint64_t*>(rq_xmax + C::kRqXmaxWords);
    off += C::kRqBytes;
  }
  off = (off + 7) & ~static_cast<size_t>(7);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + off);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + kMaxStages;
  uint64_t* tfull_bar = bars + 2 * kMaxStages;
  uint64_t* tempty_bar = tfull_bar + C::kNumPBuf;
  uint64_t* ready_bar = tempty_bar + C::kNumPBuf;  // all partials of the tile are parked
  uint64_t* consumed_bar = ready_bar + 1;          // every peer has read this CTA's partial
  uint64_t* drain_bar = consumed_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = args.wait_limit_ns;
  unsigned int* status = args.status;
  const uint32_t rank = cluster_ctarank();
  const int split = args.split;
  const int cluster_id = blockIdx.x / split;
  const int kb_lo = static_cast<int>(rank) * args.num_kb / split;
  const int kb_hi = (static_cast<int>(rank) + 1) * args.num_kb / split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < C::kNumPBuf; ++b) {
      mbar_init(smem_u32(&tfull_bar[b]), 1);
      mbar_init(smem_u32(&tempty_bar[b]), C::kEpiWarps);
    }
    mbar_init(smem_u32(ready_bar), split * C::kEpiWarps);
    mbar_init(smem_u32(consumed_bar), split * C::kEpiWarps);
    mbar_init(smem_u32(drain_bar), C::kIssuers);
    if constexpr (kQ) {
      requant_xchg_init(rq_xchg, C::kEpiWarps);
      for (int q = 0; q < 2; ++q) {
        mbar_init(smem_u32(&rq_bar[q]), split * C::kEpiWarps);  // every rank's warps have sent their maxima
        mbar_init(smem_u32(&rq_bar[2 + q]), C::kEpiWarps);      // this CTA's warps have folded theirs
      }
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  if constexpr (kQ) {
    for (uint32_t i = threadIdx.x; i < C::kRqPmaxWords; i += blockDim.x) rq_pmax[i] = 0u;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // every peer's barriers exist before any remote arrive
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  uint32_t loads_issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    uint32_t it = 0;
    bool ok = true;
    for (int nb = cluster_id; nb < args.num_nb && ok; nb += args.num_clusters) {
      for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
        const uint32_t stage = it % S;
        const uint32_t par = (it / S) & 1u;
        if (lane == 0) {
          ok = mbar_wait(smem_u32(&empty_bar[stage]), par ^ 1u, abort_flag, status, limit);
          if (ok) {
            const uint32_t fb = smem_u32(&full_bar[stage]);
            mbar_arrive_expect_tx(fb, args.a_box_bytes + C::kBTileBytes);
            tma_load_operand(smem_u32(smem_a + stage * args.a_stage_bytes), &tmap_a, fb, kb * kBK, 0, args.a_mn);
            const uint32_t bdst = smem_u32(smem_b + stage * C::kBTileBytes);
            if (args.b_mn) {
              // MN-major B: 128-column boxes (one 128-byte swizzle atom column each), 16 KB apart.
#pragma unroll
              for (int h = 0; h < BN / 128; ++h)
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
    const uint32_t me = static_cast<uint32_t>(warp - 1);
    uint32_t it = 0;
    bool ok = true;
    for (int nb = cluster_id; nb < args.num_nb && ok; nb += args.num_clusters) {
      for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
        if (it % C::kIssuers != me) continue;
        const uint32_t stage = it % S;
        const uint32_t par = (it / S) & 1u;
        const uint32_t buf = it % C::kNumPBuf;
        const uint32_t bpar = (it / C::kNumPBuf) & 1u;
        if (lane == 0) {
          ok = mbar_wait(smem_u32(&tempty_bar[buf]), bpar ^ 1u, abort_flag, status, limit) &&
               mbar_wait(smem_u32(&full_bar[stage]), par, abort_flag, status, limit);
          if (ok) {
            tc_fence_after();
            const OperandTile at{static_cast<uint32_t>(args.a_mn), 128u}, bt{static_cast<uint32_t>(args.b_mn), 128u};
            const uint64_t adesc = at.desc(smem_u32(smem_a + stage * args.a_stage_bytes));
            const uint64_t bdesc = bt.desc(smem_u32(smem_b + stage * C::kBTileBytes));
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k)
              mma_e4m3(tmem_base + buf * BN, adesc + at.kstep() * k, bdesc + bt.kstep() * k, args.idesc,
                       k > 0 ? 1u : 0u);
            mma_commit(smem_u32(&empty_bar[stage]));
            mma_commit(smem_u32(&tfull_bar[buf]));
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp >= C::kFirstEpiWarp) {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - C::kFirstEpiWarp;
    const int grp = ew >> 2;              // columns [64 grp, 64 grp + 64) of the tile
    const int lg = warp & 3;              // TMEM lane quadrant this warp may access
    const int row = lg * 32 + lane;
    const bool rows_here = lg * 32 < args.M;  // this warp holds at least one real row
    const uint32_t tmem_row = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + grp * 64;
    // Columns this CTA reduces: an 8-column-aligned share of the tile.
    const int col_lo = (static_cast<int>(rank) * (BN / 8) / split) * 8;
    const int col_hi = ((static_cast<int>(rank) + 1) * (BN / 8) / split) * 8;
    const int groups8 = (col_hi - col_lo) / 8;
    const int work = args.M * groups8;
    // Offset of this thread's row's scales (rows past M read the last row's).
    const int sa_off = args.sa_per_row ? min(row, args.M - 1) * args.ld_sa : 0;
    uint32_t it = 0;
    uint32_t tile_seq = 0;
    bool ok = true;
    for (int nb = cluster_id; nb < args.num_nb && ok; nb += args.num_clusters, ++tile_seq) {
      const int colt = nb * BN + grp * 64;
      const bool valid = colt < args.N;
      const float* sb_row = args.sb + static_cast<int64_t>(min(colt / kBK, args.nbs - 1)) * args.ld_sb;
      uint64_t acc[32];  // 64 FP32 accumulators, two per register pair
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = 0ull;
      // Tiles of up to 192 columns fetch the K blocks' scales three blocks
      // ahead: loaded in the block that uses them, their L2 latency paced every
      // block's promotion (16x24576x1536: 10.4 -> 9.5 us). The 256-column kernel
      // (96 registers a thread) spilled more with the extra registers and its
      // blocks are long enough to hide the load: it keeps the in-block load.
      constexpr bool kPf = BN < 256;
      const float* sa_p = args.sa + sa_off;
      float a0 = kPf && valid ? __ldg(sa_p + kb_lo) : 0.f, b0 = kPf && valid ? __ldg(sb_row + kb_lo) : 0.f;
      float a1 = kPf && valid && kb_lo + 1 < kb_hi ? __ldg(sa_p + kb_lo + 1) : 0.f;
      float b1 = kPf && valid && kb_lo + 1 < kb_hi ? __ldg(sb_row + kb_lo + 1) : 0.f;
      float a2 = kPf && valid && kb_lo + 2 < kb_hi ? __ldg(sa_p + kb_lo + 2) : 0.f;
      float b2 = kPf && valid && kb_lo + 2 < kb_hi ? __ldg(sb_row + kb_lo + 2) : 0.f;
      for (int kb = kb_lo; kb < kb_hi && ok; ++kb, ++it) {
        const float sv = kPf ? a0 * b0 : (valid ? __ldg(sa_p + kb) * __ldg(sb_row + kb) : 0.f);  // 0 past N
        a0 = a1; b0 = b1; a1 = a2; b1 = b2;
        a2 = kPf && valid && kb + 3 < kb_hi ? __ldg(sa_p + kb + 3) : 0.f;
        b2 = kPf && valid && kb + 3 < kb_hi ? __ldg(sb_row + kb + 3) : 0.f;
        const uint32_t buf = it % C::kNumPBuf;
        const bool w = mbar_wait(smem_u32(&tfull_bar[buf]), (it / C::kNumPBuf) & 1u, abort_flag, status, limit);
        ok = __all_sync(0xFFFFFFFFu, w);
        if (!ok) break;
        tc_fence_after();
        if (rows_here) {
          const uint64_t s2 = f32x2(__float_as_uint(sv), __float_as_uint(sv));
#pragma unroll
          for (int rd = 0; rd < 64 / C::kChunk; ++rd) {
            uint32_t r[C::kChunk];
            tmem_ld<C::kChunk>(tmem_row + buf * BN + rd * C::kChunk, r);
            tmem_wait_ld();
            if (rd == 64 / C::kChunk - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[buf]));
            }
#pragma unroll
            for (int j = 0; j < C::kChunk / 2; ++j)
              ffma2(acc[rd * (C::kChunk / 2) + j], s2, f32x2(r[2 * j], r[2 * j + 1]));
          }
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[buf]));
        }
      }
      if (!ok) break;

      if constexpr (kQ) {
        if constexpr (!kRed) {
          // No peers: the epilogue slices exchange their maxima in this CTA.
          bool unused = false;
          if (!requant_store_slice<C::kEpiWarps>(acc, row < args.M, false, lg * 32, args.M, args.N, colt, ew, lane,
                                                 tile_seq, rq_xchg, args.rq, nullptr, nullptr, unused, abort_flag,
                                                 status, limit)) {
            ok = false;
            break;
          }
          continue;
        }
      }
      if constexpr (!kRed) {
        // No peers: round this thread's row segment to bf16 and store it.
        if (row < args.M && valid) {
          __nv_bfloat16* dst = args.c + static_cast<int64_t>(row) * args.ld_c + colt;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 v0 = f32x2_split(acc[4 * j]), v1 = f32x2_split(acc[4 * j + 1]);
            const float2 v2 = f32x2_split(acc[4 * j + 2]), v3 = f32x2_split(acc[4 * j + 3]);
            store_bf16x8(dst + 8 * j, colt + 8 * j, args.N, v0, v1, v2, v3);
          }
        }
        continue;
      }

      // Push this CTA's partial (rows < M) to the ranks that reduce it, once
      // every rank has read the last tile's: each 8-column unit goes into slot
      // `rank` of its owner's buffer ([split][M][part_stride] floats, columns
      // relative to the owner's share). Remote stores do not wait for a round
      // trip the way remote loads of the peers' partials did.
      if (tile_seq > 0) {
        const bool w = mbar_wait_cluster(smem_u32(consumed_bar), (tile_seq - 1) & 1u, abort_flag, status, limit);
        ok = __all_sync(0xFFFFFFFFu, w);
        if (!ok) break;
      }
      if (row < args.M) {
        const uint32_t slot_row = smem_u32(part + (static_cast<int>(rank) * args.M + row) * args.part_stride);
        int owner = share_owner(grp * 8, C::kUnits, split);
        int lo = share_lo(owner, C::kUnits, split), hi = share_lo(owner + 1, C::kUnits, split);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int u = grp * 8 + j;
          if (u >= hi) {  // next owner (shares are at least one unit wide)
            ++owner;
            lo = hi;
            hi = share_lo(owner + 1, C::kUnits, split);
          }
          const uint32_t dst = mapa_shared(slot_row + (u - lo) * 32u, static_cast<uint32_t>(owner));
          const float2 v0 = f32x2_split(acc[4 * j]), v1 = f32x2_split(acc[4 * j + 1]);
          const float2 v2 = f32x2_split(acc[4 * j + 2]), v3 = f32x2_split(acc[4 * j + 3]);
          st_dsmem_f4(dst, make_float4(v0.x, v0.y, v1.x, v1.y));
          st_dsmem_f4(dst + 16, make_float4(v2.x, v2.y, v3.x, v3.y));
        }
      }
      // The warp's stores are ordered (warp barrier) before the releasing remote
      // arrives; lane s signals rank s, so the arrives to all ranks overlap.
      __syncwarp();
      if (lane < split) mbar_arrive_remote(mapa_shared(smem_u32(ready_bar), lane));

      // Reduce this CTA's columns over the cluster's partials, in rank order.
      {
        const bool w = mbar_wait_cluster(smem_u32(ready_bar), tile_seq & 1u, abort_flag, status, limit);
        ok = __all_sync(0xFFFFFFFFu, w);
        if (!ok) break;
      }
      if constexpr (kQ) {
        ok = requant_cluster_tile<BN>(args, part, rank, split, nb, col_lo, groups8, work, ew, lane, tile_seq,
                                      rq_pmax, rq_xmax, rq_bar, consumed_bar, abort_flag, status, limit);
        if (!ok) break;
        continue;
      }
      for (int g = ew * 32 + lane; g < work; g += C::kEpiWarps * 32) {
        const int rr = g / groups8;
        const int col = col_lo + (g % groups8) * 8;
        float sum[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) sum[q] = 0.f;
        const float* src = part + rr * args.part_stride + (col - col_lo);
        for (int s = 0; s < split; ++s) {
          const float* q = src + s * args.M * args.part_stride;
          const float4 x0 = *reinterpret_cast<const float4*>(q), x1 = *reinterpret_cast<const float4*>(q + 4);
          sum[0] += x0.x; sum[1] += x0.y; sum[2] += x0.z; sum[3] += x0.w;
          sum[4] += x1.x; sum[5] += x1.y; sum[6] += x1.z; sum[7] += x1.w;
        }
        const int gcol = nb * BN + col;
        store_bf16x8(args.c + static_cast<int64_t>(rr) * args.ld_c + gcol, gcol, args.N,
                     make_float2(sum[0], sum[1]), make_float2(sum[2], sum[3]),
                     make_float2(sum[4], sum[5]), make_float2(sum[6], sum[7]));
      }
      __syncwarp();
      if (lane < split) mbar_arrive_remote(mapa_shared(smem_u32(consumed_bar), lane));
    }
    __syncwarp();
  }

  // ------------------------------------------------------------- teardown --
  __syncthreads();
  if (*abort_flag) {
    const uint64_t drain_ns = 10000000ull;
    if (warp == 0 && lane == 0) {
      const uint32_t n = loads_issued < static_cast<uint32_t>(S) ? loads_issued : S;
      for (uint32_t j = loads_issued - n; j < loads_issued; ++j) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&full_bar[j % S]), (j / S) & 1u))
          if (global_timer_ns() - t0 > drain_ns) break;
      }
    }
    if (warp >= 1 && warp <= C::kIssuers && lane == 0) mma_commit(smem_u32(drain_bar));
    if (warp == 1 && lane == 0) {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_u32(drain_bar), 0))
        if (global_timer_ns() - t0 > drain_ns) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
  cluster_sync_all();  // no CTA leaves while a peer may still read its partial
}

// Largest number of co-resident clusters of `split` CTAs for this kernel with
// `smem` bytes of shared memory per CTA. The answer depends on the shared
// memory, which follows M, so it is cached per (device, split, smem): decode
// calls with varying M query the runtime once per distinct size.
template <int BN, bool kQ>
int max_active_clusters(int split, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, int> cache;
  if (split < 1 || split > kMaxSplit) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(dev, split, smem);
  const auto hit = cache.find(key);
  if (hit != cache.end()) return hit->second;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(split * 256, 1, 1);
  cfg.blockDim = dim3(SCfg<BN, kQ>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = split > 1 ? cudaOccupancyMaxActiveClusters(&n, fp8_gemm_splitk_kernel<BN, kQ, true>, &cfg)
                                   : cudaOccupancyMaxActiveClusters(&n, fp8_gemm_splitk_kernel<BN, kQ, false>, &cfg);
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = -1;
  }
  cache.emplace(key, n);
  return n;
}

struct Plan {
  int split = 0;
  int part_stride = 0;
  int clusters = 0;
  int stages = 0;
  size_t smem = 0;
  double cost = 1e300;
};

// Launch geometry for tile width BN: shared memory, stages, and the K split
// with the least modelled time. Returns false if BN does not fit.
template <int BN, bool kQ>
bool plan_small_m(const GemmProblem& p, int sms, SmallArgs& args, size_t& smem_out, Plan& plan) {
  using C = SCfg<BN, kQ>;
  args.num_nb = static_cast<int>((p.N + BN - 1) / BN);
  const uint32_t stage_bytes = args.a_stage_bytes + C::kBTileBytes;
  const size_t bar_bytes = (2 * kMaxStages + 2 * C::kNumPBuf + 3) * sizeof(uint64_t) + 32;
  auto ring_bytes = [&](int st) {
    return std::max<size_t>(static_cast<size_t>(st) * stage_bytes,
                            static_cast<size_t>(st - 1) * args.a_stage_bytes + kATileBytes);
  };
  // Stages and shared memory for a K split: with split >= 2 each CTA holds
  // the reduction buffer of its column share (split slots of M rows of the
  // widest share; ~100 KB at M = 128), which a CTA that reduces alone spends
  // on stages instead. `pst` is the slot row stride in floats.
  auto layout = [&](int split, int pst, int& stages_out, size_t& smem_o) {
    const size_t part_bytes =
        (split > 1 ? (static_cast<size_t>(split) * p.M * pst * sizeof(float) + 15) / 16 * 16 : 0) +
        (kQ ? C::kRqBytes : 0);
    if (part_bytes + bar_bytes + 1024 >= kMaxDynSmem) return false;
    const size_t budget = kMaxDynSmem - 1024 - part_bytes - bar_bytes;
    int stages = std::min<int>(kMaxStages, static_cast<int>(budget / stage_bytes));
    while (stages > C::kIssuers && ring_bytes(stages) > budget) --stages;
    stages = stages / C::kIssuers * C::kIssuers;  // whole stage sets per issuer
    if (stages < std::max(C::kIssuers, 4) || ring_bytes(stages) > budget) return false;
    size_t smem = 1024 + ring_bytes(stages) + part_bytes + bar_bytes;
    smem = std::max<size_t>(smem, kMinSmemPerCta);
    if (smem > kMaxDynSmem) return false;
    stages_out = stages;
    smem_o = smem;
    return true;
  };

  // Model (fitted to graph-timed sweeps of forced plans on GB300): one SM
  // streams ~45 GB/s of 128-byte TMA rows; the whole GPU streams B at ~4.4,
  // 5.2 and 4.6 TB/s with 128-, 192- and 256-column tiles as the kernel runs
  // them; A's rows (from L2) count half; a tile's cluster reduction adds
  // ~0.25 us per CTA of the split after its stream (the wait for the slowest
  // peer grows with the split). Time = max(whole-GPU stream of B, the slowest
  // cluster's K ranges) + reductions.
  const double sm_bytes_per_us = 4.5e4;
  const double gpu_bytes_per_us = (BN == 256) ? 4.6e6 : (BN == 192) ? 5.2e6 : 4.4e6;
  const double b_bytes = static_cast<double>(p.N) * static_cast<double>(p.K);
  for (int split = 1; split <= kMaxSplit; ++split) {
    if (split > args.num_kb || (BN / 8) / split < 1) break;
    // Slot rows padded by 16 bytes (conflict-free pushes), unpadded where the
    // padding would cost stages.
    const int widest = share_cols_max(C::kUnits, split);
    int pst = widest + 4, stages = 0;
    size_t smem = 0;
    if (!layout(split, pst, stages, smem)) continue;
    if (split > 1) {
      int st0 = 0;
      size_t sm0 = 0;
      if (layout(split, widest, st0, sm0) && st0 > stages) {
        pst = widest;
        stages = st0;
        smem = sm0;
      }
    }
    const int active = max_active_clusters<BN, kQ>(split, smem);
    if (active <= 0) continue;
    int clusters = std::min(active, args.num_nb);
    if (p.num_sms_cap > 0) clusters = std::min(clusters, std::max(1, p.num_sms_cap / split));
    if (clusters <= 0 || clusters * split > sms * 2) continue;
    const int waves = (args.num_nb + clusters - 1) / clusters;
    // A K split serves to fill the GPU in one wave; split plans that need
    // several ran 25-40 % slower than a smaller split in every sweep. (Under
    // an SM cap every plan needs several waves; the model chooses.)
    if (split > 1 && waves > 1 && p.num_sms_cap <= 0) continue;
    const int kbs = (args.num_kb + split - 1) / split;
    const double per_cluster =
        waves * kbs * (static_cast<double>(C::kBTileBytes) + 0.5 * args.a_box_bytes) / sm_bytes_per_us;
    const double reduce = split > 1 ? waves * 0.25 * split : 0.0;
    const double cost = (std::max(b_bytes / gpu_bytes_per_us, per_cluster) + reduce) * (1.0 + 0.01 * split);
    if (cost < plan.cost) {
      plan.cost = cost;
      plan.split = split;
      plan.clusters = clusters;
      plan.stages = stages;
      plan.part_stride = pst;
      plan.smem = smem;
    }
  }
  if (plan.split <= 0) return false;
  args.num_stages = plan.stages;
  smem_out = plan.smem;
  return true;
}

// Allows the kernel its shared memory on the current device (once per device);
// the occupancy query of the planner needs it too.
template <int BN, bool kQ>
bool set_smem_attribute() {
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (attr_set.load() & (1ull << dev)) return true;
  if (cudaFuncSetAttribute(fp8_gemm_splitk_kernel<BN, kQ, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kMaxDynSmem)) != cudaSuccess ||
      cudaFuncSetAttribute(fp8_gemm_splitk_kernel<BN, kQ, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kMaxDynSmem)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  attr_set.fetch_or(1ull << dev);
  return true;
}

template <int BN, bool kQ>
int run_small_m(const GemmProblem& p, cudaStream_t stream, SmallArgs args, size_t smem, const Plan& plan) {
  args.split = plan.split;
  args.num_clusters = plan.clusters;
  args.part_stride = plan.part_stride;
  CUtensorMap ta, tb;
  const uint32_t a_rows = args.a_box_bytes / kBK;
  if (p.a_mn) {
    // A as [K][ld_a]: 128 (M, zero-filled past M) x 128 (K) boxes.
    const uint64_t dims[2] = {static_cast<uint64_t>(p.M), static_cast<uint64_t>(p.K)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.ld_a)};
    const uint32_t box[2] = {kBM, kBK};
    if (!encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 2, dims, strides, box, true))
      return DG_ERR_CUDA;
  } else {
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.ld_a)};
    const uint32_t box[2] = {kBK, a_rows};
    if (!encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, 2, dims, strides, box, true))
      return DG_ERR_CUDA;
  }
  if (p.b_mn) {
    // B as [K][ld_b]: 128 (N) x 128 (K) boxes.
    const uint64_t dims[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.K)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.ld_b)};
    const uint32_t box[2] = {128, kBK};
    if (!encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 2, dims, strides, box, true))
      return DG_ERR_CUDA;
  } else {
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.N)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.ld_b)};
    const uint32_t box[2] = {kBK, static_cast<uint32_t>(BN)};
    if (!encode_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, 2, dims, strides, box, true))
      return DG_ERR_CUDA;
  }
  args.idesc = SCfg<BN, kQ>::kIdesc | idesc_majors(p.a_mn, p.b_mn);
  SmallArgsT<kQ> kargs;
  static_cast<SmallArgs&>(kargs) = args;
  if constexpr (kQ) kargs.rq = p.rq;
  const cudaError_t e =
      args.split > 1
          ? launch_kernel(fp8_gemm_splitk_kernel<BN, kQ, true>, dim3(args.split * args.num_clusters),
                          dim3(SCfg<BN, kQ>::kThreads), smem, stream, static_cast<unsigned>(args.split), ta, tb, kargs)
          : launch_kernel(fp8_gemm_splitk_kernel<BN, kQ, false>, dim3(args.num_clusters), dim3(SCfg<BN, kQ>::kThreads),
                          smem, stream, 1u, ta, tb, kargs);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DG_ERR_CUDA;
  }
  return DG_OK;
}

// The tile width with the least modelled time: 256 columns (fewer, larger TMA
// boxes), 128, or -- bf16 output with K-major B -- 192, whose tile count often
// fills the SMs where 256 leaves a third of them idle (24576 columns: 128
// tiles of 192 against 96 of 256; 7168 columns: 38 tiles of 192 x a K split of
// 4 = 152 CTAs).
template <bool kQ>
int plan_and_run(const GemmProblem& p, cudaStream_t stream, int sms, const SmallArgs& args) {
  if (!set_smem_attribute<256, kQ>() || !set_smem_attribute<128, kQ>()) return DG_ERR_CUDA;
  SmallArgs a256 = args, a128 = args;
  size_t s256 = 0, s128 = 0;
  Plan p256, p128;
  const bool ok256 = plan_small_m<256, kQ>(p, sms, a256, s256, p256);
  const bool ok128 = plan_small_m<128, kQ>(p, sms, a128, s128, p128);
  if constexpr (!kQ) {
    if (!p.b_mn) {
      if (!set_smem_attribute<192, kQ>()) return DG_ERR_CUDA;
      SmallArgs a192 = args;
      size_t s192 = 0;
      Plan p192;
      if (plan_small_m<192, kQ>(p, sms, a192, s192, p192) && (!ok256 || p192.cost < p256.cost) &&
          (!ok128 || p192.cost < p128.cost))
        return run_small_m<192, kQ>(p, stream, a192, s192, p192);
    }
  }
  // Requantized output takes 128-column tiles whenever they fit: the 256-column
  // requantizing kernel (19 warps, 96 registers a thread) spills in its tile
  // tail, which the model does not see (128x24576x1536: 54.9 -> 33.0 us; the
  // other decode shapes within 1 %).
  if (ok256 && !(kQ && ok128) && (!ok128 || p256.cost <= p128.cost))
    return run_small_m<256, kQ>(p, stream, a256, s256, p256);
  if (ok128) return run_small_m<128, kQ>(p, stream, a128, s128, p128);
  return DG_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace

bool small_m_supported(int64_t M, const void* m_indices) { return m_indices == nullptr && M >= 1 && M <= kBM; }

int launch_gemm_small_m(const GemmProblem& p, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DG_ERR_NO_DEVICE;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return DG_ERR_NO_DEVICE;
  unsigned int* status = device_status_word();
  if (!status) return DG_ERR_CUDA;

  SmallArgs args{};
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
  args.nbs = static_cast<int>((p.N + kBK - 1) / kBK);
  args.wait_limit_ns = kDefaultWaitLimitNs;
  // K-major A: the valid rows (a multiple of 8); MN-major A: a full 128-byte-wide box.
  const uint32_t a_rows = p.a_mn ? kBM : static_cast<uint32_t>((p.M + 7) / 8 * 8);
  args.a_box_bytes = a_rows * kBK;
  args.a_stage_bytes = (args.a_box_bytes + 1023u) / 1024u * 1024u;
  return p.rq.q ? plan_and_run<true>(p, stream, sms, args) : plan_and_run<false>(p, stream, sms, args);
}

}  // namespace dg
