// dg_pair.cuh -- pieces of the CTA-pair GEMM kernels (gemm_pair.cu): tile
// sizes, the argument structs, the grouped raster of pair tiles and its
// M-grouped units, and the bf16 output stores.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "dg_device.cuh"
#include "dg_encode.cuh"
#include "dg_internal.h"

namespace dg {
namespace {

constexpr int kBM = 128;               // rows per CTA (256 per pair)
constexpr int kBN = 128;               // columns per pair tile
constexpr int kBK = 128;               // K block = scale block
constexpr int kGroupPM = 8;            // raster group height in pair rows (A larger than L2 allows)
constexpr int64_t kRasterABytes = 16ll << 20;  // A up to this size is swept whole per N band
constexpr uint32_t kABytes = kBM * kBK;            // 16 KB
constexpr uint32_t kBoxBytes = 32 * 32 * 2;        // one warp's 32 x 32 bf16 output box
constexpr size_t kMaxDynSmem = 227 * 1024;

struct PairArgs {
  __nv_bfloat16* c;  // bf16 output (kernels without requantization)
  int64_t ld_c;
  int sa_per_row;  // sa is [M][K/128] instead of [ceil(M/128)][K/128]
  const float* sa;
  const float* sb;
  unsigned int* status;
  int M, N;
  int num_kb;   // K / 128
  int ld_sa, ld_sb;  // row strides of sa and sb (floats)
  uint32_t idesc;    // MMA instruction descriptor (shape, scale type, operand majorness)
  int a_mn, b_mn;    // MN-major A ([K][M]) / B ([K][N]) tiles
  int num_mb;   // ceil(M / 128)
  int num_pm;   // ceil(M / 256)
  int num_nb;   // ceil(N / 128)
  int group_pm; // raster group height in pair rows
  int num_stages;
  uint64_t wait_limit_ns;
};

// Arguments of the requantizing kernels. A separate type: the extra fields in
// the common struct changed the bf16 kernels' register allocation.
struct PairArgsQ : PairArgs {
  RequantOut rq;     // E4M3 output and scales
};
// M-grouped calls add the expert of each row (-1: padding) and the number of
// experts (ids outside [0, num_groups) run no MMAs). Separate types again, so
// that the dense kernels keep their argument layout.
struct PairGroups {
  const int32_t* m_indices;
  int num_groups;
};
struct PairArgsG : PairArgs, PairGroups {};
struct PairArgsQG : PairArgsQ, PairGroups {};
template <bool kQ, bool kG = false>
using PairArgsT = std::conditional_t<kG, std::conditional_t<kQ, PairArgsQG, PairArgsG>,
                                     std::conditional_t<kQ, PairArgsQ, PairArgs>>;
// K-grouped calls (one output matrix per range of K, the MoE weight gradient
// C_g = A_g^T B_g): the ranges with K > 0, in K order. Unit t of such a launch
// is tile t % T of range t / T (T = num_pm * num_nb tiles per range).
constexpr int kMaxKGroups = 256;
struct KGroups {
  int num_kg;                // ranges with K > 0
  int kb_lo[kMaxKGroups];    // first K block of the range
  int kb_n[kMaxKGroups];     // K blocks of the range (> 0)
  int g_out[kMaxKGroups];    // output matrix of the range
};
struct PairArgsKG : PairArgs, KGroups {};
template <bool kQ, bool kKG>
using PairArgsF = std::conditional_t<kKG, PairArgsKG, PairArgsT<kQ>>;

// Tile t of the raster: groups of group_pm pair rows, each swept over N with
// the pair row fastest, so the pairs at work at once share a few B column
// bands and one group's A rows. With the group spanning all of M (A small
// enough to stay in L2) every B band is read from HBM once.
__device__ __forceinline__ void pair_tile_coords(int t, int num_pm, int num_nb, int group_pm, int& pm, int& nb) {
  const int per_group = group_pm * num_nb;
  const int grp = t / per_group;
  const int first = grp * group_pm;
  const int gm = min(group_pm, num_pm - first);
  const int r = t - grp * per_group;
  pm = first + r % gm;
  nb = r / gm;
}

// A unit of a pair's persistent work: pair row pm (A rows [256 pm, +256)) and
// N tile nb. Dense calls run one slot per unit. M-grouped calls (both 128-row
// halves of a pair MMA multiply one B, so one expert) look up the experts g0,
// g1 of the row's blocks b0 = 2 pm and b1 = b0 + 1:
//   * g0 == g1 (one expert, or both padding), or no block b1: one slot, the
//     whole pair row with expert g0 (a missing b1 is discarded);
//   * otherwise two slots, slot s covering block b_s with expert g_s: CTA s
//     keeps its rows, the other CTA's half of the MMA result is discarded.
// A slot whose expert is -1 (padding) or past the last expert runs no MMAs;
// its kept rows are written as zeros.
struct PairUnit {
  int pm, nb;
  int g0, g1;
  int nslots;
};
struct PairSlot {
  int g, keep;     // expert of the MMAs; bit r set: CTA r writes its 128 rows
  bool mma, bad;   // the MMAs run; the expert id is past the last expert
};

__device__ __forceinline__ int pair_num_units(const PairArgs& a) { return a.num_pm * a.num_nb; }

// The raw ids a unit's lookup reduces (4 per lane for each of b0, b1), loaded
// one unit ahead so that their latency hides behind the current unit.
struct UnitIds {
  int4 v0, v1;
};
template <bool kGrouped, class Args>
__device__ __forceinline__ UnitIds pair_unit_ids(int t, const Args& a, int lane) {
  UnitIds r{make_int4(-1, -1, -1, -1), make_int4(-1, -1, -1, -1)};
  if constexpr (kGrouped) {
    if (t < pair_num_units(a)) {
      int pm, nb;
      pair_tile_coords(t, a.num_pm, a.num_nb, a.group_pm, pm, nb);
      const int4* ids = reinterpret_cast<const int4*>(a.m_indices);
      r.v0 = __ldg(ids + static_cast<int64_t>(2 * pm) * 32 + lane);
      if (2 * pm + 1 < a.num_mb) r.v1 = __ldg(ids + static_cast<int64_t>(2 * pm + 1) * 32 + lane);
    }
  }
  return r;
}
// Unit t from its ids (warp-collective for M-grouped calls).
template <bool kGrouped, class Args>
__device__ __forceinline__ PairUnit pair_unit(int t, const Args& a, const UnitIds& ids) {
  PairUnit u;
  pair_tile_coords(t, a.num_pm, a.num_nb, a.group_pm, u.pm, u.nb);
  u.g0 = u.g1 = 0;
  u.nslots = 1;
  if constexpr (kGrouped) {
    const int m0 = max(max(ids.v0.x, ids.v0.y), max(ids.v0.z, ids.v0.w));
    const int m1 = max(max(ids.v1.x, ids.v1.y), max(ids.v1.z, ids.v1.w));
    u.g0 = __reduce_max_sync(0xFFFFFFFFu, m0);
    const bool has1 = 2 * u.pm + 1 < a.num_mb;
    u.g1 = has1 ? __reduce_max_sync(0xFFFFFFFFu, m1) : u.g0;
    u.nslots = (has1 && u.g1 != u.g0) ? 2 : 1;
  }
  return u;
}
template <bool kGrouped, class Args>
__device__ __forceinline__ PairSlot pair_slot(const PairUnit& u, int slot, const Args& a) {
  PairSlot s{0, 3, true, false};
  if constexpr (kGrouped) {
    s.g = slot == 0 ? u.g0 : u.g1;
    s.keep = u.nslots == 1 ? 3 : (1 << slot);
    s.bad = s.g >= a.num_groups;
    s.mma = s.g >= 0 && !s.bad;
  }
  return s;
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

// bf16 epilogue of one warp: its 32 rows x EC columns of acc (two FP32 per
// 64-bit pair) -> 64-byte-swizzled 32 x 32 boxes in shared memory (16-byte
// chunk c of row r at chunk c ^ ((r / 2) % 4)) -> TMA stores, clipped at M.
// A box that crosses column N is written element by element instead: the
// swizzled store clips N only to whole 16-byte chunks.
// k3D: C is [G][M][ld_c] with a 3-D map {N, M, G}; the rows go to matrix g.
template <int EC, int kBoxes = EC / 32, bool k3D = false>
__device__ __forceinline__ void store_tile_rows(const uint64_t (&acc)[EC / 2], const CUtensorMap& tmap_c,
                                                const PairArgs& args, uint8_t* out_box, int row0, int col0,
                                                int lane, bool& stores_issued, int g = 0) {
  if (lane == 0 && stores_issued) bulk_wait_read_all();  // the last tile's stores have read the boxes
  __syncwarp();
#pragma unroll
  for (int h = 0; h < EC / 32; ++h) {
    if (kBoxes == 1 && h > 0) {  // one box, reused: its previous store must have read it
      if (lane == 0 && stores_issued) bulk_wait_read_all();
      __syncwarp();
    }
    const int bcol = col0 + 32 * h;
    if (bcol + 32 > args.N) {
      const int row = row0 + lane;
      if (row < args.M && bcol < args.N) {
        __nv_bfloat16* crow = args.c + (static_cast<int64_t>(g) * args.M + row) * args.ld_c;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 v = f32x2_split(acc[h * 16 + j]);
          if (bcol + 2 * j < args.N) crow[bcol + 2 * j] = __float2bfloat16_rn(v.x);
          if (bcol + 2 * j + 1 < args.N) crow[bcol + 2 * j + 1] = __float2bfloat16_rn(v.y);
        }
      }
      continue;
    }
    uint8_t* box = out_box + (kBoxes == 1 ? 0 : h) * kBoxBytes;
    uint8_t* my_row = box + lane * 64;
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
      if constexpr (k3D)
        tma_store_3d(&tmap_c, smem_u32(box), bcol, row0, g);
      else
        tma_store_2d(&tmap_c, smem_u32(box), bcol, row0);
      bulk_commit();
      stores_issued = true;
    }
  }
}

// bf16 epilogue of one warp with one 32 x 64 box: 128-byte rows in the
// 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)), one TMA
// store per warp and tile. A slice that crosses column N is written element
// by element.
template <bool k3D = false>
__device__ __forceinline__ void store_tile_rows64(const uint64_t (&acc)[32], const CUtensorMap& tmap_c,
                                                  const PairArgs& args, uint8_t* box, int row0, int col0, int lane,
                                                  bool& stores_issued, int g = 0) {
  if (lane == 0 && stores_issued) bulk_wait_read_all();  // the last tile's store has read the box
  __syncwarp();
  if (col0 + 64 > args.N) {
    const int row = row0 + lane;
    if (row < args.M && col0 < args.N) {
      __nv_bfloat16* crow = args.c + (static_cast<int64_t>(g) * args.M + row) * args.ld_c;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float2 v = f32x2_split(acc[j]);
        if (col0 + 2 * j < args.N) crow[col0 + 2 * j] = __float2bfloat16_rn(v.x);
        if (col0 + 2 * j + 1 < args.N) crow[col0 + 2 * j + 1] = __float2bfloat16_rn(v.y);
      }
    }
    return;
  }
  uint8_t* my_row = box + lane * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float2 v0 = f32x2_split(acc[c * 4]), v1 = f32x2_split(acc[c * 4 + 1]);
    const float2 v2 = f32x2_split(acc[c * 4 + 2]), v3 = f32x2_split(acc[c * 4 + 3]);
    uint4 pk;
    pk.x = pack_bf16(v0.x, v0.y);
    pk.y = pack_bf16(v1.x, v1.y);
    pk.z = pack_bf16(v2.x, v2.y);
    pk.w = pack_bf16(v3.x, v3.y);
    *reinterpret_cast<uint4*>(my_row + ((c ^ (lane & 7)) << 4)) = pk;
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < args.M) {
    if constexpr (k3D)
      tma_store_3d(&tmap_c, smem_u32(box), col0, row0, g);
    else
      tma_store_2d(&tmap_c, smem_u32(box), col0, row0);
    bulk_commit();
    stores_issued = true;
  }
}

// The same store for a row slice already rounded to bf16: pk[j] holds columns
// col0 + 2 j and col0 + 2 j + 1; one staging box per warp, reused for the
// second 32-column half once its first store has read it.
__device__ __forceinline__ void store_packed_rows(const uint32_t (&pk)[32], const CUtensorMap& tmap_c,
                                                  const PairArgs& args, uint8_t* box, int row0, int col0,
                                                  int lane, bool& stores_issued) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int bcol = col0 + 32 * h;
    if (bcol + 32 > args.N) {
      const int row = row0 + lane;
      if (row < args.M && bcol < args.N) {
        uint16_t* crow = reinterpret_cast<uint16_t*>(args.c + static_cast<int64_t>(row) * args.ld_c);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (bcol + 2 * j < args.N) crow[bcol + 2 * j] = static_cast<uint16_t>(pk[h * 16 + j] & 0xFFFFu);
          if (bcol + 2 * j + 1 < args.N) crow[bcol + 2 * j + 1] = static_cast<uint16_t>(pk[h * 16 + j] >> 16);
        }
      }
      continue;
    }
    if (lane == 0 && stores_issued) bulk_wait_read_all();  // the box's previous store has read it
    __syncwarp();
    uint8_t* my_row = box + lane * 64;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(my_row + ((c ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(pk[h * 16 + 4 * c], pk[h * 16 + 4 * c + 1], pk[h * 16 + 4 * c + 2], pk[h * 16 + 4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && row0 < args.M) {
      tma_store_2d(&tmap_c, smem_u32(box), bcol, row0);
      bulk_commit();
      stores_issued = true;
    }
  }
}

}  // namespace
}  // namespace dg
