// dg_encode.cuh -- E4M3 encoding shared by the quantizers and the GEMM epilogue
// that requantizes its FP32 accumulators.
//
// The arithmetic is that of the lpnh.cn DeepGEMM walkthrough §4.2 (scale =
// max|x| / 448, divide, round to the nearest E4M3 value with ties to even) and
// §5.4 (an all-zero block gets scale 1); power-of-two scales follow the packed
// UE8M0 scales of pzsr.cn "DeepGEMM: GPU上的高效BLAS内核库解析" §3.1. The GEMM
// epilogue variant applies the same steps to the FP32 accumulators before they
// leave the chip ("quantize on demand at write-back", walkthrough §2.2; fusing
// the scale computation saves a round trip through memory, §6).
#pragma once

#include <cuda_fp8.h>
#include <cstdint>

#include "dg_device.cuh"
#include "dg_internal.h"

namespace dg {

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

// Scale of a block whose largest magnitude is amax: fl32(amax / 448); 1 for an
// all-zero block (or an underflow to 0); optionally rounded up to a power of two.
__device__ __forceinline__ float block_scale(float amax, bool pow2) {
  float s = amax / 448.0f;
  if (s == 0.0f) s = 1.0f;
  return pow2 ? pow2_round_up(s) : s;
}

__device__ __forceinline__ uint32_t cvt2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// E4M3 codes of fl32(v / s) for the four values of v, packed little-endian.
// kMode 0: exact division with the r = 1/s fast path (valid for normal s);
// kMode 1: power-of-two s, v * r exact; kMode 2: plain division (tiny s).
//
// Why kMode 0 is exact: q = fl32(v r) with r = fl32(1/s) lies within
// 1.5 * 2^-23 (relative) of fl32(v / s). If q (1 - 2^-20) and q (1 + 2^-20)
// round to the same E4M3 code, every value between them -- fl32(v / s)
// included -- does too (rounding to E4M3 is monotone), so that code is exact.
// Otherwise (an E4M3 rounding boundary within 2^-20 of q, about one value in
// 2^15) the element is divided exactly.
// kMode 0 without its fallback: the codes of q (1 - 2^-20), which are exact
// when ok (no E4M3 rounding boundary near q); otherwise the caller divides.
// Products two at a time (mul.rn.f32x2: each lane rounded as a scalar multiply).
__device__ __forceinline__ uint32_t encode4_bracketed(const float4 v, float r, bool& ok) {
  const uint64_t r2 = f32x2(__float_as_uint(r), __float_as_uint(r));
  const uint64_t q01 = fmul2(f32x2(__float_as_uint(v.x), __float_as_uint(v.y)), r2);
  const uint64_t q23 = fmul2(f32x2(__float_as_uint(v.z), __float_as_uint(v.w)), r2);
  const uint64_t lo2 = f32x2(__float_as_uint(1.0f - 0x1p-20f), __float_as_uint(1.0f - 0x1p-20f));
  const uint64_t hi2 = f32x2(__float_as_uint(1.0f + 0x1p-20f), __float_as_uint(1.0f + 0x1p-20f));
  const float2 la = f32x2_split(fmul2(q01, lo2)), lb = f32x2_split(fmul2(q23, lo2));
  const float2 ha = f32x2_split(fmul2(q01, hi2)), hb = f32x2_split(fmul2(q23, hi2));
  const uint32_t lo = cvt2(la.x, la.y) | (cvt2(lb.x, lb.y) << 16);
  const uint32_t hi = cvt2(ha.x, ha.y) | (cvt2(hb.x, hb.y) << 16);
  ok = lo == hi;
  return lo;
}

template <int kMode>
__device__ __forceinline__ uint32_t encode4(const float4 v, float s, float r) {
  if constexpr (kMode == 2) {
    return cvt2(v.x / s, v.y / s) | (cvt2(v.z / s, v.w / s) << 16);
  } else if constexpr (kMode == 1) {
    return cvt2(v.x * r, v.y * r) | (cvt2(v.z * r, v.w * r) << 16);
  } else {
    bool ok;
    const uint32_t c = encode4_bracketed(v, r, ok);
    return ok ? c : encode4<2>(v, s, r);
  }
}

// encode4 over n groups at once: every group's codes are formed before any
// fallback division, so the groups' independent work can interleave.
template <int kMode, int n>
__device__ __forceinline__ void encode4_n(const float4 (&v)[n], uint32_t (&code)[n], float s, float r) {
  if constexpr (kMode == 0) {
    uint32_t bad = 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      bool ok;
      code[i] = encode4_bracketed(v[i], r, ok);
      bad |= (ok ? 0u : 1u) << i;
    }
    if (bad != 0u) {
#pragma unroll
      for (int i = 0; i < n; ++i)
        if ((bad >> i) & 1u) code[i] = encode4<2>(v[i], s, r);
    }
  } else {
#pragma unroll
    for (int i = 0; i < n; ++i) code[i] = encode4<kMode>(v[i], s, r);
  }
}

template <int kMode>
__device__ __forceinline__ uint8_t encode1(float v, float s, float r) {
  const uint32_t c = encode4<kMode>(make_float4(v, 0.f, 0.f, 0.f), s, r);
  return static_cast<uint8_t>(c & 0xFFu);
}

// E4M3 codes of fl32(v / s) for four values held as two FP32 pairs (the
// epilogue's accumulator layout), with the arithmetic of encode4 done in
// packed f32x2 multiplies. r2 = (1/s, 1/s).
__device__ __forceinline__ uint32_t encode4_pairs(uint64_t v01, uint64_t v23, float s, uint64_t r2, bool pow2) {
  const uint64_t q01 = fmul2(v01, r2), q23 = fmul2(v23, r2);
  const float2 a = f32x2_split(q01), b = f32x2_split(q23);
  const uint32_t c = cvt2(a.x, a.y) | (cvt2(b.x, b.y) << 16);
  if (pow2) return c;  // q = v / s exactly
  if (s >= 0x1p-126f) {
    const uint64_t lo2 = f32x2(__float_as_uint(1.0f - 0x1p-20f), __float_as_uint(1.0f - 0x1p-20f));
    const uint64_t hi2 = f32x2(__float_as_uint(1.0f + 0x1p-20f), __float_as_uint(1.0f + 0x1p-20f));
    const float2 la = f32x2_split(fmul2(q01, lo2)), lb = f32x2_split(fmul2(q23, lo2));
    const float2 ha = f32x2_split(fmul2(q01, hi2)), hb = f32x2_split(fmul2(q23, hi2));
    const uint32_t lo = cvt2(la.x, la.y) | (cvt2(lb.x, lb.y) << 16);
    const uint32_t hi = cvt2(ha.x, ha.y) | (cvt2(hb.x, hb.y) << 16);
    if (lo == hi) return lo;  // no E4M3 rounding boundary near q: exact
  }
  const float2 va = f32x2_split(v01), vb = f32x2_split(v23);
  return cvt2(va.x / s, va.y / s) | (cvt2(vb.x / s, vb.y / s) << 16);
}

// encode4_pairs over a 64-column row slice (16 groups of four): every group's
// codes are formed before any fallback division, so the groups' independent
// multiplies and conversions can interleave (a division branch per group
// serialized them). The codes are those of encode4_pairs.
__device__ __forceinline__ void encode64_pairs(const uint64_t (&acc)[32], uint32_t (&code)[16], float s, uint64_t r2,
                                               bool pow2) {
  if (pow2) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 a = f32x2_split(fmul2(acc[2 * j], r2)), b = f32x2_split(fmul2(acc[2 * j + 1], r2));
      code[j] = cvt2(a.x, a.y) | (cvt2(b.x, b.y) << 16);  // q = v / s exactly
    }
    return;
  }
  const uint64_t lo2 = f32x2(__float_as_uint(1.0f - 0x1p-20f), __float_as_uint(1.0f - 0x1p-20f));
  const uint64_t hi2 = f32x2(__float_as_uint(1.0f + 0x1p-20f), __float_as_uint(1.0f + 0x1p-20f));
  uint32_t bad = s >= 0x1p-126f ? 0u : 0xFFFFu;  // a subnormal scale is always divided
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint64_t q01 = fmul2(acc[2 * j], r2), q23 = fmul2(acc[2 * j + 1], r2);
    const float2 la = f32x2_split(fmul2(q01, lo2)), lb = f32x2_split(fmul2(q23, lo2));
    const float2 ha = f32x2_split(fmul2(q01, hi2)), hb = f32x2_split(fmul2(q23, hi2));
    const uint32_t lo = cvt2(la.x, la.y) | (cvt2(lb.x, lb.y) << 16);
    const uint32_t hi = cvt2(ha.x, ha.y) | (cvt2(hb.x, hb.y) << 16);
    code[j] = lo;
    bad |= (lo == hi ? 0u : 1u) << j;
  }
  if (bad != 0u) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if ((bad >> j) & 1u) {
        const float2 va = f32x2_split(acc[2 * j]), vb = f32x2_split(acc[2 * j + 1]);
        code[j] = cvt2(va.x / s, va.y / s) | (cvt2(vb.x / s, vb.y / s) << 16);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Requantizing GEMM epilogue.
//
// Each epilogue thread holds 64 FP32 accumulators: one output row, 64
// consecutive columns starting at a multiple of 64. A 128-column output block
// is covered by two such slices held by warps ew and ew ^ 4 of the same TMEM
// lane quadrant, and a 128 x 128 block by the eight warps [ew & ~7, +8).
// The slices' maxima meet in shared memory: every warp writes its values,
// arrives on the tile parity's exchange barrier (count = number of epilogue
// warps, release at CTA scope) and waits for it (bounded), then computes the
// scale, encodes and stores. Two sets of exchange slots alternate between
// tiles: a warp can only overwrite a set after every warp has arrived on the
// other set's barrier, i.e. after every read of the set's previous use.

// Shared-memory bytes of the exchange for kEpiWarps epilogue warps (8-byte aligned).
__host__ __device__ constexpr uint32_t requant_xchg_bytes(int epi_warps) {
  return 2 * 8 + 2 * epi_warps * 4 + 2 * epi_warps * 32 * 4;
}

// One epilogue warp's staging box for its 32 x 64 codes (TMA store source).
constexpr uint32_t kRequantBoxBytes = 32 * 64;

// Shared memory of the requantizing epilogue: the exchange, then one
// 1024-byte-aligned staging box per epilogue warp.
__host__ __device__ constexpr uint32_t requant_smem_bytes(int epi_warps) {
  return (requant_xchg_bytes(epi_warps) + 1023u) / 1024u * 1024u + epi_warps * kRequantBoxBytes;
}
__device__ __forceinline__ uint8_t* requant_box(uint8_t* xchg, int epi_warps, int ew) {
  return xchg + (requant_xchg_bytes(epi_warps) + 1023u) / 1024u * 1024u + ew * kRequantBoxBytes;
}

// Initializes the two exchange barriers (one thread, before the CTA's first sync).
__device__ __forceinline__ void requant_xchg_init(uint8_t* xchg, int epi_warps) {
  uint64_t* bar = reinterpret_cast<uint64_t*>(xchg);
  mbar_init(smem_u32(&bar[0]), epi_warps);
  mbar_init(smem_u32(&bar[1]), epi_warps);
}

// Requantizes one thread's slice: row `row` = row0 + lane (valid: row < M and
// not a padding row; invalid rows count as zeros and store nothing unless
// store_zero_row), columns [col0, col0 + 64) of an N-column output, tile
// sequence number tl (the same for all epilogue warps of the CTA). With a
// tensor map, whole 64-column slices leave through this warp's 2 KB staging
// box (64-byte swizzle: 16-byte chunk c of row r at chunk c ^ ((r / 2) % 4))
// and a TMA store clipped at M; without one (tmap_q == nullptr) each thread
// stores its 64 codes directly. A slice that crosses column N is stored
// element by element (the swizzled store clips N only to whole 16-byte chunks). Returns
// false if a wait failed (abort raised or timeout); then nothing is stored.
template <int kEpiWarps>
__device__ __forceinline__ bool requant_store_slice(const uint64_t (&acc)[32], bool row_valid,
                                                    bool store_zero_row, int row0, int M, int N, int col0,
                                                    int ew, int lane, uint32_t tl, uint8_t* xchg,
                                                    const RequantOut& o, const CUtensorMap* tmap_q,
                                                    uint8_t* box, bool& stores_issued, volatile int* abort,
                                                    unsigned int* status, uint64_t limit) {
  uint64_t* bar = reinterpret_cast<uint64_t*>(xchg);
  const uint32_t p = tl & 1u;
  float* xw = reinterpret_cast<float*>(xchg + 16) + p * kEpiWarps;
  float* xv = reinterpret_cast<float*>(xchg + 16 + 2 * kEpiWarps * 4) + p * kEpiWarps * 32;
  const int row = row0 + lane;

  float m = 0.f;
  if (row_valid) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float2 v = f32x2_split(acc[j]);
      m = fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y)));
    }
  }
  // Non-negative floats order like their bit patterns.
  if (o.block_rows == 1) {
    xv[ew * 32 + lane] = m;
  } else {
    const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
    if (lane == 0) xw[ew] = __uint_as_float(wm);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bar[p]));
  const bool w = mbar_wait(smem_u32(&bar[p]), (tl >> 1) & 1u, abort, status, limit);
  if (!__all_sync(0xFFFFFFFFu, w)) return false;

  float amax;
  if (o.block_rows == 1) {
    amax = fmaxf(m, xv[(ew ^ 4) * 32 + lane]);
  } else {
    const int w0 = ew & ~7;
    amax = xw[w0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, xw[w0 + i]);
  }
  const bool pow2 = o.pow2 != 0;
  const float s = block_scale(amax, pow2);
  const float r = 1.0f / s;
  const int sblk = col0 >> 7;  // 128-column block of this slice

  if (col0 >= N) return true;
  if (o.block_rows == 1) {
    if ((ew & 4) == 0 && row < M && (row_valid || store_zero_row))
      o.s[static_cast<int64_t>(row) * o.ld_s + sblk] = s;
  } else if (ew == (ew & ~7) && lane == 0 && (row0 & ~127) < M) {
    // One thread per block; the block's first row is row0 & ~127.
    o.s[static_cast<int64_t>(row0 >> 7) * o.ld_s + sblk] = s;
  }

  const uint64_t r2 = f32x2(__float_as_uint(r), __float_as_uint(r));
  uint32_t code[16];
  encode64_pairs(acc, code, s, r2, pow2);
  if (!row_valid) {
#pragma unroll
    for (int j = 0; j < 16; ++j) code[j] = 0u;
  }

  if (col0 + 64 <= N && tmap_q != nullptr) {
    if (lane == 0 && stores_issued) bulk_wait_read_all();  // the last store has read the box
    __syncwarp();
    uint8_t* my_row = box + lane * 64;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(my_row + ((c ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(code[4 * c], code[4 * c + 1], code[4 * c + 2], code[4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && row0 < M) {
      tma_store_2d(tmap_q, smem_u32(box), col0, row0);
      bulk_commit();
      stores_issued = true;
    }
    return true;
  }
  if (row >= M || !(row_valid || store_zero_row)) return true;
  uint8_t* dst = o.q + static_cast<int64_t>(row) * o.ld_q + col0;
  if (col0 + 64 <= N) {  // no TMA map: four 16-byte stores (ld_q and q are 16-byte aligned)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(code[4 * c], code[4 * c + 1], code[4 * c + 2], code[4 * c + 3]);
    return true;
  }
  const int n = N - col0;  // 1..63 valid columns
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (4 * j + 3 < n) {
      *reinterpret_cast<uint32_t*>(dst + 4 * j) = code[j];
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (4 * j + t < n) dst[4 * j + t] = static_cast<uint8_t>(code[j] >> (8 * t));
    }
  }
  return true;
}

}  // namespace dg
