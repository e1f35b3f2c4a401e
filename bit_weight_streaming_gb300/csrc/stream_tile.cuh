// Device pieces shared by the TMA-fed weight-stream kernels (the per-call
// product kernel and the persistent decode-step kernel): the unit geometry,
// the decode-and-MMA of one 16-row sub-tile, SiLU, and the host encoder of the
// 2D tensor maps the units are cut from.
//
// A unit is 128 rows x 128 bytes of each row (256 NVFP4 or 128 FP8 weights),
// loaded as four 32-row boxes with 128-byte swizzle, plus, for NVFP4, four
// 32-row x 16-byte boxes of E4M3 block scales.
#pragma once
#include <cuda.h>

#include "bws_common.cuh"
#include "bws_internal.h"

namespace bws {

constexpr int kBoxRows = 32;
constexpr int kBoxes = 4;                          // boxes per unit
constexpr int kBoxBytes = kBoxRows * 128;          // one code box
constexpr int kCodeBytes = kBoxes * kBoxBytes;     // code bytes of a unit
constexpr int kScaleBoxBytes = kBoxRows * 16;      // one NVFP4 scale box

static BWS_DEV float silu_mul_t(float g, float u) {
  const float sg = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  return __fmul_rn(sg, u);
}

// Products of one 16-row sub-tile with one unit's activations: w0 / w1 are
// the lane's chunk words of rows g / g+8, sc0 / sc1 their two block scales
// (NVFP4), xh the hi-band pieces, xl the lo band (when lo).
template <int FMT, bool LO>
BWS_DEV void sub_mma(float (&acc)[2][4], float (&accl)[4], const uint32_t (&w0)[4], const uint32_t (&w1)[4],
                     uint32_t sc0, uint32_t sc1, const uint4 (&xh)[FMT == kFmtFP8 ? 2 : 4],
                     const uint4 (&xl)[FMT == kFmtFP8 ? 2 : 4]) {
  if constexpr (FMT == kFmtFP8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t a0, a2, a1, a3;
      e4m3x4_to_f16x2x2(w0[j], a0, a2);
      e4m3x4_to_f16x2x2(w1[j], a1, a3);
      const uint4& xq = xh[j >> 1];
      mma_f16_16816(acc[j & 1], a0, a1, a2, a3, (j & 1) ? xq.z : xq.x, (j & 1) ? xq.w : xq.y);
      if (LO) {
        const uint4& lq = xl[j >> 1];
        mma_f16_16816(accl, a0, a1, a2, a3, (j & 1) ? lq.z : lq.x, (j & 1) ? lq.w : lq.y);
      }
    }
  } else {
    const uint32_t f0 = e4m3x2_to_f16x2(sc0), f1 = e4m3x2_to_f16x2(sc1);
    const uint32_t m0[2] = {bcast_lo(f0), bcast_hi(f0)};
    const uint32_t m1[2] = {bcast_lo(f1), bcast_hi(f1)};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
      e2m1x8_to_f16x2x4(w0[w], p0, p1, p2, p3);
      e2m1x8_to_f16x2x4(w1[w], q0, q1, q2, q3);
      const uint32_t sa = m0[w >> 1], sb = m1[w >> 1];
      p0 = hmul2_u32(p0, sa); p1 = hmul2_u32(p1, sa); p2 = hmul2_u32(p2, sa); p3 = hmul2_u32(p3, sa);
      q0 = hmul2_u32(q0, sb); q1 = hmul2_u32(q1, sb); q2 = hmul2_u32(q2, sb); q3 = hmul2_u32(q3, sb);
      mma_f16_16816(acc[0], p0, q0, p1, q1, xh[w].x, xh[w].y);
      mma_f16_16816(acc[1], p2, q2, p3, q3, xh[w].z, xh[w].w);
      if (LO) {
        mma_f16_16816(accl, p0, q0, p1, q1, xl[w].x, xl[w].y);
        mma_f16_16816(accl, p2, q2, p3, q3, xl[w].z, xl[w].w);
      }
    }
  }
}

// True if the driver's tensor-map encoder can be reached.
bool tensor_maps_available();
// One token, NVFP4: the products of one 16-row sub-tile with one unit, block
// scales applied to the accumulators. The activation operand is block
// diagonal: lanes with g == 2t hold their chunk's first-block activations
// (words 0, 1) and lanes with g == 2t + 1 its second-block ones (words 2, 3),
// every other lane zeros, so MMA column 2t' + e collects exactly block e of
// lane t''s chunk. Lane (g, t) then holds, for rows g and g + 8, the raw sums
// of its own chunk's two blocks and adds them, times their E4M3 scales, to y
// (y[0], y[1]: row g blocks 0, 1; y[2], y[3]: row g + 8).
template <bool LO>
BWS_DEV void sub_mma_n1(float (&y)[4], float (&yl)[4], const uint32_t (&w0)[4], const uint32_t (&w1)[4],
                        uint32_t sc0, uint32_t sc1, const uint4 (&xh)[4], const uint4 (&xl)[4]) {
  float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
  float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
    e2m1x8_to_f16x2x4(w0[w], p0, p1, p2, p3);
    e2m1x8_to_f16x2x4(w1[w], q0, q1, q2, q3);
    float (&d)[4] = w < 2 ? da : db;
    mma_f16_16816(d, p0, q0, p1, q1, xh[w].x, xh[w].y);
    mma_f16_16816(d, p2, q2, p3, q3, xh[w].z, xh[w].w);
    if (LO) {
      float (&l)[4] = w < 2 ? la : lb;
      mma_f16_16816(l, p0, q0, p1, q1, xl[w].x, xl[w].y);
      mma_f16_16816(l, p2, q2, p3, q3, xl[w].z, xl[w].w);
    }
  }
  const uint32_t f0 = e4m3x2_to_f16x2(sc0), f1 = e4m3x2_to_f16x2(sc1);
  const float s[4] = {__half2float(__ushort_as_half((unsigned short)(f0 & 0xFFFF))),
                      __half2float(__ushort_as_half((unsigned short)(f0 >> 16))),
                      __half2float(__ushort_as_half((unsigned short)(f1 & 0xFFFF))),
                      __half2float(__ushort_as_half((unsigned short)(f1 >> 16)))};
  y[0] = __fmaf_rn(s[0], da[0], y[0]);
  y[1] = __fmaf_rn(s[1], db[1], y[1]);
  y[2] = __fmaf_rn(s[2], da[2], y[2]);
  y[3] = __fmaf_rn(s[3], db[3], y[3]);
  if (LO) {
    yl[0] = __fmaf_rn(s[0], la[0], yl[0]);
    yl[1] = __fmaf_rn(s[1], lb[1], yl[1]);
    yl[2] = __fmaf_rn(s[2], la[2], yl[2]);
    yl[3] = __fmaf_rn(s[3], lb[3], yl[3]);
  }
}

// Encodes a 2D u8 tensor map [rows][inner_bytes] with the given box (128-byte
// swizzle or none). False if the driver entry point is missing or refuses.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint32_t box_inner,
               uint32_t box_rows, bool swizzle);
// A 2D tensor map of packed E2M1 codes [rows][d_in / 2 bytes] that TMA
// unpacks on the way into shared memory: each 16 codes (8 bytes) land in a
// 16-byte slot, the layout the tensor cores read 4-bit operands from. Box
// {128 codes, box_rows}, 128-byte swizzle; d_in % 128 == 0, base 32-byte
// aligned, d_in / 2 a multiple of 32.
bool encode_fp4_2d(CUtensorMap* m, const void* base, uint64_t d_in, uint64_t rows, uint32_t box_rows);
// A 3D u8 tensor map [n][rows][inner_bytes] (byte stride stride2 between the
// n planes) with box {box_inner, box_rows, 1} and 128-byte swizzle.
bool encode_3d(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint64_t n,
               uint64_t stride2, uint32_t box_inner, uint32_t box_rows);

}  // namespace bws
