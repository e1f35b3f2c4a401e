// Weight-stream products: N <= 8 token rows against NVFP4, MXFP4 or FP8
// weights, exact products, FP32 accumulation.
//
// Work decomposition ("stream-K"): a tile is 32 output rows (two 16-row MMA
// sub-tiles), a work unit is one tile x 128 consecutive k. The units of all
// tiles, in tile-major order, are split into equal contiguous ranges, one per
// warp, so every warp streams the same number of bytes whatever the shape.
// A tile cut between warps is finished by the last warp to arrive, which adds
// the pieces' partial sums in a fixed order (deterministic, no float atomics).
//
// Per unit a lane (g = lane/4, t = lane%4) holds, for rows g and g+8 of each
// sub-tile, the 32 consecutive weights k = 32t..32t+31 of the unit. MMA j
// (j = 0..7) takes physical k = 32t+4j+{0,1,2,3} as its logical k
// {2t, 2t+1, 2t+8, 2t+9}; the activations are loaded with the same mapping,
// so the permutation cancels in the dot product. Each MMA is
// mma.sync.m16n8k16 f16 x f16 -> f32 with the 8 token rows as its N dimension.
//
// Weights become exact f16: E2M1 and E4M3 codes by the hardware converters,
// NVFP4 block scales applied by an exact f16 multiply (an E2M1 value times an
// E4M3 value has at most 6 significant bits and lies in [2^-10, 2688]);
// MXFP4 block scales 2^(e - e_ref) relative to the unit's largest, with the
// unit partial sum rescaled by 2^e_ref in FP32.
#include "bws_common.cuh"
#include "bws_internal.h"

namespace bws {

namespace {

// In-flight data of one unit for one lane.
template <int FMT, bool LO>
struct Frag {
  uint4 c[2][2][FMT == kFmtFP8 ? 2 : 1];   // [sub][row g / g+8][16-byte pieces]
  uint32_t sc[2][2];                        // [sub][row g / g+8] block scale bytes
  uint4 xh[4];                              // this lane's 32 f16 activations, hi band
  uint4 xl[LO ? 4 : 1];                     // lo band
};

struct TileRows {
  int mat[2];
  int row0[2];        // first row of each sub-tile within its matrix
};

template <int EPI>
BWS_DEV TileRows tile_rows(const GemvParams& p, int tile) {
  TileRows tr;
  if (EPI == kEpiSwiGLU) {
    tr.mat[0] = 0; tr.mat[1] = 1;
    tr.row0[0] = tr.row0[1] = tile * 16;
  } else {
    int m = 0;
#pragma unroll
    for (int i = 1; i < kMaxMats; ++i)
      if (i < p.n_mats && tile >= p.mats[i].tile_begin) m = i;
    const int local = tile - p.mats[m].tile_begin;
    tr.mat[0] = tr.mat[1] = m;
    tr.row0[0] = local * 32;
    tr.row0[1] = local * 32 + 16;
  }
  return tr;
}

// Per-tile lane pointers: computed once per piece, advanced per unit.
template <int FMT>
struct LanePtrs {
  const uint8_t* c[2][2];
  const uint8_t* sc[2][2];
  const uint16_t* xh;
  const uint16_t* xl;
  uint32_t rowmask;   // bit 2*s+h: row valid
};

template <int FMT, int EPI>
BWS_DEV LanePtrs<FMT> lane_ptrs(const GemvParams& p, const TileRows& tr, int g, int t) {
  LanePtrs<FMT> L;
  L.rowmask = 0u;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const GemvMat& M = p.mats[tr.mat[s]];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = tr.row0[s] + g + 8 * h;
      const int rr = row < M.d_out ? row : 0;
      if (row < M.d_out) L.rowmask |= 1u << (2 * s + h);
      if (FMT == kFmtFP8) {
        L.c[s][h] = M.codes + (size_t)rr * p.d_in + 32 * t;
        L.sc[s][h] = nullptr;
      } else {
        L.c[s][h] = M.codes + (size_t)rr * (p.d_in >> 1) + 16 * t;
        L.sc[s][h] = FMT == kFmtNVFP4 ? M.scales + (size_t)rr * (p.d_in >> 4) + 2 * t
                                      : M.scales + (size_t)rr * (p.d_in >> 5) + t;
      }
    }
  }
  // token rows g >= N read the all-zero row kept after the N real rows
  const size_t xo = (size_t)(g < p.N ? g : p.N) * p.d_in_pad + 32 * t;
  L.xh = p.x.hi + xo;
  L.xl = p.x.lo + xo;
  return L;
}

// Loads are unpredicated: rows past d_out read row 0 (their outputs are never
// stored) and lanes past d_in read the row's last 32 weights, which meet the
// zero padding of the activations, so they add nothing.
template <int FMT, bool LO>
BWS_DEV void load_unit(const GemvParams& p, const LanePtrs<FMT>& L, int seg, int g, int t, Frag<FMT, LO>& f) {
  const int k0 = min(seg * kSegK + 32 * t, p.d_in - 32) - 32 * t;   // lane offset added in L
  const int cb = FMT == kFmtFP8 ? k0 : (k0 >> 1);
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      f.c[s][h][0] = ld_stream_v4(L.c[s][h] + cb);
      if constexpr (FMT == kFmtFP8) {
        f.c[s][h][FMT == kFmtFP8 ? 1 : 0] = ld_stream_v4(L.c[s][h] + cb + 16);
        f.sc[s][h] = 0u;
      } else if constexpr (FMT == kFmtNVFP4) {
        f.sc[s][h] = ld_stream_u16(L.sc[s][h] + (k0 >> 4));
      } else {
        f.sc[s][h] = ld_stream_u8(L.sc[s][h] + (k0 >> 5));
      }
    }
#pragma unroll
  for (int i = 0; i < 4; ++i) f.xh[i] = ld_act_v4(L.xh + seg * kSegK + 8 * i);
  if (LO) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f.xl[i] = ld_act_v4(L.xl + seg * kSegK + 8 * i);
  }
}

BWS_DEV uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// f16 2^k for k <= 0, exact down to 2^-24, 0 below.
BWS_DEV uint32_t f16x2_pow2(int k) {
  uint32_t h;
  if (k >= -14) h = (uint32_t)(k + 15) << 10;
  else if (k >= -24) h = 1u << (k + 24);
  else h = 0u;
  return h | (h << 16);
}

// Accumulators: [sub][chain][4].
constexpr int kChains = 1;
typedef float Acc[2][kChains][4];

template <int FMT, bool LO>
BWS_DEV void compute_unit(const Frag<FMT, LO>& f, Acc& acc, Acc& accl) {
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    if constexpr (FMT == kFmtFP8) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t a0, a2, a1, a3;
        e4m3x4_to_f16x2x2(word_of(f.c[s][0][j >> 2], j & 3), a0, a2);
        e4m3x4_to_f16x2x2(word_of(f.c[s][1][j >> 2], j & 3), a1, a3);
        const uint32_t b0 = word_of(f.xh[j >> 1], 2 * (j & 1));
        const uint32_t b1 = word_of(f.xh[j >> 1], 2 * (j & 1) + 1);
        mma_f16_16816(acc[s][(j & 1) % kChains], a0, a1, a2, a3, b0, b1);
        if (LO) {
          const uint32_t c0 = word_of(f.xl[j >> 1], 2 * (j & 1));
          const uint32_t c1 = word_of(f.xl[j >> 1], 2 * (j & 1) + 1);
          mma_f16_16816(accl[s][(j & 1) % kChains], a0, a1, a2, a3, c0, c1);
        }
      }
    } else {
      uint32_t mg[2], m8[2];   // multipliers for the two 16-weight halves
      float sref_g = 0.f, sref_8 = 0.f;
      if constexpr (FMT == kFmtNVFP4) {
        const uint32_t sg = e4m3x2_to_f16x2(f.sc[s][0]);
        const uint32_t s8 = e4m3x2_to_f16x2(f.sc[s][1]);
        mg[0] = bcast_lo(sg); mg[1] = bcast_hi(sg);
        m8[0] = bcast_lo(s8); m8[1] = bcast_hi(s8);
      } else {
        // MXFP4: the lane's 32 weights are one E8M0 block; scale relative to
        // the largest block of the row in this unit, rescale the sum in FP32.
        const int eg = (int)f.sc[s][0] - 127;
        const int e8 = (int)f.sc[s][1] - 127;
        int rg = max(eg, __shfl_xor_sync(0xffffffffu, eg, 1));
        rg = max(rg, __shfl_xor_sync(0xffffffffu, rg, 2));
        int r8 = max(e8, __shfl_xor_sync(0xffffffffu, e8, 1));
        r8 = max(r8, __shfl_xor_sync(0xffffffffu, r8, 2));
        mg[0] = mg[1] = f16x2_pow2(eg - rg);
        m8[0] = m8[1] = f16x2_pow2(e8 - r8);
        sref_g = exp2i(rg);
        sref_8 = exp2i(r8);
      }
      float dm[kChains][4] = {};
      float dml[kChains][4] = {};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
        e2m1x8_to_f16x2x4(word_of(f.c[s][0][0], w), p0, p1, p2, p3);
        e2m1x8_to_f16x2x4(word_of(f.c[s][1][0], w), q0, q1, q2, q3);
        const uint32_t sa = mg[w >> 1], sb = m8[w >> 1];
        p0 = hmul2_u32(p0, sa); p1 = hmul2_u32(p1, sa); p2 = hmul2_u32(p2, sa); p3 = hmul2_u32(p3, sa);
        q0 = hmul2_u32(q0, sb); q1 = hmul2_u32(q1, sb); q2 = hmul2_u32(q2, sb); q3 = hmul2_u32(q3, sb);
        float(&D0)[4] = FMT == kFmtMXFP4 ? dm[0] : acc[s][0];
        float(&D1)[4] = FMT == kFmtMXFP4 ? dm[1 % kChains] : acc[s][1 % kChains];
        mma_f16_16816(D0, p0, q0, p1, q1, f.xh[w].x, f.xh[w].y);
        mma_f16_16816(D1, p2, q2, p3, q3, f.xh[w].z, f.xh[w].w);
        if (LO) {
          float(&L0)[4] = FMT == kFmtMXFP4 ? dml[0] : accl[s][0];
          float(&L1)[4] = FMT == kFmtMXFP4 ? dml[1 % kChains] : accl[s][1 % kChains];
          mma_f16_16816(L0, p0, q0, p1, q1, f.xl[w].x, f.xl[w].y);
          mma_f16_16816(L1, p2, q2, p3, q3, f.xl[w].z, f.xl[w].w);
        }
      }
      if constexpr (FMT == kFmtMXFP4) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) {
          acc[s][c][0] = __fmaf_rn(dm[c][0], sref_g, acc[s][c][0]);
          acc[s][c][1] = __fmaf_rn(dm[c][1], sref_g, acc[s][c][1]);
          acc[s][c][2] = __fmaf_rn(dm[c][2], sref_8, acc[s][c][2]);
          acc[s][c][3] = __fmaf_rn(dm[c][3], sref_8, acc[s][c][3]);
          if (LO) {
            accl[s][c][0] = __fmaf_rn(dml[c][0], sref_g, accl[s][c][0]);
            accl[s][c][1] = __fmaf_rn(dml[c][1], sref_g, accl[s][c][1]);
            accl[s][c][2] = __fmaf_rn(dml[c][2], sref_8, accl[s][c][2]);
            accl[s][c][3] = __fmaf_rn(dml[c][3], sref_8, accl[s][c][3]);
          }
        }
      }
    }
  }
}

BWS_DEV float silu_mul(float g, float u) {
  const float sg = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  return __fmul_rn(sg, u);
}

// Scale raw sums v[sub][4] to outputs and store them.
template <int FMT, int EPI>
BWS_DEV void finish_tile(const GemvParams& p, const TileRows& tr, int g, int t,
                         const float (&v)[2][4], const int (&xexp)[2]) {
  float val[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const GemvMat& M = p.mats[tr.mat[s]];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = tr.row0[s] + g + 8 * (i >> 1);
      float sc = 1.0f;
      if (FMT == kFmtNVFP4) sc = __ldg(M.scale32);
      if (FMT == kFmtFP8) sc = row < M.d_out ? __ldg(M.scale32 + row) : 0.0f;
      val[s][i] = ldexp_exact(__fmul_rn(v[s][i], sc), xexp[i & 1] - 14);
    }
  }
  if constexpr (EPI == kEpiSwiGLU) {
    const int d_out = p.mats[0].d_out;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = tr.row0[0] + g + 8 * (i >> 1);
      const int tok = 2 * t + (i & 1);
      if (row < d_out && tok < p.N) {
        const float h = silu_mul(val[0][i], val[1][i]);
        reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t)tok * p.out_ld + row] = __float2bfloat16_rn(h);
      }
    }
  } else {
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const GemvMat& M = p.mats[tr.mat[s]];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = tr.row0[s] + g + 8 * (i >> 1);
      const int tok = 2 * t + (i & 1);
      if (row < M.d_out && tok < p.N) {
        const size_t o = (size_t)tok * p.out_ld + M.out_row_off + row;
        if (EPI == kEpiStoreBF16)
          reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(val[s][i]);
        else if (EPI == kEpiStoreF32)
          reinterpret_cast<float*>(p.out)[o] = val[s][i];
        else
          reinterpret_cast<float*>(p.out)[o] = __fadd_rn(reinterpret_cast<float*>(p.out)[o], val[s][i]);
      }
    }
  }
  }
}

BWS_DEV long long owner_warp(long long u, long long U, long long W) {
  return ((u + 1) * W - 1) / U;
}
BWS_DEV long long range_begin(long long w, long long U, long long W) { return w * U / W; }

// End of a warp's piece of a tile: finish directly, or deposit the partial
// sums and let the last contributor finish the tile.
template <int FMT, int EPI>
BWS_DEV void end_piece(const GemvParams& p, int tile, long long warp_id, bool whole,
                       float (&v)[2][4], const int (&xexp)[2], int lane) {
  const int g = lane >> 2, t = lane & 3;
  const TileRows tr = tile_rows<EPI>(p, tile);
  if (whole) {
    finish_tile<FMT, EPI>(p, tr, g, t, v, xexp);
    return;
  }
  const long long U = p.n_units, W = p.n_warps;
  float4* slot = reinterpret_cast<float4*>(p.partials) + (size_t)(tile + warp_id) * (kSlotFloats / 4);
  slot[lane] = make_float4(v[0][0], v[0][1], v[0][2], v[0][3]);
  slot[32 + lane] = make_float4(v[1][0], v[1][1], v[1][2], v[1][3]);
  __threadfence();
  __syncwarp();
  const long long w0 = owner_warp((long long)tile * p.nseg, U, W);
  const long long w1 = owner_warp((long long)(tile + 1) * p.nseg - 1, U, W);
  uint32_t prev = 0;
  if (lane == 0) prev = atomicAdd(p.counters + tile, 1u);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != (uint32_t)(w1 - w0)) return;
  __threadfence();
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  for (long long w = w0; w <= w1; ++w) {
    const float4* o = reinterpret_cast<const float4*>(p.partials) + (size_t)(tile + w) * (kSlotFloats / 4);
    float4 a, b;
    if (w == warp_id) {
      a = make_float4(v[0][0], v[0][1], v[0][2], v[0][3]);
      b = make_float4(v[1][0], v[1][1], v[1][2], v[1][3]);
    } else {
      a = ld_cg_f4(o + lane);
      b = ld_cg_f4(o + 32 + lane);
    }
    s[0][0] += a.x; s[0][1] += a.y; s[0][2] += a.z; s[0][3] += a.w;
    s[1][0] += b.x; s[1][1] += b.y; s[1][2] += b.z; s[1][3] += b.w;
  }
  finish_tile<FMT, EPI>(p, tr, g, t, s, xexp);
  if (lane == 0) p.counters[tile] = 0u;
}

// Pull unit u's weights of this warp's 32 rows towards L2 (lane l: row l).
template <int FMT, int EPI>
BWS_DEV void prefetch_unit(const GemvParams& p, long long u, int lane) {
  const int tile = (int)(u / p.nseg);
  const int seg = (int)(u % p.nseg);
  const TileRows tr = tile_rows<EPI>(p, tile);
  const int s = lane >> 4;
  const GemvMat& M = p.mats[tr.mat[s]];
  const int row = tr.row0[s] + (lane & 15);
  if (row >= M.d_out) return;
  if (FMT == kFmtFP8) {
    const uint8_t* a = M.codes + (size_t)row * p.d_in + seg * kSegK;
    const int nb = min(kSegK, p.d_in - seg * kSegK);
    if (nb >= 16) prefetch_l2_bulk(a, (uint32_t)(nb & ~15));
  } else {
    const uint8_t* a = M.codes + (size_t)row * (p.d_in >> 1) + seg * (kSegK / 2);
    const int nb = min(kSegK / 2, (p.d_in >> 1) - seg * (kSegK / 2));
    if (nb >= 16) prefetch_l2_bulk(a, (uint32_t)(nb & ~15));
    const uint8_t* sa = FMT == kFmtNVFP4 ? M.scales + (size_t)row * (p.d_in >> 4) + seg * (kSegK / 16)
                                         : M.scales + (size_t)row * (p.d_in >> 5) + seg * (kSegK / 32);
    asm volatile("prefetch.global.L2 [%0];" :: "l"(sa));
  }
}

// Lane l pulls row l's bytes of units [sa, sb] of a tile into L2 (one op).
template <int FMT>
BWS_DEV void prefetch_rows(const GemvParams& p, const TileRows& tr, int sa, int sb, int lane) {
  const int sub = lane >> 4;
  const GemvMat& M = p.mats[tr.mat[sub]];
  const int row = tr.row0[sub] + (lane & 15);
  if (row >= M.d_out || sb < sa) return;
  const int per = FMT == kFmtFP8 ? kSegK : kSegK / 2;
  const size_t row_bytes = FMT == kFmtFP8 ? (size_t)p.d_in : (size_t)(p.d_in >> 1);
  const size_t kb0 = (size_t)sa * per;
  size_t nb = (size_t)(sb - sa + 1) * per;
  if (kb0 + nb > row_bytes) nb = row_bytes - kb0;
  if (nb >= 16) prefetch_l2_bulk(M.codes + (size_t)row * row_bytes + kb0, (uint32_t)(nb & ~(size_t)15));
}

// One piece: units [seg0, seg1] of one tile, software-pipelined two deep.
template <int FMT, int EPI, bool LO>
BWS_DEV void run_piece(const GemvParams& p, int tile, int seg0, int seg1, long long warp_id, int lane,
                       const int (&xexp)[2]) {
  const int g = lane >> 2, t = lane & 3;
  const TileRows tr = tile_rows<EPI>(p, tile);
  const LanePtrs<FMT> L = lane_ptrs<FMT, EPI>(p, tr, g, t);
  Acc acc = {}, accl = {};
  if (LO) {
    // rare path (two activation bands): one unit at a time
    for (int seg = seg0; seg <= seg1; ++seg) {
      Frag<FMT, true> f;
      load_unit<FMT, true>(p, L, seg, g, t, f);
      compute_unit<FMT, true>(f, acc, accl);
    }
  } else {
    Frag<FMT, false> fa, fb;
    const int P = p.prefetch_ahead;           // L2 prefetch window in units
    if (P > 0) prefetch_rows<FMT>(p, tr, seg0, min(seg1, seg0 + P - 1), lane);
    load_unit<FMT, false>(p, L, seg0, g, t, fa);
    for (int seg = seg0; seg <= seg1; seg += 2) {
      if (seg + 1 <= seg1) load_unit<FMT, false>(p, L, seg + 1, g, t, fb);
      // every P/2 units, extend the prefetched window to P units ahead
      if (P > 0 && ((seg - seg0) % (P >> 1)) < 2 && ((seg - seg0) % (P >> 1)) == 0 && seg + P <= seg1)
        prefetch_rows<FMT>(p, tr, seg + P - (P >> 1) + 1, min(seg1, seg + P), lane);
      compute_unit<FMT, false>(fa, acc, accl);
      if (seg + 1 > seg1) break;
      if (seg + 2 <= seg1) load_unit<FMT, false>(p, L, seg + 2, g, t, fa);
      compute_unit<FMT, false>(fb, acc, accl);
    }
  }
  float v[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float a = acc[s][0][i], al = accl[s][0][i];
#pragma unroll
      for (int c = 1; c < kChains; ++c) { a = __fadd_rn(a, acc[s][c][i]); al = __fadd_rn(al, accl[s][c][i]); }
      v[s][i] = LO ? __fmaf_rn(al, 0x1p-29f, a) : a;
    }
  const bool whole = seg0 == 0 && seg1 == p.nseg - 1;
  end_piece<FMT, EPI>(p, tile, warp_id, whole, v, xexp, lane);
}

// The two-band path is rare; keep it out of line so that its register
// needs do not constrain the common path.
template <int FMT, int EPI, bool LO>
__device__ __noinline__ void run_range_lo(const GemvParams& p, long long u, long long u_end, long long warp_id,
                                          int lane, int xe0, int xe1);

template <int FMT, int EPI, bool LO>
BWS_DEV void run_range(const GemvParams& p, long long u, long long u_end, long long warp_id, int lane,
                       const int (&xexp)[2]) {
  while (u < u_end) {
    const int tile = (int)(u / p.nseg);
    const int seg0 = (int)(u % p.nseg);
    const long long left = u_end - u;
    const int seg1 = (long long)(p.nseg - 1 - seg0) < left ? p.nseg - 1 : seg0 + (int)left - 1;
    run_piece<FMT, EPI, LO>(p, tile, seg0, seg1, warp_id, lane, xexp);
    u += seg1 - seg0 + 1;
  }
}

template <int FMT, int EPI, bool LO>
__device__ __noinline__ void run_range_lo(const GemvParams& p, long long u, long long u_end, long long warp_id,
                                          int lane, int xe0, int xe1) {
  const int xexp[2] = {xe0, xe1};
  run_range<FMT, EPI, true>(p, u, u_end, warp_id, lane, xexp);
}

#ifndef BWS_GEMV_MIN_BLOCKS
#define BWS_GEMV_MIN_BLOCKS 2
#endif

template <int FMT, int EPI>
__global__ void __launch_bounds__(kWarpsPerCta * 32, BWS_GEMV_MIN_BLOCKS) gemv_kernel(const __grid_constant__ GemvParams p) {
  const int lane = threadIdx.x & 31;
  const long long warp_id = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  pdl_launch_dependents();
  if (warp_id >= p.n_warps) { pdl_wait(); return; }
  const long long U = p.n_units, W = p.n_warps;
  const long long u0 = range_begin(warp_id, U, W);
  const long long u1 = range_begin(warp_id + 1, U, W);

  // Weights do not depend on earlier kernels: start pulling the first units
  // of this warp's range into L2 before waiting for the activations (one bulk
  // prefetch per lane, lane l covering row l of the first tile piece).
  if (p.prefetch_units > 0) {
    const int tile = (int)(u0 / p.nseg);
    const int seg = (int)(u0 % p.nseg);
    long long nu = p.nseg - seg;
    if (nu > p.prefetch_units) nu = p.prefetch_units;
    if (nu > u1 - u0) nu = u1 - u0;
    const TileRows tr = tile_rows<EPI>(p, tile);
    const int sub = lane >> 4;
    const GemvMat& M = p.mats[tr.mat[sub]];
    const int row = tr.row0[sub] + (lane & 15);
    if (row < M.d_out && nu > 0) {
      const int per = FMT == kFmtFP8 ? kSegK : kSegK / 2;
      const size_t row_bytes = FMT == kFmtFP8 ? (size_t)p.d_in : (size_t)(p.d_in >> 1);
      const size_t kb0 = (size_t)seg * per;
      size_t nb = (size_t)nu * per;
      if (kb0 + nb > row_bytes) nb = row_bytes - kb0;
      if (nb >= 16) prefetch_l2_bulk(M.codes + (size_t)row * row_bytes + kb0, (uint32_t)(nb & ~(size_t)15));
    }
  }
  pdl_wait();

  int xexp[2];
  uint32_t flags = 0u;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int tok = 2 * (lane & 3) + i;
    xexp[i] = tok < p.N ? __ldg(p.x.exp + tok) : 0;
  }
  for (int tok = 0; tok < p.N; ++tok) flags |= __ldg(p.x.flags + tok);
  if (flags & 1u)
    run_range_lo<FMT, EPI, true>(p, u0, u1, warp_id, lane, xexp[0], xexp[1]);
  else
    run_range<FMT, EPI, false>(p, u0, u1, warp_id, lane, xexp);
}

// ---- activation prep ----------------------------------------------------------

// One CTA per token: E = floor(log2 max|x|), then the two f16 bands. Each
// thread handles 8-element chunks (d_in % 32 == 0, so a chunk never straddles
// d_in). Also zeroes the counters of the product that follows.
constexpr int kPrepThreads = 1024;
__global__ void __launch_bounds__(kPrepThreads) prep_x_kernel(const uint16_t* __restrict__ x, int N, int d_in,
                                                              int d_in_pad, uint16_t* __restrict__ xhi,
                                                              uint16_t* __restrict__ xlo, int* __restrict__ xexp,
                                                              uint32_t* __restrict__ xflags, uint32_t* __restrict__ hdr,
                                                              uint32_t* __restrict__ zero_ptr, int zero_words) {
  pdl_launch_dependents();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < zero_words; i += gridDim.x * blockDim.x)
    zero_ptr[i] = 0u;
  if (blockIdx.x == 0) {   // the all-zero token row N read by unused MMA columns
    uint4* zh = reinterpret_cast<uint4*>(xhi + (size_t)N * d_in_pad);
    uint4* zl = reinterpret_cast<uint4*>(xlo + (size_t)N * d_in_pad);
    for (int c = threadIdx.x; c < (d_in_pad >> 3); c += blockDim.x) {
      zh[c] = make_uint4(0, 0, 0, 0);
      zl[c] = make_uint4(0, 0, 0, 0);
    }
  }
  const int tok = blockIdx.x;
  if (tok >= N) return;
  if (tok == 0 && threadIdx.x == 0) hdr[0] = (uint32_t)N;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)tok * d_in);
  const int nchunk = d_in >> 3, nchunk_pad = d_in_pad >> 3;
  float m = 0.0f;
  for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
    const uint4 v = __ldg(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
  }
  m = warp_max(m);
  __shared__ float sm[kPrepThreads / 32];
  __shared__ uint32_t sf[kPrepThreads / 32];
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = m;
  __syncthreads();
  float mx = 0.0f;
#pragma unroll 8
  for (int i = 0; i < kPrepThreads / 32; ++i) mx = fmaxf(mx, sm[i]);
  const int E = mx > 0.0f ? floor_log2_abs(mx) : 0;
  uint32_t flags = 0u;
  uint4* hi4 = reinterpret_cast<uint4*>(xhi + (size_t)tok * d_in_pad);
  uint4* lo4 = reinterpret_cast<uint4*>(xlo + (size_t)tok * d_in_pad);
  for (int c = threadIdx.x; c < nchunk_pad; c += blockDim.x) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (c < nchunk) v = __ldg(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t hh[2], ll[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float f = __uint_as_float(j == 0 ? (w[i] << 16) : (w[i] & 0xFFFF0000u));
        const float a = ldexp_exact(f, 14 - E);
        hh[j] = 0u;
        ll[j] = 0u;
        if (fabsf(a) >= 0x1p-14f) {
          hh[j] = __half_as_ushort(__float2half_rn(a));
        } else if (f != 0.0f) {
          const float b = ldexp_exact(f, 43 - E);
          if (fabsf(b) >= 0x1p-14f) {
            ll[j] = __half_as_ushort(__float2half_rn(b));
            flags |= 1u;
          } else {
            flags |= 2u;
          }
        }
      }
      h[i] = hh[0] | (hh[1] << 16);
      l[i] = ll[0] | (ll[1] << 16);
    }
    hi4[c] = make_uint4(h[0], h[1], h[2], h[3]);
    lo4[c] = make_uint4(l[0], l[1], l[2], l[3]);
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if ((threadIdx.x & 31) == 0) sf[threadIdx.x >> 5] = flags;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t f = 0u;
    for (int i = 0; i < kPrepThreads / 32; ++i) f |= sf[i];
    xexp[tok] = E;
    xflags[tok] = f;
  }
}

template <int FMT, int EPI>
cudaError_t launch_one(const GemvParams& p, cudaStream_t st, bool pdl) {
  const long long ctas = (p.n_warps + kWarpsPerCta - 1) / kWarpsPerCta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.stream = st;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<FMT, EPI>, p);
}

}  // namespace

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 152;
  }
  return n;
}

long long gemv_max_warps() { return (long long)num_sms() * BWS_GEMV_MIN_BLOCKS * kWarpsPerCta; }

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

GemvWorkspace gemv_workspace_layout(int N, int d_in, int n_tiles, long long max_warps) {
  GemvWorkspace w;
  const size_t d_pad = (size_t)((d_in + kSegK - 1) / kSegK) * kSegK;
  size_t o = 0;
  w.off_hdr = o; o += 256;
  w.off_exp = o; o += align256(sizeof(int) * kMaxTokens);
  w.off_flags = o; o += align256(sizeof(uint32_t) * kMaxTokens);
  w.off_hi = o; o += align256(2 * d_pad * (N + 1));   // N tokens + one zero row
  w.off_lo = o; o += align256(2 * d_pad * (N + 1));
  w.off_counters = o; o += align256(sizeof(uint32_t) * (size_t)n_tiles);
  w.off_partials = o; o += align256(sizeof(float) * kSlotFloats * ((size_t)n_tiles + max_warps));
  w.total = o;
  return w;
}

cudaError_t launch_prep_x(const uint16_t* x, int N, int d_in, int d_in_pad, uint16_t* xhi, uint16_t* xlo,
                          int* xexp, uint32_t* xflags, uint32_t* hdr, uint32_t* zero_ptr, int zero_words,
                          cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)N);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prep_x_kernel, x, N, d_in, d_in_pad, xhi, xlo, xexp, xflags, hdr,
                            zero_ptr, zero_words);
}

cudaError_t launch_gemv(int fmt, int epi, const GemvParams& p, cudaStream_t st, bool pdl) {
#define BWS_CASE(F, E) \
  if (fmt == F && epi == E) return launch_one<F, E>(p, st, pdl);
  BWS_CASE(kFmtNVFP4, kEpiStoreBF16)
  BWS_CASE(kFmtNVFP4, kEpiResidF32)
  BWS_CASE(kFmtNVFP4, kEpiSwiGLU)
  BWS_CASE(kFmtNVFP4, kEpiStoreF32)
  BWS_CASE(kFmtMXFP4, kEpiStoreBF16)
  BWS_CASE(kFmtMXFP4, kEpiResidF32)
  BWS_CASE(kFmtMXFP4, kEpiSwiGLU)
  BWS_CASE(kFmtMXFP4, kEpiStoreF32)
  BWS_CASE(kFmtFP8, kEpiStoreF32)
  BWS_CASE(kFmtFP8, kEpiStoreBF16)
#undef BWS_CASE
  return cudaErrorInvalidValue;
}

}  // namespace bws
