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
#include "moe_route.cuh"

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

// Where a tile's two sub-tiles live.
struct TileInfo {
  const uint8_t* codes[2];
  const uint8_t* scales[2];
  const float* scale32[2];
  int d_out[2];        // rows of the matrix (rows >= d_out are padding)
  int row0[2];         // first row of the sub-tile within its matrix
  int out_row_off[2];  // output row of the matrix's row 0
  int slot;
};

template <int FMT, int EPI>
BWS_DEV TileInfo tile_info(const GemvParams& p, int tile) {
  TileInfo ti;
  if (p.slots.n_slots != nullptr) {
    const SlotMode& S = p.slots;
    const int slot = tile / S.tiles_per_slot;
    const int rt = tile - slot * S.tiles_per_slot;
    const int e = __ldg(S.slot_expert + slot);
    const uint8_t* c = e < 0 ? S.shared_codes : S.codes + (size_t)e * S.codes_stride;
    const uint8_t* sc = e < 0 ? S.shared_scales : S.scales + (size_t)e * S.scales_stride;
    const size_t row_bytes = FMT == kFmtFP8 ? (size_t)p.d_in : (size_t)(p.d_in >> 1);
    const size_t srow_bytes = FMT == kFmtNVFP4 ? (size_t)(p.d_in >> 4) : (size_t)(p.d_in >> 5);
    ti.slot = slot;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int half = (EPI == kEpiSwiGLU && s == 1) ? S.up_row_off : 0;
      ti.codes[s] = c + (size_t)half * row_bytes;
      ti.scales[s] = sc + (size_t)half * srow_bytes;
      ti.scale32[s] = nullptr;
      ti.d_out[s] = S.rows;
      ti.row0[s] = EPI == kEpiSwiGLU ? rt * 16 : rt * 32 + 16 * s;
      ti.out_row_off[s] = 0;
    }
    return ti;
  }
  ti.slot = 0;
  if (EPI == kEpiSwiGLU) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      ti.codes[s] = p.mats[s].codes;
      ti.scales[s] = p.mats[s].scales;
      ti.scale32[s] = p.mats[s].scale32;
      ti.d_out[s] = p.mats[s].d_out;
      ti.row0[s] = tile * 16;
      ti.out_row_off[s] = 0;
    }
    return ti;
  }
  int m = 0;
#pragma unroll
  for (int i = 1; i < kMaxMats; ++i)
    if (i < p.n_mats && tile >= p.mats[i].tile_begin) m = i;
  const GemvMat& M = p.mats[m];
  const int local = tile - M.tile_begin;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    ti.codes[s] = M.codes;
    ti.scales[s] = M.scales;
    ti.scale32[s] = M.scale32;
    ti.d_out[s] = M.d_out;
    ti.row0[s] = local * 32 + 16 * s;
    ti.out_row_off[s] = M.out_row_off;
  }
  return ti;
}

BWS_DEV int x_block(const GemvParams& p, int slot) { return p.x.shared ? 0 : slot; }

// Per-piece lane pointers.
template <int FMT>
struct LanePtrs {
  const uint8_t* c[2][2];
  const uint8_t* sc[2][2];
  const uint16_t* xh;
  const uint16_t* xl;
};

template <int FMT>
BWS_DEV LanePtrs<FMT> lane_ptrs(const GemvParams& p, const TileInfo& ti, int g, int t) {
  LanePtrs<FMT> L;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = ti.row0[s] + g + 8 * h;
      const int rr = row < ti.d_out[s] ? row : 0;   // padding rows read row 0
      if (FMT == kFmtFP8) {
        L.c[s][h] = ti.codes[s] + (size_t)rr * p.d_in + 32 * t;
        L.sc[s][h] = nullptr;
      } else {
        L.c[s][h] = ti.codes[s] + (size_t)rr * (p.d_in >> 1) + 16 * t;
        L.sc[s][h] = FMT == kFmtNVFP4 ? ti.scales[s] + (size_t)rr * (p.d_in >> 4) + 2 * t
                                      : ti.scales[s] + (size_t)rr * (p.d_in >> 5) + t;
      }
    }
  }
  // token rows g >= N read the all-zero row after the N real rows
  const size_t xo = ((size_t)x_block(p, ti.slot) * (p.N + 1) + (g < p.N ? g : p.N)) * p.d_in_pad + 32 * t;
  L.xh = p.x.hi + xo;
  L.xl = p.x.lo + xo;
  return L;
}

// Loads are unpredicated: rows past d_out read row 0 (their outputs are never
// stored) and lanes past d_in read the row's last 32 weights, which meet the
// zero padding of the activations, so they add nothing.
template <int FMT, bool LO>
BWS_DEV void load_unit(const GemvParams& p, const LanePtrs<FMT>& L, int seg, int t, Frag<FMT, LO>& f) {
  const int k0 = min(seg * kSegK + 32 * t, p.d_in - 32) - 32 * t;   // lane offset is in L
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

typedef float Acc[2][4];   // [sub][4 accumulator registers]

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
        mma_f16_16816(acc[s], a0, a1, a2, a3, b0, b1);
        if (LO) {
          const uint32_t c0 = word_of(f.xl[j >> 1], 2 * (j & 1));
          const uint32_t c1 = word_of(f.xl[j >> 1], 2 * (j & 1) + 1);
          mma_f16_16816(accl[s], a0, a1, a2, a3, c0, c1);
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
      float dm[4] = {0.f, 0.f, 0.f, 0.f};
      float dml[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
        e2m1x8_to_f16x2x4(word_of(f.c[s][0][0], w), p0, p1, p2, p3);
        e2m1x8_to_f16x2x4(word_of(f.c[s][1][0], w), q0, q1, q2, q3);
        const uint32_t sa = mg[w >> 1], sb = m8[w >> 1];
        p0 = hmul2_u32(p0, sa); p1 = hmul2_u32(p1, sa); p2 = hmul2_u32(p2, sa); p3 = hmul2_u32(p3, sa);
        q0 = hmul2_u32(q0, sb); q1 = hmul2_u32(q1, sb); q2 = hmul2_u32(q2, sb); q3 = hmul2_u32(q3, sb);
        float(&D)[4] = FMT == kFmtMXFP4 ? dm : acc[s];
        mma_f16_16816(D, p0, q0, p1, q1, f.xh[w].x, f.xh[w].y);
        mma_f16_16816(D, p2, q2, p3, q3, f.xh[w].z, f.xh[w].w);
        if (LO) {
          float(&DL)[4] = FMT == kFmtMXFP4 ? dml : accl[s];
          mma_f16_16816(DL, p0, q0, p1, q1, f.xl[w].x, f.xl[w].y);
          mma_f16_16816(DL, p2, q2, p3, q3, f.xl[w].z, f.xl[w].w);
        }
      }
      if constexpr (FMT == kFmtMXFP4) {
        acc[s][0] = __fmaf_rn(dm[0], sref_g, acc[s][0]);
        acc[s][1] = __fmaf_rn(dm[1], sref_g, acc[s][1]);
        acc[s][2] = __fmaf_rn(dm[2], sref_8, acc[s][2]);
        acc[s][3] = __fmaf_rn(dm[3], sref_8, acc[s][3]);
        if (LO) {
          accl[s][0] = __fmaf_rn(dml[0], sref_g, accl[s][0]);
          accl[s][1] = __fmaf_rn(dml[1], sref_g, accl[s][1]);
          accl[s][2] = __fmaf_rn(dml[2], sref_8, accl[s][2]);
          accl[s][3] = __fmaf_rn(dml[3], sref_8, accl[s][3]);
        }
      }
    }
  }
}

BWS_DEV float silu_mul(float g, float u) {
  const float sg = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  return __fmul_rn(sg, u);
}

// Scale raw sums v[sub][4] to outputs and store them. Register i of a lane
// holds (row g + 8*(i>>1), token 2t + (i&1)).
template <int FMT, int EPI>
BWS_DEV void finish_tile(const GemvParams& p, const TileInfo& ti, int g, int t, const float (&v)[2][4]) {
  const int xb = x_block(p, ti.slot);
  int xexp[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int tok = 2 * t + i;
    xexp[i] = tok < p.N ? __ldg(p.x.exp + xb * p.N + tok) : 0;
  }
  float val[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = ti.row0[s] + g + 8 * (i >> 1);
      float sc = 1.0f;
      if (FMT == kFmtNVFP4 && ti.scale32[s] != nullptr) sc = __ldg(ti.scale32[s]);
      if (FMT == kFmtFP8) sc = row < ti.d_out[s] ? __ldg(ti.scale32[s] + row) : 0.0f;
      val[s][i] = ldexp_exact(__fmul_rn(v[s][i], sc), xexp[i & 1] - 14);
    }
  }
  char* out = reinterpret_cast<char*>(p.out);
  if constexpr (EPI == kEpiSwiGLU) {
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(out) + (size_t)ti.slot * p.out_slot_stride;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = ti.row0[0] + g + 8 * (i >> 1);
      const int tok = 2 * t + (i & 1);
      if (row < ti.d_out[0] && tok < p.N)
        h[(size_t)tok * p.out_ld + row] = __float2bfloat16_rn(silu_mul(val[0][i], val[1][i]));
    }
  } else {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = ti.row0[s] + g + 8 * (i >> 1);
        const int tok = 2 * t + (i & 1);
        if (row < ti.d_out[s] && tok < p.N) {
          const size_t o = (size_t)ti.slot * p.out_slot_stride + (size_t)tok * p.out_ld + ti.out_row_off[s] + row;
          if (EPI == kEpiStoreBF16)
            reinterpret_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(val[s][i]);
          else if (EPI == kEpiStoreF32)
            reinterpret_cast<float*>(out)[o] = val[s][i];
          else
            reinterpret_cast<float*>(out)[o] = __fadd_rn(reinterpret_cast<float*>(out)[o], val[s][i]);
        }
      }
    }
  }
}

BWS_DEV long long owner_warp(long long u, long long U, long long W) { return ((u + 1) * W - 1) / U; }
BWS_DEV long long range_begin(long long w, long long U, long long W) { return w * U / W; }

// End of a warp's piece of a tile: finish directly, or deposit the partial
// sums and let the last contributor finish the tile.
template <int FMT, int EPI>
BWS_DEV void end_piece(const GemvParams& p, const TileInfo& ti, int tile, long long warp_id, bool whole,
                       const float (&v)[2][4], long long U, long long W, int lane) {
  const int g = lane >> 2, t = lane & 3;
  if (whole) {
    finish_tile<FMT, EPI>(p, ti, g, t, v);
    return;
  }
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
    float4 a, b;
    if (w == warp_id) {
      a = make_float4(v[0][0], v[0][1], v[0][2], v[0][3]);
      b = make_float4(v[1][0], v[1][1], v[1][2], v[1][3]);
    } else {
      const float4* o = reinterpret_cast<const float4*>(p.partials) + (size_t)(tile + w) * (kSlotFloats / 4);
      a = ld_cg_f4(o + lane);
      b = ld_cg_f4(o + 32 + lane);
    }
    s[0][0] += a.x; s[0][1] += a.y; s[0][2] += a.z; s[0][3] += a.w;
    s[1][0] += b.x; s[1][1] += b.y; s[1][2] += b.z; s[1][3] += b.w;
  }
  finish_tile<FMT, EPI>(p, ti, g, t, s);
  if (lane == 0) p.counters[tile] = 0u;
}

// One piece: units [seg0, seg1] of one tile, software-pipelined two deep
// (one unit at a time on the rare two-band path).
template <int FMT, int EPI, bool LO>
BWS_DEV void run_piece(const GemvParams& p, int tile, int seg0, int seg1, long long warp_id, long long U,
                       long long W, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const TileInfo ti = tile_info<FMT, EPI>(p, tile);
  const LanePtrs<FMT> L = lane_ptrs<FMT>(p, ti, g, t);
  Acc acc = {}, accl = {};
  if (LO) {
    for (int seg = seg0; seg <= seg1; ++seg) {
      Frag<FMT, true> f;
      load_unit<FMT, true>(p, L, seg, t, f);
      compute_unit<FMT, true>(f, acc, accl);
    }
  } else {
    Frag<FMT, false> fa, fb;
    load_unit<FMT, false>(p, L, seg0, t, fa);
    for (int seg = seg0; seg <= seg1; seg += 2) {
      if (seg + 1 <= seg1) load_unit<FMT, false>(p, L, seg + 1, t, fb);
      compute_unit<FMT, false>(fa, acc, accl);
      if (seg + 1 > seg1) break;
      if (seg + 2 <= seg1) load_unit<FMT, false>(p, L, seg + 2, t, fa);
      compute_unit<FMT, false>(fb, acc, accl);
    }
  }
  float v[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int i = 0; i < 4; ++i) v[s][i] = LO ? __fmaf_rn(accl[s][i], 0x1p-29f, acc[s][i]) : acc[s][i];
  const bool whole = seg0 == 0 && seg1 == p.nseg - 1;
  end_piece<FMT, EPI>(p, ti, tile, warp_id, whole, v, U, W, lane);
}

// The two-band path is rare; keep it out of line so that its register needs
// do not constrain the common path.
template <int FMT, int EPI>
__device__ __noinline__ void run_piece_lo(const GemvParams& p, int tile, int seg0, int seg1, long long warp_id,
                                          long long U, long long W, int lane) {
  run_piece<FMT, EPI, true>(p, tile, seg0, seg1, warp_id, U, W, lane);
}

template <int FMT, int EPI>
BWS_DEV bool piece_needs_lo(const GemvParams& p, int tile) {
  const int slot = p.slots.n_slots != nullptr ? tile / p.slots.tiles_per_slot : 0;
  const int xb = x_block(p, slot);
  uint32_t f = 0u;
  for (int tok = 0; tok < p.N; ++tok) f |= __ldg(p.x.flags + xb * p.N + tok);
  return (f & 1u) != 0u;
}

#ifndef BWS_GEMV_MIN_BLOCKS
#define BWS_GEMV_MIN_BLOCKS 2
#endif

template <int FMT, int EPI>
__global__ void __launch_bounds__(kWarpsPerCta * 32, BWS_GEMV_MIN_BLOCKS) gemv_kernel(const __grid_constant__ GemvParams p) {
  const int lane = threadIdx.x & 31;
  const long long warp_id = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  pdl_launch_dependents();
  long long U, W;
  if (p.slots.n_slots == nullptr) {
    U = p.n_units;
    W = p.n_warps;
    if (warp_id >= W) {
      pdl_wait();
      return;
    }
    // Weights do not depend on earlier kernels: start pulling the first units
    // of this warp's range into L2 before waiting for the activations (one
    // bulk prefetch per lane, lane l covering row l of the first piece).
    const long long u0 = range_begin(warp_id, U, W), u1 = range_begin(warp_id + 1, U, W);
    if (p.prefetch_units > 0) {
      const int tile = (int)(u0 / p.nseg);
      const int seg = (int)(u0 % p.nseg);
      long long nu = p.nseg - seg;
      if (nu > p.prefetch_units) nu = p.prefetch_units;
      if (nu > u1 - u0) nu = u1 - u0;
      const TileInfo ti = tile_info<FMT, EPI>(p, tile);
      const int sub = lane >> 4;
      const int row = ti.row0[sub] + (lane & 15);
      if (row < ti.d_out[sub] && nu > 0) {
        const int per = FMT == kFmtFP8 ? kSegK : kSegK / 2;
        const size_t row_bytes = FMT == kFmtFP8 ? (size_t)p.d_in : (size_t)(p.d_in >> 1);
        const size_t kb0 = (size_t)seg * per;
        size_t nb = (size_t)nu * per;
        if (kb0 + nb > row_bytes) nb = row_bytes - kb0;
        if (nb >= 16) prefetch_l2_bulk(ti.codes[sub] + (size_t)row * row_bytes + kb0, (uint32_t)(nb & ~(size_t)15));
      }
    }
    pdl_wait();
  } else {
    pdl_wait();
    const long long n_slots = __ldg(p.slots.n_slots);
    U = n_slots * p.slots.tiles_per_slot * p.nseg;
    // A short k range (at most 8 units, like an expert's down projection):
    // each warp takes whole tiles rather than slicing every tile between
    // warps, whose partial sums would then all go through the fix-up.
    const long long per = p.nseg <= 8 ? p.nseg : 1;
    const long long want = (U + per - 1) / per;
    W = p.n_warps < want ? p.n_warps : want;
    if (warp_id >= W) return;
  }
  long long u = range_begin(warp_id, U, W);
  const long long u_end = range_begin(warp_id + 1, U, W);
  while (u < u_end) {
    const int tile = (int)(u / p.nseg);
    const int seg0 = (int)(u % p.nseg);
    const long long left = u_end - u;
    const int seg1 = (long long)(p.nseg - 1 - seg0) < left ? p.nseg - 1 : seg0 + (int)left - 1;
    if (piece_needs_lo<FMT, EPI>(p, tile))
      run_piece_lo<FMT, EPI>(p, tile, seg0, seg1, warp_id, U, W, lane);
    else
      run_piece<FMT, EPI, false>(p, tile, seg0, seg1, warp_id, U, W, lane);
    u += seg1 - seg0 + 1;
  }
}

// ---- launches ------------------------------------------------------------------

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                            cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

template <int FMT, int EPI>
cudaError_t launch_one(const GemvParams& p, cudaStream_t st, bool pdl) {
  const long long ctas = (p.n_warps + kWarpsPerCta - 1) / kWarpsPerCta;
  if (ctas <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((unsigned)ctas), dim3(kWarpsPerCta * 32), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, gemv_kernel<FMT, EPI>, p);
}

// ---- MoE routing and combine -------------------------------------------------

// One CTA of 128 threads (N * topk <= 64 routed entries): the shared expert in
// slot 0, then the distinct routed experts in ascending id order, and the
// combine weight of every (slot, token) pair.
__global__ void __launch_bounds__(128) moe_route_kernel(const MoeRoute m) {
  pdl_launch_dependents();
  pdl_wait();
  moe_route_body(m);
}

__global__ void __launch_bounds__(256) moe_combine_kernel(const float* __restrict__ ys, const float* __restrict__ cw,
                                                          const int* __restrict__ n_slots_p, int N, int d,
                                                          void* __restrict__ out, int out_mode) {
  pdl_launch_dependents();
  pdl_wait();
  const int tok = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  const int ns = __ldg(n_slots_p);
  float acc = 0.0f;
  for (int s = 0; s < ns; ++s) {
    const float w = __ldg(cw + s * N + tok);
    if (w != 0.0f) acc = __fmaf_rn(w, __ldg(ys + ((size_t)s * N + tok) * d + i), acc);
  }
  if (out_mode == kEpiStoreBF16)
    reinterpret_cast<__nv_bfloat16*>(out)[(size_t)tok * d + i] = __float2bfloat16_rn(acc);
  else
    reinterpret_cast<float*>(out)[(size_t)tok * d + i] =
        __fadd_rn(reinterpret_cast<float*>(out)[(size_t)tok * d + i], acc);
}

}  // namespace

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

int num_sms() {
  // per device: a process may drive GPUs of different SM counts
  static std::atomic<int> n[kMaxDevices];
  const int dev = current_device();
  int v = n[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      v = 152;
    }
    n[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

long long gemv_max_warps() { return (long long)num_sms() * BWS_GEMV_MIN_BLOCKS * kWarpsPerCta; }

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

GemvWorkspace gemv_workspace_layout(int N, int d_in, int n_tiles, long long max_warps, int slots) {
  GemvWorkspace w;
  const size_t d_pad = (size_t)((d_in + kSegK - 1) / kSegK) * kSegK;
  size_t o = 0;
  w.off_hdr = o; o += 256;
  w.off_exp = o; o += align256(sizeof(int) * (size_t)kMaxTokens * slots);
  w.off_flags = o; o += align256(sizeof(uint32_t) * (size_t)kMaxTokens * slots);
  w.off_hi = o; o += align256(2 * d_pad * (size_t)(N + 1) * slots);
  w.off_lo = o; o += align256(2 * d_pad * (size_t)(N + 1) * slots);
  w.off_counters = o;   // tile counters, then (8-byte aligned) the argmax keys of the output layer
  o += align256(sizeof(uint32_t) * (size_t)argmax_key_word(n_tiles) + sizeof(unsigned long long) * kMaxTokens);
  w.off_partials = o; o += align256(sizeof(float) * kSlotFloats * ((size_t)n_tiles + max_warps));
  w.total = o;
  return w;
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
  BWS_CASE(kFmtFP8, kEpiResidF32)
  BWS_CASE(kFmtFP8, kEpiSwiGLU)
#undef BWS_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_moe_route(const MoeRoute& m, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(1), dim3(128), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, moe_route_kernel, m);
}

cudaError_t launch_moe_combine(const float* ys, const float* cw, const int* n_slots, int N, int d, void* out,
                               int out_mode, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((unsigned)((d + 255) / 256), (unsigned)N), dim3(256), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, moe_combine_kernel, ys, cw, n_slots, N, d, out, out_mode);
}

}  // namespace bws
