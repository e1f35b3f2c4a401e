// Weight-stream products fed by TMA: one producer warp per CTA streams weight
// tiles into a ring of shared-memory stages with cp.async.bulk.tensor; eight
// consumer warps decode them and run the MMAs. The producer gives the first
// stages their weights before the kernel waits on its inputs (weights never
// depend on earlier kernels); the weight copies carry an L2 evict-first
// policy (read once per step, they should not push out what later kernels
// read back).
//
// Tiles and units. A tile is 128 output rows (8 MMA sub-tiles of 16): rows
// [128i, 128i+128) of one matrix, or, for the fused SwiGLU, 64 gate rows and
// the same 64 up rows. A unit is a tile x 128 bytes of each row (256 NVFP4
// weights, 128 FP8 weights) and arrives as four 32-row TMA boxes with 128-byte
// swizzle (plus four 32 x 16-byte boxes of E4M3 block scales for NVFP4) and,
// through 1D bulk copies, the unit's activations of every token. Units are
// dealt to CTAs in contiguous ranges (stream-K, SplitK); a tile cut between
// CTAs is finished by the last CTA to arrive, adding partial sums in CTA
// order. In deposit mode (the layer stack) every tile piece only writes its
// raw sums to the slot of its (tile, CTA) pair, and the prep that reads the
// rows next finishes them the same way.
//
// Consumer warp w takes box b = w%4 (two sub-tiles) and half h = w/4 of every
// unit's 128 bytes: lane (g, t) reads the 16-byte chunk c = 2t + h of rows g,
// g+8, g+16, g+24 of the box, which puts the 8 lanes of each shared-memory
// access phase on 8 distinct swizzled chunks (no bank conflicts). A chunk is
// 32 NVFP4 weights (two 16-weight blocks) or 16 FP8 weights; MMA j takes its
// 4 consecutive weights 4j..4j+3 as logical k {2t, 2t+1, 2t+8, 2t+9}, and the
// activations, laid out by the prep kernel so that chunk c's pieces sit at
// c * 16 + q * 128, are read with the same mapping. The two halves of a
// sub-tile are added through shared memory at the end of each tile piece.
#include <cuda.h>

#include <cstddef>
#include <cstring>

#include "bws_common.cuh"
#include "bws_internal.h"
#include "stream_tile.cuh"
#include "trace.cuh"

namespace bws {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreadsTma = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 16;
constexpr int kSmemBudget = 100 * 1024;            // stages per CTA: two CTAs share an SM
constexpr uint32_t kMaxPolls = 1u << 24;           // bounded waits (seconds)
constexpr uint32_t kStatusTimeout = 0x100u;
constexpr int kPartialBytes = kBoxes * 2 * 32 * 16;   // one (tile, CTA) slot of partial sums

struct TmaMat {
  CUtensorMap codes;    // u8 [d_out][row_bytes], box {128, 32}, 128B swizzle
  CUtensorMap scales;   // u8 [d_out][d_in/16], box {16, 32} (NVFP4)
  const float* scale32;
  int d_out;
  int out_row_off;
  int tile_begin;
};

struct TmaParams {
  TmaMat mats[kMaxMats];
  int n_mats;
  int N, d_in, d_in_pad, nks;   // nks: units per tile (128-byte steps of a row)
  int n_tiles;
  long long n_units;
  int n_ctas;
  int lf, num, den;   // the split's lighter CTAs (SplitK)
  XPrep x;
  void* out;
  int out_ld;
  float* partials;
  uint32_t* counters;
  uint32_t* status;
  // shared-memory stage layout: code boxes at 0, scale boxes at kCodeBytes
  // (NVFP4), one activation block per token at x_off + tok * x_blk
  int n_stages, stage_bytes, x_off, x_blk, x_bytes;
  int n_prime;   // stages given their weights before the inputs are ready
  int deposit;   // 1: each tile piece writes its raw sums to its partial slot, nothing else
  unsigned long long* amax_key;   // StoreF32, optional: greedy argmax keys [N] (GemvParams)
  int no_store;
};

// Shared memory after the stages (which end on a 1024-byte boundary).
struct Tail {
  float4 red[kBoxes][2][32];   // half-pair reduction (box, sub-tile, lane)
  float4 swi[2][2][32];        // SwiGLU: up sums handed to the gate warps
  uint4 zero_x[33];             // zero activation pieces (one-token block-diagonal operand),
                                // used from element 1 on (see consume)
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  unsigned long long akey[kMaxTokens];   // the CTA's best argmax keys
  uint32_t flag;
#ifdef BWS_TRACE
  unsigned long long tr[4];   // producer's wait returned, consumers' wait returned, first stage, loop done
#endif
};
static_assert(offsetof(Tail, zero_x) % 128 == 0, "zero pieces must start on a 128-byte boundary");

// Matrix and first row of box b of a tile.
template <int EPI>
BWS_DEV void box_of(const TmaParams& p, int tile, int b, int& m, int& row) {
  if (EPI == kEpiSwiGLU) {
    m = b >> 1;
    row = tile * 64 + 32 * (b & 1);
    return;
  }
  m = 0;
#pragma unroll
  for (int i = 1; i < kMaxMats; ++i)
    if (i < p.n_mats && tile >= p.mats[i].tile_begin) m = i;
  row = (tile - p.mats[m].tile_begin) * 128 + 32 * b;
}

BWS_DEV SplitK split_of(const TmaParams& p) {
  SplitK s;
  s.n_units = p.n_units;
  s.n_ctas = p.n_ctas;
  s.lf = p.lf;
  s.num = p.num;
  s.den = p.den;
  return s;
}

// Inputs of a tile's stores that live in global memory, read when the tile
// piece ends, before its reductions and the fix-up handshake, so that they
// arrive meanwhile: per sub-tile s and register i (row g + 8*(i>>1), token
// 2t + (i&1)) the residual a ResidF32 store adds to and, for FP8, the row's
// scale; the tensor scales of the matrices (loaded once per CTA).
struct EpiIn {
  float r[2][4];
  float rs[2][2];    // FP8: row scales of the stored rows (SwiGLU: the gate rows)
  float rsu[2][2];   // FP8 SwiGLU: row scales of the matching up rows
  float ts[kMaxMats];
};

template <int FMT, int EPI>
BWS_DEV void epi_read(const TmaParams& p, int tile, int b, int g, int t, EpiIn& in) {
  int mi, row_b;
  box_of<EPI>(p, tile, b, mi, row_b);
  const TmaMat& M = p.mats[mi];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = row_b + 16 * s + g + 8 * (i >> 1);
      const int tok = 2 * t + (i & 1);
      const bool ok = row < M.d_out && tok < p.N;
      if (EPI == kEpiResidF32)
        in.r[s][i] = ok ? reinterpret_cast<const float*>(p.out)[(size_t)tok * p.out_ld + M.out_row_off + row] : 0.0f;
      if (FMT == kFmtFP8 && (i & 1) == 0) {
        in.rs[s][i >> 1] = row < M.d_out ? __ldg(M.scale32 + row) : 0.0f;
        if (EPI == kEpiSwiGLU) in.rsu[s][i >> 1] = row < p.mats[1].d_out ? __ldg(p.mats[1].scale32 + row) : 0.0f;
      }
    }
  }
}

// Store v (raw sums of sub-tile s of box b; register i = row g + 8*(i>>1),
// token 2t + (i&1)). SwiGLU: b is a gate box and vu the matching up sums.
template <int FMT, int EPI>
BWS_DEV void store_sub(const TmaParams& p, int tile, int b, int s, int g, int t, const float (&v)[4],
                       const float (&vu)[4], const int (&xexp)[2], const EpiIn& in, unsigned long long (&ak)[2]) {
  int mi, row_b;
  box_of<EPI>(p, tile, b, mi, row_b);
  const TmaMat& M = p.mats[mi];
  const int row0 = row_b + 16 * s;
  const float tsm = mi == 0 ? in.ts[0] : mi == 1 ? in.ts[1] : mi == 2 ? in.ts[2] : in.ts[kMaxMats - 1];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = row0 + g + 8 * (i >> 1);
    const int tok = 2 * t + (i & 1);
    if (row >= M.d_out || tok >= p.N) continue;
    float sc = 1.0f;
    if (FMT == kFmtNVFP4) sc = tsm;
    if (FMT == kFmtFP8) sc = in.rs[s][i >> 1];
    const float val = ldexp_exact(__fmul_rn(v[i], sc), xexp[i & 1] - 14);
    if (EPI == kEpiSwiGLU) {
      const float su = FMT == kFmtFP8 ? in.rsu[s][i >> 1] : in.ts[1];
      const float up = ldexp_exact(__fmul_rn(vu[i], su), xexp[i & 1] - 14);
      reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t)tok * p.out_ld + row] =
          __float2bfloat16_rn(silu_mul_t(val, up));
    } else {
      const size_t o = (size_t)tok * p.out_ld + M.out_row_off + row;
      if (EPI == kEpiStoreBF16) {
        reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(val);
      } else if (EPI == kEpiStoreF32) {
        if (!p.no_store) reinterpret_cast<float*>(p.out)[o] = val;
        if (p.amax_key != nullptr) {
          const unsigned long long k = argmax_key(val, M.out_row_off + row);
          ak[i & 1] = k > ak[i & 1] ? k : ak[i & 1];
        }
      } else
        reinterpret_cast<float*>(p.out)[o] = __fadd_rn(in.r[s][i], val);
    }
  }
}

// The consumer warps' loop over units u0..u1 (LO: the two-band activation
// path, taken when some token has elements below the hi band's range).
template <int FMT, int EPI, bool LO, bool N1>
BWS_DEV void consume(const TmaParams& p, Tail& T, uint32_t stage0, long long u0, long long u1, int warp, int lane,
                     const uint16_t* xrow_l) {
  const int NS = p.n_stages;
  constexpr int kUnitK = FMT == kFmtFP8 ? 128 : 256;
  constexpr int kXv = FMT == kFmtFP8 ? 2 : 4;     // 16-byte activation pieces per unit
  const int b = warp & 3, half = warp >> 2;
  const int g = lane >> 2, t = lane & 3;
  const int c = 2 * t + half;                     // this lane's 16-byte chunk
  // exponents of this lane's two output tokens (inputs are ready: loaded once)
  int xexp[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) xexp[i] = 2 * t + i < p.N ? __ldg(p.x.exp + 2 * t + i) : 0;
  EpiIn ein;
#pragma unroll
  for (int i = 0; i < kMaxMats; ++i) ein.ts[i] = (FMT != kFmtFP8 && i < p.n_mats) ? __ldg(p.mats[i].scale32) : 1.0f;
  // rows g + 8j of box b (j = 0..3) share the swizzle phase g
  const uint32_t coff = b * kBoxBytes + g * 128 + ((c ^ g) << 4);
  const uint32_t soff = kCodeBytes + b * kScaleBoxBytes + g * 16 + 2 * c;
  // activations of token g (absent tokens read token 0's: their MMA columns
  // are never stored), pieces at q * 128
  const int xg = g < p.N ? g : 0;
  const uint32_t xoff = (uint32_t)(p.x_off + xg * p.x_blk + c * 16);
  xrow_l += (size_t)xg * p.d_in_pad;
  // one token: lanes g == 2t feed their chunk's first block, g == 2t + 1 its
  // second, the rest read zeros (see sub_mma_n1)
  const bool m01 = g == 2 * t, m23 = g == 2 * t + 1;
  // the zero pieces sit 16 bytes past a 128-byte boundary while the stages'
  // activation blocks sit on one, so a phase's zero reads and real reads fall
  // in different banks
  const uint32_t zaddr = smem_u32(&T.zero_x[1]) + c * 16;
  float acc[2][2][4] = {}, accl[2][4] = {};   // N1: acc[st][0] holds y, accl[st] the lo band's
  unsigned long long ak[2] = {0ull, 0ull};     // StoreF32 with argmax: best keys of tokens 2t, 2t+1
  uint4 xh[kXv], xl[kXv];
  bool dead = false;   // a wait ran out: keep the control flow (barriers), skip the work
  int tile = (int)(u0 / p.nks), ks = (int)(u0 % p.nks);
  int s = 0;
  uint32_t ph = 0u;
  bool piece_whole = ks == 0;   // the piece starts at the tile's first unit
  for (long long u = u0; u < u1; ++u) {
    if (LO) {   // two-band path: the lo band comes from global memory
#pragma unroll
      for (int q = 0; q < kXv; ++q) {
        xl[q] = ld_act_v4(xrow_l + (size_t)ks * kUnitK + q * 64 + c * 8);
        if (N1 && !(q < 2 ? m01 : m23)) xl[q] = make_uint4(0, 0, 0, 0);
      }
    }
    if (!dead && !mbar_wait_bounded(smem_u32(&T.full[s]), ph, kMaxPolls)) {
      if (lane == 0) atomicOr(p.status, kStatusTimeout);
      dead = true;
    }
#ifdef BWS_TRACE
    if (u == u0 && threadIdx.x == 0) T.tr[2] = trace_now();
#endif
    const uint32_t base = stage0 + (uint32_t)s * p.stage_bytes;
    uint4 cw[4];
    uint32_t sc[4];
    if (!dead) {
#pragma unroll
      for (int j = 0; j < 4; ++j) cw[j] = lds_v4(base + coff + j * 1024);
      if (FMT == kFmtNVFP4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[j] = lds_u16(base + soff + j * 128);
      }
      if constexpr (N1) {
        const uint32_t xb = base + xoff;
        const uint32_t a01 = m01 ? xb : zaddr, a23 = m23 ? xb : zaddr;
        xh[0] = lds_v4(a01);
        xh[1] = lds_v4(a01 + 128);
        xh[2] = lds_v4(a23 + 256);
        xh[3] = lds_v4(a23 + 384);
      } else {
#pragma unroll
        for (int q = 0; q < kXv; ++q) xh[q] = lds_v4(base + xoff + q * 128);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) { cw[j] = make_uint4(0, 0, 0, 0); sc[j] = 0u; }
#pragma unroll
      for (int q = 0; q < kXv; ++q) xh[q] = make_uint4(0, 0, 0, 0);
    }
    // the stage's shared memory has been read: hand it back to the producer
    __syncwarp();
    if (lane == 0 && !dead) mbar_arrive(smem_u32(&T.empty[s]));
    if (++s == NS) { s = 0; ph ^= 1u; }
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const uint32_t w0[4] = {cw[2 * st].x, cw[2 * st].y, cw[2 * st].z, cw[2 * st].w};
      const uint32_t w1[4] = {cw[2 * st + 1].x, cw[2 * st + 1].y, cw[2 * st + 1].z, cw[2 * st + 1].w};
      if constexpr (N1)
        sub_mma_n1<LO>(acc[st][0], accl[st], w0, w1, sc[2 * st], sc[2 * st + 1], xh, xl);
      else
        sub_mma<FMT, LO>(acc[st], accl[st], w0, w1, sc[2 * st], sc[2 * st + 1], xh, xl);
    }
    // ---- end of a tile piece ----
    const bool last_of_tile = ks == p.nks - 1;
    const int cur_tile = tile;
    if (++ks == p.nks) { ks = 0; ++tile; }
    if (!last_of_tile && u + 1 < u1) continue;
    float v[2][4];
    if constexpr (N1) {
      // rows g and g + 8: this lane's two blocks, then the four chunks of the half
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        float yg = __fadd_rn(acc[st][0][0], acc[st][0][1]), y8 = __fadd_rn(acc[st][0][2], acc[st][0][3]);
        if (LO) {
          yg = __fmaf_rn(__fadd_rn(accl[st][0], accl[st][1]), 0x1p-29f, yg);
          y8 = __fmaf_rn(__fadd_rn(accl[st][2], accl[st][3]), 0x1p-29f, y8);
        }
        yg += __shfl_xor_sync(0xffffffffu, yg, 1);
        y8 += __shfl_xor_sync(0xffffffffu, y8, 1);
        yg += __shfl_xor_sync(0xffffffffu, yg, 2);
        y8 += __shfl_xor_sync(0xffffffffu, y8, 2);
        v[st][0] = yg; v[st][1] = 0.f; v[st][2] = y8; v[st][3] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[st][0][r] = accl[st][r] = 0.f;
      }
    } else {
#pragma unroll
      for (int st = 0; st < 2; ++st) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float a = __fadd_rn(acc[st][0][r], acc[st][1][r]);
          v[st][r] = LO ? __fmaf_rn(accl[st][r], 0x1p-29f, a) : a;
          acc[st][0][r] = acc[st][1][r] = accl[st][r] = 0.f;
        }
      }
    }
    // the stores' global inputs of the storing warps, in flight during the reductions
    if (half == 0 && (EPI == kEpiResidF32 || FMT == kFmtFP8) && !p.deposit)
      epi_read<FMT, EPI>(p, cur_tile, b, g, t, ein);
    // add the two halves: warps 4..7 hand their sums to warps 0..3
    if (half == 1) {
#pragma unroll
      for (int st = 0; st < 2; ++st) T.red[b][st][lane] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
    }
    named_bar_sync(1, kConsumerWarps * 32);
    if (half == 0) {
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        const float4 o = T.red[b][st][lane];
        v[st][0] += o.x; v[st][1] += o.y; v[st][2] += o.z; v[st][3] += o.w;
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);
    const bool whole = piece_whole && last_of_tile;
    piece_whole = true;   // later pieces start at a tile's first unit
    if (half == 1) continue;
    if (p.deposit) {
      // the piece's raw sums, row-major per token in the slot of (tile, CTA):
      // the next prep adds a tile's slots in CTA order and finishes the rows
      float* slot = p.partials + (size_t)(cur_tile + blockIdx.x) * p.N * 128;
#pragma unroll
      for (int st = 0; st < 2; ++st) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = 32 * b + 16 * st + g + 8 * (i >> 1);
          const int tok = N1 ? 0 : 2 * t + (i & 1);
          if (N1 ? (t == 0 && (i & 1) == 0) : tok < p.N) slot[tok * 128 + row] = v[st][i];
        }
      }
      continue;
    }
    // warps 0..3: finish or deposit
    if (!whole) {
      float4* slot = reinterpret_cast<float4*>(p.partials) + ((size_t)(cur_tile + blockIdx.x) * kBoxes + b) * 64;
#pragma unroll
      for (int st = 0; st < 2; ++st) slot[st * 32 + lane] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
      // the four warps' deposits, then one acquire-release count: it publishes
      // them (release, cumulative over the barrier) and, for the last arriver,
      // makes the other CTAs' deposits visible (acquire)
      named_bar_sync(2, 4 * 32);
      const long long c0 = splitk_owner(split_of(p), (long long)cur_tile * p.nks);
      const long long c1 = splitk_owner(split_of(p), (long long)(cur_tile + 1) * p.nks - 1);
      if (threadIdx.x == 0) T.flag = atom_add_acq_rel_gpu(p.counters + cur_tile, 1u);
      named_bar_sync(2, 4 * 32);
      const uint32_t prev = T.flag;
      named_bar_sync(2, 4 * 32);
      if (prev != (uint32_t)(c1 - c0)) continue;
      // the tile's pieces in CTA order; their loads are issued kFix pieces at a
      // time, so the tail of a product waits for a few L2 round trips, not one
      // per piece
      constexpr int kFix = 4;
      float a8[2][4] = {};
      const float4* slots = reinterpret_cast<const float4*>(p.partials) + (size_t)cur_tile * kBoxes * 64 + b * 64 + lane;
      for (long long cc0 = c0; cc0 <= c1; cc0 += kFix) {
        float4 o[kFix][2];
#pragma unroll
        for (int k = 0; k < kFix; ++k) {
          const long long cc = cc0 + k;
#pragma unroll
          for (int st = 0; st < 2; ++st) {
            if (cc > c1)
              o[k][st] = make_float4(0.f, 0.f, 0.f, 0.f);
            else if (cc == blockIdx.x)
              o[k][st] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
            else
              o[k][st] = ld_cg_f4(slots + (size_t)cc * kBoxes * 64 + st * 32);
          }
        }
#pragma unroll
        for (int k = 0; k < kFix; ++k) {
          if (cc0 + k > c1) break;
#pragma unroll
          for (int st = 0; st < 2; ++st) {
            a8[st][0] += o[k][st].x; a8[st][1] += o[k][st].y; a8[st][2] += o[k][st].z; a8[st][3] += o[k][st].w;
          }
        }
      }
#pragma unroll
      for (int st = 0; st < 2; ++st)
#pragma unroll
        for (int r = 0; r < 4; ++r) v[st][r] = a8[st][r];
      if (threadIdx.x == 0) p.counters[cur_tile] = 0u;
    }
    if (EPI == kEpiSwiGLU) {
      // boxes 2, 3 (up rows) meet boxes 0, 1 (gate rows) of the same rows
      if (b >= 2) {
#pragma unroll
        for (int st = 0; st < 2; ++st) T.swi[b - 2][st][lane] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
      }
      named_bar_sync(3, 4 * 32);
      if (b < 2) {
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          const float4 o = T.swi[b][st][lane];
          const float vu[4] = {o.x, o.y, o.z, o.w};
          store_sub<FMT, EPI>(p, cur_tile, b, st, g, t, v[st], vu, xexp, ein, ak);
        }
      }
      named_bar_sync(3, 4 * 32);
    } else {
      const float none[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int st = 0; st < 2; ++st) store_sub<FMT, EPI>(p, cur_tile, b, st, g, t, v[st], none, xexp, ein, ak);
    }
  }
#ifdef BWS_TRACE
  if (threadIdx.x == 0) T.tr[3] = trace_now();
#endif
  if (EPI == kEpiStoreF32 && p.amax_key != nullptr) {
    // the warp's best key per token (lanes of one t hold the same tokens), into the CTA's
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const unsigned long long q = __shfl_xor_sync(0xffffffffu, ak[k], o);
        ak[k] = q > ak[k] ? q : ak[k];
      }
      if (g == 0 && 2 * t + k < p.N) atomicMax(&T.akey[2 * t + k], ak[k]);
    }
  }
}

// The rare two-band loop, out of line so that its registers do not weigh on
// the main loop.
template <int FMT, int EPI, bool N1>
__device__ __noinline__ void consume_lo(const TmaParams& p, Tail& T, uint32_t stage0, long long u0, long long u1,
                                        int warp, int lane, const uint16_t* xrow_l) {
  consume<FMT, EPI, true, N1>(p, T, stage0, u0, u1, warp, lane, xrow_l);
}

template <int FMT, int EPI, bool N1>
__global__ void __launch_bounds__(kThreadsTma, 2) gemv_tma_kernel(const __grid_constant__ TmaParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
#ifdef BWS_TRACE
  const unsigned long long tr_start = trace_now();
#endif
  // 128-byte swizzled TMA boxes need 1024-byte aligned destinations
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* sbase = smem_raw + ((1024u - mis) & 1023u);
  Tail& T = *reinterpret_cast<Tail*>(sbase + (size_t)p.n_stages * p.stage_bytes);
  const uint32_t stage0 = smem_u32(sbase);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long u0 = splitk_begin(split_of(p), blockIdx.x), u1 = splitk_begin(split_of(p), blockIdx.x + 1);
  const int NS = p.n_stages;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&T.full[i]), 1);
      mbar_init(smem_u32(&T.empty[i]), kConsumerWarps);
    }
    T.flag = 0u;
    mbar_fence_init();
  }
  for (int i = threadIdx.x; i < 33; i += blockDim.x) T.zero_x[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x < kMaxTokens) T.akey[threadIdx.x] = 0ull;
  __syncthreads();
  constexpr int kUnitK = FMT == kFmtFP8 ? 128 : 256;

  if (warp == kConsumerWarps) {
    // ---- producer: weights before the inputs are ready, activations after ----
    if (lane == 0) {
      for (int i = 0; i < p.n_mats; ++i) {
        tma_prefetch_desc(&p.mats[i].codes);
        if (FMT == kFmtNVFP4) tma_prefetch_desc(&p.mats[i].scales);
      }
      const uint32_t w_tx = FMT == kFmtNVFP4 ? kCodeBytes + kBoxes * kScaleBoxBytes : kCodeBytes;
      const uint64_t pol = l2_evict_first();   // weights are read once per step
      // weights of unit (tile, ks) into stage s (the stage's full barrier also
      // expects the unit's activation bytes)
      auto issue_weights = [&](int tile, int ks, int s) {
        const uint32_t full = smem_u32(&T.full[s]);
        const uint32_t dst = stage0 + (uint32_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(full, w_tx + (uint32_t)p.x_bytes);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b) {
          int m, row;
          box_of<EPI>(p, tile, b, m, row);
          tma_load_2d_hint(dst + b * kBoxBytes, &p.mats[m].codes, ks * 128, row, full, pol);
          if (FMT == kFmtNVFP4)
            tma_load_2d_hint(dst + kCodeBytes + b * kScaleBoxBytes, &p.mats[m].scales, ks * 16, row, full, pol);
        }
      };
      auto issue_x = [&](int ks, int s) {
        const uint32_t full = smem_u32(&T.full[s]);
        const uint32_t dst = stage0 + (uint32_t)s * p.stage_bytes + p.x_off;
        const uint16_t* src = p.x.hi + (size_t)ks * kUnitK;
        for (int tok = 0; tok < p.N; ++tok)
          bulk_load(dst + tok * p.x_blk, src + (size_t)tok * p.d_in_pad, kUnitK * 2, full);
      };
      // Prime the first n_prime stages with weights before waiting for the
      // activations (the weights never depend on the kernels before this
      // one), then fill the rest of the ring.
      const int n_ring = (u1 - u0) < NS ? (int)(u1 - u0) : NS;
      const int n_pre = n_ring < p.n_prime ? n_ring : p.n_prime;
      {
        int tile = (int)(u0 / p.nks), ks = (int)(u0 % p.nks);
        for (int k = 0; k < n_pre; ++k) {
          issue_weights(tile, ks, k);
          if (++ks == p.nks) { ks = 0; ++tile; }
        }
        pdl_wait();
#ifdef BWS_TRACE
        T.tr[0] = trace_now();
#endif
        tile = (int)(u0 / p.nks);
        ks = (int)(u0 % p.nks);
        for (int k = 0; k < n_ring; ++k) {
          if (k >= n_pre) issue_weights(tile, ks, k);
          issue_x(ks, k);
          if (++ks == p.nks) { ks = 0; ++tile; }
        }
      }
      // The loop runs only when the ring was filled (n_ring == NS): unit
      // n_ring + j reuses stage j % NS after its (j / NS)-th release.
      int s = 0;
      uint32_t ph = 0u;   // parity of the release to wait for
      long long issued = n_ring;
      int tile = (int)((u0 + n_ring) / p.nks), ks = (int)((u0 + n_ring) % p.nks);
      for (long long u = u0 + n_ring; u < u1; ++u, ++issued) {
        if (!mbar_wait_bounded(smem_u32(&T.empty[s]), ph, kMaxPolls)) {
          atomicOr(p.status, kStatusTimeout);
          // let copies already issued land before the CTA's shared memory goes away
          for (long long k = (issued > NS ? issued - NS : 0); k < issued; ++k)
            mbar_wait_bounded(smem_u32(&T.full[k % NS]), (uint32_t)(k / NS) & 1u, kMaxPolls);
          break;
        }
        issue_weights(tile, ks, s);
        issue_x(ks, s);
        if (++s == NS) { s = 0; ph ^= 1u; }
        if (++ks == p.nks) { ks = 0; ++tile; }
      }
    }
    return;
  }

  // ---- consumers ----
  pdl_wait();
#ifdef BWS_TRACE
  if (threadIdx.x == 0) T.tr[1] = trace_now();
#endif
  uint32_t fl = 0u;
  for (int tok = 0; tok < p.N; ++tok) fl |= __ldg(p.x.flags + tok);
  if (fl & 1u)
    consume_lo<FMT, EPI, N1>(p, T, stage0, u0, u1, warp, lane, p.x.lo);
  else
    consume<FMT, EPI, false, N1>(p, T, stage0, u0, u1, warp, lane, p.x.lo);
  if (EPI == kEpiStoreF32 && p.amax_key != nullptr) {
    // the CTA's best keys into the call's, one atomic per token
    named_bar_sync(1, kConsumerWarps * 32);
    if (threadIdx.x < p.N) atomicMax(p.amax_key + threadIdx.x, T.akey[threadIdx.x]);
  }
#ifdef BWS_TRACE
  named_bar_sync(1, kConsumerWarps * 32);
  if (threadIdx.x == 0) {
    const unsigned long long t[6] = {tr_start, T.tr[0], T.tr[1], T.tr[2], T.tr[3], trace_now()};
    trace_put(1000u + 100u * FMT + 10u * EPI + (p.deposit ? 1u : 0u), t);
  }
#endif
}

template <int FMT, int EPI, bool N1>
cudaError_t launch_tma_one(const TmaParams& p, cudaStream_t st, bool pdl) {
  const int smem = p.n_stages * p.stage_bytes + (int)sizeof(Tail) + 1024;
  static std::atomic<unsigned long long> attr{0};
  {
    const cudaError_t e = set_smem_once(attr, gemv_tma_kernel<FMT, EPI, N1>, kSmemBudget + (int)sizeof(Tail) + 1024);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_ctas);
  cfg.blockDim = dim3(kThreadsTma);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_tma_kernel<FMT, EPI, N1>, p);
}

}  // namespace

bool gemv_tma_eligible(int fmt, const GemvParams& p) {
  if (p.slots.n_slots != nullptr || !tensor_maps_available()) return false;
  if (fmt == kFmtNVFP4) {
    if (p.d_in % 256 != 0) return false;
  } else if (fmt == kFmtFP8) {
    if (p.d_in % 128 != 0) return false;
  } else {
    return false;
  }
  for (int i = 0; i < p.n_mats; ++i) {
    if (((uintptr_t)p.mats[i].codes & 15) != 0) return false;
    if (fmt == kFmtNVFP4 && ((uintptr_t)p.mats[i].scales & 15) != 0) return false;
  }
  return true;
}

TmaGeom gemv_tma_geometry(int fmt, int epi, const GemvParams& g) {
  TmaGeom t;
  t.nks = fmt == kFmtFP8 ? g.d_in / 128 : g.d_in / 256;
  t.n_tiles = gemv_tma_tiles(epi, g.mats, g.n_mats);
  SplitK& s = t.split;
  s.n_units = (long long)t.n_tiles * t.nks;
  const long long ctas = 2LL * num_sms();   // two CTAs per SM
  s.n_ctas = (int)(s.n_units < ctas ? s.n_units : ctas);
  s.lf = s.n_ctas;
  s.num = s.den = 1;
  // CTAs that start when the inputs are ready (behind the prep's slots) are
  // about 1.5 us, two units of streaming, behind the others: their share is
  // cut by that much, within [1/4, 1] of the others'
  // (one token only: with more tokens fewer stages are primed, so the late
  // CTAs lose less, and measured, lighter shares made those steps slower)
  const int light = g.N == 1 ? g.split_light : 0;
  if (light > 0 && light < s.n_ctas / 4 && s.n_ctas == ctas) {
    const double per = (double)s.n_units / s.n_ctas;
    int num = (int)(16.0 * (1.0 - 2.0 / per) + 0.5);
    num = num < 4 ? 4 : num;
    const long long w = 16LL * (s.n_ctas - light) + (long long)num * light;
    if (num < 16 && (long long)num * s.n_units >= w) {   // every range keeps a unit
      s.lf = s.n_ctas - light;
      s.num = num;
      s.den = 16;
    }
  }
  return t;
}

bool gemv_tma_deposit_fits(const TmaGeom& t, const GemvParams& g) {
  return ((long long)t.n_tiles + t.split.n_ctas) * g.N * 128 * (long long)sizeof(float) <=
         ((long long)g.n_tiles + gemv_max_warps()) * kSlotFloats * (long long)sizeof(float);
}

int gemv_tma_tiles(int epi, const GemvMat* mats, int n_mats) {
  if (epi == kEpiSwiGLU) return (mats[0].d_out + 63) / 64;
  int t = 0;
  for (int i = 0; i < n_mats; ++i) t += (mats[i].d_out + 127) / 128;
  return t;
}

// Runs the product described by g (plain mode, activations already prepared)
// with the TMA kernel, in the scratch a product workspace provides: g.counters
// (g.n_tiles words, zero) and g.partials ((g.n_tiles + gemv_max_warps()) KiB).
cudaError_t launch_gemv_tma(int fmt, int epi, const GemvParams& g, uint32_t* status, cudaStream_t st, bool pdl) {
  TmaParams p;
  memset(&p, 0, sizeof(p));
  p.n_mats = g.n_mats;
  int tile = 0, row = 0;
  for (int i = 0; i < g.n_mats; ++i) {
    const GemvMat& M = g.mats[i];
    const uint64_t row_bytes = fmt == kFmtFP8 ? (uint64_t)g.d_in : (uint64_t)g.d_in / 2;
    if (!encode_2d(&p.mats[i].codes, M.codes, row_bytes, (uint64_t)M.d_out, 128, kBoxRows, true))
      return cudaErrorInvalidValue;
    if (fmt == kFmtNVFP4 &&
        !encode_2d(&p.mats[i].scales, M.scales, (uint64_t)g.d_in / 16, (uint64_t)M.d_out, 16, kBoxRows, false))
      return cudaErrorInvalidValue;
    p.mats[i].scale32 = M.scale32;
    p.mats[i].d_out = M.d_out;
    p.mats[i].out_row_off = epi == kEpiSwiGLU ? 0 : row;
    p.mats[i].tile_begin = tile;
    row += M.d_out;
    tile += (M.d_out + 127) / 128;
  }
  p.N = g.N;
  p.d_in = g.d_in;
  p.d_in_pad = g.d_in_pad;
  const TmaGeom geo = gemv_tma_geometry(fmt, epi, g);
  p.nks = geo.nks;
  p.n_tiles = geo.n_tiles;
  p.n_units = geo.split.n_units;
  p.n_ctas = geo.split.n_ctas;
  p.lf = geo.split.lf;
  p.num = geo.split.num;
  p.den = geo.split.den;
  p.deposit = g.deposit;
  p.amax_key = epi == kEpiStoreF32 ? g.amax_key : nullptr;
  p.no_store = p.amax_key != nullptr && g.no_store;
  if (p.deposit && (epi == kEpiStoreF32 || !gemv_tma_deposit_fits(geo, g))) return cudaErrorInvalidValue;
  p.x = g.x;
  p.out = g.out;
  p.out_ld = g.out_ld;
  p.partials = g.partials;
  p.counters = g.counters;
  p.status = status;
  // the scratch of the product workspace must cover this kernel's counters and partial sums
  if (p.n_tiles > g.n_tiles ||
      ((long long)p.n_tiles + p.n_ctas) * kPartialBytes >
          ((long long)g.n_tiles + gemv_max_warps()) * kSlotFloats * (long long)sizeof(float))
    return cudaErrorInvalidValue;
  const int unit_k = fmt == kFmtFP8 ? 128 : 256;
  p.x_off = fmt == kFmtNVFP4 ? kCodeBytes + kBoxes * kScaleBoxBytes : kCodeBytes;
  p.x_blk = unit_k * 2 + 16;                    // one token's slice, skewed by 16 bytes
  p.x_bytes = g.N * unit_k * 2;
  p.stage_bytes = ((p.x_off + g.N * p.x_blk) + 1023) / 1024 * 1024;
  p.n_stages = kSmemBudget / p.stage_bytes;
  if (p.n_stages > kMaxStages) p.n_stages = kMaxStages;
  if (p.n_stages < 2) return cudaErrorInvalidValue;
  // Weights primed before the inputs are ready: every CTA of the product
  // starts while the previous kernels finish, and a full ring of weight
  // copies from all of them (about 30 MB) queues ahead of those kernels'
  // last loads and stores, which decide when the inputs are ready. A stage
  // keeps the overlap without the queue (measured on the 27B-shape step,
  // one token, 1 / 2 / 3 / 4 stages: 5.16 / 5.23 / 5.31 / 5.37 ms; eight
  // tokens, 0 / 1 / 2: 6.90 / 6.99 / 7.07 ms; 2-4 tokens best with 1).
  p.n_prime = p.N <= 4 ? 1 : 0;
  if (p.n_ctas <= 0) return cudaSuccess;
  // one NVFP4 token: the block-diagonal operand (block scales on the accumulators)
  const bool n1 = fmt == kFmtNVFP4 && p.N == 1;
#define BWS_CASE(F, E)                                                              \
  if (fmt == F && epi == E)                                                         \
    return n1 ? launch_tma_one<F, E, (F == kFmtNVFP4)>(p, st, pdl) : launch_tma_one<F, E, false>(p, st, pdl);
  BWS_CASE(kFmtNVFP4, kEpiStoreBF16)
  BWS_CASE(kFmtNVFP4, kEpiResidF32)
  BWS_CASE(kFmtNVFP4, kEpiSwiGLU)
  BWS_CASE(kFmtNVFP4, kEpiStoreF32)
  BWS_CASE(kFmtFP8, kEpiStoreF32)
  BWS_CASE(kFmtFP8, kEpiStoreBF16)
  BWS_CASE(kFmtFP8, kEpiResidF32)
  BWS_CASE(kFmtFP8, kEpiSwiGLU)
#undef BWS_CASE
  return cudaErrorInvalidValue;
}

}  // namespace bws

#ifdef BWS_TRACE
extern "C" int bws_trace_read_tma(void* host, int cap) { return bws::trace_read(host, cap); }
#endif
