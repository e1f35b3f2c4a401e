// Persistent decode-step kernel for dense NVFP4 layer stacks (NVFP4 or FP8
// output layer): one cooperative launch runs every product of the step.
//
// Why one kernel. A decode step is a chain of a few hundred weight-stream
// products, each needing the whole output of the one before. As separate
// launches each product pays the ramp of filling the memory pipeline and the
// drain at its end, and the activation prep between them is a launch of its
// own. Here every CTA stays resident: its producer warp streams the weight
// units of all its products, in order, through a ring of shared-memory stages
// without ever waiting for activations (weights never depend on them), so the
// stream runs on across product boundaries while the consumer warps wait for
// the previous product to finish and prepare their activations.
//
// Work of one product. Its d_in is cut into S k-slabs of whole units (S is
// chosen so that one slab's activations of all N tokens fit in shared
// memory); the CTAs are dealt to the slabs in equal contiguous groups, and
// within a slab the (tile, k-unit) pairs, tile-major, are dealt to the group's
// CTAs in equal contiguous ranges (stream-K). A CTA therefore needs the
// activations of one slab only, and builds them itself: after the previous
// product's completion counter reaches its tile count, the consumer warps read
// the slab's raw inputs (the FP32 residual through RMSNorm, or a BF16 vector)
// from L2, form the f16 bands with the slab's own per-token exponent, and
// write them to shared memory in the layout the MMA lanes read. Partial sums
// of a tile, one per (slab, CTA) piece, are scaled back to true units and
// added by the last piece to arrive, in a fixed (slab, CTA) order.
//
// Completion and stats. The CTA that finishes a tile writes its outputs and
// the tile's per-token statistics of what it stored (the largest magnitude,
// and for a residual update the sum of squares of the new residual), then
// increments the product's completion counter. The next product's CTAs take
// from these, in a fixed order, the RMSNorm scale and the f16 band exponent
// of their input, so building a slab is a single pass over the input. All
// counters are zeroed by the step's init kernel; every wait is bounded and
// sets a status bit.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <new>
#include <vector>

#include "bws_common.cuh"
#include "bws_internal.h"
#include "step.h"
#include "stream_tile.cuh"

namespace bws {

namespace {

constexpr int kSW = 8;                                  // consumer warps
constexpr int kStepThreads = (kSW + 1) * 32;
constexpr int kConsumerThreads = kSW * 32;
constexpr int kStages = 4;
constexpr int kStageBytes = kCodeBytes + kBoxes * kScaleBoxBytes;   // one NVFP4 unit, 18 KiB
constexpr int kXBytes = 24 * 1024;                      // one slab of activations
constexpr uint32_t kPolls = 1u << 24;                   // bounded waits
constexpr uint32_t kStatusTimeout = 0x100u;
constexpr int kSlotF4 = kBoxes * 2 * 32;                // float4s in one partial-sum slot
constexpr int kStatRows = 128;                          // rows per residual sum-of-squares partial

struct StepMat {   // 64-byte aligned through CUtensorMap
  CUtensorMap codes;     // u8 [d_out][row bytes], box {128, 32}, 128B swizzle
  CUtensorMap scales;    // NVFP4: u8 [d_out][d_in/16], box {16, 32}
  const float* scale32;  // NVFP4 tensor scale [1]; FP8 row scales [d_out]
  int d_out, out_row_off, tile_begin;
};

constexpr int kSrcNorm = 0;   // the product reads bf16(RMSNorm(r))
constexpr int kSrcBF16 = 1;   // the product reads BF16 rows of the workspace

struct StepProduct {
  int fmt, epi, n_mats, mat0;
  int d_in, nks, n_tiles, n_slabs;
  int src, x_ld, stats_tiles, out_ld;
  long long x_off;          // kSrcBF16: workspace offset of the source rows
  long long stats_off;      // workspace offset of the input's [stats_tiles][N] (sum of squares, max |v|)
  long long out_off;        // workspace offset of the output, -1: the logits
  long long stats_out_off;  // workspace offset of the output's [n_tiles][N] statistics (not for logits)
};

struct StepParams {
  const StepProduct* prods;
  const StepMat* mats;
  int n_prods, N, hidden, G;
  float eps;
  char* ws;
  float* logits;
  const uint16_t* x0;
  long long r_off, done_off, counters_off, partials_off, lo_off, stats0_off;
  long long slab_stride;    // partial-sum slots per slab
  int max_tiles;
};

// Shared memory after the ring and the activation slab.
struct StepTail {
  float4 red[kBoxes][2][32];   // half-pair reduction (box, sub-tile, lane)
  float4 swi[2][2][32];        // SwiGLU: up sums handed to the gate warps
  uint64_t full[kStages];
  uint64_t empty[kStages];
  float inv_rms[kMaxTokens];
  int E[kMaxTokens];
  float hs[kMaxTokens];        // 2^(14 - E) when a normal float, else 0
  uint32_t maxbits[kMaxTokens];
  float2 stat[4][kMaxTokens];
  uint32_t xflags;
  uint32_t prev;
  uint32_t dead;
};

// Where CTA c works in a product: its slab, the slab's k-units and its range of
// the slab's (tile, k-unit) pairs.
struct SlabPos {
  int s, k0, nk, l, gs;
  long long units, u0, u1;
};

__host__ __device__ inline long long owner_of(long long u, long long U, long long G) { return ((u + 1) * G - 1) / U; }

__host__ __device__ inline SlabPos slab_pos(int T, int K, int S, int c, int G) {
  SlabPos q;
  q.s = (int)owner_of(c, G, S);
  const int c0 = (int)((long long)q.s * G / S), c1 = (int)((long long)(q.s + 1) * G / S);
  q.l = c - c0;
  q.k0 = (int)((long long)q.s * K / S);
  q.nk = (int)((long long)(q.s + 1) * K / S) - q.k0;
  q.units = (long long)T * q.nk;
  // a slab with fewer units than CTAs uses only as many CTAs as it has units,
  // so that every working CTA has at least one
  q.gs = (long long)(c1 - c0) < q.units ? c1 - c0 : (int)q.units;
  if (q.l < q.gs) {
    q.u0 = q.l * q.units / q.gs;
    q.u1 = (q.l + 1) * q.units / q.gs;
  } else {
    q.u0 = q.u1 = 0;
  }
  return q;
}

// Matrix and first row of box b of a tile.
BWS_DEV void step_box(const StepProduct& P, const StepMat* M, int tile, int b, int& m, int& row) {
  if (P.epi == kEpiSwiGLU) {
    m = P.mat0 + (b >> 1);
    row = tile * 64 + 32 * (b & 1);
    return;
  }
  int mi = 0;
  for (int i = 1; i < P.n_mats; ++i)
    if (tile >= __ldg(&M[P.mat0 + i].tile_begin)) mi = i;
  m = P.mat0 + mi;
  row = (tile - __ldg(&M[m].tile_begin)) * 128 + 32 * b;
}

BWS_DEV float bf16_to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }

BWS_DEV uint32_t ld_cg_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
BWS_DEV float ld_cg_f32(const float* p) { return __uint_as_float(ld_cg_u32(reinterpret_cast<const uint32_t*>(p))); }
BWS_DEV uint2 ld_cg_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
BWS_DEV uint4 ld_cg_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
BWS_DEV uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Raw input of piece i (8 consecutive k of one token) of the slab: 8 FP32
// residual values (kSrcNorm) or 8 BF16 values in raw.x..w (kSrcBF16).
struct RawPiece {
  uint4 a, b;
};
BWS_DEV RawPiece load_piece(const StepParams& p, const StepProduct& P, int n, int k) {
  RawPiece r;
  if (P.src == kSrcNorm) {
    const float* x = reinterpret_cast<const float*>(p.ws + p.r_off) + (size_t)n * p.hidden + k;
    r.a = ld_cg_u4(x);
    r.b = ld_cg_u4(x + 4);
  } else {
    r.a = ld_cg_u4(reinterpret_cast<const uint16_t*>(p.ws + P.x_off) + (size_t)n * P.x_ld + k);
    r.b = make_uint4(0, 0, 0, 0);
  }
  return r;
}

// The piece as BF16 bit patterns (the product's input is BF16 by definition).
BWS_DEV void piece_bf16(const StepProduct& P, const RawPiece& r, float inv_rms, uint32_t (&w)[4]) {
  if (P.src == kSrcNorm) {
    const uint32_t v[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__uint_as_float(v[2 * i]), inv_rms)));
      const uint32_t hi =
          __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__uint_as_float(v[2 * i + 1]), inv_rms)));
      w[i] = lo | (hi << 16);
    }
  } else {
    w[0] = r.a.x; w[1] = r.a.y; w[2] = r.a.z; w[3] = r.a.w;
  }
}

// f16 bands of a piece with exponent E: the hi band, and band flags (bit 0: an
// element needs the lo band, bit 1: an element is below both).
BWS_DEV uint4 piece_hi(const uint32_t (&w)[4], int E, uint32_t& flags) {
  uint32_t h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t hh[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float f = bf16_to_f32(e == 0 ? (w[j] & 0xFFFF) : (w[j] >> 16));
      const float a = ldexp_exact(f, 14 - E);
      hh[e] = 0u;
      if (fabsf(a) >= 0x1p-14f)
        hh[e] = __half_as_ushort(__float2half_rn(a));
      else if (f != 0.0f)
        flags |= fabsf(ldexp_exact(f, 43 - E)) >= 0x1p-14f ? 1u : 2u;
    }
    h[j] = hh[0] | (hh[1] << 16);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}
// The same with the scale 2^(14 - E) given as a float (14 - E in the normal
// range): one multiply per element, exact (a power of two; results below
// 2^-14 leave the hi band whatever their rounding).
BWS_DEV uint4 piece_hi_fast(const uint32_t (&w)[4], float hs, int E, uint32_t& flags) {
  uint32_t h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float f0 = __uint_as_float(w[j] << 16), f1 = __uint_as_float(w[j] & 0xFFFF0000u);
    float a0 = __fmul_rn(f0, hs), a1 = __fmul_rn(f1, hs);
    if (fabsf(a0) < 0x1p-14f) {
      if (f0 != 0.0f) flags |= fabsf(ldexp_exact(f0, 43 - E)) >= 0x1p-14f ? 1u : 2u;
      a0 = 0.0f;
    }
    if (fabsf(a1) < 0x1p-14f) {
      if (f1 != 0.0f) flags |= fabsf(ldexp_exact(f1, 43 - E)) >= 0x1p-14f ? 1u : 2u;
      a1 = 0.0f;
    }
    const __half2 v = __floats2half2_rn(a0, a1);
    h[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}
BWS_DEV uint4 piece_lo(const uint32_t (&w)[4], int E) {
  uint32_t l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t ll[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float f = bf16_to_f32(e == 0 ? (w[j] & 0xFFFF) : (w[j] >> 16));
      ll[e] = 0u;
      if (fabsf(ldexp_exact(f, 14 - E)) < 0x1p-14f && f != 0.0f) {
        const float b = ldexp_exact(f, 43 - E);
        if (fabsf(b) >= 0x1p-14f) ll[e] = __half_as_ushort(__float2half_rn(b));
      }
    }
    l[j] = ll[0] | (ll[1] << 16);
  }
  return make_uint4(l[0], l[1], l[2], l[3]);
}

constexpr int kBatch = 4;   // pieces a thread loads before converting

// Builds the CTA's activation slab for product P (consumer threads only): the
// hi band in shared memory at xs, the lo band (when some element needs it) in
// the CTA's global scratch. The per-token RMSNorm scale and band exponent come
// from the statistics the input's producer left per tile (for RMSNorm,
// max |BF16(r * s)| = BF16(max |r| * s), rounding being monotone), so the
// slab's inputs are read once, their loads issued before the statistics are
// reduced. Returns the CTA's band flags.
__device__ __noinline__ uint32_t build_slab(const StepParams& p, const StepProduct& P, const SlabPos& pos,
                                            StepTail& T, uint8_t* xs, uint8_t* lo_glob, int tid) {
  const int N = p.N;
  const int UK = P.fmt == kFmtFP8 ? 128 : 256;
  const int xblk = UK * 2 + 16;
  const int u8 = UK / 8;                 // pieces per unit
  const int lk = UK / 64;                // pieces per lane chunk
  const int n8 = pos.nk * u8;            // pieces per token
  const int total = N * n8;
  const int kbase = pos.k0 * UK;
  const int warp = tid >> 5, lane = tid & 31;
  // first batch of this thread's pieces, in flight while the statistics are reduced
  RawPiece raw[kBatch];
#pragma unroll
  for (int k = 0; k < kBatch; ++k) {
    const int i = tid + k * kConsumerThreads;
    if (i < total) {
      const int n = i / n8;
      raw[k] = load_piece(p, P, n, kbase + (i - n * n8) * 8);
    }
  }
  if (warp < N) {
    // the tiles' statistics of this token, eight per lane in flight at once
    const float2* st = reinterpret_cast<const float2*>(p.ws + P.stats_off) + warp;
    const int tiles = P.stats_tiles;
    float sq = 0.0f, mx = 0.0f;
    for (int t0 = lane; t0 < tiles; t0 += 8 * 32) {
      uint2 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = t0 + k * 32;
        v[k] = t < tiles ? ld_cg_u2(st + (size_t)t * N) : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        sq = __fadd_rn(sq, __uint_as_float(v[k].x));
        mx = fmaxf(mx, __uint_as_float(v[k].y));
      }
    }
    sq = warp_sum(sq);
    mx = warp_max(mx);
    if (lane == 0) {
      float inv = 1.0f, amax = mx;
      if (P.src == kSrcNorm) {
        inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sq, (float)p.hidden), p.eps)));
        amax = __bfloat162float(__float2bfloat16_rn(__fmul_rn(mx, inv)));
      }
      T.inv_rms[warp] = inv;
      const int E = amax > 0.0f ? floor_log2_abs(amax) : 0;
      T.E[warp] = E;
      T.hs[warp] = (14 - E >= -126 && 14 - E <= 127) ? exp2i(14 - E) : 0.0f;   // 0: exact slow path
    }
  }
  if (tid == 0) T.xflags = 0u;
  named_bar_sync(4, kConsumerThreads);
  uint32_t flags = 0u;
  for (int i0 = tid; i0 < total; i0 += kBatch * kConsumerThreads) {
    if (i0 != tid) {
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int i = i0 + k * kConsumerThreads;
        if (i < total) {
          const int n = i / n8;
          raw[k] = load_piece(p, P, n, kbase + (i - n * n8) * 8);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = i0 + k * kConsumerThreads;
      if (i >= total) break;
      const int n = i / n8, i8 = i - n * n8;
      uint32_t w[4];
      piece_bf16(P, raw[k], T.inv_rms[n], w);
      const int j = i8 / u8, kl8 = i8 - j * u8;
      const int off = (j * N + n) * xblk + (kl8 / lk) * 16 + (kl8 % lk) * 128;
      const float hs = T.hs[n];
      *reinterpret_cast<uint4*>(xs + off) = hs != 0.0f ? piece_hi_fast(w, hs, T.E[n], flags) : piece_hi(w, T.E[n], flags);
    }
  }
  if (flags) atomicOr(&T.xflags, flags);
  named_bar_sync(4, kConsumerThreads);
  const uint32_t fl = T.xflags;
  if (fl & 1u) {
    // (rare) the lo band, same layout, in global scratch
    for (int i = tid; i < total; i += kConsumerThreads) {
      const int n = i / n8, i8 = i - n * n8;
      const RawPiece r = load_piece(p, P, n, kbase + i8 * 8);
      uint32_t w[4];
      piece_bf16(P, r, T.inv_rms[n], w);
      const int j = i8 / u8, kl8 = i8 - j * u8;
      const int off = (j * N + n) * xblk + (kl8 / lk) * 16 + (kl8 % lk) * 128;
      *reinterpret_cast<uint4*>(lo_glob + off) = piece_lo(w, T.E[n]);
    }
    __threadfence_block();
    named_bar_sync(4, kConsumerThreads);
  }
  return fl;
}

// Where CTA c works in product Pp.
BWS_DEV SlabPos pos_of(const StepProduct* Pp, int c, int G) {
  return slab_pos(__ldg(&Pp->n_tiles), __ldg(&Pp->nks), __ldg(&Pp->n_slabs), c, G);
}

// Pieces of tile t over all slabs.
BWS_DEV int tile_pieces(const StepProduct* Pp, int t, int G) {
  const int S = __ldg(&Pp->n_slabs), T = __ldg(&Pp->n_tiles), K = __ldg(&Pp->nks);
  int n = 0;
  for (int s = 0; s < S; ++s) {
    const SlabPos q = slab_pos(T, K, S, (int)((long long)s * G / S), G);
    n += (int)(owner_of((long long)t * q.nk + q.nk - 1, q.units, q.gs) - owner_of((long long)t * q.nk, q.units, q.gs)) + 1;
  }
  return n;
}

// Final outputs of sub-tile st of box b (v: true-unit sums before the matrix
// scale; register i = row g + 8*(i>>1), token 2t + (i&1)); adds to ss / mx
// (tokens 2t, 2t+1) the squares (residual updates) and the largest magnitude
// of the values stored.
BWS_DEV void step_store(const StepParams& p, const StepProduct& P, int tile, int b, int st, int g, int t,
                        const float (&v)[4], const float (&vu)[4], float (&ss)[2], float (&mx)[2]) {
  int mi, row_b;
  step_box(P, p.mats, tile, b, mi, row_b);
  const StepMat& M = p.mats[mi];
  const int d_out = __ldg(&M.d_out);
  const int row0 = row_b + 16 * st;
  const float* s32 = M.scale32;
  const float su = P.epi == kEpiSwiGLU ? __ldg(p.mats[P.mat0 + 1].scale32) : 1.0f;
  char* outb = P.out_off < 0 ? reinterpret_cast<char*>(p.logits) : p.ws + P.out_off;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = row0 + g + 8 * (i >> 1);
    const int tok = 2 * t + (i & 1);
    if (row >= d_out || tok >= p.N) continue;
    const float sc = P.fmt == kFmtFP8 ? __ldg(s32 + row) : __ldg(s32);
    const float val = __fmul_rn(v[i], sc);
    if (P.epi == kEpiSwiGLU) {
      const float up = __fmul_rn(vu[i], su);
      const __nv_bfloat16 h = __float2bfloat16_rn(silu_mul_t(val, up));
      reinterpret_cast<__nv_bfloat16*>(outb)[(size_t)tok * P.out_ld + row] = h;
      mx[i & 1] = fmaxf(mx[i & 1], fabsf(__bfloat162float(h)));
    } else {
      const size_t o = (size_t)tok * P.out_ld + __ldg(&M.out_row_off) + row;
      if (P.epi == kEpiStoreBF16) {
        const __nv_bfloat16 y = __float2bfloat16_rn(val);
        reinterpret_cast<__nv_bfloat16*>(outb)[o] = y;
        mx[i & 1] = fmaxf(mx[i & 1], fabsf(__bfloat162float(y)));
      } else if (P.epi == kEpiStoreF32) {
        reinterpret_cast<float*>(outb)[o] = val;
      } else {
        float* r = reinterpret_cast<float*>(outb) + o;
        const float nr = __fadd_rn(ld_cg_f32(r), val);
        *r = nr;
        ss[i & 1] = __fmaf_rn(nr, nr, ss[i & 1]);
        mx[i & 1] = fmaxf(mx[i & 1], fabsf(nr));
      }
    }
  }
}

// End of a tile piece of product pi for warps 0..3 (v0 / v1: sub-tiles 0 and
// 1 of box b, sums in true units): deposit it, and if it is the tile's last
// piece add all pieces, store the outputs and statistics and count the tile
// done. Out of line, with scalar arguments: it runs once per piece, and the
// unit loop keeps its registers.
__device__ __noinline__ void piece_end(const StepParams& p, int pi, StepTail& T, int cur, bool whole, float4 v0,
                                       float4 v1) {
  const StepProduct P = p.prods[pi];
  const int N = p.N;
  const int lane = threadIdx.x & 31, b = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
  float v[2][4] = {{v0.x, v0.y, v0.z, v0.w}, {v1.x, v1.y, v1.z, v1.w}};
  float* partials = reinterpret_cast<float*>(p.ws + p.partials_off);
  uint32_t* counters = reinterpret_cast<uint32_t*>(p.ws + p.counters_off);
  uint32_t* done = reinterpret_cast<uint32_t*>(p.ws + p.done_off);
  if (!whole) {
    const SlabPos pos = slab_pos(P.n_tiles, P.nks, P.n_slabs, blockIdx.x, p.G);
    float4* slot = reinterpret_cast<float4*>(partials) + ((size_t)pos.s * p.slab_stride + cur + pos.l) * kSlotF4 + b * 64;
    slot[lane] = v0;
    slot[32 + lane] = v1;
    __threadfence();
    named_bar_sync(2, 4 * 32);
    if (threadIdx.x == 0) T.prev = atomicAdd(counters + cur, 1u);
    named_bar_sync(2, 4 * 32);
    const uint32_t prev = T.prev;
    named_bar_sync(2, 4 * 32);
    if (prev + 1 != (uint32_t)tile_pieces(p.prods + pi, cur, p.G)) return;
    __threadfence();
    // all pieces of the tile, added in (slab, CTA) order, two slots' loads in flight
    float a8[2][4] = {};
    for (int s2 = 0; s2 < P.n_slabs; ++s2) {
      const SlabPos q = slab_pos(P.n_tiles, P.nks, P.n_slabs, (int)((long long)s2 * p.G / P.n_slabs), p.G);
      const int l0 = (int)owner_of((long long)cur * q.nk, q.units, q.gs);
      const int l1 = (int)owner_of((long long)cur * q.nk + q.nk - 1, q.units, q.gs);
      const float4* src0 =
          reinterpret_cast<const float4*>(partials) + ((size_t)s2 * p.slab_stride + cur) * kSlotF4 + b * 64 + lane;
      for (int l = l0; l <= l1; l += 2) {
        const bool two = l + 1 <= l1;
        const float4 o0 = ld_cg_f4(src0 + (size_t)l * kSlotF4), o1 = ld_cg_f4(src0 + (size_t)l * kSlotF4 + 32);
        float4 o2 = make_float4(0.f, 0.f, 0.f, 0.f), o3 = o2;
        if (two) {
          o2 = ld_cg_f4(src0 + (size_t)(l + 1) * kSlotF4);
          o3 = ld_cg_f4(src0 + (size_t)(l + 1) * kSlotF4 + 32);
        }
        a8[0][0] += o0.x; a8[0][1] += o0.y; a8[0][2] += o0.z; a8[0][3] += o0.w;
        a8[1][0] += o1.x; a8[1][1] += o1.y; a8[1][2] += o1.z; a8[1][3] += o1.w;
        if (two) {
          a8[0][0] += o2.x; a8[0][1] += o2.y; a8[0][2] += o2.z; a8[0][3] += o2.w;
          a8[1][0] += o3.x; a8[1][1] += o3.y; a8[1][2] += o3.z; a8[1][3] += o3.w;
        }
      }
    }
#pragma unroll
    for (int st = 0; st < 2; ++st)
#pragma unroll
      for (int r = 0; r < 4; ++r) v[st][r] = a8[st][r];
    if (threadIdx.x == 0) counters[cur] = 0u;
  }
  float ss[2] = {0.f, 0.f}, mx[2] = {0.f, 0.f};
  const float none[4] = {0.f, 0.f, 0.f, 0.f};
  if (P.epi == kEpiSwiGLU) {
    if (b >= 2) {
#pragma unroll
      for (int st = 0; st < 2; ++st) T.swi[b - 2][st][lane] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
    }
    named_bar_sync(2, 4 * 32);
    if (b < 2) {
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        const float4 o = T.swi[b][st][lane];
        const float vu[4] = {o.x, o.y, o.z, o.w};
        step_store(p, P, cur, b, st, g, t, v[st], vu, ss, mx);
      }
    }
  } else {
#pragma unroll
    for (int st = 0; st < 2; ++st) step_store(p, P, cur, b, st, g, t, v[st], none, ss, mx);
  }
  if (P.epi != kEpiStoreF32) {
    // the tile's per-token statistics, reduced in a fixed order
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], o));
      }
    }
    if (g == 0) {
      T.stat[b][2 * t] = make_float2(ss[0], mx[0]);
      T.stat[b][2 * t + 1] = make_float2(ss[1], mx[1]);
    }
    named_bar_sync(2, 4 * 32);
    if (threadIdx.x < (unsigned)N) {
      const int n = threadIdx.x;
      float2* so = reinterpret_cast<float2*>(p.ws + P.stats_out_off);
      so[(size_t)cur * N + n] =
          make_float2(__fadd_rn(__fadd_rn(T.stat[0][n].x, T.stat[1][n].x), __fadd_rn(T.stat[2][n].x, T.stat[3][n].x)),
                      fmaxf(fmaxf(T.stat[0][n].y, T.stat[1][n].y), fmaxf(T.stat[2][n].y, T.stat[3][n].y)));
    }
  }
  __threadfence();
  named_bar_sync(2, 4 * 32);
  if (threadIdx.x == 0) atomicAdd(done + pi, 1u);
}

// The consumer warps' units [u0, u1) of product pi (slab k-units nk; tiles
// whole if the product has one slab); LO: the two-band path. Keeps little
// state in registers: everything else is reread at the piece ends.
template <int FMT, bool LO>
BWS_DEV void step_units(const StepParams& p, int pi, long long u0, long long u1, int nk, bool one_slab, StepTail& T,
                        uint32_t stage0, uint32_t xs0, const uint8_t* lo_glob, int& s, uint32_t& ph) {
  constexpr int kUnitK = FMT == kFmtFP8 ? 128 : 256;
  constexpr int kXv = FMT == kFmtFP8 ? 2 : 4;
  const int N = p.N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int xblk = kUnitK * 2 + 16;
  const int b = warp & 3, half = warp >> 2;
  const int g = lane >> 2, t = lane & 3;
  const int c = 2 * t + half;
  const uint32_t coff = b * kBoxBytes + g * 128 + ((c ^ g) << 4);
  const uint32_t soff = kCodeBytes + b * kScaleBoxBytes + g * 16 + 2 * c;
  const int xg = g < N ? g : 0;
  const uint32_t xlane = xs0 + (uint32_t)(xg * xblk + c * 16);
  const uint32_t xstep = (uint32_t)(N * xblk);

  float acc[2][2][4] = {}, accl[2][4] = {};
  uint4 xh[kXv], xl[kXv];
  int tile = (int)(u0 / nk), kl = (int)(u0 % nk);
  bool piece_whole = kl == 0;
  for (long long u = u0; u < u1; ++u) {
    const uint32_t xu = xlane + (uint32_t)kl * xstep;
    if (LO) {
#pragma unroll
      for (int q = 0; q < kXv; ++q) xl[q] = ld_cg_u4(lo_glob + (xu - xs0) + q * 128);
    }
    // once a wait has run out nothing is waited for or released any more, so
    // the producer runs out of released stages and stops (no copy is ever
    // issued into a stage that a copy may still be filling)
    bool have = !T.dead;
    if (have && !mbar_wait_bounded(smem_u32(&T.full[s]), ph, kPolls)) {
      if (lane == 0) atomicOr(reinterpret_cast<uint32_t*>(p.ws) + 1, kStatusTimeout);
      T.dead = 1u;
      have = false;
    }
    const uint32_t base = stage0 + (uint32_t)s * kStageBytes;
    uint4 cw[4];
    uint32_t sc[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) cw[j] = lds_v4(base + coff + j * 1024);
    if (FMT == kFmtNVFP4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[j] = lds_u16(base + soff + j * 128);
    }
#pragma unroll
    for (int q = 0; q < kXv; ++q) xh[q] = lds_v4(xu + q * 128);
    __syncwarp();
    if (lane == 0 && have) mbar_arrive(smem_u32(&T.empty[s]));
    if (++s == kStages) { s = 0; ph ^= 1u; }
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const uint32_t w0[4] = {cw[2 * st].x, cw[2 * st].y, cw[2 * st].z, cw[2 * st].w};
      const uint32_t w1[4] = {cw[2 * st + 1].x, cw[2 * st + 1].y, cw[2 * st + 1].z, cw[2 * st + 1].w};
      sub_mma<FMT, LO>(acc[st], accl[st], w0, w1, sc[2 * st], sc[2 * st + 1], xh, xl);
    }
    const bool last_of_tile = kl == nk - 1;
    const int cur = tile;
    if (++kl == nk) { kl = 0; ++tile; }
    if (!last_of_tile && u + 1 < u1) continue;
    // ---- end of a tile piece: the two halves added, sums in true units ----
    float v[2][4];
#pragma unroll
    for (int st = 0; st < 2; ++st) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float a = __fadd_rn(acc[st][0][r], acc[st][1][r]);
        v[st][r] = LO ? __fmaf_rn(accl[st][r], 0x1p-29f, a) : a;
        acc[st][0][r] = acc[st][1][r] = accl[st][r] = 0.f;
      }
    }
    if (half == 1) {
#pragma unroll
      for (int st = 0; st < 2; ++st) T.red[b][st][lane] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
    }
    named_bar_sync(1, kConsumerThreads);
    const bool whole = piece_whole && last_of_tile && one_slab;
    piece_whole = true;
    if (half == 0) {
      const int e0 = (2 * t < N ? T.E[2 * t] : 0) - 14, e1 = (2 * t + 1 < N ? T.E[2 * t + 1] : 0) - 14;
      float4 w[2];
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        const float4 o = T.red[b][st][lane];
        w[st] = make_float4(ldexp_exact(v[st][0] + o.x, e0), ldexp_exact(v[st][1] + o.y, e1),
                            ldexp_exact(v[st][2] + o.z, e0), ldexp_exact(v[st][3] + o.w, e1));
      }
      named_bar_sync(1, kConsumerThreads);   // T.red read: warps 4..7 may go on
      piece_end(p, pi, T, cur, whole, w[0], w[1]);
    } else {
      named_bar_sync(1, kConsumerThreads);
    }
  }
}

// The two-band unit loops, out of line (rare; their registers stay out of the
// main loops).
template <int FMT>
__device__ __noinline__ void step_units_lo(const StepParams& p, int pi, long long u0, long long u1, int nk,
                                           bool one_slab, StepTail& T, uint32_t stage0, uint32_t xs0,
                                           const uint8_t* lo_glob, int& s, uint32_t& ph) {
  step_units<FMT, true>(p, pi, u0, u1, nk, one_slab, T, stage0, xs0, lo_glob, s, ph);
}

// A position in this CTA's sequence of weight units (products in order, each
// product's units tile-major within its slab). pi == n_prods: past the end.
struct UnitCursor {
  int pi, tile, kl, nk, k0;
  long long u, u1;
};

BWS_DEV void cursor_product(const StepParams& p, UnitCursor& c) {
  for (; c.pi < p.n_prods; ++c.pi) {
    const SlabPos q = pos_of(p.prods + c.pi, blockIdx.x, p.G);
    if (q.u1 > q.u0) {
      c.u = q.u0;
      c.u1 = q.u1;
      c.nk = q.nk;
      c.k0 = q.k0;
      c.tile = (int)(q.u0 / q.nk);
      c.kl = (int)(q.u0 % q.nk);
      return;
    }
  }
}
BWS_DEV void cursor_start(const StepParams& p, UnitCursor& c) {
  c.pi = 0;
  cursor_product(p, c);
}
BWS_DEV void cursor_next(const StepParams& p, UnitCursor& c) {
  if (++c.kl == c.nk) { c.kl = 0; ++c.tile; }
  if (++c.u == c.u1) {
    ++c.pi;
    cursor_product(p, c);
  }
}

// The unit at the cursor into the stage at dst, completing on bar.
BWS_DEV void issue_unit(const StepParams& p, const UnitCursor& c, uint32_t dst, uint32_t bar) {
  const StepProduct P = p.prods[c.pi];
  const int ks = c.k0 + c.kl;
  mbar_arrive_expect_tx(bar, P.fmt == kFmtNVFP4 ? kStageBytes : kCodeBytes);
#pragma unroll
  for (int b = 0; b < kBoxes; ++b) {
    int m, row;
    step_box(P, p.mats, c.tile, b, m, row);
    tma_load_2d(dst + b * kBoxBytes, &p.mats[m].codes, ks * 128, row, bar);
    if (P.fmt == kFmtNVFP4) tma_load_2d(dst + kCodeBytes + b * kScaleBoxBytes, &p.mats[m].scales, ks * 16, row, bar);
  }
}

__global__ void __launch_bounds__(kStepThreads, 2) step_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* sbase = smem_raw + ((1024u - mis) & 1023u);
  uint8_t* xs = sbase + kStages * kStageBytes;
  StepTail& T = *reinterpret_cast<StepTail*>(xs + kXBytes);
  const uint32_t stage0 = smem_u32(sbase);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&T.full[i]), 1);
      mbar_init(smem_u32(&T.empty[i]), kSW);
    }
    T.dead = 0u;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kSW) {
    // ---- producer: the weight units of every product, in order ----
    if (lane == 0) {
      UnitCursor ld;
      cursor_start(p, ld);
      int s = 0;
      uint32_t ph = 0u;
      long long issued = 0;
      for (; ld.pi < p.n_prods; ++issued) {
        if (issued >= kStages && !mbar_wait_bounded(smem_u32(&T.empty[s]), ph ^ 1u, kPolls)) {
          atomicOr(reinterpret_cast<uint32_t*>(p.ws) + 1, kStatusTimeout);
          break;
        }
        issue_unit(p, ld, stage0 + (uint32_t)s * kStageBytes, smem_u32(&T.full[s]));
        cursor_next(p, ld);
        if (++s == kStages) { s = 0; ph ^= 1u; }
      }
      // let copies in flight land before the CTA's shared memory goes away
      for (long long k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
        mbar_wait_bounded(smem_u32(&T.full[k % kStages]), (uint32_t)(k / kStages) & 1u, kPolls);
    }
    return;
  }

  // ---- consumers ----
  pdl_wait();
  const int tid = threadIdx.x;
  uint32_t* done = reinterpret_cast<uint32_t*>(p.ws + p.done_off);
  uint32_t* status = reinterpret_cast<uint32_t*>(p.ws) + 1;
  uint8_t* lo_glob = reinterpret_cast<uint8_t*>(p.ws + p.lo_off) + (size_t)blockIdx.x * kXBytes;
  const uint32_t xs0 = smem_u32(xs);
  int s = 0;
  uint32_t ph = 0u;
  for (int pi = 0; pi < p.n_prods; ++pi) {
    const StepProduct* Pp = p.prods + pi;
    const SlabPos pos = pos_of(Pp, blockIdx.x, p.G);
    if (pos.u1 <= pos.u0) continue;
    if (pi > 0) {
      // the previous product's outputs (this product's input) are complete
      if (tid == 0 && !T.dead) {
        const uint32_t want = (uint32_t)__ldg(&p.prods[pi - 1].n_tiles);
        uint32_t k = 0;
        while (ld_acquire_u32(done + pi - 1) < want) {
          if (++k == kPolls) {
            atomicOr(status, kStatusTimeout);
            T.dead = 1u;
            break;
          }
          __nanosleep(32);
        }
      }
      named_bar_sync(4, kConsumerThreads);
    }
    const uint32_t fl = build_slab(p, *Pp, pos, T, xs, lo_glob, tid);
    if (tid == 0 && fl) atomicOr(status, fl);
    const bool fp8 = __ldg(&Pp->fmt) == kFmtFP8;
    const bool one_slab = __ldg(&Pp->n_slabs) == 1;
    if (fl & 1u) {
      if (fp8)
        step_units_lo<kFmtFP8>(p, pi, pos.u0, pos.u1, pos.nk, one_slab, T, stage0, xs0, lo_glob, s, ph);
      else
        step_units_lo<kFmtNVFP4>(p, pi, pos.u0, pos.u1, pos.nk, one_slab, T, stage0, xs0, lo_glob, s, ph);
    } else {
      if (fp8)
        step_units<kFmtFP8, false>(p, pi, pos.u0, pos.u1, pos.nk, one_slab, T, stage0, xs0, lo_glob, s, ph);
      else
        step_units<kFmtNVFP4, false>(p, pi, pos.u0, pos.u1, pos.nk, one_slab, T, stage0, xs0, lo_glob, s, ph);
    }
  }
}

// r = x0 (FP32), the first RMSNorm's per-128-row sums of squares, and zeroed
// counters and status. Block (tile, n), 128 threads.
__global__ void __launch_bounds__(128) step_init_kernel(const __grid_constant__ StepParams p) {
  pdl_launch_dependents();   // the step kernel's producers may start streaming weights
  const int n = blockIdx.y, tile = blockIdx.x;
  const int i = tile * kStatRows + threadIdx.x;
  float* r = reinterpret_cast<float*>(p.ws + p.r_off);
  float v = 0.0f;
  if (i < p.hidden) {
    v = __uint_as_float((uint32_t)p.x0[(size_t)n * p.hidden + i] << 16);
    r[(size_t)n * p.hidden + i] = v;
  }
  const float s = warp_sum(__fmul_rn(v, v));
  const float m = warp_max(fabsf(v));
  __shared__ float2 ws4[4];
  if ((threadIdx.x & 31) == 0) ws4[threadIdx.x >> 5] = make_float2(s, m);
  __syncthreads();
  if (threadIdx.x == 0) {
    float2* st = reinterpret_cast<float2*>(p.ws + p.stats0_off);
    st[(size_t)tile * p.N + n] = make_float2(__fadd_rn(__fadd_rn(ws4[0].x, ws4[1].x), __fadd_rn(ws4[2].x, ws4[3].x)),
                                             fmaxf(fmaxf(ws4[0].y, ws4[1].y), fmaxf(ws4[2].y, ws4[3].y)));
  }
  if (tile == 0 && n == 0) {
    uint32_t* done = reinterpret_cast<uint32_t*>(p.ws + p.done_off);
    uint32_t* counters = reinterpret_cast<uint32_t*>(p.ws + p.counters_off);
    for (int k = threadIdx.x; k < p.n_prods; k += blockDim.x) done[k] = 0u;
    for (int k = threadIdx.x; k < p.max_tiles; k += blockDim.x) counters[k] = 0u;
    if (threadIdx.x < 2) reinterpret_cast<uint32_t*>(p.ws)[threadIdx.x] = 0u;
  }
}

}  // namespace

// ---- host: the program of a stack -------------------------------------------

struct StepProgram {
  int N, hidden, G, n_prods, n_mats, max_tiles;
  float eps;
  void* dev;               // [StepProduct x n_prods][StepMat x n_mats]
  StepProduct* d_prods;
  StepMat* d_mats;
  long long r_off, done_off, counters_off, partials_off, lo_off, stats0_off, slab_stride;
  size_t ws_bytes;
  int smem;
};

namespace {

size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

int step_smem() { return kStages * kStageBytes + kXBytes + (int)sizeof(StepTail) + 1024; }

bool qualifies(const bws_matrix& m, int d_in) {
  if (m.d_in != d_in || m.d_out < 1 || !m.codes || ((uintptr_t)m.codes & 15)) return false;
  if (m.format == BWS_FMT_NVFP4) return d_in % 256 == 0 && m.scales && !((uintptr_t)m.scales & 15) && m.scale32;
  if (m.format == BWS_FMT_FP8_ROW) return d_in % 128 == 0 && m.scale32;
  return false;
}

}  // namespace

StepProgram* step_program_create(int N, int hidden, float eps, const bws_layer* layers, int n_layers,
                                 const bws_matrix& head) {
  if (N < 1 || N > kMaxTokens || hidden % 128 != 0 || !tensor_maps_available()) return nullptr;
  int dev = 0, sms = 0, nb = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
  int coop = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return nullptr;
  const int smem = step_smem();
  if (cudaFuncSetAttribute(step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, step_kernel, kStepThreads, smem) != cudaSuccess || nb < 1) {
    cudaGetLastError();
    return nullptr;
  }
  const int G = (nb > 2 ? 2 : nb) * sms;

  // matrices and products
  std::vector<StepMat> mats;
  std::vector<StepProduct> prods;
  std::vector<int> prod_outputs;   // for validation only
  long long max_u = 8, max_inter = 8;
  bool ok = true;
  auto add_mats = [&](const bws_matrix* ms, int n, int epi, int d_in) -> int {
    const int first = (int)mats.size();
    int tile = 0, row = 0;
    for (int i = 0; i < n; ++i) {
      if (!qualifies(ms[i], d_in) || ms[i].format != ms[0].format) { ok = false; return first; }
      StepMat m;
      memset(&m, 0, sizeof(m));
      const bool fp8 = ms[i].format == BWS_FMT_FP8_ROW;
      const uint64_t row_bytes = fp8 ? (uint64_t)d_in : (uint64_t)d_in / 2;
      if (!encode_2d(&m.codes, ms[i].codes, row_bytes, (uint64_t)ms[i].d_out, 128, kBoxRows, true)) ok = false;
      if (!fp8 && !encode_2d(&m.scales, ms[i].scales, (uint64_t)d_in / 16, (uint64_t)ms[i].d_out, 16, kBoxRows, false))
        ok = false;
      m.scale32 = ms[i].scale32;
      m.d_out = ms[i].d_out;
      m.out_row_off = epi == kEpiSwiGLU ? 0 : row;
      m.tile_begin = tile;
      row += ms[i].d_out;
      tile += (ms[i].d_out + 127) / 128;
      mats.push_back(m);
    }
    return first;
  };
  // workspace offsets are filled in below; products refer to them by role
  enum Role { kRoleR, kRoleU, kRoleH, kRoleLogits, kRoleStats0, kRoleStatsP };
  struct Pending { int role_x, role_out; };
  std::vector<Pending> roles;
  auto add_prod = [&](const bws_matrix* ms, int n, int epi, int d_in, int src, int role_x, int role_out) {
    StepProduct P;
    memset(&P, 0, sizeof(P));
    P.mat0 = add_mats(ms, n, epi, d_in);
    if (!ok) return;
    P.fmt = ms[0].format == BWS_FMT_FP8_ROW ? kFmtFP8 : kFmtNVFP4;
    P.epi = epi;
    P.n_mats = n;
    P.d_in = d_in;
    const int UK = P.fmt == kFmtFP8 ? 128 : 256;
    P.nks = d_in / UK;
    int tiles = 0;
    if (epi == kEpiSwiGLU) {
      tiles = (ms[0].d_out + 63) / 64;
    } else {
      for (int i = 0; i < n; ++i) tiles += (ms[i].d_out + 127) / 128;
    }
    P.n_tiles = tiles;
    const int xblk = UK * 2 + 16;
    const int max_units = kXBytes / (N * xblk);
    int S = (P.nks + max_units - 1) / max_units;
    if (S < 1) S = 1;
    if (S > G || S > P.nks) { ok = false; return; }
    P.n_slabs = S;
    P.src = src;
    int out_w = 0;
    for (int i = 0; i < n; ++i) out_w += ms[i].d_out;
    P.out_ld = role_out == kRoleR ? hidden : (epi == kEpiSwiGLU ? ms[0].d_out : out_w);
    prods.push_back(P);
    roles.push_back({role_x, role_out});
  };
  for (int li = 0; li < n_layers && ok; ++li) {
    const bws_layer& L = layers[li];
    if (L.kind == BWS_LAYER_MIXER_MLP) {
      if (L.n_mixer_in < 1 || L.n_mixer_in > kMaxMats) { ok = false; break; }
      int sum_out = 0;
      for (int i = 0; i < L.n_mixer_in; ++i) sum_out += L.mixer_in[i].d_out;
      // BF16 rows of u and h are read in 16-byte pieces
      if (L.mixer_out.d_in > sum_out || L.mixer_out.d_out != hidden || sum_out % 8) { ok = false; break; }
      max_u = sum_out > max_u ? sum_out : max_u;
      add_prod(L.mixer_in, L.n_mixer_in, kEpiStoreBF16, hidden, kSrcNorm, kRoleR, kRoleU);
      add_prod(&L.mixer_out, 1, kEpiResidF32, L.mixer_out.d_in, kSrcBF16, kRoleU, kRoleR);
    } else if (L.kind != BWS_LAYER_MLP) {
      ok = false;
      break;
    }
    if (!ok) break;
    if (L.up.d_out != L.gate.d_out || L.down.d_out != hidden || L.down.d_in != L.gate.d_out || L.gate.d_out % 8) {
      ok = false;
      break;
    }
    const bws_matrix gu[2] = {L.gate, L.up};
    max_inter = L.gate.d_out > max_inter ? L.gate.d_out : max_inter;
    add_prod(gu, 2, kEpiSwiGLU, hidden, kSrcNorm, kRoleR, kRoleH);
    add_prod(&L.down, 1, kEpiResidF32, L.down.d_in, kSrcBF16, kRoleH, kRoleR);
  }
  if (ok) add_prod(&head, 1, kEpiStoreF32, hidden, kSrcNorm, kRoleR, kRoleLogits);
  if (!ok || prods.empty()) return nullptr;

  // workspace: [status 256][r][u][h][stats0][stats per residual product][done][counters][partials][lo]
  StepProgram* S = new (std::nothrow) StepProgram();
  if (!S) return nullptr;
  S->N = N;
  S->hidden = hidden;
  S->eps = eps;
  S->G = G;
  S->smem = smem;
  size_t o = 256;
  S->r_off = (long long)o; o += al256(sizeof(float) * (size_t)N * hidden);
  const long long u_off = (long long)o; o += al256(2 * (size_t)N * max_u);
  const long long h_off = (long long)o; o += al256(2 * (size_t)N * max_inter);
  const int t0 = hidden / kStatRows;
  S->stats0_off = (long long)o; o += al256(sizeof(float2) * (size_t)t0 * N);
  long long resid_stats = S->stats0_off;   // statistics of the current residual
  int resid_tiles = t0;
  int max_tiles = 1;
  long long stride = 1;
  size_t partial_slabs = 1;
  for (size_t i = 0; i < prods.size(); ++i) {
    StepProduct& P = prods[i];
    const Pending& R = roles[i];
    if (R.role_x == kRoleR) {
      P.stats_off = resid_stats;
      P.stats_tiles = resid_tiles;
    } else {
      P.x_off = R.role_x == kRoleU ? u_off : h_off;
      P.x_ld = prods[i - 1].out_ld;
      P.stats_off = prods[i - 1].stats_out_off;
      P.stats_tiles = prods[i - 1].n_tiles;
    }
    if (R.role_out != kRoleLogits) {
      P.stats_out_off = (long long)o;
      o += al256(sizeof(float2) * (size_t)P.n_tiles * N);
    }
    if (R.role_out == kRoleR) {
      P.out_off = S->r_off;
      resid_stats = P.stats_out_off;
      resid_tiles = P.n_tiles;
      if (P.n_tiles * 128 < hidden) { delete S; return nullptr; }
    } else if (R.role_out == kRoleU) {
      P.out_off = u_off;
    } else if (R.role_out == kRoleH) {
      P.out_off = h_off;
    } else {
      P.out_off = -1;
    }
    max_tiles = P.n_tiles > max_tiles ? P.n_tiles : max_tiles;
    const long long gs = (G + P.n_slabs - 1) / P.n_slabs;
    stride = P.n_tiles + gs > stride ? P.n_tiles + gs : stride;
    partial_slabs = (size_t)P.n_slabs > partial_slabs ? (size_t)P.n_slabs : partial_slabs;
  }
  S->slab_stride = stride;
  S->max_tiles = max_tiles;
  S->n_prods = (int)prods.size();
  S->n_mats = (int)mats.size();
  S->done_off = (long long)o; o += al256(sizeof(uint32_t) * (size_t)S->n_prods);
  S->counters_off = (long long)o; o += al256(sizeof(uint32_t) * (size_t)max_tiles);
  S->partials_off = (long long)o; o += al256((size_t)partial_slabs * stride * kSlotF4 * sizeof(float4));
  S->lo_off = (long long)o; o += al256((size_t)G * kXBytes);
  S->ws_bytes = o;

  // device tables
  const size_t pb = al256(sizeof(StepProduct) * prods.size());
  const size_t mb = sizeof(StepMat) * mats.size();
  if (cudaMalloc(&S->dev, pb + mb) != cudaSuccess) {
    cudaGetLastError();
    delete S;
    return nullptr;
  }
  S->d_prods = static_cast<StepProduct*>(S->dev);
  S->d_mats = reinterpret_cast<StepMat*>(static_cast<char*>(S->dev) + pb);
  if (cudaMemcpy(S->d_prods, prods.data(), sizeof(StepProduct) * prods.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(S->d_mats, mats.data(), mb, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(S->dev);
    delete S;
    return nullptr;
  }
  return S;
}

void step_program_destroy(StepProgram* S) {
  if (!S) return;
  if (S->dev) cudaFree(S->dev);
  delete S;
}

size_t step_program_workspace(const StepProgram* S) { return S ? S->ws_bytes : 0; }

int step_program_grid(const StepProgram* S) { return S ? S->G : 0; }

cudaError_t step_program_enqueue(const StepProgram* S, const uint16_t* x0, float* logits, void* ws, cudaStream_t st) {
  StepParams p;
  memset(&p, 0, sizeof(p));
  p.prods = S->d_prods;
  p.mats = S->d_mats;
  p.n_prods = S->n_prods;
  p.N = S->N;
  p.hidden = S->hidden;
  p.G = S->G;
  p.eps = S->eps;
  p.ws = static_cast<char*>(ws);
  p.logits = logits;
  p.x0 = x0;
  p.r_off = S->r_off;
  p.done_off = S->done_off;
  p.counters_off = S->counters_off;
  p.partials_off = S->partials_off;
  p.lo_off = S->lo_off;
  p.stats0_off = S->stats0_off;
  p.slab_stride = S->slab_stride;
  p.max_tiles = S->max_tiles;
  step_init_kernel<<<dim3(S->hidden / kStatRows, S->N), 128, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)S->G);
  cfg.blockDim = dim3(kStepThreads);
  cfg.dynamicSmemBytes = (size_t)S->smem;
  cfg.stream = st;
  cudaLaunchAttribute a[2];
  a[0].id = cudaLaunchAttributeCooperative;
  a[0].val.cooperative = 1;
  a[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, step_kernel, p);
}

}  // namespace bws
