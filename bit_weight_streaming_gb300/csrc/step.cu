// Persistent decode-step kernel for dense layer stacks (NVFP4 layers, NVFP4
// or FP8 output layer): one cooperative launch runs every product of the step.
//
// Why one kernel. A decode step is a chain of a few hundred weight-stream
// products, each needing the whole output of the one before ([Spark27B]
// "Decode speed is bytes divided by bandwidth": every weight is read once per
// step, in layer order). As separate launches each product pays the ramp of
// filling the memory pipeline, the drain at its end and a kernel boundary for
// the activation prep. Here every CTA stays resident: its producer warp
// streams the weight units of all its products, in order, into a ring of
// shared-memory stages and never waits for activations (weights never depend
// on them), so the stream runs on across product boundaries while the
// consumer warps wait for their inputs.
//
// One CTA per SM (the unit loop needs more registers than two CTAs of
// 288 threads leave it) with a deep ring. The producer issues one 128-row
// box of codes and one of scales per unit, from fields of the current
// product it keeps in registers, and may be limited to `inflight` units of
// copies in flight: fewer copies in flight keep the memory queues short for
// the dependent loads of a product boundary, at the cost of streaming rate.
//
// Work of one product. Its d_in is cut into S k-slabs of whole units (S is
// chosen so that the activations a CTA needs fit its shared-memory slab); the
// CTAs are dealt to the slabs in equal contiguous groups and within a slab the
// (tile, k-unit) pairs, tile-major, to the group's CTAs in contiguous ranges
// (stream-K). A CTA builds, in shared memory, the f16 bands of just the
// k-units its range touches.
//
// Hand-off without a fix-up. Every tile piece a CTA computes is deposited as
// raw FP32 sums in true units (before the matrix scale) in a slot of its own,
// followed by a release count on the tile. Nothing waits at the end of a
// product. The next product's CTAs read what they need:
//   * a copy input (the BF16 outputs of a mixer input projection, or the
//     SwiGLU activations of the gate/up product) is finished by every CTA
//     that reads it, from the deposits of the tiles covering its k-units:
//     the tile's slots added in a fixed (slab, CTA) order, scaled, rounded to
//     BF16; the CTA's own exponent of its slab sets the f16 bands;
//   * a normalised input BF16(RMSNorm(r)) needs the whole row's sum of
//     squares: one designated CTA per tile of the residual update finishes
//     its 128 rows (r += y, written to the other of two residual buffers)
//     and their statistics, then counts the tile done; every CTA waits for
//     all tiles' statistics and reads its slab of the new residual.
// Deposits go to a ring of four buffers; a product reuses a buffer only after
// every CTA has read the inputs of the product three before it, and a
// residual buffer is overwritten only after every CTA has read the input it
// held. The output layer's tiles are finished at the end by one warp each.
// Every wait is bounded and sets a status bit instead of hanging; all
// counters are zeroed by the step's init kernel.
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
constexpr int kMaxStages = 12;
#ifndef BWS_STEP_CTAS
#define BWS_STEP_CTAS 1
#endif
constexpr int kCtasPerSm = BWS_STEP_CTAS;              // CTAs per SM
constexpr int kStageBytes = kCodeBytes + kBoxes * kScaleBoxBytes;   // one NVFP4 unit, 18 KiB
constexpr uint32_t kStatusTimeout = 0x100u;
constexpr int kStatRows = 128;                          // rows per statistics tile of x0
constexpr int kPBufs = 4;                               // ring of deposit buffers
constexpr int kMaxPieces = 96;                          // deposits a tile may collect

constexpr int kInNorm = 0;    // the product reads BF16(RMSNorm(r))
constexpr int kInCopy = 1;    // the product reads the previous product's outputs

struct StepMat {   // 64-byte aligned through CUtensorMap
  CUtensorMap codes;     // u8 [d_out][row bytes], box {128, 32}, 128B swizzle
  CUtensorMap scales;    // NVFP4: u8 [d_out][d_in/16], box {16, 32}
  const float* scale32;  // NVFP4 tensor scale [1]; FP8 row scales [d_out]
  int d_out, out_row_off, tile_begin;
};

struct StepProduct {
  int fmt, epi, n_mats, mat0;
  int d_in, nks, n_tiles, n_slabs;
  int in_kind;     // kInNorm / kInCopy
  int in_prod;     // kInCopy: the product whose outputs are the input; kInNorm: the residual
                   // update whose result is normalised (-1: x0)
  int r_in;        // kInNorm: the residual buffer read
  int r_src, r_dst;   // residual updates: buffer read and buffer written by the finishing
  int r_guard;     // residual updates: product whose input r_dst held (-1: none)
  int pbuf;        // deposit buffer (kPBufs: the output layer's own)
  int cnt_off;     // first of this product's tile counters
  int out_ld;      // the output layer: logits row length
  long long stats_off;   // residual updates: [n_tiles][N] (sum of squares, max |r|) of the new r
};

struct StepParams {
  CUtensorMap head_codes, head_scales;   // the output layer's maps (kernel parameters)
  const StepProduct* prods;
  const StepMat* mats;
  int n_prods, N, hidden, G;
  float eps;
  char* ws;
  float* logits;
  const uint16_t* x0;
  long long r_off[2];
  long long stats0_off;                  // [hidden / 128][N] statistics of x0
  long long cnt_off, stats_cnt_off, read_done_off;   // uint32 counter arrays
  int n_zero_words;                      // counters zeroed by the init kernel (from cnt_off on)
  long long pbuf_off[kPBufs + 1];
  long long slab_stride;                 // deposit slots per slab
  long long lo_off;                      // per-CTA lo-band scratch, x_bytes each
  int n_stages, x_bytes, inflight;
  uint32_t max_polls;
  long long trace_off;                   // >= 0: per (CTA, product) timestamps [G][n_prods][4] (measurement aid)
};

// Shared memory after the ring and the activation slab.
struct StepTail {
  uint4 zero_x[33];            // zeros read by the one-token block-diagonal operand (from element 1 on)
  float4 red[kBoxes][2][32];   // half-pair reduction (box, sub-tile, lane)
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  float inv_rms[kMaxTokens];
  int E[kMaxTokens];
  float hs[kMaxTokens];        // 2^(14 - E) when a normal float, else 0
  float wpart[kSW][kMaxTokens][2];   // per-warp (sum, max) of a reduction
  int pieces[kMaxPieces];      // deposit slots of the tile being finished
  int n_pieces;
  uint32_t xflags;
  uint32_t dead;
};

// ---- positions ------------------------------------------------------------

__host__ __device__ inline long long owner_of(long long u, long long U, long long G) { return ((u + 1) * G - 1) / U; }

// Where CTA c works in a product of T tiles of K k-units cut into S slabs:
// slab s (its k-units [k0, k0 + nk)), local index l in the slab's group of
// gs working CTAs, its units [u0, u1) of the slab, and the k-units its range
// touches: cnt of them from kl0 on (mod nk).
struct SlabPos {
  int s, k0, nk, l, gs;
  long long units, u0, u1;
  int kl0, cnt;
};

__host__ __device__ inline SlabPos slab_pos(int T, int K, int S, int c, int G) {
  SlabPos q;
  q.s = (int)owner_of(c, G, S);
  const int c0 = (int)((long long)q.s * G / S), c1 = (int)((long long)(q.s + 1) * G / S);
  q.l = c - c0;
  q.k0 = (int)((long long)q.s * K / S);
  q.nk = (int)((long long)(q.s + 1) * K / S) - q.k0;
  q.units = (long long)T * q.nk;
  // a slab with fewer units than CTAs uses only as many CTAs as it has units
  q.gs = (long long)(c1 - c0) < q.units ? c1 - c0 : (int)q.units;
  if (q.l < q.gs) {
    q.u0 = q.l * q.units / q.gs;
    q.u1 = (q.l + 1) * q.units / q.gs;
  } else {
    q.u0 = q.u1 = 0;
  }
  if (q.u1 - q.u0 >= q.nk) {
    q.kl0 = 0;
    q.cnt = q.nk;
  } else {
    q.kl0 = (int)(q.u0 % q.nk);
    q.cnt = (int)(q.u1 - q.u0);
  }
  return q;
}

// The deposit slots of tile t, in the order they are added: slabs in order,
// each slab's CTAs in order. Returns their number (at most cap written).
__host__ __device__ inline int tile_slots(int T, int K, int S, int G, long long stride, int t, int* out, int cap) {
  int n = 0;
  for (int s = 0; s < S; ++s) {
    const SlabPos q = slab_pos(T, K, S, (int)((long long)s * G / S), G);
    const int l0 = (int)owner_of((long long)t * q.nk, q.units, q.gs);
    const int l1 = (int)owner_of((long long)t * q.nk + q.nk - 1, q.units, q.gs);
    for (int l = l0; l <= l1; ++l) {
      if (n < cap && out) out[n] = (int)(s * stride + t + l);
      ++n;
    }
  }
  return n;
}

// ---- small device helpers -------------------------------------------------

BWS_DEV float bf16_to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }

BWS_DEV uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
BWS_DEV void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
BWS_DEV uint4 ld_cg_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
BWS_DEV float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
BWS_DEV float2 ld_cg_f2(const float2* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}

// Polls *f until it reaches target (acquire); false after max_polls reads.
BWS_DEV bool poll_ge(const uint32_t* f, uint32_t target, uint32_t max_polls) {
  for (uint32_t i = 0; i < max_polls; ++i) {
    if (ld_acquire_u32(f) >= target) return true;
    if (i > 32) __nanosleep(64);
  }
  return false;
}

BWS_DEV uint32_t* status_of(const StepParams& p) { return reinterpret_cast<uint32_t*>(p.ws) + 1; }

// Optional trace: the global timer's low word at four points of a product
// (start, residual share finished, slab built, units done), per CTA.
BWS_DEV void trace(const StepParams& p, int pi, int k) {
  if (p.trace_off < 0) return;
  uint32_t t;
  asm volatile("mov.u32 %0, %%globaltimer_lo;" : "=r"(t));
  reinterpret_cast<uint32_t*>(p.ws + p.trace_off)[((size_t)blockIdx.x * p.n_prods + pi) * 4 + k] = t;
}
BWS_DEV uint32_t* counters(const StepParams& p) { return reinterpret_cast<uint32_t*>(p.ws + p.cnt_off); }
BWS_DEV uint32_t* stats_cnt(const StepParams& p) { return reinterpret_cast<uint32_t*>(p.ws + p.stats_cnt_off); }
BWS_DEV uint32_t* read_done(const StepParams& p) { return reinterpret_cast<uint32_t*>(p.ws + p.read_done_off); }
BWS_DEV float* pbuf_of(const StepParams& p, int b) { return reinterpret_cast<float*>(p.ws + p.pbuf_off[b]); }

// Consumer thread 0 waits for *f >= target, then every consumer thread
// continues (named barrier 4). After a wait has run out, nothing is waited
// for any more.
BWS_DEV void consumers_wait(const StepParams& p, StepTail& T, const uint32_t* f, uint32_t target, int tid) {
  if (tid == 0 && !T.dead && !poll_ge(f, target, p.max_polls)) {
    atomicOr(status_of(p), kStatusTimeout);
    T.dead = 1u;
  }
  named_bar_sync(4, kConsumerThreads);
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

// Output row j of product P: its tile, row within the tile and matrix.
BWS_DEV void row_tile(const StepParams& p, const StepProduct& P, int j, int& tile, int& rit, int& m) {
  if (P.epi == kEpiSwiGLU) {
    tile = j >> 6;
    rit = j & 63;
    m = P.mat0;
    return;
  }
  int mi = 0;
  for (int i = 1; i < P.n_mats; ++i)
    if (j >= __ldg(&p.mats[P.mat0 + i].out_row_off)) mi = i;
  m = P.mat0 + mi;
  const int lr = j - __ldg(&p.mats[m].out_row_off);
  tile = __ldg(&p.mats[m].tile_begin) + (lr >> 7);
  rit = lr & 127;
}

BWS_DEV int pieces_of(const StepParams& p, const StepProduct& P, int t) {
  return tile_slots(P.n_tiles, P.nks, P.n_slabs, p.G, p.slab_stride, t, nullptr, 0);
}

// ---- f16 bands ---------------------------------------------------------------

// f16 hi band of 8 BF16 values (bit patterns w) with exponent E (scale hs =
// 2^(14 - E) when that is a normal float, else the exact slow path); flags:
// bit 0 an element needs the lo band, bit 1 an element is below both.
BWS_DEV uint4 band_hi(const uint32_t (&w)[4], float hs, int E, uint32_t& flags) {
  uint32_t h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float f0 = __uint_as_float(w[j] << 16), f1 = __uint_as_float(w[j] & 0xFFFF0000u);
    float a0 = hs != 0.0f ? __fmul_rn(f0, hs) : ldexp_exact(f0, 14 - E);
    float a1 = hs != 0.0f ? __fmul_rn(f1, hs) : ldexp_exact(f1, 14 - E);
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
BWS_DEV uint4 band_lo(const uint32_t (&w)[4], int E) {
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
BWS_DEV uint32_t pack_bf16x2(float a, float b) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// Byte offset in the slab of 8-value piece i of the CTA's slab activations
// (token n, k-unit position v, piece kl8 of the unit): unit blocks of xblk
// bytes per (position, token); within a unit, the piece of lane chunk
// kl8 / lk sits at (kl8 / lk) * 16 + (kl8 % lk) * 128 (the layout the MMA
// lanes read).
struct SlabGeo {
  int N, UK, u8, lk, xblk, cnt, per_tok;
};
BWS_DEV SlabGeo slab_geo(const StepProduct& P, const SlabPos& pos, int N) {
  SlabGeo g;
  g.N = N;
  g.UK = P.fmt == kFmtFP8 ? 128 : 256;
  g.u8 = g.UK / 8;
  g.lk = g.UK / 64;
  g.xblk = g.UK * 2 + 16;
  g.cnt = pos.cnt;
  g.per_tok = pos.cnt * g.u8;
  return g;
}
// piece i -> token n, global k of its first value, byte offset in the slab
BWS_DEV void slab_piece(const SlabGeo& g, const SlabPos& pos, int i, int& n, int& k, int& off) {
  n = i / g.per_tok;
  const int r = i - n * g.per_tok;
  const int v = r / g.u8, kl8 = r - v * g.u8;
  int kl = pos.kl0 + v;
  if (kl >= pos.nk) kl -= pos.nk;
  k = (pos.k0 + kl) * g.UK + kl8 * 8;
  off = (v * g.N + n) * g.xblk + (kl8 / g.lk) * 16 + (kl8 % g.lk) * 128;
}

// ---- inputs ------------------------------------------------------------------

// Per-token exponent E and hi-band scale from the largest magnitude amax.
BWS_DEV void set_exponent(StepTail& T, int n, float amax) {
  const int E = amax > 0.0f ? floor_log2_abs(amax) : 0;
  T.E[n] = E;
  T.hs[n] = (14 - E >= -126 && 14 - E <= 127) ? exp2i(14 - E) : 0.0f;
}

// The lo band of the whole slab (rare: some element below the hi band's
// range) into the CTA's global scratch, same layout; reads the BF16 values
// back with get(i, w).
template <typename Get>
BWS_DEV void slab_lo(const SlabGeo& g, const SlabPos& pos, StepTail& T, uint8_t* lo_glob, int tid, Get get) {
  const int total = g.N * g.per_tok;
  for (int i = tid; i < total; i += kConsumerThreads) {
    int n, k, off;
    slab_piece(g, pos, i, n, k, off);
    uint32_t w[4];
    get(i, n, k, w);
    *reinterpret_cast<uint4*>(lo_glob + off) = band_lo(w, T.E[n]);
  }
  __threadfence_block();
}

// The slab of a normalised input: BF16(r * inv_rms) of the k-units the
// CTA's range touches, as f16 bands. The per-token RMSNorm scale and band
// exponent come from the statistics of the residual update (for RMSNorm,
// max |BF16(r s)| = BF16(max |r| s), rounding being monotone). Returns the
// band flags.
__device__ __noinline__ uint32_t build_norm(const StepParams& p, const StepProduct& P, const SlabPos& pos,
                                            StepTail& T, uint8_t* xs, uint8_t* lo_glob, int tid) {
  const int N = p.N;
  const int q = P.in_prod;
  const float2* st;
  int tiles;
  if (q >= 0) {
    const StepProduct& Q = p.prods[q];
    consumers_wait(p, T, stats_cnt(p) + q, (uint32_t)Q.n_tiles, tid);
    st = reinterpret_cast<const float2*>(p.ws + Q.stats_off);
    tiles = Q.n_tiles;
  } else {
    st = reinterpret_cast<const float2*>(p.ws + p.stats0_off);
    tiles = p.hidden / kStatRows;
  }
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < N) {
    float sq = 0.0f, mx = 0.0f;
    for (int t = lane; t < tiles; t += 32) {
      const float2 v = ld_cg_f2(st + (size_t)t * N + warp);
      sq = __fadd_rn(sq, v.x);
      mx = fmaxf(mx, v.y);
    }
    sq = warp_sum(sq);
    mx = warp_max(mx);
    if (lane == 0) {
      const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sq, (float)p.hidden), p.eps)));
      T.inv_rms[warp] = inv;
      set_exponent(T, warp, __bfloat162float(__float2bfloat16_rn(__fmul_rn(mx, inv))));
    }
  }
  if (tid == 0) T.xflags = 0u;
  named_bar_sync(4, kConsumerThreads);
  const SlabGeo g = slab_geo(P, pos, N);
  const float* r = reinterpret_cast<const float*>(p.ws + p.r_off[P.r_in]);
  auto get = [&](int, int n, int k, uint32_t (&w)[4]) {
    const float* x = r + (size_t)n * p.hidden + k;
    const uint4 a = ld_cg_u4(x), b = ld_cg_u4(x + 4);
    const float inv = T.inv_rms[n];
    w[0] = pack_bf16x2(__fmul_rn(__uint_as_float(a.x), inv), __fmul_rn(__uint_as_float(a.y), inv));
    w[1] = pack_bf16x2(__fmul_rn(__uint_as_float(a.z), inv), __fmul_rn(__uint_as_float(a.w), inv));
    w[2] = pack_bf16x2(__fmul_rn(__uint_as_float(b.x), inv), __fmul_rn(__uint_as_float(b.y), inv));
    w[3] = pack_bf16x2(__fmul_rn(__uint_as_float(b.z), inv), __fmul_rn(__uint_as_float(b.w), inv));
  };
  const int total = N * g.per_tok;
  uint32_t flags = 0u;
  constexpr int kB = 4;   // pieces in flight per thread
  for (int i0 = tid; i0 < total; i0 += kB * kConsumerThreads) {
    uint4 ra[kB], rb[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int i = i0 + b * kConsumerThreads;
      if (i < total) {
        int n, k, off;
        slab_piece(g, pos, i, n, k, off);
        const float* x = r + (size_t)n * p.hidden + k;
        ra[b] = ld_cg_u4(x);
        rb[b] = ld_cg_u4(x + 4);
      }
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int i = i0 + b * kConsumerThreads;
      if (i >= total) break;
      int n, k, off;
      slab_piece(g, pos, i, n, k, off);
      const float inv = T.inv_rms[n];
      uint32_t w[4];
      w[0] = pack_bf16x2(__fmul_rn(__uint_as_float(ra[b].x), inv), __fmul_rn(__uint_as_float(ra[b].y), inv));
      w[1] = pack_bf16x2(__fmul_rn(__uint_as_float(ra[b].z), inv), __fmul_rn(__uint_as_float(ra[b].w), inv));
      w[2] = pack_bf16x2(__fmul_rn(__uint_as_float(rb[b].x), inv), __fmul_rn(__uint_as_float(rb[b].y), inv));
      w[3] = pack_bf16x2(__fmul_rn(__uint_as_float(rb[b].z), inv), __fmul_rn(__uint_as_float(rb[b].w), inv));
      *reinterpret_cast<uint4*>(xs + off) = band_hi(w, T.hs[n], T.E[n], flags);
    }
  }
  if (flags) atomicOr(&T.xflags, flags);
  named_bar_sync(4, kConsumerThreads);
  const uint32_t fl = T.xflags;
  if (fl & 1u) {
    slab_lo(g, pos, T, lo_glob, tid, get);
    named_bar_sync(4, kConsumerThreads);
  }
  return fl;
}

// Values j .. j+7 (one 8-row chunk of a tile) of token n of product Q's
// outputs, finished from its deposits: the tile's slots added in order, the
// matrix scale, and for SwiGLU SiLU(gate) * up; returned as BF16 bits.
BWS_DEV void finish_chunk(const StepParams& p, const StepProduct& Q, int n, int j, uint32_t (&w)[4]) {
  int tile, rit, m;
  row_tile(p, Q, j, tile, rit, m);
  const bool swi = Q.epi == kEpiSwiGLU;
  const float* buf = pbuf_of(p, Q.pbuf);
  float a[8], u[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = u[i] = 0.0f;
  const int N = p.N;
  for (int s = 0; s < Q.n_slabs; ++s) {
    const SlabPos q = slab_pos(Q.n_tiles, Q.nks, Q.n_slabs, (int)((long long)s * p.G / Q.n_slabs), p.G);
    const int l0 = (int)owner_of((long long)tile * q.nk, q.units, q.gs);
    const int l1 = (int)owner_of((long long)tile * q.nk + q.nk - 1, q.units, q.gs);
    constexpr int kB = 2;
    for (int lb = l0; lb <= l1; lb += kB) {
      float4 o[kB][4];
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        if (lb + b <= l1) {
          const float* slot = buf + ((size_t)(s * p.slab_stride + tile + lb + b) * N + n) * 128 + rit;
          o[b][0] = ld_cg_f4(reinterpret_cast<const float4*>(slot));
          o[b][1] = ld_cg_f4(reinterpret_cast<const float4*>(slot) + 1);
          if (swi) {
            o[b][2] = ld_cg_f4(reinterpret_cast<const float4*>(slot + 64));
            o[b][3] = ld_cg_f4(reinterpret_cast<const float4*>(slot + 64) + 1);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        if (lb + b > l1) break;
        a[0] += o[b][0].x; a[1] += o[b][0].y; a[2] += o[b][0].z; a[3] += o[b][0].w;
        a[4] += o[b][1].x; a[5] += o[b][1].y; a[6] += o[b][1].z; a[7] += o[b][1].w;
        if (swi) {
          u[0] += o[b][2].x; u[1] += o[b][2].y; u[2] += o[b][2].z; u[3] += o[b][2].w;
          u[4] += o[b][3].x; u[5] += o[b][3].y; u[6] += o[b][3].z; u[7] += o[b][3].w;
        }
      }
    }
  }
  float v[8];
  if (swi) {
    const float sg = __ldg(p.mats[Q.mat0].scale32), su = __ldg(p.mats[Q.mat0 + 1].scale32);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = silu_mul_t(__fmul_rn(a[i], sg), __fmul_rn(u[i], su));
  } else if (Q.fmt == kFmtFP8) {
    const float* rs = p.mats[m].scale32 + (j - __ldg(&p.mats[m].out_row_off));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(a[i], __ldg(rs + i));
  } else {
    const float ts = __ldg(p.mats[m].scale32);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(a[i], ts);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

// The slab of a copy input (the previous product's outputs), finished from
// that product's deposits: wait for the tiles covering the CTA's k-units,
// finish each 8-value chunk into the slab as BF16 (first pass, with the
// per-token largest magnitude), then turn the slab into f16 bands in place
// with the CTA's own per-token exponent (second pass). Returns the flags.
__device__ __noinline__ uint32_t build_copy(const StepParams& p, const StepProduct& P, const SlabPos& pos,
                                            StepTail& T, uint8_t* xs, uint8_t* lo_glob, int tid) {
  const int N = p.N;
  const StepProduct& Q = p.prods[P.in_prod];
  const SlabGeo g = slab_geo(P, pos, N);
  const int rpt = Q.epi == kEpiSwiGLU ? 64 : 128;   // rows per tile of Q
  const int tpu = g.UK / rpt;                      // Q tiles per k-unit
  // one thread per covered tile waits for its deposits
  bool ok = true;
  if (tid < g.cnt * tpu && !T.dead) {
    const int v = tid / tpu, sub = tid - v * tpu;
    int kl = pos.kl0 + v;
    if (kl >= pos.nk) kl -= pos.nk;
    int tile, rit, m;
    row_tile(p, Q, (pos.k0 + kl) * g.UK + sub * rpt, tile, rit, m);
    ok = poll_ge(counters(p) + Q.cnt_off + tile, (uint32_t)pieces_of(p, Q, tile), p.max_polls);
  }
  if (!ok) {
    atomicOr(status_of(p), kStatusTimeout);
    T.dead = 1u;
  }
  if (tid == 0) T.xflags = 0u;
  named_bar_sync(4, kConsumerThreads);
  // pass 1: finish the chunks, BF16 into the slab; per-token maxima
  const int total = N * g.per_tok;
  float mx[kMaxTokens];
#pragma unroll
  for (int n = 0; n < kMaxTokens; ++n) mx[n] = 0.0f;
  if (!T.dead) {
    for (int i = tid; i < total; i += kConsumerThreads) {
      int n, k, off;
      slab_piece(g, pos, i, n, k, off);
      uint32_t w[4];
      finish_chunk(p, Q, n, k, w);
      *reinterpret_cast<uint4*>(xs + off) = make_uint4(w[0], w[1], w[2], w[3]);
      float m8 = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) m8 = fmaxf(m8, fmaxf(fabsf(bf16_to_f32(w[e] & 0xFFFF)), fabsf(bf16_to_f32(w[e] >> 16))));
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t)
        if (t == n) mx[t] = fmaxf(mx[t], m8);
    }
  }
  const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int n = 0; n < kMaxTokens; ++n) {
    const float m = warp_max(mx[n]);
    if (lane == 0) T.wpart[warp][n][1] = m;
  }
  named_bar_sync(4, kConsumerThreads);
  if (tid < N) {
    float m = 0.0f;
    for (int w2 = 0; w2 < kSW; ++w2) m = fmaxf(m, T.wpart[w2][tid][1]);
    set_exponent(T, tid, m);
  }
  named_bar_sync(4, kConsumerThreads);
  // pass 2: the bands, in place
  uint32_t flags = 0u;
  for (int i = tid; i < total; i += kConsumerThreads) {
    int n, k, off;
    slab_piece(g, pos, i, n, k, off);
    const uint4 b = *reinterpret_cast<const uint4*>(xs + off);
    const uint32_t w[4] = {b.x, b.y, b.z, b.w};
    *reinterpret_cast<uint4*>(xs + off) = band_hi(w, T.hs[n], T.E[n], flags);
  }
  if (flags) atomicOr(&T.xflags, flags);
  named_bar_sync(4, kConsumerThreads);
  const uint32_t fl = T.xflags;
  if (fl & 1u) {
    // (rare) the lo band: the values are finished again from the deposits
    slab_lo(g, pos, T, lo_glob, tid, [&](int, int n, int k, uint32_t (&w)[4]) { finish_chunk(p, Q, n, k, w); });
    named_bar_sync(4, kConsumerThreads);
  }
  return fl;
}

// The residual update of product q for the tiles this CTA finishes (tile t
// goes to CTA t * G / n_tiles): r_dst = r_src + scale * (the tile's deposits
// added in order), and the tile's per-token sum of squares and largest
// magnitude of the new residual; each tile is then counted in stats_cnt[q].
__device__ __noinline__ void finish_residual(const StepParams& p, int q, StepTail& T, int tid) {
  const StepProduct& Q = p.prods[q];
  const int nt = Q.n_tiles, G = p.G, c = blockIdx.x;
  const int t0 = (int)(((long long)c * nt + G - 1) / G), t1 = (int)(((long long)(c + 1) * nt + G - 1) / G);
  if (t0 >= t1) return;
  const int N = p.N;
  // the buffer written held the input of product r_guard: wait until every CTA has read it
  if (Q.r_guard >= 0) consumers_wait(p, T, read_done(p) + Q.r_guard, (uint32_t)G, tid);
  const float* r_src = reinterpret_cast<const float*>(p.ws + p.r_off[Q.r_src]);
  float* r_dst = reinterpret_cast<float*>(p.ws + p.r_off[Q.r_dst]);
  const float* buf = pbuf_of(p, Q.pbuf);
  float2* stats = reinterpret_cast<float2*>(p.ws + Q.stats_off);
  const int warp = tid >> 5, lane = tid & 31;
  for (int t = t0; t < t1; ++t) {
    if (tid == 0) T.n_pieces = tile_slots(nt, Q.nks, Q.n_slabs, G, p.slab_stride, t, T.pieces, kMaxPieces);
    named_bar_sync(4, kConsumerThreads);
    consumers_wait(p, T, counters(p) + Q.cnt_off + t, (uint32_t)T.n_pieces, tid);
    const int np = T.n_pieces;
    const int m = Q.mat0;   // one output matrix of hidden rows
    const bool fp8 = Q.fmt == kFmtFP8;
    const float ts = fp8 ? 0.0f : __ldg(p.mats[m].scale32);
    float ss[kMaxTokens / 2], mx[kMaxTokens / 2];
#pragma unroll
    for (int i = 0; i < kMaxTokens / 2; ++i) ss[i] = mx[i] = 0.0f;
    if (!T.dead) {
#pragma unroll
      for (int i = 0; i < kMaxTokens / 2; ++i) {
        const int e = tid + i * kConsumerThreads;
        const int n = e >> 7, row = e & 127;
        const int grow = t * 128 + row;
        if (n >= N || grow >= p.hidden) continue;
        float acc = 0.0f;
        constexpr int kB = 8;
        for (int k0 = 0; k0 < np; k0 += kB) {
          float o[kB];
#pragma unroll
          for (int b = 0; b < kB; ++b)
            o[b] = k0 + b < np ? ld_cg_f32(buf + ((size_t)T.pieces[k0 + b] * N + n) * 128 + row) : 0.0f;
#pragma unroll
          for (int b = 0; b < kB; ++b)
            if (k0 + b < np) acc += o[b];
        }
        const float y = __fmul_rn(acc, fp8 ? __ldg(p.mats[m].scale32 + grow) : ts);
        const float nr = __fadd_rn(ld_cg_f32(r_src + (size_t)n * p.hidden + grow), y);
        r_dst[(size_t)n * p.hidden + grow] = nr;
        ss[i] = __fmul_rn(nr, nr);
        mx[i] = fabsf(nr);
      }
    }
    // per token: threads 0..127 hold tokens 0, 2, 4, 6; threads 128..255 tokens 1, 3, 5, 7
#pragma unroll
    for (int i = 0; i < kMaxTokens / 2; ++i) {
      const float s2 = warp_sum(ss[i]), m2 = warp_max(mx[i]);
      if (lane == 0) {
        T.wpart[warp][i][0] = s2;
        T.wpart[warp][i][1] = m2;
      }
    }
    named_bar_sync(4, kConsumerThreads);
    if (tid < N) {
      const int h = tid & 1, i = tid >> 1;
      float s2 = 0.0f, m2 = 0.0f;
      for (int w2 = 4 * h; w2 < 4 * h + 4; ++w2) {
        s2 = __fadd_rn(s2, T.wpart[w2][i][0]);
        m2 = fmaxf(m2, T.wpart[w2][i][1]);
      }
      stats[(size_t)t * N + tid] = make_float2(s2, m2);
    }
    named_bar_sync(4, kConsumerThreads);
    if (tid == 0) red_release_add(stats_cnt(p) + q, 1u);
  }
}

// ---- the unit loop -------------------------------------------------------------

// Deposit of one tile piece by warps 0..3 (v: sums of sub-tiles 0 and 1 of
// box b in band units; register i = row g + 8*(i>>1), token 2t + (i&1), or
// with N1 row g / g + 8 of token 0 in registers 0 / 2 of lanes t == 0), in
// true units, then the tile's release count.
template <bool N1>
BWS_DEV void deposit_piece(const StepParams& p, float* buf, uint32_t* cnt, int slot0, const StepTail& T, int tile,
                           int b, int g, int t, const float (&v)[2][4]) {
  const int N = p.N;
  float* slot = buf + (size_t)(slot0 + tile) * N * 128;
#pragma unroll
  for (int st = 0; st < 2; ++st) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = 32 * b + 16 * st + g + 8 * (i >> 1);
      const int tok = N1 ? 0 : 2 * t + (i & 1);
      if (N1 ? (t == 0 && (i & 1) == 0) : tok < N) slot[tok * 128 + row] = ldexp_exact(v[st][i], T.E[tok] - 14);
    }
  }
  named_bar_sync(2, 4 * 32);
  if (threadIdx.x == 0) red_release_add(cnt + tile, 1u);
}

// The consumer warps' units [u0, u1) of product P (slab position pos); LO:
// the two-band path; N1: one NVFP4 token with the block-diagonal operand.
// The ring position (stage, phase) goes in and comes back packed as
// stage | phase << 16.
template <int FMT, bool LO, bool N1>
BWS_DEV uint32_t step_units(const StepParams& p, float* buf, uint32_t* cnt, int slot0, int u0, int u1, int nk,
                            int kl0, StepTail& T, uint32_t stage0, uint32_t xs0, const uint8_t* lo_glob,
                            uint32_t ring) {
  int s = (int)(ring & 0xFFFFu);
  uint32_t ph = ring >> 16;
  constexpr int kUnitK = FMT == kFmtFP8 ? 128 : 256;
  constexpr int kXv = FMT == kFmtFP8 ? 2 : 4;
  const int N = p.N;
  const int NS = p.n_stages;
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
  const bool m01 = g == 2 * t, m23 = g == 2 * t + 1;
  const uint32_t zaddr = smem_u32(&T.zero_x[1]) + c * 16;
  float acc[2][2][4] = {}, accl[2][4] = {};
  uint4 xh[kXv], xl[kXv];
  int tile = u0 / nk, kl = u0 - tile * nk;
  for (int u = u0; u < u1; ++u) {
    const uint32_t xu = xlane + (uint32_t)(kl >= kl0 ? kl - kl0 : kl + nk - kl0) * xstep;
    if (LO) {
#pragma unroll
      for (int q = 0; q < kXv; ++q) {
        xl[q] = ld_cg_u4(lo_glob + (xu - xs0) + q * 128);
        if (N1 && !(q < 2 ? m01 : m23)) xl[q] = make_uint4(0, 0, 0, 0);
      }
    }
    // once a wait has run out nothing is waited for or released any more, so
    // the producer runs out of released stages and stops
    bool have = !T.dead;
    if (have && !mbar_wait_bounded(smem_u32(&T.full[s]), ph, p.max_polls)) {
      if (lane == 0) atomicOr(status_of(p), kStatusTimeout);
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
    if constexpr (N1) {
      const uint32_t a01 = m01 ? xu : zaddr, a23 = m23 ? xu : zaddr;
      xh[0] = lds_v4(a01);
      xh[1] = lds_v4(a01 + 128);
      xh[2] = lds_v4(a23 + 256);
      xh[3] = lds_v4(a23 + 384);
    } else {
#pragma unroll
      for (int q = 0; q < kXv; ++q) xh[q] = lds_v4(xu + q * 128);
    }
    __syncwarp();
    if (lane == 0 && have) mbar_arrive(smem_u32(&T.empty[s]));
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
    const bool last_of_tile = kl == nk - 1;
    const int cur = tile;
    if (++kl == nk) { kl = 0; ++tile; }
    if (!last_of_tile && u + 1 < u1) continue;
    // ---- end of a tile piece ----
    float v[2][4];
    if constexpr (N1) {
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
    if (half == 1) {
#pragma unroll
      for (int st = 0; st < 2; ++st) T.red[b][st][lane] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
    }
    named_bar_sync(1, kConsumerThreads);
    if (half == 0) {
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        const float4 o = T.red[b][st][lane];
        v[st][0] += o.x; v[st][1] += o.y; v[st][2] += o.z; v[st][3] += o.w;
      }
    }
    named_bar_sync(1, kConsumerThreads);   // T.red read: warps 4..7 may go on
    if (half == 0) deposit_piece<N1>(p, buf, cnt, slot0, T, cur, b, g, t, v);
  }
  return (uint32_t)s | (ph << 16);
}

// The rare paths out of line: the two-band loops, and the output layer's
// format when it differs from the layers' (their registers stay out of the
// main loop).
template <int FMT, bool LO, bool N1>
__device__ __noinline__ uint32_t step_units_ool(const StepParams& p, float* buf, uint32_t* cnt, int slot0, int u0,
                                                int u1, int nk, int kl0, StepTail& T, uint32_t stage0, uint32_t xs0,
                                                const uint8_t* lo_glob, uint32_t ring) {
  return step_units<FMT, LO, N1>(p, buf, cnt, slot0, u0, u1, nk, kl0, T, stage0, xs0, lo_glob, ring);
}

// The output layer's tiles, finished from their deposits by one warp each
// (tile t by warp t / G of CTA t % G): logits = row scale * the tile's
// deposits added in order.
__device__ __noinline__ void finish_head(const StepParams& p, const StepProduct& P, StepTail& T, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int N = p.N, G = p.G;
  const float* buf = pbuf_of(p, P.pbuf);
  const bool fp8 = P.fmt == kFmtFP8;
  for (int t = blockIdx.x + warp * G; t < P.n_tiles; t += kSW * G) {
    const int np = pieces_of(p, P, t);
    bool ok = true;
    if (lane == 0 && !T.dead) ok = poll_ge(counters(p) + P.cnt_off + t, (uint32_t)np, p.max_polls);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) {
      if (lane == 0) atomicOr(status_of(p), kStatusTimeout);
      T.dead = 1u;
      return;
    }
    int m, row0;
    step_box(P, p.mats, t, 0, m, row0);
    const int d_out = __ldg(&p.mats[m].d_out), off = __ldg(&p.mats[m].out_row_off);
    const float ts = fp8 ? 0.0f : __ldg(p.mats[m].scale32);
    for (int e = lane; e < 128 * N; e += 32) {
      const int n = e >> 7, row = e & 127;
      if (row0 + row >= d_out) continue;
      float acc = 0.0f;
      for (int s = 0; s < P.n_slabs; ++s) {
        const SlabPos q = slab_pos(P.n_tiles, P.nks, P.n_slabs, (int)((long long)s * G / P.n_slabs), G);
        const int l0 = (int)owner_of((long long)t * q.nk, q.units, q.gs);
        const int l1 = (int)owner_of((long long)t * q.nk + q.nk - 1, q.units, q.gs);
        for (int l = l0; l <= l1; ++l) acc += ld_cg_f32(buf + ((size_t)(s * p.slab_stride + t + l) * N + n) * 128 + row);
      }
      const float y = __fmul_rn(acc, fp8 ? __ldg(p.mats[m].scale32 + row0 + row) : ts);
      p.logits[(size_t)n * P.out_ld + off + row0 + row] = y;
    }
  }
}

// ---- the producer --------------------------------------------------------------

// A position in this CTA's sequence of weight units (products in order, each
// product's units tile-major within its slab), with the fields of the
// current product the copies need (read once per product, so that issuing a
// unit reads no memory). pi == n_prods: past the end.
struct UnitCursor {
  int pi, tile, kl, nk, k0, u, u1;
  int fmt, swiglu, mat0, tb1, tb2, tb3;   // tb*: first tile of matrices 1..3 (INT_MAX: absent)
  const CUtensorMap* codes0;              // tensor maps of the product's matrices
};

BWS_DEV void cursor_product(const StepParams& p, UnitCursor& c) {
  for (; c.pi < p.n_prods; ++c.pi) {
    const StepProduct* Pp = p.prods + c.pi;
    const SlabPos q = slab_pos(__ldg(&Pp->n_tiles), __ldg(&Pp->nks), __ldg(&Pp->n_slabs), blockIdx.x, p.G);
    if (q.u1 > q.u0) {
      c.u = (int)q.u0;
      c.u1 = (int)q.u1;
      c.nk = q.nk;
      c.k0 = q.k0;
      c.tile = (int)(q.u0 / q.nk);
      c.kl = (int)(q.u0 % q.nk);
      c.fmt = __ldg(&Pp->fmt);
      c.swiglu = __ldg(&Pp->epi) == kEpiSwiGLU;
      c.mat0 = __ldg(&Pp->mat0);
      const int nm = __ldg(&Pp->n_mats);
      c.tb1 = nm > 1 ? __ldg(&p.mats[c.mat0 + 1].tile_begin) : 0x7FFFFFFF;
      c.tb2 = nm > 2 ? __ldg(&p.mats[c.mat0 + 2].tile_begin) : 0x7FFFFFFF;
      c.tb3 = nm > 3 ? __ldg(&p.mats[c.mat0 + 3].tile_begin) : 0x7FFFFFFF;
      // the output layer's maps are kernel parameters
      c.codes0 = c.pi == p.n_prods - 1 ? &p.head_codes : &p.mats[c.mat0].codes;
      for (int i = 0; i < nm; ++i) {
        const StepMat* M = p.mats + c.mat0 + i;
        tma_prefetch_desc(c.pi == p.n_prods - 1 ? (const void*)&p.head_codes : (const void*)&M->codes);
        if (c.fmt == kFmtNVFP4)
          tma_prefetch_desc(c.pi == p.n_prods - 1 ? (const void*)&p.head_scales : (const void*)&M->scales);
      }
      return;
    }
  }
}
BWS_DEV void cursor_next(const StepParams& p, UnitCursor& c) {
  if (++c.kl == c.nk) { c.kl = 0; ++c.tile; }
  if (++c.u == c.u1) {
    ++c.pi;
    cursor_product(p, c);
  }
}

// The unit at the cursor into the stage at dst, completing on bar: one
// 128-row box of codes and one of scales (SwiGLU: 64 gate and 64 up rows,
// two of each). A 128-row box with 128-byte swizzle lands exactly as four
// 32-row boxes would (the swizzle pattern repeats every 8 rows), so the
// consumers read the same layout.
BWS_DEV void issue_unit(const StepParams& p, const UnitCursor& c, uint32_t dst, uint32_t bar, uint64_t pol) {
  const int ks = c.k0 + c.kl;
  const bool nv = c.fmt == kFmtNVFP4;
  mbar_arrive_expect_tx(bar, nv ? kStageBytes : kCodeBytes);
  constexpr int kMatStride = (int)sizeof(StepMat);   // consecutive StepMat entries
  const bool head = c.codes0 == &p.head_codes;
  if (c.swiglu) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const char* cm = reinterpret_cast<const char*>(c.codes0) + (size_t)m * kMatStride;
      tma_load_2d_hint(dst + m * 2 * kBoxBytes, cm, ks * 128, c.tile * 64, bar, pol);
      if (nv)
        tma_load_2d_hint(dst + kCodeBytes + m * 2 * kScaleBoxBytes, cm + offsetof(StepMat, scales), ks * 16,
                         c.tile * 64, bar, pol);
    }
    return;
  }
  const int mi = (c.tile >= c.tb1) + (c.tile >= c.tb2) + (c.tile >= c.tb3);
  const int t0 = mi == 0 ? 0 : (mi == 1 ? c.tb1 : (mi == 2 ? c.tb2 : c.tb3));
  const char* cm = reinterpret_cast<const char*>(c.codes0) + (size_t)mi * kMatStride;
  const int row = (c.tile - t0) * 128;
  tma_load_2d_hint(dst, cm, ks * 128, row, bar, pol);
  if (nv) {
    const void* sm = head ? (const void*)&p.head_scales : (const void*)(cm + offsetof(StepMat, scales));
    tma_load_2d_hint(dst + kCodeBytes, sm, ks * 16, row, bar, pol);
  }
}

// N1: one token (the block-diagonal operand in the NVFP4 loop).
template <bool N1>
__global__ void __launch_bounds__(kStepThreads, kCtasPerSm) step_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* sbase = smem_raw + ((1024u - mis) & 1023u);
  const int NS = p.n_stages;
  uint8_t* xs = sbase + NS * kStageBytes;
  StepTail& T = *reinterpret_cast<StepTail*>(xs + p.x_bytes);
  const uint32_t stage0 = smem_u32(sbase);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&T.full[i]), 1);
      mbar_init(smem_u32(&T.empty[i]), kSW);
    }
    T.dead = 0u;
    mbar_fence_init();
  }
  for (int i = threadIdx.x; i < 33; i += blockDim.x) T.zero_x[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  if (warp == kSW) {
    // ---- producer: the weight units of every product, in order, at most
    // `inflight` of them in flight ----
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();   // weights are read once per step
      UnitCursor ld;
      memset(&ld, 0, sizeof(ld));
      cursor_product(p, ld);
      int s = 0;
      uint32_t ph = 0u;
      long long issued = 0;
      bool ok = true;
      for (; ld.pi < p.n_prods; ++issued) {
        if (issued >= NS && !mbar_wait_bounded(smem_u32(&T.empty[s]), ph ^ 1u, p.max_polls)) ok = false;
        if (ok && p.inflight < NS && issued >= p.inflight) {
          const long long k = issued - p.inflight;
          ok = mbar_wait_bounded(smem_u32(&T.full[k % NS]), (uint32_t)(k / NS) & 1u, p.max_polls);
        }
        if (!ok) {
          atomicOr(status_of(p), kStatusTimeout);
          break;
        }
        issue_unit(p, ld, stage0 + (uint32_t)s * kStageBytes, smem_u32(&T.full[s]), pol);
        cursor_next(p, ld);
        if (++s == NS) { s = 0; ph ^= 1u; }
      }
      // let copies in flight land before the CTA's shared memory goes away
      for (long long k = (issued > NS ? issued - NS : 0); k < issued; ++k)
        mbar_wait_bounded(smem_u32(&T.full[k % NS]), (uint32_t)(k / NS) & 1u, p.max_polls);
    }
    return;
  }

  // ---- consumers ----
  pdl_wait();
  const int tid = threadIdx.x;
  uint8_t* lo_glob = reinterpret_cast<uint8_t*>(p.ws + p.lo_off) + (size_t)blockIdx.x * p.x_bytes;
  const uint32_t xs0 = smem_u32(xs);
  uint32_t ring = 0u;   // the consumers' ring position: stage | phase << 16
  for (int pi = 0; pi < p.n_prods; ++pi) {
    const StepProduct* Pp = p.prods + pi;
    const StepProduct P = *Pp;
    const SlabPos pos = slab_pos(P.n_tiles, P.nks, P.n_slabs, blockIdx.x, p.G);
    if (tid == 0) trace(p, pi, 0);
    // this CTA's share of the residual update the product normalises
    if (P.in_kind == kInNorm && P.in_prod >= 0) finish_residual(p, P.in_prod, T, tid);
    if (tid == 0) trace(p, pi, 1);
    uint32_t fl = 0u;
    if (pos.u1 > pos.u0) {
      fl = P.in_kind == kInNorm ? build_norm(p, P, pos, T, xs, lo_glob, tid)
                                : build_copy(p, P, pos, T, xs, lo_glob, tid);
      if (tid == 0 && fl) atomicOr(reinterpret_cast<uint32_t*>(p.ws), fl);
    }
    // every CTA has read this product's inputs when read_done reaches G
    named_bar_sync(4, kConsumerThreads);
    if (tid == 0) {
      red_release_add(read_done(p) + pi, 1u);
      trace(p, pi, 2);
    }
    if (pos.u1 <= pos.u0) continue;
    // the deposit buffer was last filled by product pi - kPBufs, whose
    // deposits product pi - kPBufs + 1 reads
    if (P.pbuf < kPBufs && pi >= kPBufs - 1) consumers_wait(p, T, read_done(p) + pi - (kPBufs - 1), (uint32_t)p.G, tid);
    const bool fp8 = P.fmt == kFmtFP8;
    const bool n1 = !fp8 && N1;
    float* buf = pbuf_of(p, P.pbuf);
    uint32_t* cnt = counters(p) + P.cnt_off;
    const int slot0 = (int)(pos.s * p.slab_stride + pos.l), u0 = (int)pos.u0, u1 = (int)pos.u1;
    if (fl & 1u) {
      if (fp8)
        ring = step_units_ool<kFmtFP8, true, false>(p, buf, cnt, slot0, u0, u1, pos.nk, pos.kl0, T, stage0, xs0, lo_glob, ring);
      else if (n1)
        ring = step_units_ool<kFmtNVFP4, true, true>(p, buf, cnt, slot0, u0, u1, pos.nk, pos.kl0, T, stage0, xs0, lo_glob, ring);
      else
        ring = step_units_ool<kFmtNVFP4, true, false>(p, buf, cnt, slot0, u0, u1, pos.nk, pos.kl0, T, stage0, xs0, lo_glob, ring);
    } else if (fp8) {
      ring = step_units_ool<kFmtFP8, false, false>(p, buf, cnt, slot0, u0, u1, pos.nk, pos.kl0, T, stage0, xs0, lo_glob, ring);
    } else if (N1) {
#if BWS_STEP_CTAS > 1
      ring = step_units_ool<kFmtNVFP4, false, true>(p, buf, cnt, slot0, u0, u1, pos.nk, pos.kl0, T, stage0, xs0, lo_glob, ring);
#else
      ring = step_units<kFmtNVFP4, false, true>(p, buf, cnt, slot0, u0, u1, pos.nk, pos.kl0, T, stage0, xs0, lo_glob, ring);
#endif
    } else {
#if BWS_STEP_CTAS > 1
      ring = step_units_ool<kFmtNVFP4, false, false>(p, buf, cnt, slot0, u0, u1, pos.nk, pos.kl0, T, stage0, xs0, lo_glob, ring);
#else
      ring = step_units<kFmtNVFP4, false, false>(p, buf, cnt, slot0, u0, u1, pos.nk, pos.kl0, T, stage0, xs0, lo_glob, ring);
#endif
    }
    if (tid == 0) trace(p, pi, 3);
  }
  finish_head(p, p.prods[p.n_prods - 1], T, tid);
}

// r = x0 (FP32) in residual buffer 0, the first RMSNorm's per-128-row
// statistics, zeroed counters and status. Block (tile, n), 128 threads.
__global__ void __launch_bounds__(128) step_init_kernel(const __grid_constant__ StepParams p) {
  pdl_launch_dependents();   // the step kernel's producers may start streaming weights
  const int n = blockIdx.y, tile = blockIdx.x;
  const int i = tile * kStatRows + threadIdx.x;
  float* r = reinterpret_cast<float*>(p.ws + p.r_off[0]);
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
  const int nb = gridDim.x * gridDim.y, b = blockIdx.y * gridDim.x + blockIdx.x;
  uint32_t* z = reinterpret_cast<uint32_t*>(p.ws + p.cnt_off);
  for (int k = b * 128 + threadIdx.x; k < p.n_zero_words; k += nb * 128) z[k] = 0u;
  if (b == 0 && threadIdx.x < 2) reinterpret_cast<uint32_t*>(p.ws)[threadIdx.x] = 0u;
}

}  // namespace

// ---- host: the program of a stack -------------------------------------------

struct StepProgram {
  int N, hidden, G, n_prods, n_mats;
  float eps;
  void* dev;               // [StepProduct x n_prods][StepMat x n_mats]
  StepProduct* d_prods;
  StepMat* d_mats;
  StepParams proto;        // every field but the pointers of one call
  size_t ws_bytes;
  int smem;
};

namespace {

size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

int step_smem(int n_stages, int x_bytes) { return n_stages * kStageBytes + x_bytes + (int)sizeof(StepTail) + 1024; }

bool qualifies(const bws_matrix& m, int d_in) {
  if (m.d_in != d_in || m.d_out < 1 || !m.codes || ((uintptr_t)m.codes & 15)) return false;
  if (m.format == BWS_FMT_NVFP4) return d_in % 256 == 0 && m.scales && !((uintptr_t)m.scales & 15) && m.scale32;
  if (m.format == BWS_FMT_FP8_ROW) return d_in % 128 == 0 && m.scale32;
  return false;
}

// Tunables read from the environment at plan creation (measurement aids):
// BWS_STEP_INFLIGHT (weight units in flight per CTA), BWS_STEP_TRACE=1 (per
// CTA and product timestamps at the end of the workspace).
int env_int(const char* name, int dflt, int lo, int hi) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  const int x = atoi(v);
  return x < lo ? lo : (x > hi ? hi : x);
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
  // ring and slab: the slab holds the activations of the k-units a CTA
  // touches; with more tokens it takes a larger share of shared memory
  const int n_stages = kCtasPerSm == 1 ? (N == 1 ? 11 : 10) : (N == 1 ? 5 : 4);
  const int x_bytes = N == 1 ? 12 * 1024 : 24 * 1024;
  const int smem = step_smem(n_stages, x_bytes);
  auto kernel = N == 1 ? step_kernel<true> : step_kernel<false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kStepThreads, smem) != cudaSuccess || nb < 1) {
    cudaGetLastError();
    return nullptr;
  }
  const int G = (nb > kCtasPerSm ? kCtasPerSm : nb) * sms;

  std::vector<StepMat> mats;
  std::vector<StepProduct> prods;
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
      const uint32_t box_rows = epi == kEpiSwiGLU ? 64 : 128;   // one box per unit (per half for SwiGLU)
      if (!encode_2d(&m.codes, ms[i].codes, row_bytes, (uint64_t)ms[i].d_out, 128, box_rows, true)) ok = false;
      if (!fp8 && !encode_2d(&m.scales, ms[i].scales, (uint64_t)d_in / 16, (uint64_t)ms[i].d_out, 16, box_rows, false))
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
  auto add_prod = [&](const bws_matrix* ms, int n, int epi, int d_in, int in_kind) {
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
    int tiles = 0, out_w = 0;
    if (epi == kEpiSwiGLU) {
      tiles = (ms[0].d_out + 63) / 64;
    } else {
      for (int i = 0; i < n; ++i) tiles += (ms[i].d_out + 127) / 128;
    }
    for (int i = 0; i < n; ++i) out_w += ms[i].d_out;
    P.n_tiles = tiles;
    // the fewest slabs whose k-units a CTA touches fit the slab buffer
    const int xblk = UK * 2 + 16;
    const int max_units = x_bytes / (N * xblk);
    if (max_units < 1) { ok = false; return; }
    int S = 1;
    for (;; ++S) {
      if (S > G || S > P.nks) { ok = false; return; }
      int need = 0;
      for (int c = 0; c < G; ++c) {
        const SlabPos q = slab_pos(P.n_tiles, P.nks, S, c, G);
        need = q.cnt > need ? q.cnt : need;
      }
      if (need <= max_units) break;
    }
    P.n_slabs = S;
    P.in_kind = in_kind;
    P.in_prod = in_kind == kInCopy ? (int)prods.size() - 1 : -1;
    P.r_guard = -1;
    P.out_ld = out_w;
    prods.push_back(P);
  };
  for (int li = 0; li < n_layers && ok; ++li) {
    const bws_layer& L = layers[li];
    if (L.kind == BWS_LAYER_MIXER_MLP) {
      if (L.n_mixer_in < 1 || L.n_mixer_in > kMaxMats) { ok = false; break; }
      int sum_out = 0;
      for (int i = 0; i < L.n_mixer_in; ++i) {
        sum_out += L.mixer_in[i].d_out;
        if (L.mixer_in[i].d_out % 128) ok = false;   // the deposits of a tile come from one matrix
      }
      if (L.mixer_out.d_in > sum_out || L.mixer_out.d_out != hidden) ok = false;
      if (!ok) break;
      add_prod(L.mixer_in, L.n_mixer_in, kEpiStoreBF16, hidden, kInNorm);
      add_prod(&L.mixer_out, 1, kEpiResidF32, L.mixer_out.d_in, kInCopy);
    } else if (L.kind != BWS_LAYER_MLP) {
      ok = false;
      break;
    }
    if (!ok) break;
    if (L.up.d_out != L.gate.d_out || L.down.d_out != hidden || L.down.d_in != L.gate.d_out || L.gate.d_out % 64) {
      ok = false;
      break;
    }
    const bws_matrix gu[2] = {L.gate, L.up};
    add_prod(gu, 2, kEpiSwiGLU, hidden, kInNorm);
    add_prod(&L.down, 1, kEpiResidF32, L.down.d_in, kInCopy);
  }
  if (ok) add_prod(&head, 1, kEpiStoreF32, hidden, kInNorm);
  if (!ok || prods.empty()) return nullptr;

  // residual chain: every normalised input reads the residual of the last
  // update before it; updates alternate between the two buffers
  {
    int last = -1, cur_buf = 0, last_norm_of[2] = {-1, -1};   // the product that read each buffer last
    for (size_t i = 0; i < prods.size(); ++i) {
      StepProduct& P = prods[i];
      if (P.in_kind == kInNorm) {
        P.in_prod = last;
        P.r_in = cur_buf;
        last_norm_of[cur_buf] = (int)i;
      }
      if (P.epi == kEpiResidF32) {
        if (P.n_tiles * 128 < hidden) { ok = false; break; }
        P.r_src = cur_buf;
        P.r_dst = cur_buf ^ 1;
        P.r_guard = last_norm_of[cur_buf ^ 1];
        cur_buf ^= 1;
        last = (int)i;
        // the product after a residual update must normalise it (its finishing runs there)
        if (i + 1 >= prods.size() || prods[i + 1].in_kind != kInNorm) { ok = false; break; }
      }
    }
  }
  if (!ok) return nullptr;
  const int np = (int)prods.size();
  prods[np - 1].pbuf = kPBufs;
  for (int i = 0; i < np - 1; ++i) prods[i].pbuf = i % kPBufs;

  // deposits: slots and pieces per tile
  long long stride = 1;
  for (auto& P : prods) {
    const long long gs = (G + P.n_slabs - 1) / P.n_slabs;
    stride = P.n_tiles + gs > stride ? P.n_tiles + gs : stride;
  }
  size_t pbuf_floats[kPBufs + 1] = {0, 0, 0, 0, 0};
  int cnt = 0;
  for (auto& P : prods) {
    const size_t f = (size_t)P.n_slabs * stride * N * 128;
    pbuf_floats[P.pbuf] = f > pbuf_floats[P.pbuf] ? f : pbuf_floats[P.pbuf];
    P.cnt_off = cnt;
    cnt += P.n_tiles;
    for (int t = 0; t < P.n_tiles; ++t) {
      const int n_p = tile_slots(P.n_tiles, P.nks, P.n_slabs, G, stride, t, nullptr, 0);
      if (n_p > kMaxPieces) ok = false;
    }
  }
  // every slot a CTA deposits into lies inside its buffer (checked here, on the host)
  for (auto& P : prods) {
    for (int c = 0; c < G && ok; ++c) {
      const SlabPos q = slab_pos(P.n_tiles, P.nks, P.n_slabs, c, G);
      if (q.u1 <= q.u0) continue;
      const long long last_tile = (q.u1 - 1) / q.nk;
      if ((q.s * stride + last_tile + q.l + 1) * N * 128 > (long long)pbuf_floats[P.pbuf]) ok = false;
      if (q.cnt * (long long)N * (P.fmt == kFmtFP8 ? 272 : 528) > x_bytes) ok = false;
      // the copy input's covered tiles are waited for by one consumer thread each
      if (P.in_kind == kInCopy) {
        const int rpt = prods[P.in_prod].epi == kEpiSwiGLU ? 64 : 128;
        const int UK = P.fmt == kFmtFP8 ? 128 : 256;
        if (q.cnt * (UK / rpt) > kConsumerThreads) ok = false;
      }
    }
  }
  if (!ok) return nullptr;

  // workspace: [status 256][r0][r1][stats0][stats of each update][counters: tiles, stats, read][deposit buffers][lo]
  StepProgram* S = new (std::nothrow) StepProgram();
  if (!S) return nullptr;
  memset(&S->proto, 0, sizeof(S->proto));
  StepParams& q = S->proto;
  S->N = N;
  S->hidden = hidden;
  S->eps = eps;
  S->G = G;
  S->smem = smem;
  size_t o = 256;
  q.r_off[0] = (long long)o; o += al256(sizeof(float) * (size_t)N * hidden);
  q.r_off[1] = (long long)o; o += al256(sizeof(float) * (size_t)N * hidden);
  q.stats0_off = (long long)o; o += al256(sizeof(float2) * (size_t)(hidden / kStatRows) * N);
  for (auto& P : prods) {
    if (P.epi == kEpiResidF32) {
      P.stats_off = (long long)o;
      o += al256(sizeof(float2) * (size_t)P.n_tiles * N);
    }
  }
  q.cnt_off = (long long)o; o += sizeof(uint32_t) * (size_t)cnt;
  q.stats_cnt_off = (long long)o; o += sizeof(uint32_t) * (size_t)np;
  q.read_done_off = (long long)o; o += sizeof(uint32_t) * (size_t)np;
  q.n_zero_words = cnt + 2 * np;
  o = al256(o);
  for (int b = 0; b <= kPBufs; ++b) {
    q.pbuf_off[b] = (long long)o;
    o += al256(sizeof(float) * pbuf_floats[b]);
  }
  q.slab_stride = stride;
  q.lo_off = (long long)o; o += al256((size_t)G * x_bytes);
  q.trace_off = -1;
  if (env_int("BWS_STEP_TRACE", 0, 0, 1)) {
    q.trace_off = (long long)o;
    o += al256(sizeof(uint32_t) * 4 * (size_t)G * np);
  }
  S->ws_bytes = o;
  q.n_prods = np;
  q.N = N;
  q.hidden = hidden;
  q.G = G;
  q.eps = eps;
  q.n_stages = n_stages;
  q.x_bytes = x_bytes;
  q.inflight = env_int("BWS_STEP_INFLIGHT", 4, 1, n_stages);
  q.max_polls = 1u << 24;
  S->n_prods = np;
  S->n_mats = (int)mats.size();

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
  q.prods = S->d_prods;
  q.mats = S->d_mats;
  q.head_codes = mats.back().codes;
  q.head_scales = mats.back().scales;
  return S;
}

void step_program_destroy(StepProgram* S) {
  if (!S) return;
  if (S->dev) cudaFree(S->dev);
  delete S;
}

size_t step_program_workspace(const StepProgram* S) { return S ? S->ws_bytes : 0; }

int step_program_grid(const StepProgram* S) { return S ? S->G : 0; }

long long step_program_trace(const StepProgram* S, int* n_prods) {
  if (!S) return -1;
  if (n_prods) *n_prods = S->n_prods;
  return S->proto.trace_off;
}

cudaError_t step_program_enqueue(const StepProgram* S, const uint16_t* x0, float* logits, void* ws, cudaStream_t st) {
  StepParams p = S->proto;
  p.ws = static_cast<char*>(ws);
  p.logits = logits;
  p.x0 = x0;
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
  return S->N == 1 ? cudaLaunchKernelEx(&cfg, step_kernel<true>, p) : cudaLaunchKernelEx(&cfg, step_kernel<false>, p);
}

}  // namespace bws
