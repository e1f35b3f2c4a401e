// Activation prep: for each (slot, token) row, optionally r = x0, then
// BF16(RMSNorm(r)) or the BF16 input itself, its exponent E = floor(log2
// max|x|) and the two f16 bands x * 2^(14 - E) / x * 2^(43 - E) the product
// kernels read. Also zeroes the tile counters of the product that follows.
//
// A long row (d > 8192) gets a thread-block cluster of 8 CTAs of 256 threads:
// each CTA takes a contiguous share of the row's 8-element chunks, and the
// row's sum of squares, largest magnitude and band flags are exchanged through
// distributed shared memory, combined in CTA-rank order (deterministic), so
// the row costs one pass of loads spread over 8 SMs. A shorter row gets one
// CTA of 1024 threads (a cluster of one): it starts sooner while the previous
// product's CTAs still hold most SMs.
#include <cooperative_groups.h>

#include "bws_common.cuh"
#include "bws_internal.h"
#include "moe_route.cuh"
#include "stream_tile.cuh"
#include "trace.cuh"

namespace cg = cooperative_groups;

namespace bws {

namespace {

constexpr int kLongRow = 8192;    // longer rows get a cluster

BWS_DEV float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// The row's values as BF16 bit patterns, chunk c (8 values); for RMSNorm, the
// FP32 residual times inv_rms rounded to BF16.
template <bool FIN>
BWS_DEV void chunk_bf16(const PrepParams& q, int c, const float* rr, const uint4* xr, float inv_rms,
                        uint32_t (&w)[4]) {
  // a copied row that this kernel finished and wrote (fin_partials) is read
  // back through L2, not the read-only path
  if (q.mode == kPrepRmsNorm) {
    const float4 a = reinterpret_cast<const float4*>(rr)[2 * c];
    const float4 b = reinterpret_cast<const float4*>(rr)[2 * c + 1];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(v[2 * i], inv_rms)));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(v[2 * i + 1], inv_rms)));
      w[i] = lo | (hi << 16);
    }
  } else {
    const uint4 b = FIN ? __ldcg(xr + c) : __ldg(xr + c);
    w[0] = b.x; w[1] = b.y; w[2] = b.z; w[3] = b.w;
  }
}

// Elements e..e+7 of token tok of the previous product's output (one 8-element
// chunk: never across a tile), finished from its CTAs' deposits the way the
// product kernel's last arriving CTA finishes a tile: the tile's slots added
// in CTA order from zero, times the matrix's scale, times 2^(E - 14) of the
// product's input; SwiGLU (SWI): SiLU(gate) * up. Only the finishing
// instantiations of the prep use it.
template <bool SWI, int KB>
__device__ __forceinline__ void finish_chunk(const PrepParams& q, int tok, int e, float (&out)[8]) {
  int m = 0;
  for (int i = 1; i < q.fin_n_mats; ++i)
    if (e >= q.fin_row_off[i]) m = i;
  const int lrow = e - q.fin_row_off[m];
  constexpr int kRows = SWI ? 64 : 128;
  const int tile = (SWI ? 0 : q.fin_tile_begin[m]) + lrow / kRows, rit = lrow % kRows;
  // the CTAs that hold the tile's first and last units
  const int cc0 = splitk_owner(q.fin_split, (long long)tile * q.fin_nks);
  const int cc1 = splitk_owner(q.fin_split, (long long)(tile + 1) * q.fin_nks - 1);
  float a[8], au[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = au[i] = 0.0f;
  // KB slots' loads in flight per batch
  constexpr int kB = KB, kV = SWI ? 4 : 2;
  for (int cb = cc0; cb <= cc1; cb += kB) {
    float4 o[kB][kV];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      // the chunk's 8 values (32 bytes) in one request; SwiGLU: gate, then up 64 rows on
      const float* base = q.fin_partials + ((size_t)(tile + cb + k) * q.N + tok) * 128 + rit;
#pragma unroll
      for (int j = 0; j < kV; j += 2) {
        if (cb + k <= cc1) {
          ld_cg_f8(base + 64 * (j >> 1), o[k][j], o[k][j + 1]);
        } else {
          o[k][j] = o[k][j + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      if (cb + k > cc1) break;
#pragma unroll
      for (int j = 0; j < kV; ++j) {
        float* d = (j >> 1) ? au : a;
        const int h = 4 * (j & 1);
        d[h] += o[k][j].x;
        d[h + 1] += o[k][j].y;
        d[h + 2] += o[k][j].z;
        d[h + 3] += o[k][j].w;
      }
    }
  }
  const int xe = __ldg(q.fin_xexp + tok) - 14;
  if (SWI) {
    // NVFP4: the two tensor scales; FP8: the gate and up rows' own scales
    const bool fp8 = q.fin_fmt == kFmtFP8;
    const float tg = fp8 ? 0.0f : __ldg(q.fin_scale[0]), tu = fp8 ? 0.0f : __ldg(q.fin_scale[1]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float sg = fp8 ? __ldg(q.fin_scale[0] + lrow + i) : tg;
      const float su = fp8 ? __ldg(q.fin_scale[1] + lrow + i) : tu;
      out[i] = silu_mul_t(ldexp_exact(__fmul_rn(a[i], sg), xe), ldexp_exact(__fmul_rn(au[i], su), xe));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float sc = q.fin_fmt == kFmtFP8 ? __ldg(q.fin_scale[m] + lrow + i) : __ldg(q.fin_scale[m]);
      out[i] = ldexp_exact(__fmul_rn(a[i], sc), xe);
    }
  }
}


// The previous MoE layer's combine for chunk c of token tok, in slot order,
// added to the residual r, which it writes back (v: the updated chunk). The
// residual is loaded here, in the same round of loads as the slots' outputs.
// Out of line: its registers stay out of the prep's main path.
__device__ __noinline__ void combine_chunk(const PrepParams& q, int tok, int c, float (&v)[8], float* rr) {
  const float4 ra = reinterpret_cast<const float4*>(rr)[2 * c];
  const float4 rb = reinterpret_cast<const float4*>(rr)[2 * c + 1];
  const float r8[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
  // the slot count, weights and outputs of nine slots at a time are loaded
  // together, whatever the slot count turns out to be (every slot up to the
  // layer's maximum is in bounds); slots past the count or with weight 0 (a
  // slot the token does not use, whose outputs may be stale) are then
  // skipped, the rest added in slot order
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  constexpr int kB = 9;
  if (q.comb_tok_slots != nullptr && q.comb_max_slots > kB) {
    // more slots than one batch (several tokens): the token's own slots, the
    // shared one, then its routed ones ascending (at most 1 + 8 = kB), their
    // weights and outputs loaded together; the slots it does not use have
    // weight 0, so the sum equals the one over every live slot in slot order.
    // (With one batch of slots in all, the loads below need no slot list.)
    const int nk = q.comb_has_shared + q.comb_topk;
    float wt[kB];
    float4 ya[kB], yb[kB];
    int live[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      int sl = -1;
      if (k < nk) sl = (q.comb_has_shared && k == 0) ? 0 : __ldg(q.comb_tok_slots + tok * q.comb_topk + k - q.comb_has_shared);
      live[k] = sl >= 0;
      const int s2 = sl >= 0 ? sl : 0;
      wt[k] = __ldg(q.comb_cw + s2 * q.N + tok);
      const float4* yp = reinterpret_cast<const float4*>(q.comb_ys + ((size_t)s2 * q.N + tok) * q.d_in) + 2 * c;
      ya[k] = __ldg(yp);
      yb[k] = __ldg(yp + 1);
    }
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      if (!live[k] || wt[k] == 0.0f) continue;
      const float y8[8] = {ya[k].x, ya[k].y, ya[k].z, ya[k].w, yb[k].x, yb[k].y, yb[k].z, yb[k].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(wt[k], y8[i], acc[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fadd_rn(r8[i], acc[i]);
    reinterpret_cast<float4*>(rr)[2 * c] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(rr)[2 * c + 1] = make_float4(v[4], v[5], v[6], v[7]);
    return;
  }
  const int ns = __ldg(q.comb_n_slots);
  for (int s0 = 0; s0 < q.comb_max_slots; s0 += kB) {
    float wt[kB];
    float4 ya[kB], yb[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const int sl = s0 + k < q.comb_max_slots ? s0 + k : s0;
      wt[k] = __ldg(q.comb_cw + sl * q.N + tok);
      const float4* yp = reinterpret_cast<const float4*>(q.comb_ys + ((size_t)sl * q.N + tok) * q.d_in) + 2 * c;
      ya[k] = __ldg(yp);
      yb[k] = __ldg(yp + 1);
    }
    if (s0 >= ns) break;
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      if (s0 + k >= ns || wt[k] == 0.0f) continue;
      const float y8[8] = {ya[k].x, ya[k].y, ya[k].z, ya[k].w, yb[k].x, yb[k].y, yb[k].z, yb[k].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(wt[k], y8[i], acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fadd_rn(r8[i], acc[i]);
  reinterpret_cast<float4*>(rr)[2 * c] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(rr)[2 * c + 1] = make_float4(v[4], v[5], v[6], v[7]);
}

// The routing CTA, out of line for the same reason.
__device__ __noinline__ void route_cta(const MoeRoute& m) { moe_route_body(m); }

// The row's sum (of squares) and largest magnitude over the cluster: each
// warp reduces its lanes, warp 0 the CTA's warps, then every CTA adds the
// CTAs' values in rank order through their `slot`s. The shuffle trees are
// fixed, so the result is the same on every run and in every thread.
template <int CL, int THREADS>
BWS_DEV float2 cluster_sum_max(float2* slot, float s, float m, float2* warp_part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  s = warp_sum(s);
  m = warp_max(m);
  if (lane == 0) warp_part[warp] = make_float2(s, m);
  __syncthreads();
  if (warp == 0) {
    const float2 v = lane < THREADS / 32 ? warp_part[lane] : make_float2(0.0f, 0.0f);
    s = warp_sum(v.x);
    m = warp_max(v.y);
    if (lane == 0) *slot = make_float2(s, m);
  }
  if (CL == 1) {
    __syncthreads();
    return *slot;
  }
  cg::cluster_group cl = cg::this_cluster();
  cl.sync();
  float2 r = *cl.map_shared_rank(slot, 0);
  for (int k = 1; k < CL; ++k) {
    const float2 o = *cl.map_shared_rank(slot, k);
    r.x += o.x;
    r.y = fmaxf(r.y, o.y);
  }
  // this CTA is done with the others' slots; the matching wait at the end of
  // the kernel keeps every CTA alive until all have read
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  return r;
}

// E4M3 code of a (RN) and its value.
BWS_DEV uint32_t e4m3_code(float a, float& dec) {
  const uint32_t c = f32x2_to_e4m3x2(0.0f, a) & 0xFFu;
  dec = e4m3_to_f32(c);
  return c;
}

// The tensor-core kernel's activation image of one token (gemv_umma.cu):
// a = x * 2^(7-E) splits into E4M3 bands, a = hi0 + lo0 for |a| >= 2^-2,
// a = 2^-10 (hi1 + lo1) below (exact down to |a| = 2^-12, rounded under
// that, flag 8). Per 256-value unit 2 KB: MMA kk (blocks 2kk, 2kk+1) owns
// bytes [256kk, 256kk + 256), two 8-row x 16-byte core matrices (K chunk 0
// then 1); rows 0-3 of the first hold block 2kk's bands (hi0, lo0, hi1, lo1),
// rows 4-7 of the second block 2kk+1's, the other rows are zero. Out of
// line: its registers stay out of the prep's main path. Returns the flags.
template <bool FIN>
__device__ __noinline__ uint32_t image_chunks(const PrepParams& q, int c0, int c1, const float* rr, const uint4* xr,
                                              float inv_rms, int E) {
  uint8_t* img = reinterpret_cast<uint8_t*>(q.hi);
  uint32_t flags = 0u;
  for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
    uint32_t w[4];
    chunk_bf16<FIN>(q, c, rr, xr, inv_rms, w);
    uint32_t band[4][2] = {{0u, 0u}, {0u, 0u}, {0u, 0u}, {0u, 0u}};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float f = bf16_bits_to_f32(i & 1 ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu));
      const float a = ldexp_exact(f, 7 - E);
      const int pair = fabsf(a) >= 0.25f ? 0 : 1;
      const float b = pair == 0 ? a : ldexp_exact(a, 10);
      float dh, dl;
      const uint32_t h = e4m3_code(b, dh);
      const float rest = __fsub_rn(b, dh);
      const uint32_t l = e4m3_code(rest, dl);
      if (dl != rest) flags |= 8u;
      band[2 * pair][i >> 2] |= h << (8 * (i & 3));
      band[2 * pair + 1][i >> 2] |= l << (8 * (i & 3));
    }
    const int u = c >> 5, j = (c >> 1) & 15, half = c & 1;
    uint8_t* unit = img + (size_t)u * 2048;
    uint8_t* piece = unit + 256 * (j >> 1) + (j & 1) * 192 + half * 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) *reinterpret_cast<uint2*>(piece + 16 * k) = make_uint2(band[k][0], band[k][1]);
    if ((j & 1) == 0) {
      uint4* z = reinterpret_cast<uint4*>(unit + 256 * (j >> 1) + 64 + 64 * half);
#pragma unroll
      for (int k = 0; k < 4; ++k) z[k] = make_uint4(0, 0, 0, 0);
    }
  }
  return flags;
}

// The f16 bands of one 8-value chunk (BF16 bit patterns w) at exponent E,
// stored at chunk position dst of the row's band arrays; flags: bit 0 an
// element needs the lo band, bit 1 an element is below both.
BWS_DEV void store_bands(const uint32_t (&w)[4], int E, uint4* hi4, uint4* lo4, int dst, uint32_t& flags) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t hh[2], ll[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float f = bf16_bits_to_f32(j == 0 ? (w[i] & 0xFFFF) : (w[i] >> 16));
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
  hi4[dst] = make_uint4(h[0], h[1], h[2], h[3]);
  lo4[dst] = make_uint4(l[0], l[1], l[2], l[3]);
}

// Chunk position of chunk c in the TMA kernel's layout: within each unit of
// K_u values, the 8-value chunk j of lane chunk cl (cl = 0..7, lane chunks of
// K_u/8 values) moves to j * 8 + cl, so that the 8 lanes of a shared-memory
// phase read 8 different banks.
BWS_DEV int band_pos(int c, int interleave) {
  if (!interleave) return c;
  const int ku8 = interleave / 8, lk8 = interleave / 64;
  const int u = c / ku8, r8 = c - u * ku8;
  return u * ku8 + (r8 % lk8) * 8 + r8 / lk8;
}

// MOE: the body with the routing CTA and the folded combine.
template <int CL, int THREADS, bool MOE>
__device__ __forceinline__ void prep_body(const PrepParams& q) {
  constexpr bool FIN = false;
#ifdef BWS_TRACE
  unsigned long long tr[6] = {trace_now(), 0, 0, 0, 0, 0};
#endif
  pdl_launch_dependents();
  // the routing CTA, the last of the grid (with clusters, the last cluster
  // holds it and CL - 1 CTAs that only pad the cluster): with a ready flag it
  // reads only ids and weights, so it need not wait for the kernels before
  const bool rcl = MOE && q.has_route && (int)blockIdx.x >= (int)gridDim.x - CL;
  const bool route = rcl && blockIdx.x == gridDim.x - 1;
  const bool early = rcl && q.route.ready != nullptr;
  if (early) {
    if (route) route_cta(q.route);
    return;
  }
  pdl_wait();
#ifdef BWS_TRACE
  tr[1] = trace_now();
#endif
  const int rank = CL == 1 ? 0 : (int)cg::this_cluster().block_rank();
  const int zctas = gridDim.x - (MOE && q.has_route && q.route.ready != nullptr ? CL : 0);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < q.zero_words; i += zctas * blockDim.x)
    q.zero_ptr[i] = 0u;
  if (rcl) {
    if (route) route_cta(q.route);
    return;
  }
  const int row = blockIdx.x / CL;
  const int slot = row / q.N;
  const int tok = row - slot * q.N;
  const int n_slots = q.n_slots != nullptr ? __ldg(q.n_slots) : 1;
  if (slot >= n_slots) return;   // the whole cluster returns together
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (q.hdr != nullptr) q.hdr[0] = (uint32_t)q.N;
    if (q.status_clear != nullptr) q.status_clear[0] = q.status_clear[1] = 0u;
  }
  __shared__ float2 warp_part[THREADS / 32];
  __shared__ float2 xch;     // this CTA's values in the cluster exchange
  __shared__ uint32_t cta_flags;
  if (threadIdx.x == 0) cta_flags = 0u;   // ordered before its use by the statistics' barriers
  // the row's band flags are OR-ed into global memory by the warps that find
  // any; the cluster barrier below orders this clearing store before them
  if (rank == 0 && threadIdx.x == 0) q.flags[slot * q.N + tok] = 0u;
  const int nchunk = q.d_in >> 3, nchunk_pad = q.d_in_pad >> 3;
  // this CTA's chunks [c0, c1)
  const int per = (nchunk_pad + CL - 1) / CL;
  const int c0 = rank * per < nchunk_pad ? rank * per : nchunk_pad;
  const int c1 = c0 + per < nchunk_pad ? c0 + per : nchunk_pad;
  const size_t rowbase = ((size_t)slot * (q.N + 1)) * q.d_in_pad;
  if (tok == 0 && q.interleave != kLayoutImage) {   // this slot's all-zero row
    uint4* zh = reinterpret_cast<uint4*>(q.hi + rowbase + (size_t)q.N * q.d_in_pad);
    uint4* zl = reinterpret_cast<uint4*>(q.lo + rowbase + (size_t)q.N * q.d_in_pad);
    for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
      zh[c] = make_uint4(0, 0, 0, 0);
      zl[c] = make_uint4(0, 0, 0, 0);
    }
  }
  // One pass of statistics: the sum of squares (RMSNorm) and the largest
  // magnitude of the values the bands are cut from. Rounding to BF16 after a
  // multiplication by inv_rms > 0 is monotone and odd, so the largest
  // normalised magnitude is the normalisation of the largest raw one, and
  // the exponent E needs no second pass.
  float inv_rms = 1.0f;
  const uint4* xr = nullptr;
  float* rr = nullptr;
  float ss = 0.0f, ma = 0.0f;
  if (q.mode == kPrepRmsNorm) {
    rr = q.r + (size_t)tok * q.d_in;
    const uint4* x0 = q.x0 != nullptr ? reinterpret_cast<const uint4*>(q.x0 + (size_t)tok * q.d_in) : nullptr;
    for (int c = c0 + threadIdx.x; c < c1 && c < nchunk; c += blockDim.x) {
      float v[8];
      if (x0 != nullptr) {
        const uint4 b = __ldg(x0 + c);
        const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFF);
          v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
        }
        reinterpret_cast<float4*>(rr)[2 * c] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(rr)[2 * c + 1] = make_float4(v[4], v[5], v[6], v[7]);
      } else if (MOE && q.comb_ys != nullptr) {
        combine_chunk(q, tok, c, v, rr);
      } else {
        const float4 a = reinterpret_cast<const float4*>(rr)[2 * c];
        const float4 b = reinterpret_cast<const float4*>(rr)[2 * c + 1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss = __fmaf_rn(v[i], v[i], ss);
        ma = fmaxf(ma, fabsf(v[i]));
      }
    }
  } else {
    xr = reinterpret_cast<const uint4*>(q.x + (size_t)slot * q.x_slot_stride + (size_t)tok * q.ld);
    for (int c = c0 + threadIdx.x; c < c1 && c < nchunk; c += blockDim.x) {
      const uint4 b = __ldg(xr + c);
      const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ma = fmaxf(ma, fmaxf(fabsf(bf16_bits_to_f32(w[i] & 0xFFFF)), fabsf(bf16_bits_to_f32(w[i] >> 16))));
    }
  }
#ifdef BWS_TRACE
  tr[2] = trace_now();
#endif
  const float2 st = cluster_sum_max<CL, THREADS>(&xch, ss, ma, warp_part);
#ifdef BWS_TRACE
  tr[3] = trace_now();
#endif
  float mx = st.y;
  if (q.mode == kPrepRmsNorm) {
    const float ms = __fdiv_rn(st.x, (float)q.d_in);
    inv_rms = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, q.eps)));
    mx = __bfloat162float(__float2bfloat16_rn(__fmul_rn(mx, inv_rms)));
  }
  const int E = mx > 0.0f ? floor_log2_abs(mx) : 0;
  uint32_t flags = 0u;
  if (q.interleave == kLayoutImage) {
    flags = image_chunks<FIN>(q, c0, c1, rr, xr, inv_rms, E);
  } else {
  uint4* hi4 = reinterpret_cast<uint4*>(q.hi + rowbase + (size_t)tok * q.d_in_pad);
  uint4* lo4 = reinterpret_cast<uint4*>(q.lo + rowbase + (size_t)tok * q.d_in_pad);
  for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (c < nchunk) {
      chunk_bf16<FIN>(q, c, rr, xr, inv_rms, w);
      if (q.tap_x != nullptr)   // verification tap: the BF16 row as formed
        reinterpret_cast<uint4*>(q.tap_x + (size_t)tok * q.d_in)[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    store_bands(w, E, hi4, lo4, band_pos(c, q.interleave), flags);
  }
  }
  // the band flags: the warps' into the CTA's word, then one atomic per CTA
  const uint32_t wf = __reduce_or_sync(0xffffffffu, flags);
  if (wf != 0u && (threadIdx.x & 31) == 0) atomicOr(&cta_flags, wf);
  __syncthreads();
  if (threadIdx.x == 0 && cta_flags != 0u) atomicOr(q.flags + slot * q.N + tok, cta_flags);
  if (rank == 0 && threadIdx.x == 0) q.exp[slot * q.N + tok] = E;
#ifdef BWS_TRACE
  tr[4] = trace_now();
#endif
  if (CL > 1) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
#ifdef BWS_TRACE
  if (threadIdx.x == 0) {
    tr[5] = trace_now();
    trace_put(3000u + (MOE ? 100u : 0u) + CL, tr);
  }
#endif
}

// The prep that finishes the previous product's rows (one slot; a cluster of
// CL CTAs, one 8-value chunk per thread): RMS, the RMSNorm of r += y (the
// product a residual update), else a copy of y (SWI: SiLU(g) * u). Each
// thread keeps its chunk in registers from the statistics to the bands, and
// each warp's statistics are pushed into every CTA's table before one cluster
// barrier, after which each CTA reads only its own shared memory.
// KB: slots per batch of loads (a tile of the product's split has about
// nks * CTAs / units + 1 slots).
template <int CL, int THREADS, int KB, bool RMS, bool SWI>
__device__ __forceinline__ void prep_fin_body(const PrepParams& q) {
  constexpr int kW = THREADS / 32;
#ifdef BWS_TRACE
  unsigned long long tr[6] = {trace_now(), 0, 0, 0, 0, 0};
#endif
  pdl_launch_dependents();
  pdl_wait();
#ifdef BWS_TRACE
  tr[1] = trace_now();
#endif
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < q.zero_words; i += gridDim.x * blockDim.x)
    q.zero_ptr[i] = 0u;
  const int tok = blockIdx.x / CL;
  // the band flags are OR-ed in by the warps that find any; the cluster
  // barrier below orders this clearing store before them
  if (rank == 0 && threadIdx.x == 0) q.flags[tok] = 0u;
  const int nchunk = q.d_in >> 3, nchunk_pad = q.d_in_pad >> 3;
  const int per = (nchunk_pad + CL - 1) / CL;   // <= THREADS (launch_prep)
  const int c0 = rank * per < nchunk_pad ? rank * per : nchunk_pad;
  const int c1 = c0 + per < nchunk_pad ? c0 + per : nchunk_pad;
  const int c = c0 + threadIdx.x;
  const bool live = c < c1 && c < nchunk;
  if (tok == 0 && q.interleave != kLayoutImage && c < c1) {   // the all-zero row
    reinterpret_cast<uint4*>(q.hi + (size_t)q.N * q.d_in_pad)[c] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(q.lo + (size_t)q.N * q.d_in_pad)[c] = make_uint4(0, 0, 0, 0);
  }
  float* rr = RMS ? q.r + (size_t)tok * q.d_in : nullptr;
  uint4* xr = RMS ? nullptr : const_cast<uint4*>(reinterpret_cast<const uint4*>(q.x + (size_t)tok * q.ld));
  float v[8];
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  float ss = 0.0f, ma = 0.0f;
  if (live) {
    if (RMS) {   // r += y
      float4 a, b;
      ld_cg_f8(rr + 8 * c, a, b);
      float f[8];
      finish_chunk<false, KB>(q, tok, 8 * c, f);
      v[0] = __fadd_rn(a.x, f[0]); v[1] = __fadd_rn(a.y, f[1]); v[2] = __fadd_rn(a.z, f[2]);
      v[3] = __fadd_rn(a.w, f[3]); v[4] = __fadd_rn(b.x, f[4]); v[5] = __fadd_rn(b.y, f[5]);
      v[6] = __fadd_rn(b.z, f[6]); v[7] = __fadd_rn(b.w, f[7]);
      reinterpret_cast<float4*>(rr)[2 * c] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4*>(rr)[2 * c + 1] = make_float4(v[4], v[5], v[6], v[7]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss = __fmaf_rn(v[i], v[i], ss);
        ma = fmaxf(ma, fabsf(v[i]));
      }
    } else {     // y as the product would have stored it
      finish_chunk<SWI, KB>(q, tok, 8 * c, v);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i])) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1])) << 16);
      xr[c] = make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ma = fmaxf(ma, fmaxf(fabsf(bf16_bits_to_f32(w[i] & 0xFFFF)), fabsf(bf16_bits_to_f32(w[i] >> 16))));
    }
  }
  // the statistics: each warp's pushed into the table of every CTA of the
  // cluster (remote stores, posted), one cluster barrier, then every warp adds
  // its own CTA's table in the same fixed order
  __shared__ float2 parts[CL * kW];
  __shared__ uint32_t cta_flags;
  if (threadIdx.x == 0) cta_flags = 0u;
#ifdef BWS_TRACE
  tr[2] = trace_now();
#endif
  ss = warp_sum(ss);
  ma = warp_max(ma);
  if (lane < CL) *cl.map_shared_rank(&parts[rank * kW + warp], lane) = make_float2(ss, ma);
  cl.sync();
#ifdef BWS_TRACE
  tr[3] = trace_now();
#endif
  // every remote store into this CTA's table came before the barrier: from
  // here on no CTA of the cluster touches another's shared memory
  float ts = 0.0f, tm = 0.0f;
  for (int i = lane; i < CL * kW; i += 32) {
    const float2 o = parts[i];
    ts += o.x;
    tm = fmaxf(tm, o.y);
  }
  ts = warp_sum(ts);
  tm = warp_max(tm);
  float inv_rms = 1.0f, mx = tm;
  if (RMS) {
    inv_rms = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ts, (float)q.d_in), q.eps)));
    mx = __bfloat162float(__float2bfloat16_rn(__fmul_rn(mx, inv_rms)));
  }
  const int E = mx > 0.0f ? floor_log2_abs(mx) : 0;
  uint32_t flags = 0u;
  if (q.interleave == kLayoutImage) {   // the tensor-core kernel's image reads the row back
    flags = image_chunks<true>(q, c0, c1, rr, xr, inv_rms, E);
  } else if (c < c1) {
    if (live && RMS) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(v[2 * i], inv_rms))) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(v[2 * i + 1], inv_rms))) << 16);
      if (q.tap_x != nullptr)   // verification tap: the BF16 row as formed
        reinterpret_cast<uint4*>(q.tap_x + (size_t)tok * q.d_in)[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    uint4* hi4 = reinterpret_cast<uint4*>(q.hi + (size_t)tok * q.d_in_pad);
    uint4* lo4 = reinterpret_cast<uint4*>(q.lo + (size_t)tok * q.d_in_pad);
    store_bands(w, E, hi4, lo4, band_pos(c, q.interleave), flags);
  }
  // the band flags: the warps' into the CTA's word, then one atomic per CTA
  // (rows of small values set them in most warps; one global address for
  // every warp of the cluster would serialise their atomics)
  const uint32_t wf = __reduce_or_sync(0xffffffffu, flags);
  if (wf != 0u && lane == 0) atomicOr(&cta_flags, wf);
  __syncthreads();
  if (threadIdx.x == 0 && cta_flags != 0u) atomicOr(q.flags + tok, cta_flags);
  if (rank == 0 && threadIdx.x == 0) q.exp[tok] = E;
#ifdef BWS_TRACE
  tr[4] = trace_now();
#endif
#ifdef BWS_TRACE
  if (threadIdx.x == 0) {
    tr[5] = trace_now();
    trace_put(2000u + (RMS ? 10u : 0u) + (SWI ? 1u : 0u) + 100u * CL, tr);
  }
#endif
}

// The plain instantiations keep few registers, so that they fit beside
// running product CTAs; the finishing ones are capped to fit beside one.
template <int CL, int THREADS, bool MOE>
__global__ void __launch_bounds__(THREADS) prep_kernel(const __grid_constant__ PrepParams q) {
  prep_body<CL, THREADS, MOE>(q);
}

template <int CL, int THREADS, int KB, bool RMS, bool SWI, int MINB = 2>
__global__ void __launch_bounds__(THREADS, MINB) prep_fin_kernel(const __grid_constant__ PrepParams q) {
  prep_fin_body<CL, THREADS, KB, RMS, SWI>(q);
}

}  // namespace

bool prep_can_finish(int d) { return (d + 127) / 128 * 128 <= 3 * kLongRow; }

int prep_ctas_per_row(int d, bool fin) { return (d + 127) / 128 * 128 > kLongRow ? 8 : (fin ? 4 : 1); }

cudaError_t launch_prep(const PrepParams& q, cudaStream_t st, bool pdl) {
  const int slots = q.n_slots != nullptr ? q.max_slots : 1;
  const bool long_row = q.d_in_pad > kLongRow;
  const bool moe = q.has_route || q.comb_ys != nullptr;
  const bool fin = q.fin_partials != nullptr;
  if (q.has_route && long_row) return cudaErrorInvalidValue;   // an MoE prep row is one cluster of 4
  // rows: one CTA of 1024 threads; 8192 on, a cluster of 8 x 256. Finishing
  // a product (one slot, no x0, status or combine): a chunk per thread, and
  // registers for a tile's slots in one batch of loads: a cluster of 4 x 256
  // (8 x 384 from 8192 on, to 24576). The residual update takes up to 13
  // slots at once (the 5120-row products with a lighter split have up to 13
  // CTAs per tile), at 159 registers.
  if (fin) {
    const bool rms = q.mode == kPrepRmsNorm;
    if (moe || q.n_slots != nullptr || q.x0 != nullptr || q.hdr != nullptr || q.status_clear != nullptr ||
        rms != (q.fin_epi == kEpiResidF32) || q.d_in_pad > 3 * kLongRow)
      return cudaErrorInvalidValue;
  }
  // An MoE layer's prep (the previous layer's combine, RMSNorm, the routing
  // CTA): a cluster per token row, so that the combine's loads of every
  // slot's outputs are spread over several SMs; the routing CTA is the last
  // of one more cluster, whose other CTAs return at once. Several tokens: 4
  // x 128 (measured, MoE step at one token 1.266 -> 1.250 ms against one CTA
  // of 512; four tokens unchanged). One token with its routing CTA: 8 x 64,
  // whose CTAs (126 registers) also fit beside two expert-product CTAs on an
  // SM, so that neither waits for the other (one token 1.254-1.274 ->
  // 1.236-1.250 ms; at four tokens 2.267 -> 2.275 ms; with a router kernel
  // after the prep instead of the routing CTA 1.749 -> 1.778 ms, so not there).
  const bool moe8 = moe && !long_row && q.N == 1 && q.has_route;
  const int cl = long_row ? 8 : (moe8 ? 8 : (fin || moe ? 4 : 1));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(slots * q.N * cl + (q.has_route ? cl : 0)));
  cfg.blockDim = dim3(long_row ? (fin ? 384 : 256) : (fin ? 256 : (moe ? (moe8 ? 64 : 128) : 1024)));
  cfg.stream = st;
  cudaLaunchAttribute a[2];
  int na = 0;
  if (pdl) {
    a[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cl > 1) {
    a[na].id = cudaLaunchAttributeClusterDimension;
    a[na].val.clusterDim.x = cl;
    a[na].val.clusterDim.y = 1;
    a[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = a;
  cfg.numAttrs = na;
  if (fin) {
    const bool swi = q.fin_epi == kEpiSwiGLU;
    if (q.mode == kPrepRmsNorm)
      return long_row ? cudaLaunchKernelEx(&cfg, prep_fin_kernel<8, 384, 4, true, false>, q)
                      : cudaLaunchKernelEx(&cfg, prep_fin_kernel<4, 256, 13, true, false, 1>, q);
    if (swi)
      return long_row ? cudaLaunchKernelEx(&cfg, prep_fin_kernel<8, 384, 3, false, true>, q)
                      : cudaLaunchKernelEx(&cfg, prep_fin_kernel<4, 256, 4, false, true>, q);
    return long_row ? cudaLaunchKernelEx(&cfg, prep_fin_kernel<8, 384, 4, false, false>, q)
                    : cudaLaunchKernelEx(&cfg, prep_fin_kernel<4, 256, 10, false, false>, q);
  }
  if (long_row)
    return moe ? cudaLaunchKernelEx(&cfg, prep_kernel<8, 256, true>, q)
               : cudaLaunchKernelEx(&cfg, prep_kernel<8, 256, false>, q);
  if (moe8) return cudaLaunchKernelEx(&cfg, prep_kernel<8, 64, true>, q);
  if (moe) return cudaLaunchKernelEx(&cfg, prep_kernel<4, 128, true>, q);
  // the rows of an MoE layer's expert slots (768 values): one 256-thread CTA
  // each, whose reductions are cheaper (measured, MoE step at four tokens
  // 2.288 -> 2.263 ms, one token 1.290 -> 1.287 ms)
  if (q.n_slots != nullptr && q.d_in_pad <= 2048) {
    cfg.blockDim = dim3(256);
    return cudaLaunchKernelEx(&cfg, prep_kernel<1, 256, false>, q);
  }
  return cudaLaunchKernelEx(&cfg, prep_kernel<1, 1024, false>, q);
}

}  // namespace bws

#ifdef BWS_TRACE
extern "C" int bws_trace_read_prep(void* host, int cap) { return bws::trace_read(host, cap); }
#endif
