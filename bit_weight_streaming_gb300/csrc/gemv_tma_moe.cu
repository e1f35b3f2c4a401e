// MXFP4 expert products of an MoE layer fed by TMA: the same producer /
// consumer ring as the dense TMA kernel (gemv_tma.cu), over the live slots of
// a device-side slot table.
//
// Experts. A layer's experts are stacked tensors [E][rows][d_in/2]; the codes
// are cut with a 3D tensor map (box {128 bytes, 32 rows, 1 expert}) whose
// expert coordinate comes from the slot table, the shared expert through a 2D
// map of its own. A tile is 128 output rows of one slot (SwiGLU: 64 gate rows
// and the same 64 up rows); a unit is a tile x 128 bytes of each row (256
// weights, eight E8M0 blocks of 32). Units of all live slots are dealt to the
// CTAs stream-K, as in the dense kernel.
//
// Block scales. MXFP4 scale rows are d_in / 32 bytes (24 for the down
// projection), a row stride TMA cannot take, so the producer warp's 32 lanes
// copy a unit's 128 x 8 scale bytes into the stage with 8-byte cp.async, one
// row of each box per lane; their completions count as 32 arrivals on the
// stage's full barrier, beside the TMA bytes. With one token the scales multiply the FP32
// accumulators (block-diagonal operand, as in the dense kernel); with several
// they become f16 multipliers 2^(e - e_ref) relative to the largest block of
// the warp's row quad in the unit, whose sum is rescaled by 2^e_ref in FP32.
#include <cuda.h>

#include <cstddef>
#include <cstring>

#include "bws_common.cuh"
#include "bws_internal.h"
#include "stream_tile.cuh"
#include "trace.cuh"

namespace bws {

namespace {

constexpr int kCW = 8;                          // consumer warps
constexpr int kThreadsMoe = (kCW + 1) * 32;
constexpr int kMaxStagesMoe = 16;
constexpr int kSmemBudgetMoe = 100 * 1024;
constexpr uint32_t kPollsMoe = 1u << 24;
constexpr uint32_t kStatusTimeoutMoe = 0x100u;
constexpr int kSlotBytesMoe = kBoxes * 2 * 32 * 16;   // one partial-sum slot
constexpr int kScaleBytesMoe = kBoxes * 32 * 8;       // a unit's E8M0 bytes, [box][row][block]

struct MoeTmaParams {
  CUtensorMap experts;    // u8 [E][rows_total][d_in/2], box {128, 32, 1}, 128B swizzle
  CUtensorMap shared;     // u8 [rows_total][d_in/2], box {128, 32}, 128B swizzle
  int has_shared;
  const uint8_t* scales;  // E8M0, expert e at scales + e * scales_stride, [rows_total][d_in/32]
  size_t scales_stride;
  const uint8_t* shared_scales;
  const int* n_slots;
  const int* slot_expert;
  const uint32_t* ready;  // optional: the slot table may be read once this is set (SlotMode::ready)
  int n_prime;            // with ready: stages given their weights before the inputs are ready
  int max_slots;
  int rows;               // rows of one output matrix (inter for gate/up, hidden for down)
  int up_row_off;         // SwiGLU: first up row in the expert tensor
  int tiles_per_slot;
  int N, d_in, d_in_pad, nks;
  XPrep x;                // x.shared: every slot reads slot 0's activations
  void* out;
  int out_ld;
  size_t out_slot_stride;
  float* partials;
  uint32_t* counters;
  uint32_t* status;
  int n_ctas;
  int n_stages, stage_bytes, x_off, x_blk;
};

struct MoeTail {
  float4 red[kBoxes][2][32];
  float4 swi[2][2][32];
  uint4 zero_x[33];             // zero activation pieces, used from element 1 on
  uint64_t full[kMaxStagesMoe];
  uint64_t empty[kMaxStagesMoe];
  int slot_expert[kMaxTokens * kMaxTopk + 1];
  uint32_t flag;
  int n_slots;
#ifdef BWS_TRACE
  unsigned long long tr[4];   // table read, consumers' wait returned, first stage, loop done
#endif
};
static_assert(offsetof(MoeTail, zero_x) % 128 == 0, "zero pieces must start on a 128-byte boundary");

BWS_DEV long long owner_m(long long u, long long U, long long G) { return ((u + 1) * G - 1) / U; }
BWS_DEV long long begin_m(long long c, long long U, long long G) { return c * U / G; }

// First row (in the expert tensor) of box b of local tile lt.
template <int EPI>
BWS_DEV int box_row(const MoeTmaParams& p, int lt, int b) {
  if (EPI == kEpiSwiGLU) return (b < 2 ? 0 : p.up_row_off) + lt * 64 + 32 * (b & 1);
  return lt * 128 + 32 * b;
}
// Rows of the box that exist (the rest of the box is zero-filled by TMA).
template <int EPI>
BWS_DEV int box_limit(const MoeTmaParams& p, int b) {
  return EPI == kEpiSwiGLU ? (b < 2 ? p.rows : p.up_row_off + p.rows) : p.rows;
}

BWS_DEV const uint8_t* scale_base(const MoeTmaParams& p, int e) {
  return e < 0 ? p.shared_scales : p.scales + (size_t)e * p.scales_stride;
}

// f16 2^k for k <= 0, exact down to 2^-24, 0 below.
BWS_DEV uint32_t f16x2_pow2_m(int k) {
  uint32_t h;
  if (k >= -14) h = (uint32_t)(k + 15) << 10;
  else if (k >= -24) h = 1u << (k + 24);
  else h = 0u;
  return h | (h << 16);
}

// One 16-row sub-tile, several tokens: E8M0 codes eg / e8 of rows g / g+8.
template <bool LO>
BWS_DEV void sub_mma_mx(float (&acc)[4], float (&accl)[4], const uint32_t (&w0)[4], const uint32_t (&w1)[4],
                        int eg, int e8, const uint4 (&xh)[4], const uint4 (&xl)[4]) {
  int rg = max(eg, __shfl_xor_sync(0xffffffffu, eg, 1));
  rg = max(rg, __shfl_xor_sync(0xffffffffu, rg, 2));
  int r8 = max(e8, __shfl_xor_sync(0xffffffffu, e8, 1));
  r8 = max(r8, __shfl_xor_sync(0xffffffffu, r8, 2));
  const uint32_t sa = f16x2_pow2_m(eg - rg), sb = f16x2_pow2_m(e8 - r8);
  float d[4] = {0.f, 0.f, 0.f, 0.f}, dl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t p0, p1, p2, p3, q0, q1, q2, q3;
    e2m1x8_to_f16x2x4(w0[w], p0, p1, p2, p3);
    e2m1x8_to_f16x2x4(w1[w], q0, q1, q2, q3);
    p0 = hmul2_u32(p0, sa); p1 = hmul2_u32(p1, sa); p2 = hmul2_u32(p2, sa); p3 = hmul2_u32(p3, sa);
    q0 = hmul2_u32(q0, sb); q1 = hmul2_u32(q1, sb); q2 = hmul2_u32(q2, sb); q3 = hmul2_u32(q3, sb);
    mma_f16_16816(d, p0, q0, p1, q1, xh[w].x, xh[w].y);
    mma_f16_16816(d, p2, q2, p3, q3, xh[w].z, xh[w].w);
    if (LO) {
      mma_f16_16816(dl, p0, q0, p1, q1, xl[w].x, xl[w].y);
      mma_f16_16816(dl, p2, q2, p3, q3, xl[w].z, xl[w].w);
    }
  }
  const float sg = exp2i(rg - 127), s8 = exp2i(r8 - 127);
  acc[0] = __fmaf_rn(d[0], sg, acc[0]);
  acc[1] = __fmaf_rn(d[1], sg, acc[1]);
  acc[2] = __fmaf_rn(d[2], s8, acc[2]);
  acc[3] = __fmaf_rn(d[3], s8, acc[3]);
  if (LO) {
    accl[0] = __fmaf_rn(dl[0], sg, accl[0]);
    accl[1] = __fmaf_rn(dl[1], sg, accl[1]);
    accl[2] = __fmaf_rn(dl[2], s8, accl[2]);
    accl[3] = __fmaf_rn(dl[3], s8, accl[3]);
  }
}

// One 16-row sub-tile, one token: block-diagonal operand (see sub_mma_n1);
// the lane's 32 weights of a row are one block, scale 2^(e - 127).
template <bool LO>
BWS_DEV void sub_mma_mx_n1(float (&y)[4], float (&yl)[4], const uint32_t (&w0)[4], const uint32_t (&w1)[4], int eg,
                           int e8, const uint4 (&xh)[4], const uint4 (&xl)[4]) {
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
  const float sg = exp2i(eg - 127), s8 = exp2i(e8 - 127);
  y[0] = __fmaf_rn(sg, da[0], y[0]);
  y[1] = __fmaf_rn(sg, db[1], y[1]);
  y[2] = __fmaf_rn(s8, da[2], y[2]);
  y[3] = __fmaf_rn(s8, db[3], y[3]);
  if (LO) {
    yl[0] = __fmaf_rn(sg, la[0], yl[0]);
    yl[1] = __fmaf_rn(sg, lb[1], yl[1]);
    yl[2] = __fmaf_rn(s8, la[2], yl[2]);
    yl[3] = __fmaf_rn(s8, lb[3], yl[3]);
  }
}

// Store v (raw sums of sub-tile st of box b; register i = row g + 8*(i>>1),
// token 2t + (i&1)). SwiGLU: b is a gate box and vu the matching up sums.
template <int EPI>
BWS_DEV void store_moe(const MoeTmaParams& p, int tile, int b, int st, int g, int t, const float (&v)[4],
                       const float (&vu)[4]) {
  const int slot = tile / p.tiles_per_slot, lt = tile - slot * p.tiles_per_slot;
  const int xb = p.x.shared ? 0 : slot;
  const int row0 = (EPI == kEpiSwiGLU ? lt * 64 + 32 * b : lt * 128 + 32 * b) + 16 * st;
  int xexp[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int tok = 2 * t + i;
    xexp[i] = tok < p.N ? __ldg(p.x.exp + xb * p.N + tok) : 0;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = row0 + g + 8 * (i >> 1);
    const int tok = 2 * t + (i & 1);
    if (row >= p.rows || tok >= p.N) continue;
    const float val = ldexp_exact(v[i], xexp[i & 1] - 14);
    if (EPI == kEpiSwiGLU) {
      const float up = ldexp_exact(vu[i], xexp[i & 1] - 14);
      reinterpret_cast<__nv_bfloat16*>(p.out)[slot * p.out_slot_stride + (size_t)tok * p.out_ld + row] =
          __float2bfloat16_rn(silu_mul_t(val, up));
    } else {
      reinterpret_cast<float*>(p.out)[slot * p.out_slot_stride + (size_t)tok * p.out_ld + row] = val;
    }
  }
}

template <int EPI, bool LO, bool N1>
BWS_DEV void consume_moe(const MoeTmaParams& p, MoeTail& T, uint32_t stage0, long long u0, long long u1,
                         long long U, long long G, int warp, int lane) {
  const int NS = p.n_stages;
  const int b = warp & 3, half = warp >> 2;
  const int g = lane >> 2, t = lane & 3;
  const int c = 2 * t + half;
  const uint32_t coff = b * kBoxBytes + g * 128 + ((c ^ g) << 4);
  const int xg = g < p.N ? g : 0;
  const uint32_t xoff = (uint32_t)(p.x_off + xg * p.x_blk + c * 16);
  const bool m01 = g == 2 * t, m23 = g == 2 * t + 1;
  const uint32_t zaddr = smem_u32(&T.zero_x[1]) + c * 16;
  float acc[2][2][4] = {}, accl[2][4] = {};   // N1: acc[st][0] holds y
  uint4 xh[4], xl[4];
  bool dead = false;
  int tile = (int)(u0 / p.nks), ks = (int)(u0 % p.nks);
  int s = 0;
  uint32_t ph = 0u;
  bool piece_whole = ks == 0;
  // this lane's scale bytes in a stage: rows g + 8j of box b, block c
  const uint32_t soff = (uint32_t)(kCodeBytes + b * 256 + g * 8 + c);
  for (long long u = u0; u < u1; ++u) {
    const int slot = tile / p.tiles_per_slot;
    if (LO) {
      const uint16_t* xrow_l = p.x.lo + ((size_t)(p.x.shared ? 0 : slot) * (p.N + 1) + xg) * p.d_in_pad;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xl[q] = ld_act_v4(xrow_l + (size_t)ks * 256 + q * 64 + c * 8);
        if (N1 && !(q < 2 ? m01 : m23)) xl[q] = make_uint4(0, 0, 0, 0);
      }
    }
    if (!dead && !mbar_wait_bounded(smem_u32(&T.full[s]), ph, kPollsMoe)) {
      if (lane == 0) atomicOr(p.status, kStatusTimeoutMoe);
      dead = true;
    }
#ifdef BWS_TRACE
    if (u == u0 && threadIdx.x == 0) T.tr[2] = trace_now();
#endif
    const uint32_t base = stage0 + (uint32_t)s * p.stage_bytes;
    uint4 cw[4];
    uint32_t sc = 0u;
    if (!dead) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        cw[j] = lds_v4(base + coff + j * 1024);
        sc |= lds_u8(base + soff + j * 64) << (8 * j);
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
        for (int q = 0; q < 4; ++q) xh[q] = lds_v4(base + xoff + q * 128);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) cw[j] = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < 4; ++q) xh[q] = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
    if (lane == 0 && !dead) mbar_arrive(smem_u32(&T.empty[s]));
    if (++s == NS) { s = 0; ph ^= 1u; }
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const uint32_t w0[4] = {cw[2 * st].x, cw[2 * st].y, cw[2 * st].z, cw[2 * st].w};
      const uint32_t w1[4] = {cw[2 * st + 1].x, cw[2 * st + 1].y, cw[2 * st + 1].z, cw[2 * st + 1].w};
      const int eg = (int)((sc >> (16 * st)) & 0xFFu), e8 = (int)((sc >> (16 * st + 8)) & 0xFFu);
      if constexpr (N1)
        sub_mma_mx_n1<LO>(acc[st][0], accl[st], w0, w1, eg, e8, xh, xl);
      else
        sub_mma_mx<LO>(acc[st][0], accl[st], w0, w1, eg, e8, xh, xl);
    }
    const bool last_of_tile = ks == p.nks - 1;
    const int cur_tile = tile;
    if (++ks == p.nks) { ks = 0; ++tile; }
    if (!last_of_tile && u + 1 < u1) continue;
    float v[2][4];
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      if constexpr (N1) {
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
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) v[st][r] = LO ? __fmaf_rn(accl[st][r], 0x1p-29f, acc[st][0][r]) : acc[st][0][r];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[st][0][r] = acc[st][1][r] = accl[st][r] = 0.f;
    }
    if (half == 1) {
#pragma unroll
      for (int st = 0; st < 2; ++st) T.red[b][st][lane] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
    }
    named_bar_sync(1, kCW * 32);
    if (half == 0) {
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        const float4 o = T.red[b][st][lane];
        v[st][0] += o.x; v[st][1] += o.y; v[st][2] += o.z; v[st][3] += o.w;
      }
    }
    named_bar_sync(1, kCW * 32);
    const bool whole = piece_whole && last_of_tile;
    piece_whole = true;
    if (half == 1) continue;
    if (!whole) {
      float4* slot4 = reinterpret_cast<float4*>(p.partials) + ((size_t)(cur_tile + blockIdx.x) * kBoxes + b) * 64;
#pragma unroll
      for (int st = 0; st < 2; ++st) slot4[st * 32 + lane] = make_float4(v[st][0], v[st][1], v[st][2], v[st][3]);
      named_bar_sync(2, 4 * 32);   // deposits, then an acquire-release count (see gemv_tma.cu)
      const long long c0 = owner_m((long long)cur_tile * p.nks, U, G);
      const long long c1 = owner_m((long long)(cur_tile + 1) * p.nks - 1, U, G);
      if (threadIdx.x == 0) T.flag = atom_add_acq_rel_gpu(p.counters + cur_tile, 1u);
      named_bar_sync(2, 4 * 32);
      const uint32_t prev = T.flag;
      named_bar_sync(2, 4 * 32);
      if (prev != (uint32_t)(c1 - c0)) continue;
      float a8[2][4] = {};
      const float4* slots = reinterpret_cast<const float4*>(p.partials) + (size_t)cur_tile * kBoxes * 64 + b * 64 + lane;
      for (long long cc = c0; cc <= c1; ++cc) {
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          const float4 o = cc == blockIdx.x ? make_float4(v[st][0], v[st][1], v[st][2], v[st][3])
                                            : ld_cg_f4(slots + (size_t)cc * kBoxes * 64 + st * 32);
          a8[st][0] += o.x; a8[st][1] += o.y; a8[st][2] += o.z; a8[st][3] += o.w;
        }
      }
#pragma unroll
      for (int st = 0; st < 2; ++st)
#pragma unroll
        for (int r = 0; r < 4; ++r) v[st][r] = a8[st][r];
      if (threadIdx.x == 0) p.counters[cur_tile] = 0u;
    }
    if (EPI == kEpiSwiGLU) {
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
          store_moe<EPI>(p, cur_tile, b, st, g, t, v[st], vu);
        }
      }
      named_bar_sync(3, 4 * 32);
    } else {
      const float none[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int st = 0; st < 2; ++st) store_moe<EPI>(p, cur_tile, b, st, g, t, v[st], none);
    }
  }
#ifdef BWS_TRACE
  if (threadIdx.x == 0) T.tr[3] = trace_now();
#endif
}

template <int EPI, bool N1>
__device__ __noinline__ void consume_moe_lo(const MoeTmaParams& p, MoeTail& T, uint32_t stage0, long long u0,
                                            long long u1, long long U, long long G, int warp, int lane) {
  consume_moe<EPI, true, N1>(p, T, stage0, u0, u1, U, G, warp, lane);
}

template <int EPI, bool N1>
__global__ void __launch_bounds__(kThreadsMoe, 2) gemv_tma_moe_kernel(const __grid_constant__ MoeTmaParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
#ifdef BWS_TRACE
  const unsigned long long tr_start = trace_now();
#endif
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* sbase = smem_raw + ((1024u - mis) & 1023u);
  MoeTail& T = *reinterpret_cast<MoeTail*>(sbase + (size_t)p.n_stages * p.stage_bytes);
  const uint32_t stage0 = smem_u32(sbase);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = p.n_stages;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&T.full[i]), 1 + 32);
      mbar_init(smem_u32(&T.empty[i]), kCW);
    }
    T.flag = 0u;
    mbar_fence_init();
  }
  for (int i = threadIdx.x; i < 33; i += blockDim.x) T.zero_x[i] = make_uint4(0, 0, 0, 0);
  // the slot table: with a ready flag, written by a routing CTA that does not
  // wait for the kernels before, so it is read (and the first weight stages
  // issued) before this kernel waits for them; else the previous kernel's output
  const bool early = p.ready != nullptr;
  if (early) {
    if (threadIdx.x == 0 && !poll_acquire(p.ready, kPollsMoe)) atomicOr(p.status, kStatusTimeoutMoe);
    __syncthreads();   // the table reads below follow thread 0's acquire
  } else {
    pdl_wait();
  }
  if (threadIdx.x == 0) {
    // (read through L2: with a ready flag the table is written while this kernel runs)
    int n = early ? __ldcg(p.n_slots) : __ldg(p.n_slots);
    n = n < 0 ? 0 : (n > p.max_slots ? p.max_slots : n);
    T.n_slots = n;
  }
  for (int i = threadIdx.x; i < p.max_slots; i += blockDim.x)
    T.slot_expert[i] = early ? __ldcg(p.slot_expert + i) : __ldg(p.slot_expert + i);
  __syncthreads();
#ifdef BWS_TRACE
  if (threadIdx.x == 0) T.tr[0] = trace_now();
#endif
  // units dealt over G = min(CTAs, units) CTAs, so that every CTA that
  // shares a tile holds at least one unit of it; the rest have none
  const long long U = (long long)T.n_slots * p.tiles_per_slot * p.nks;
  const long long G = U < p.n_ctas ? U : p.n_ctas;
  const long long u0 = blockIdx.x < G ? begin_m(blockIdx.x, U, G) : U;
  const long long u1 = blockIdx.x < G ? begin_m(blockIdx.x + 1, U, G) : U;

  if (warp == kCW) {
    // ---- producer warp: lane 0 the TMA code boxes and activations of each
    // unit, every lane one scale row of each box ----
    const int rb = p.d_in >> 5;
    const uint64_t pol = l2_evict_first();   // expert weights are read once per step
    // the weights of unit (tile, ks) into stage s (the full barrier also
    // expects the unit's activation bytes), and its activations
    auto issue_w = [&](int tile, int ks, int s) {
      const int slot = tile / p.tiles_per_slot, lt = tile - slot * p.tiles_per_slot;
      const int e = T.slot_expert[slot];
      const uint32_t full = smem_u32(&T.full[s]);
      const uint32_t dst = stage0 + (uint32_t)s * p.stage_bytes;
      if (lane == 0) {
        mbar_arrive_expect_tx(full, (uint32_t)(kCodeBytes + p.N * 512));
#pragma unroll
        for (int b = 0; b < kBoxes; ++b) {
          const int row = box_row<EPI>(p, lt, b);
          if (e < 0)
            tma_load_2d_hint(dst + b * kBoxBytes, &p.shared, ks * 128, row, full, pol);
          else
            tma_load_3d_hint(dst + b * kBoxBytes, &p.experts, ks * 128, row, e, full, pol);
        }
      }
      const uint8_t* sb = scale_base(p, e) + ks * 8;
#pragma unroll
      for (int b = 0; b < kBoxes; ++b) {
        const int row = box_row<EPI>(p, lt, b) + lane;
        const bool in = row < box_limit<EPI>(p, b);
        cp_async8_zfill_hint(dst + kCodeBytes + b * 256 + lane * 8, sb + (size_t)(in ? row : 0) * rb, in ? 8u : 0u,
                             pol);
      }
      cp_async_mbar_arrive(full);
    };
    auto issue_x = [&](int tile, int ks, int s) {
      if (lane != 0) return;
      const int slot = tile / p.tiles_per_slot;
      const uint32_t full = smem_u32(&T.full[s]);
      const uint32_t dst = stage0 + (uint32_t)s * p.stage_bytes;
      const uint16_t* src = p.x.hi + (size_t)(p.x.shared ? 0 : slot) * (p.N + 1) * p.d_in_pad + (size_t)ks * 256;
      for (int tok = 0; tok < p.N; ++tok)
        bulk_load(dst + p.x_off + tok * p.x_blk, src + (size_t)tok * p.d_in_pad, 512, full);
    };
    int tile = (int)(u0 / p.nks), ks = (int)(u0 % p.nks);
    int s = 0;
    uint32_t ph = 0u;
    long long issued = 0;
    if (early) {   // weights of the first stages, then the wait, then their activations
      const long long n_pre = (u1 - u0) < p.n_prime ? (u1 - u0) : p.n_prime;
      for (long long k = 0; k < n_pre; ++k) {
        issue_w(tile, ks, s);
        if (++ks == p.nks) { ks = 0; ++tile; }
        ++s;
      }
      pdl_wait();
      tile = (int)(u0 / p.nks);
      ks = (int)(u0 % p.nks);
      for (long long k = 0; k < n_pre; ++k) {
        issue_x(tile, ks, (int)k);
        if (++ks == p.nks) { ks = 0; ++tile; }
      }
      issued = n_pre;   // n_prime < NS: the stages after them are still free
      if (s == NS) { s = 0; ph ^= 1u; }
    }
    for (long long u = u0 + issued; u < u1; ++u, ++issued) {
      if (issued >= NS) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(smem_u32(&T.empty[s]), ph ^ 1u, kPollsMoe);
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          if (lane == 0) atomicOr(p.status, kStatusTimeoutMoe);
          break;
        }
      }
      issue_w(tile, ks, s);
      issue_x(tile, ks, s);
      if (++s == NS) { s = 0; ph ^= 1u; }
      if (++ks == p.nks) { ks = 0; ++tile; }
    }
    // copies in flight land before the CTA's shared memory goes away
    if (lane == 0)
      for (long long k = (issued > NS ? issued - NS : 0); k < issued; ++k)
        mbar_wait_bounded(smem_u32(&T.full[k % NS]), (uint32_t)(k / NS) & 1u, kPollsMoe);
    __syncwarp();
    return;
  }

  // ---- consumers ----
  if (early) pdl_wait();   // the activations are the previous kernel's output
#ifdef BWS_TRACE
  if (threadIdx.x == 0) T.tr[1] = trace_now();
#endif
  // the lo band is needed if any activation row this CTA reads has one
  uint32_t fl = 0u;
  if (u0 < u1) {
    const int per = p.tiles_per_slot * p.nks;
    const int s0 = p.x.shared ? 0 : (int)(u0 / per), s1 = p.x.shared ? 0 : (int)((u1 - 1) / per);
    for (int i = s0 * p.N + lane; i < (s1 + 1) * p.N; i += 32) fl |= __ldg(p.x.flags + i);
    fl = __reduce_or_sync(0xffffffffu, fl);
  }
  if (fl & 1u)
    consume_moe_lo<EPI, N1>(p, T, stage0, u0, u1, U, G, warp, lane);
  else
    consume_moe<EPI, false, N1>(p, T, stage0, u0, u1, U, G, warp, lane);
#ifdef BWS_TRACE
  if (threadIdx.x == 0) {
    const unsigned long long t[6] = {tr_start, T.tr[0], T.tr[1], T.tr[2], T.tr[3], trace_now()};
    trace_put(4000u + 10u * EPI + (early ? 1u : 0u), t);
  }
#endif
}

template <int EPI, bool N1>
cudaError_t launch_moe_one(const MoeTmaParams& p, cudaStream_t st, bool pdl) {
  const int smem = p.n_stages * p.stage_bytes + (int)sizeof(MoeTail) + 1024;
  static std::atomic<unsigned long long> attr{0};
  {
    const cudaError_t e = set_smem_once(attr, gemv_tma_moe_kernel<EPI, N1>, kSmemBudgetMoe + (int)sizeof(MoeTail) + 1024);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_ctas);
  cfg.blockDim = dim3(kThreadsMoe);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_tma_moe_kernel<EPI, N1>, p);
}

}  // namespace

bool moe_tma_shape_ok(const uint8_t* codes, size_t codes_stride, const uint8_t* shared_codes, const uint8_t* scales,
                      size_t scales_stride, const uint8_t* shared_scales, int d_in, int N) {
  if (!tensor_maps_available()) return false;
  if (d_in % 256 != 0 || N < 1 || N > kMaxTokens) return false;
  if (((uintptr_t)codes & 15) || (codes_stride & 15)) return false;
  if (shared_codes && ((uintptr_t)shared_codes & 15)) return false;
  // 8-byte scale copies
  if (((uintptr_t)scales & 7) || (scales_stride & 7) || (shared_scales && ((uintptr_t)shared_scales & 7))) return false;
  return true;
}

int moe_tma_tiles_per_slot(int epi, int rows) { return epi == kEpiSwiGLU ? (rows + 63) / 64 : (rows + 127) / 128; }

size_t moe_tma_partials_bytes(int epi, int rows, int max_slots) {
  return ((size_t)moe_tma_tiles_per_slot(epi, rows) * max_slots + 2 * (size_t)num_sms()) * kSlotBytesMoe;
}

bool moe_tma_eligible(int epi, const GemvParams& g) {
  if (g.slots.n_slots == nullptr || g.slots.max_slots > kMaxTokens * kMaxTopk + 1) return false;
  // scratch of the caller's workspace: a counter per tile, a partial slot
  // per tile and CTA
  const long long tiles = (long long)g.slots.max_slots * moe_tma_tiles_per_slot(epi, g.slots.rows);
  if (tiles > g.n_tiles || g.partials_bytes < moe_tma_partials_bytes(epi, g.slots.rows, g.slots.max_slots))
    return false;
  return moe_tma_shape_ok(g.slots.codes, g.slots.codes_stride, g.slots.shared_codes, g.slots.scales,
                          g.slots.scales_stride, g.slots.shared_scales, g.d_in, g.N);
}

// The MXFP4 expert product described by g (slot mode; activations prepared
// in the TMA layout of 256-weight units), in the scratch of the MoE workspace:
// g.counters (tiles_per_slot * max_slots words, zero) and g.partials.
cudaError_t launch_gemv_tma_moe(int epi, const GemvParams& g, uint32_t* status, cudaStream_t st, bool pdl) {
  MoeTmaParams p;
  memset(&p, 0, sizeof(p));
  const SlotMode& S = g.slots;
  const uint64_t rb = (uint64_t)g.d_in / 2;
  const uint64_t rows_total = epi == kEpiSwiGLU ? (uint64_t)S.up_row_off + S.rows : (uint64_t)S.rows;
  if (!encode_3d(&p.experts, S.codes, rb, rows_total, (uint64_t)S.n_experts, (uint64_t)S.codes_stride, 128,
                 kBoxRows))
    return cudaErrorInvalidValue;
  p.has_shared = S.shared_codes != nullptr;
  if (p.has_shared && !encode_2d(&p.shared, S.shared_codes, rb, rows_total, 128, kBoxRows, true))
    return cudaErrorInvalidValue;
  p.scales = S.scales;
  p.scales_stride = S.scales_stride;
  p.shared_scales = S.shared_scales;
  p.n_slots = S.n_slots;
  p.slot_expert = S.slot_expert;
  p.ready = S.ready;
  p.max_slots = S.max_slots;
  p.rows = S.rows;
  p.up_row_off = S.up_row_off;
  p.tiles_per_slot = moe_tma_tiles_per_slot(epi, S.rows);
  p.N = g.N;
  p.d_in = g.d_in;
  p.d_in_pad = g.d_in_pad;
  p.nks = g.d_in / 256;
  p.x = g.x;
  p.out = g.out;
  p.out_ld = g.out_ld;
  p.out_slot_stride = g.out_slot_stride;
  p.partials = g.partials;
  p.counters = g.counters;
  p.status = status;
  // scratch: counters for every (slot, tile), partial slots for tiles + CTAs
  if (!moe_tma_eligible(epi, g)) return cudaErrorInvalidValue;
  p.n_ctas = 2 * num_sms();
  p.x_off = kCodeBytes + kScaleBytesMoe;
  p.x_blk = 512 + 16;
  p.stage_bytes = ((p.x_off + g.N * p.x_blk) + 1023) / 1024 * 1024;
  p.n_stages = kSmemBudgetMoe / p.stage_bytes;
  if (p.n_stages > kMaxStagesMoe) p.n_stages = kMaxStagesMoe;
  if (p.n_stages < 2) return cudaErrorInvalidValue;
  // weights ahead of the inputs: one stage at one token; with more tokens
  // none (measured, MoE step at one token, 0 / 1 / 2 / 3 / 5 stages: 1.329 /
  // 1.277 / 1.292 / 1.308 / 1.307 ms; at four tokens 0 / 1 / 2: 2.450 /
  // 2.482 / 2.477 ms; the table still read early)
  p.n_prime = g.N == 1 ? 1 : 0;
  if (p.n_prime > p.n_stages) p.n_prime = p.n_stages;
  const bool n1 = g.N == 1;
  if (epi == kEpiSwiGLU) return n1 ? launch_moe_one<kEpiSwiGLU, true>(p, st, pdl) : launch_moe_one<kEpiSwiGLU, false>(p, st, pdl);
  if (epi == kEpiStoreF32)
    return n1 ? launch_moe_one<kEpiStoreF32, true>(p, st, pdl) : launch_moe_one<kEpiStoreF32, false>(p, st, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace bws

#ifdef BWS_TRACE
extern "C" int bws_trace_read_moe(void* host, int cap) { return bws::trace_read(host, cap); }
#endif
