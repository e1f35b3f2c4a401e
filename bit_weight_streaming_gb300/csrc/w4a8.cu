// W4A8 products on the fifth-generation tensor cores: MXFP4 weights (E2M1
// codes, one E8M0 scale per 32 weights) times MXFP8 activations (E4M3 codes,
// one E8M0 scale per 32 values) for N <= 8 tokens, FP32 accumulation
// ([LingMoE] section 3: the MoE baseline runs W4A8, MXFP4 weights with 8-bit
// activations; the activation quantizer is read from the OCP MX rule).
//
// Both operands' scale blocks are 32 long, which is the K of one
// tcgen05.mma.kind::f8f6f4 instruction (M = 128 rows, N = 16, K = 32). So each
// MMA multiplies one scale block of 128 weight rows by the same block of
// every token, with no scale inside its sum: the E2M1 x E4M3 products are
// exact and the tensor cores add 32 of them in FP32. The epilogue warps then
// apply the block's two power-of-two scales, 2^(sw - 127) 2^(sx - 127), whose
// product is exact, with one fused multiply-add per block and token.
//
// Operands: TMA unpacks every 16 E2M1 codes into a 16-byte slot on the way
// into shared memory (the layout kind::f8f6f4 reads 4-bit operands in),
// 128B-swizzled, as the NVFP4 tensor-core kernel does. The activations are
// quantized once per call into an image laid out the way the MMA reads its
// B operand: per unit of 256 K values, per MMA, two 8x16-byte core matrices
// (K halves) of eight token rows; tokens past N are zero, and the operand's
// second eight rows read a zero area of the stage. The unit's 64 activation
// scale bytes follow its image. The weight scales (8 bytes per row and unit)
// are too narrow for a TMA box, so the producer warp's lanes copy them with
// 8-byte cp.async, four rows per lane.
//
// Roles, one CTA of ten warps per SM: warp 0 streams units (tile of 128 rows
// x 256 K) into a ring of stages; warp 1 owns 512 TMEM columns (four D
// buffers of 8 MMAs x 16 columns), copies each unit's scales to a ring in
// shared memory and issues its eight MMAs; warps 2-9 fold the products, two
// warps per TMEM lane quarter (one output row per thread), one per K half of
// the unit. Units are dealt to the CTAs stream-K with the deterministic
// last-arriver fix-up of the other kernels.
#include <cuda.h>

#include <cstddef>
#include <cstring>

#include "bws_abi_util.h"
#include "bws_common.cuh"
#include "bws_internal.h"
#include "stream_tile.cuh"

namespace bws {

namespace {

constexpr int kWWarps = 10;                  // producer, MMA, eight epilogue warps
constexpr int kWThreads = kWWarps * 32;
constexpr int kWRows = 128;                  // tile rows, the MMA's M
constexpr int kWHalf = kWRows * 128;         // one K half of a unit's unpacked codes
constexpr int kWA = 2 * kWHalf;              // the unit's codes
constexpr int kWImg = 2048;                  // 8 MMAs x two 8-row x 16-byte core matrices
constexpr int kWXs = 64;                     // the unit's activation scales [MMA][token]
constexpr int kWImgU = kWImg + kWXs;         // a unit's activation bytes in global memory
constexpr int kOffImg = kWA;
constexpr int kOffXs = kOffImg + kWImg;
constexpr int kOffZero = kOffXs + 128;       // the B operand's second row group (zeros)
constexpr int kOffWs = kOffZero + kWImg;     // weight scales [row][8]
constexpr int kWStageUsed = kOffWs + kWRows * 8;
constexpr int kWStage = (kWStageUsed + 1023) / 1024 * 1024;
constexpr int kWMaxStages = 8;
constexpr int kWNumStages = (190 * 1024) / kWStage;   // the CTA has the SM to itself
static_assert(kWNumStages <= kWMaxStages, "barrier arrays");
constexpr int kWDCols = 128;                 // TMEM columns of one unit (8 MMAs x N = 16)
constexpr int kWDBufs = 4;
constexpr int kWTmemCols = kWDBufs * kWDCols;
constexpr int kWEpi = 8 * 32;
constexpr uint32_t kWTx = kWHalf + kWImgU;   // TMA bytes a stage receives (codes counted packed)
constexpr uint32_t kWPolls = 1u << 24;
constexpr uint32_t kWTimeout = 0x100u;

// Instruction descriptor: D FP32, A E2M1, B E4M3, both K-major, M = 128, N = 16.
constexpr uint32_t kWIdesc = (1u << 4) | (5u << 7) | (0u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

struct WParams {
  CUtensorMap codes;    // E2M1 [d_out][d_in / 2], unpacked to 16-byte slots, box {128 codes, 32 rows}
  const uint8_t* wscales;   // E8M0 [d_out][d_in / 32]
  int d_out, d_in, N;
  int nks, n_tiles;
  long long n_units;
  int n_ctas, n_stages;
  const uint8_t* img;   // activation image, kWImgU bytes per unit
  uint16_t* y;          // bf16 [N][d_out]
  float* partials;      // [(n_tiles + n_ctas)][8][128]
  uint32_t* counters;   // [n_tiles], zero on entry, left zero
  uint32_t* status;
};

struct WTail {
  uint2 wsc[kWDBufs][kWRows];      // weight scale bytes of the units in the D buffers, one row each
  float4 xsf[kWDBufs][16];         // their activation scales 2^(e - 127) [MMA][token]
  float red[kMaxTokens][kWRows];   // the second K half's sums handed to the first
  uint64_t full[kWMaxStages];
  uint64_t empty[kWMaxStages];
  uint64_t dfull[kWDBufs], dempty[kWDBufs], drain;
  uint32_t tmem;
  uint32_t flag;
};

BWS_DEV long long w_owner(long long u, long long U, long long G) { return ((u + 1) * G - 1) / U; }
BWS_DEV long long w_begin(long long c, long long U, long long G) { return c * U / G; }

BWS_DEV uint64_t w_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46) | ((uint64_t)layout << 61);
}
BWS_DEV void w_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
BWS_DEV void w_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
BWS_DEV void w_mma(uint32_t d, uint64_t a, uint64_t b) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(kWIdesc), "r"(0u)
      : "memory");
}
BWS_DEV void w_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
BWS_DEV void w_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
BWS_DEV void w_wait_ld(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
        "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// MXFP8 quantization of the activations, one warp per (token slot, block of
// 32 values), lane j holding value j: amax by a warp reduction over the
// values' magnitude bits, e = clamp(floor(log2 amax) - 8, -127, 127), codes
// E4M3(x * 2^-e) (nearest even, saturating; the scaling is exact). With img
// the codes and scale bytes also go to the product's image, where the token
// slots N..7 are zero. Zeroes n_zero words at zero (the product's counters).
__global__ void __launch_bounds__(256) mxfp8_kernel(const uint16_t* __restrict__ x, int N, int d,
                                                   uint8_t* codes, uint8_t* scales, uint8_t* img, uint32_t* zero,
                                                   int n_zero, uint32_t* hdr) {
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero[i] = 0u;
  if (hdr != nullptr && blockIdx.x == 0 && threadIdx.x < 2) hdr[threadIdx.x] = 0u;   // no flags; status clear
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  const int nb = d >> 5;
  const int slots = img != nullptr ? kMaxTokens : N;
  if (gw >= slots * nb) return;
  const int tok = gw / nb, b = gw - tok * nb;
  const int k = b * 32 + lane;
  uint32_t code = 0u, sc = 0u;
  if (tok < N) {
    const float v = __uint_as_float((uint32_t)x[(size_t)tok * d + k] << 16);
    const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7FFFFFFFu);
    if (amax != 0u) {
      int e = floor_log2_abs(__uint_as_float(amax)) - 8;
      e = e < -127 ? -127 : (e > 127 ? 127 : e);
      code = f32x2_to_e4m3x2(0.0f, ldexp_exact(v, -e)) & 0xFFu;
      sc = (uint32_t)(e + 127);
    }
    if (codes != nullptr) codes[(size_t)tok * d + k] = (uint8_t)code;
    if (scales != nullptr && lane == 0) scales[(size_t)tok * nb + b] = (uint8_t)sc;
  }
  if (img != nullptr) {
    const int ks = k >> 8, kk = (k >> 5) & 7, half = (k >> 4) & 1;
    uint8_t* u = img + (size_t)ks * kWImgU;
    u[kk * 256 + half * 128 + tok * 16 + (k & 15)] = (uint8_t)code;
    if (lane == 0) u[kWImg + kk * 8 + tok] = (uint8_t)sc;
  }
}

__global__ void __launch_bounds__(kWThreads, 1) w4a8_kernel(const __grid_constant__ WParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* sbase = smem_raw + ((1024u - mis) & 1023u);
  const int NS = p.n_stages;
  WTail& T = *reinterpret_cast<WTail*>(sbase + (size_t)NS * kWStage);
  const uint32_t stage0 = smem_u32(sbase);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&T.tmem)),
                 "n"(kWTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&T.full[i]), 1 + 32);   // the TMA bytes' arrival and each lane's scale copies
      mbar_init(smem_u32(&T.empty[i]), 1);
    }
    for (int d = 0; d < kWDBufs; ++d) {
      mbar_init(smem_u32(&T.dfull[d]), 2);    // the scale copy and the MMA commit
      mbar_init(smem_u32(&T.dempty[d]), 8);   // the eight epilogue warps
    }
    mbar_init(smem_u32(&T.drain), 1);
    T.flag = 0u;
    mbar_fence_init();
  }
  // the B operand's second eight rows (token columns 8..15) read zeros
  for (int i = threadIdx.x; i < NS * (kWImg / 16); i += blockDim.x) {
    const int s = i / (kWImg / 16), o = i - s * (kWImg / 16);
    *reinterpret_cast<uint4*>(sbase + (size_t)s * kWStage + kOffZero + 16 * o) = make_uint4(0, 0, 0, 0);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  w_fence_before();
  __syncthreads();
  w_fence_after();
  const long long U = p.n_units, G = p.n_ctas;
  const long long u0 = w_begin(blockIdx.x, U, G), u1 = w_begin(blockIdx.x + 1, U, G);
  const int nks = p.nks;
  const int rb = p.d_in >> 5;   // scale bytes per weight row

  if (warp == 0) {
    // ---- producer: the weights of the first stages before the activations are ready ----
    const uint64_t pol = l2_evict_first();   // weights are read once
    if (lane == 0) tma_prefetch_desc(&p.codes);
    auto issue_w = [&](int tile, int ks, int s) {
      const uint32_t full = smem_u32(&T.full[s]);
      const uint32_t dst = stage0 + (uint32_t)s * kWStage;
      if (lane == 0) {
        mbar_arrive_expect_tx(full, kWTx);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b) {
          const int row = tile * kWRows + kBoxRows * b;
          tma_load_2d_hint(dst + b * kBoxBytes, &p.codes, ks * 256, row, full, pol);
          tma_load_2d_hint(dst + kWHalf + b * kBoxBytes, &p.codes, ks * 256 + 128, row, full, pol);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = lane * 4 + q, row = tile * kWRows + r;
        const bool in = row < p.d_out;
        cp_async8_zfill_hint(dst + kOffWs + r * 8, p.wscales + (size_t)(in ? row : 0) * rb + ks * 8, in ? 8u : 0u,
                             pol);
      }
      cp_async_mbar_arrive(full);
    };
    auto issue_x = [&](int ks, int s) {
      if (lane == 0)
        bulk_load(stage0 + (uint32_t)s * kWStage + kOffImg, p.img + (size_t)ks * kWImgU, kWImgU,
                  smem_u32(&T.full[s]));
    };
    const int n_pre = (u1 - u0) < NS ? (int)(u1 - u0) : NS;
    int tile = (int)(u0 / nks), ks = (int)(u0 % nks);
    for (int k = 0; k < n_pre; ++k) {
      issue_w(tile, ks, k);
      if (++ks == nks) { ks = 0; ++tile; }
    }
    pdl_wait();   // the activation image is the quantizer's output
    ks = (int)(u0 % nks);
    for (int k = 0; k < n_pre; ++k) {
      issue_x(ks, k);
      if (++ks == nks) ks = 0;
    }
    int s = 0;
    uint32_t ph = 0u;
    long long issued = n_pre;
    tile = (int)((u0 + n_pre) / nks);
    ks = (int)((u0 + n_pre) % nks);
    for (long long u = u0 + n_pre; u < u1; ++u, ++issued) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(smem_u32(&T.empty[s]), ph, kWPolls);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
        if (lane == 0) atomicOr(p.status, kWTimeout);
        break;
      }
      issue_w(tile, ks, s);
      issue_x(ks, s);
      if (++s == NS) { s = 0; ph ^= 1u; }
      if (++ks == nks) { ks = 0; ++tile; }
    }
    // copies in flight land before the CTA's shared memory goes away
    if (lane == 0)
      for (long long k = (issued > NS ? issued - NS : 0); k < issued; ++k)
        mbar_wait_bounded(smem_u32(&T.full[k % NS]), (uint32_t)(k / NS) & 1u, kWPolls);
    __syncwarp();
    return;
  }

  const uint32_t tmem = T.tmem;
  if (warp == 1) {
    // ---- scales to the ring, then the unit's eight MMAs ----
    long long i = 0;
    for (long long u = u0; u < u1; ++u, ++i) {
      const int s = (int)(i % NS), d = (int)(i % kWDBufs);
      bool ok = mbar_wait_bounded(smem_u32(&T.full[s]), (uint32_t)(i / NS) & 1u, kWPolls);
      if (ok && i >= kWDBufs)
        ok = mbar_wait_bounded(smem_u32(&T.dempty[d]), (uint32_t)(i / kWDBufs - 1) & 1u, kWPolls);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(p.status, kWTimeout);
        break;
      }
      const uint8_t* st = sbase + (size_t)s * kWStage;
      const uint2* ws = reinterpret_cast<const uint2*>(st + kOffWs);
#pragma unroll
      for (int q = 0; q < 4; ++q) T.wsc[d][lane * 4 + q] = ws[lane * 4 + q];
      {   // lane l: MMA l / 4, tokens 2 (l % 4) and 2 (l % 4) + 1
        const uint32_t b2 = *reinterpret_cast<const uint16_t*>(st + kOffXs + 2 * lane);
        float* xf = reinterpret_cast<float*>(&T.xsf[d][0]);
        xf[2 * lane] = exp2i((int)(b2 & 0xFFu) - 127);
        xf[2 * lane + 1] = exp2i((int)(b2 >> 8) - 127);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&T.dfull[d]));
        w_fence_after();
        const uint32_t a0 = stage0 + (uint32_t)s * kWStage, b0 = a0 + kOffImg;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = w_desc(a0 + (kk >> 2) * kWHalf + (kk & 3) * 32, 16, 1024, 2);
          const uint64_t bd = w_desc(b0 + kk * 256, 128, kOffZero - kOffImg, 0);
          w_mma(tmem + (uint32_t)(d * kWDCols + 16 * kk), ad, bd);
        }
        w_commit(smem_u32(&T.empty[s]));
        w_commit(smem_u32(&T.dfull[d]));
      }
      __syncwarp();
    }
    // every MMA has finished before the columns are released
    if (lane == 0) {
      w_commit(smem_u32(&T.drain));
      mbar_wait_bounded(smem_u32(&T.drain), 0u, kWPolls);
    }
    __syncwarp();
    w_fence_before();
    named_bar_sync(2, 32 + kWEpi);
    w_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kWTmemCols) : "memory");
    return;
  }

  // ---- epilogue warps: row R of every tile, K half kh of every unit ----
  pdl_wait();
  const int R = 32 * (warp & 3) + lane, kh = (warp - 2) >> 2;
  const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const int N = p.N;
  float y[kMaxTokens];
#pragma unroll
  for (int t = 0; t < kMaxTokens; ++t) y[t] = 0.0f;
  bool dead = false;
  int tile = (int)(u0 / nks), ks = (int)(u0 % nks);
  bool piece_whole = ks == 0;
  long long i = 0;
  for (long long u = u0; u < u1; ++u, ++i) {
    const int d = (int)(i % kWDBufs);
    if (!dead) {
      const bool ok = mbar_wait_bounded(smem_u32(&T.dfull[d]), (uint32_t)(i / kWDBufs) & 1u, kWPolls);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(p.status, kWTimeout);
        dead = true;
      }
    }
    uint32_t r[32];
    uint2 sw = make_uint2(0u, 0u);
    float4 sx[8];   // MMA 4 kh + k: tokens 0..3, then 4..7
#pragma unroll
    for (int k = 0; k < 8; ++k) sx[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!dead) {
      w_fence_after();
      sw = T.wsc[d][R];   // the scales are read before the buffer is released
#pragma unroll
      for (int k = 0; k < 8; ++k) sx[k] = T.xsf[d][8 * kh + k];
#pragma unroll
      for (int k = 0; k < 4; ++k) w_ld8(tq + (uint32_t)(d * kWDCols + 16 * (4 * kh + k)), &r[8 * k]);
      w_wait_ld(r);
      w_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&T.dempty[d]));
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) r[k] = 0u;
    }
    const uint32_t swb = kh == 0 ? sw.x : sw.y;   // the weight scale bytes of MMAs 4 kh .. 4 kh + 3
    // y += D * 2^(ew - 127) * 2^(ex - 127): the product of the two powers of two is exact
    // (short of underflow below 2^-149), so the fused multiply-add rounds once, as the add would
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float swf = exp2i((int)((swb >> (8 * k)) & 0xFFu) - 127);
      const float xs[8] = {sx[2 * k].x, sx[2 * k].y, sx[2 * k].z, sx[2 * k].w,
                           sx[2 * k + 1].x, sx[2 * k + 1].y, sx[2 * k + 1].z, sx[2 * k + 1].w};
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t)
        if (t < N) y[t] = __fmaf_rn(__uint_as_float(r[8 * k + t]), __fmul_rn(swf, xs[t]), y[t]);
    }
    // ---- end of a tile piece ----
    const bool last_of_tile = ks == nks - 1;
    const int cur_tile = tile;
    if (++ks == nks) { ks = 0; ++tile; }
    if (!last_of_tile && u + 1 < u1) continue;
    const bool whole = piece_whole && last_of_tile;
    piece_whole = true;
    // the two K halves of the row, added in that order
    if (kh == 1) {
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t)
        if (t < N) T.red[t][R] = y[t];
    }
    named_bar_sync(3, kWEpi);
    float v[kMaxTokens];
#pragma unroll
    for (int t = 0; t < kMaxTokens; ++t) v[t] = (kh == 0 && t < N) ? __fadd_rn(y[t], T.red[t][R]) : 0.0f;
    named_bar_sync(3, kWEpi);
#pragma unroll
    for (int t = 0; t < kMaxTokens; ++t) y[t] = 0.0f;
    if (kh == 1) continue;
    if (!whole) {
      float* slot = p.partials + (size_t)(cur_tile + blockIdx.x) * kMaxTokens * kWRows;
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t)
        if (t < N) slot[t * kWRows + R] = v[t];
      named_bar_sync(1, 128);   // deposits, then an acquire-release count
      const long long c0 = w_owner((long long)cur_tile * nks, U, G);
      const long long c1 = w_owner((long long)(cur_tile + 1) * nks - 1, U, G);
      if (warp == 2 && lane == 0) T.flag = atom_add_acq_rel_gpu(p.counters + cur_tile, 1u);
      named_bar_sync(1, 128);
      const uint32_t prev = T.flag;
      if (prev != (uint32_t)(c1 - c0)) continue;
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t) {
        if (t < N) {
          float a = 0.0f;
          for (long long cc = c0; cc <= c1; ++cc)
            a += cc == blockIdx.x ? v[t]
                                  : __ldcg(p.partials + ((size_t)(cur_tile + cc) * kMaxTokens + t) * kWRows + R);
          v[t] = a;
        }
      }
      if (warp == 2 && lane == 0) p.counters[cur_tile] = 0u;
    }
    const int row = cur_tile * kWRows + R;
    if (row < p.d_out) {
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t)
        if (t < N) reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)t * p.d_out + row] = __float2bfloat16_rn(v[t]);
    }
  }
  w_fence_before();
  named_bar_sync(2, 32 + kWEpi);
}

}  // namespace

// Workspace of one W4A8 call: status word, activation image, tile counters,
// partial sums (256-byte aligned pieces).
struct W4a8Layout {
  size_t off_img, off_counters, off_partials, total;
  int nks, n_tiles, n_ctas;
};

cudaError_t launch_mxfp8(const uint16_t* x, int N, int d, uint8_t* codes, uint8_t* scales, uint8_t* img,
                         uint32_t* zero, int n_zero, uint32_t* hdr, cudaStream_t st) {
  const long long slots = img != nullptr ? kMaxTokens : N;
  const long long threads = slots * (d / 32) * 32;
  const unsigned blocks = (unsigned)((threads + 255) / 256 > 0 ? (threads + 255) / 256 : 1);
  mxfp8_kernel<<<blocks, 256, 0, st>>>(x, N, d, codes, scales, img, zero, n_zero, hdr);
  return cudaGetLastError();
}

cudaError_t launch_w4a8(const WParams& p, cudaStream_t st) {
  const int smem = p.n_stages * kWStage + (int)sizeof(WTail) + 1024;
  static std::atomic<unsigned long long> attr{0};
  {
    const cudaError_t e = set_smem_once(attr, w4a8_kernel, kWNumStages * kWStage + (int)sizeof(WTail) + 1024);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_ctas);
  cfg.blockDim = dim3(kWThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w4a8_kernel, p);
}

W4a8Layout w4a8_layout(int N, int d_out, int d_in) {
  (void)N;
  W4a8Layout L;
  L.nks = d_in / 256;
  L.n_tiles = (d_out + kWRows - 1) / kWRows;
  const long long units = (long long)L.n_tiles * L.nks;
  const long long sms = num_sms();
  L.n_ctas = (int)(units < sms ? units : sms);
  size_t o = 256;
  L.off_img = o; o += align256((size_t)L.nks * kWImgU);
  L.off_counters = o; o += align256(sizeof(uint32_t) * (size_t)L.n_tiles);
  L.off_partials = o; o += align256(sizeof(float) * (size_t)(L.n_tiles + L.n_ctas) * kMaxTokens * kWRows);
  L.total = o;
  return L;
}

}  // namespace bws

extern "C" {

int bws_mxfp8_quantize(const uint16_t* x, int N, int d, uint8_t* codes, uint8_t* scales, void* stream) {
  using namespace bws;
  const char* name = "bws_mxfp8_quantize";
  if (N == 0) return BWS_OK;
  if (!x || !codes || !scales) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (N < 0) return fail(BWS_ERR_INVALID_ARG, "%s: N = %d", name, N);
  if (d < 32 || d % 32) return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: d = %d must be a positive multiple of 32", name, d);
  if (!aligned(x, 2)) return fail(BWS_ERR_MISALIGNED, "%s: x must be 2-byte aligned", name);
  return cuda_status(launch_mxfp8(x, N, d, codes, scales, nullptr, nullptr, 0, nullptr, as_stream(stream)), name);
}

size_t bws_w4a8_workspace_size(int N, int d_out, int d_in) {
  using namespace bws;
  if (N < 1 || N > kMaxTokens || d_out < 1 || d_in < 256 || d_in % 256) return 0;
  return w4a8_layout(N, d_out, d_in).total;
}

int bws_mxfp4_w4a8_gemv(const uint8_t* codes, const uint8_t* scales, const uint16_t* x, int N, int d_out, int d_in,
                        uint16_t* y, void* workspace, size_t workspace_bytes, void* stream) {
  using namespace bws;
  const char* name = "bws_mxfp4_w4a8_gemv";
  if (N == 0 || d_out == 0) return BWS_OK;
  if (!codes || !scales || !x || !y) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (N < 1 || N > kMaxTokens) return fail(BWS_ERR_INVALID_ARG, "%s: N = %d must be in [1, %d]", name, N, kMaxTokens);
  if (d_out < 0 || d_in < 256 || d_in % 256)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: d_in = %d must be a positive multiple of 256", name, d_in);
  if (!aligned(codes, 32) || !aligned(scales, 8) || !aligned(x, 2) || !aligned(y, 2))
    return fail(BWS_ERR_MISALIGNED, "%s: codes 32-byte, scales 8-byte, x and y 2-byte alignment needed", name);
  const W4a8Layout L = w4a8_layout(N, d_out, d_in);
  if (!workspace || workspace_bytes < L.total)
    return fail(BWS_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, L.total, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(BWS_ERR_MISALIGNED, "%s: workspace must be 256-byte aligned", name);
  if (!tensor_maps_available()) return fail(BWS_ERR_CUDA, "%s: the driver's tensor-map encoder is unavailable", name);
  char* w = static_cast<char*>(workspace);
  WParams p;
  memset(&p, 0, sizeof(p));
  if (!encode_fp4_2d(&p.codes, codes, (uint64_t)d_in, (uint64_t)d_out, kBoxRows))
    return fail(BWS_ERR_CUDA, "%s: tensor map encoding failed", name);
  p.wscales = scales;
  p.d_out = d_out;
  p.d_in = d_in;
  p.N = N;
  p.nks = L.nks;
  p.n_tiles = L.n_tiles;
  p.n_units = (long long)L.n_tiles * L.nks;
  p.n_ctas = L.n_ctas;
  p.n_stages = kWNumStages;
  p.img = reinterpret_cast<const uint8_t*>(w + L.off_img);
  p.y = y;
  p.partials = reinterpret_cast<float*>(w + L.off_partials);
  p.counters = reinterpret_cast<uint32_t*>(w + L.off_counters);
  p.status = reinterpret_cast<uint32_t*>(w) + 1;
  cudaStream_t st = as_stream(stream);
  cudaError_t e = launch_mxfp8(x, N, d_in, nullptr, nullptr, reinterpret_cast<uint8_t*>(w + L.off_img), p.counters,
                               L.n_tiles, reinterpret_cast<uint32_t*>(w), st);
  if (e == cudaSuccess) e = launch_w4a8(p, st);
  return cuda_status(e, name);
}

}  // extern "C"
