// Weight-stream products on the fifth-generation tensor cores for one token:
// NVFP4 weights (E2M1 codes, one E4M3 scale per 16 weights, FP32 tensor
// scale) times a BF16 activation row, FP32 accumulation.
//
// No thread decodes a weight. TMA unpacks every 16 E2M1 codes into a 16-byte
// slot on the way into shared memory, the layout tcgen05.mma kind::f8f6f4
// reads 4-bit operands in, and the tensor cores multiply the codes as they
// are. What the tensor cores cannot do is apply one scale per 16 weights
// inside a K sum, so the activation operand is block-diagonal: each MMA
// covers K = 32 (two 16-weight blocks), and its B operand has, for each of
// the two blocks, four columns that are nonzero only on that block's 16 K
// positions. One MMA (M = 128 rows, N = 16, K = 32) per block pair leaves the
// per-block partial products of all 128 rows in TMEM, and the epilogue warps
// fold them with the block scales in FP32.
//
// The four columns of a block are E4M3 "bands" of the activations, written
// by the prep kernel: with E = floor(log2 max|x|) of the token's row, every
// a = x * 2^(7-E) (|a| < 2^8) is split exactly into hi0 + lo0 when
// |a| >= 2^-2, or into 2^-10 (hi1 + lo1) when 2^-12 <= |a| < 2^-2 (each an
// E4M3 number: 4 significant bits, subnormals down to 2^-9); smaller values
// are rounded to the nearest multiple of 2^-19 and flagged. A block's
// product is then (D_hi0 + D_lo0) + 2^-10 (D_hi1 + D_lo1), and
// y = 2^(E-7) * s_t * sum over blocks of s_j * that.
//
// Roles, one CTA of ten warps per SM: warp 0 issues the TMA copies of each
// unit (codes, block scales, the unit's 2 KB activation image) into a ring of
// stages; warp 1 owns all 512 TMEM columns (four D buffers), copies each
// unit's scales into a four-entry ring and one of its threads issues the
// unit's eight MMAs, committing the stage back to the producer and the D
// buffer to the epilogue; warps 2-9 fold the products, two warps per TMEM
// lane quarter (one output row per thread), one per K half of the unit. Tiles are 128 rows (or 64 gate + 64 up rows for
// the fused SwiGLU), units a tile x 256 weights, dealt to the CTAs stream-K
// with the deterministic last-arriver fixup of the other TMA kernels.
//
// Status: opt-in (BWS_PRODUCT_KERNEL=tcgen05). Measured on GB300 it streams
// the 46336 x 5120 product in 54 us against 35 us for the mma.sync kernel
// (gemv_tma.cu). Neither the MMAs nor the unpacking are the limit (skipping
// the MMAs, or loading the same bytes through a plain byte map, changes
// little); the stream is: the unpacked codes take twice the shared memory,
// so a CTA keeps half the bytes in flight, and the unpacking copy needs
// 64-byte box rows, which stream at about half the rate of 128-byte rows
// (the same bytes as 128-byte rows: 44 us without MMAs). L2 prefetch ahead
// of the ring, by TMA or by plain loads, made it slower.
#include <cuda.h>

#include <cstddef>
#include <cstdlib>
#include <cstring>

#include "bws_common.cuh"
#include "bws_internal.h"
#include "stream_tile.cuh"

namespace bws {

namespace {

constexpr int kUWarps = 10;                  // producer, MMA, eight epilogue warps
constexpr int kUThreads = kUWarps * 32;
constexpr int kURows = 128;                  // tile rows, the MMA's M
constexpr int kUHalf = kURows * 128;         // one K half of a unit's codes in shared memory (128 codes a row)
constexpr int kUA = 2 * kUHalf;
constexpr int kUImg = 2048;                  // a unit's activation image: 8 MMAs x two 8-row core pairs
constexpr int kUB = 2 * kUImg;               // the image, then the zero rows read as the operand's second row group
constexpr int kUS = kURows * 16;             // the unit's E4M3 block scales, [row][16]
constexpr int kUStage = kUA + kUB + kUS;
constexpr int kUMaxStages = 8;
constexpr int kUNumStages = (190 * 1024) / kUStage;   // five stages: the CTA has the SM to itself
static_assert(kUNumStages <= kUMaxStages, "barrier arrays");
constexpr int kUDCols = 128;                 // TMEM columns of one unit's products (8 MMAs x N = 16)
constexpr int kUDBufs = 4;                   // D buffers in TMEM (and entries of the scale ring)
constexpr int kUTmemCols = kUDBufs * kUDCols;
constexpr int kUEpi = 8 * 32;                // epilogue threads
constexpr uint32_t kUTx = kUHalf + kUS + kUImg;   // bytes a stage receives (codes packed)
constexpr uint32_t kUPolls = 1u << 24;
constexpr uint32_t kUTimeout = 0x100u;
static_assert(kUStage % 1024 == 0, "stages must keep the 1024-byte alignment of the swizzled code boxes");

// Instruction descriptor: D FP32, A E2M1, B E4M3, both K-major, M = 128, N = 16.
constexpr uint32_t kUIdesc = (1u << 4) | (5u << 7) | (0u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

struct UMat {
  CUtensorMap codes;    // E2M1 [d_out][d_in / 2] unpacked to 16-byte slots, box {128 codes, 32 rows}, 128B swizzle
  CUtensorMap scales;   // u8 [d_out][d_in / 16], box {16, 32}
  const float* scale32;
  int d_out;
  int out_row_off;
  int tile_begin;
};

struct UParams {
  UMat mats[kMaxMats];
  int n_mats;
  int nks;              // units per tile
  int n_tiles;
  long long n_units;
  int n_ctas, n_stages;
  const uint8_t* img;   // activation image, kUImg bytes per unit
  const int* xexp;      // E of the token's row
  void* out;
  int out_ld;
  float* partials;      // [(n_tiles + n_ctas) * 128]
  uint32_t* counters;   // [n_tiles], zero on entry, left zero
  uint32_t* status;
};

struct UTail {
  uint4 scales[kUDBufs][kURows];   // block scales of the units in the D buffers, one row each
  float red[kURows];               // the second K half's row sums handed to the first
  float swi[64];                   // SwiGLU: up rows handed to the gate rows
  uint64_t full[kUMaxStages];
  uint64_t empty[kUMaxStages];
  uint64_t dfull[kUDBufs], dempty[kUDBufs], drain;
  uint32_t tmem;
  uint32_t flag;
};

template <int EPI>
BWS_DEV void ubox_of(const UParams& p, int tile, int b, int& m, int& row) {
  if (EPI == kEpiSwiGLU) {
    m = b >> 1;
    row = tile * 64 + 32 * (b & 1);
    return;
  }
  m = 0;
#pragma unroll
  for (int i = 1; i < kMaxMats; ++i)
    if (i < p.n_mats && tile >= p.mats[i].tile_begin) m = i;
  row = (tile - p.mats[m].tile_begin) * kURows + 32 * b;
}

BWS_DEV long long u_owner(long long u, long long U, long long G) { return ((u + 1) * G - 1) / U; }
BWS_DEV long long u_begin(long long c, long long U, long long G) { return c * U / G; }

// Shared-memory matrix descriptor (tcgen05): start, leading / stride byte
// offsets, version 1, layout (0: no swizzle, 2: 128-byte swizzle).
BWS_DEV uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46) | ((uint64_t)layout << 61);
}
BWS_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
BWS_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
// D = A * B^T (no accumulation into D)
BWS_DEV void tc_mma(uint32_t d, uint64_t a, uint64_t b) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(kUIdesc), "r"(0u)
      : "memory");
}
// One arrival on the mbarrier when every MMA this thread issued so far is done.
BWS_DEV void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// Eight consecutive TMEM columns of this warp's 32 lanes.
BWS_DEV void tc_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
// Waits for this thread's TMEM loads; the registers are tied to the wait so
// that no use of them moves above it.
BWS_DEV void tc_wait_ld(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
        "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// Final value of row R of a tile (sum v over the units), stored per EPI.
template <int EPI>
BWS_DEV void ustore(const UParams& p, UTail& T, int tile, int R, float v, int E) {
  int m, row_b;
  ubox_of<EPI>(p, tile, R >> 5, m, row_b);
  const int row = row_b + (R & 31);
  const float val = ldexp_exact(__fmul_rn(v, __ldg(p.mats[m].scale32)), E - 7);
  if (EPI == kEpiSwiGLU) {
    if (R >= 64) T.swi[R - 64] = val;
    named_bar_sync(1, 128);
    if (R < 64 && row < p.mats[0].d_out)
      reinterpret_cast<__nv_bfloat16*>(p.out)[row] = __float2bfloat16_rn(silu_mul_t(val, T.swi[R]));
    named_bar_sync(1, 128);
    return;
  }
  if (row >= p.mats[m].d_out) return;
  const size_t o = (size_t)p.mats[m].out_row_off + row;
  if (EPI == kEpiStoreBF16)
    reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(val);
  else if (EPI == kEpiStoreF32)
    reinterpret_cast<float*>(p.out)[o] = val;
  else
    reinterpret_cast<float*>(p.out)[o] = __fadd_rn(reinterpret_cast<float*>(p.out)[o], val);
}

template <int EPI>
__global__ void __launch_bounds__(kUThreads, 1) gemv_umma_kernel(const __grid_constant__ UParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  uint8_t* sbase = smem_raw + ((1024u - mis) & 1023u);
  const int NS = p.n_stages;
  UTail& T = *reinterpret_cast<UTail*>(sbase + (size_t)NS * kUStage);
  const uint32_t stage0 = smem_u32(sbase);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&T.tmem)),
                 "n"(kUTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&T.full[i]), 1);
      mbar_init(smem_u32(&T.empty[i]), 1);
    }
    for (int d = 0; d < kUDBufs; ++d) {
      mbar_init(smem_u32(&T.dfull[d]), 2);    // the scale copy and the MMA commit
      mbar_init(smem_u32(&T.dempty[d]), 8);   // the eight epilogue warps
    }
    mbar_init(smem_u32(&T.drain), 1);
    T.flag = 0u;
    mbar_fence_init();
  }
  // the operand's second row group (a second token's columns) stays zero
  for (int i = threadIdx.x; i < NS * (kUImg / 16); i += blockDim.x) {
    const int s = i / (kUImg / 16), o = i - s * (kUImg / 16);
    *reinterpret_cast<uint4*>(sbase + (size_t)s * kUStage + kUA + kUImg + 16 * o) = make_uint4(0, 0, 0, 0);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const long long U = p.n_units, G = p.n_ctas;
  const long long u0 = u_begin(blockIdx.x, U, G), u1 = u_begin(blockIdx.x + 1, U, G);
  const int nks = p.nks;

  if (warp == 0) {
    // ---- producer: the weights of the first stages before the inputs are ready ----
    if (lane == 0) {
      for (int i = 0; i < p.n_mats; ++i) {
        tma_prefetch_desc(&p.mats[i].codes);
        tma_prefetch_desc(&p.mats[i].scales);
      }
      auto issue_w = [&](int tile, int ks, int s) {
        const uint32_t full = smem_u32(&T.full[s]);
        const uint32_t dst = stage0 + (uint32_t)s * kUStage;
        mbar_arrive_expect_tx(full, kUTx);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b) {
          int m, row;
          ubox_of<EPI>(p, tile, b, m, row);
          tma_load_2d(dst + b * kBoxBytes, &p.mats[m].codes, ks * 256, row, full);
          tma_load_2d(dst + kUHalf + b * kBoxBytes, &p.mats[m].codes, ks * 256 + 128, row, full);
          tma_load_2d(dst + kUA + kUB + b * kScaleBoxBytes, &p.mats[m].scales, ks * 16, row, full);
        }
      };
      auto issue_x = [&](int ks, int s) {
        bulk_load(stage0 + (uint32_t)s * kUStage + kUA, p.img + (size_t)ks * kUImg, kUImg, smem_u32(&T.full[s]));
      };
      const int n_pre = (u1 - u0) < NS ? (int)(u1 - u0) : NS;
      int tile = (int)(u0 / nks), ks = (int)(u0 % nks);
      for (int k = 0; k < n_pre; ++k) {
        issue_w(tile, ks, k);
        if (++ks == nks) { ks = 0; ++tile; }
      }
      pdl_wait();
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
        if (!mbar_wait_bounded(smem_u32(&T.empty[s]), ph, kUPolls)) {
          atomicOr(p.status, kUTimeout);
          break;
        }
        issue_w(tile, ks, s);
        issue_x(ks, s);
        if (++s == NS) { s = 0; ph ^= 1u; }
        if (++ks == nks) { ks = 0; ++tile; }
      }
      // copies in flight land before the CTA's shared memory goes away
      for (long long k = (issued > NS ? issued - NS : 0); k < issued; ++k)
        mbar_wait_bounded(smem_u32(&T.full[k % NS]), (uint32_t)(k / NS) & 1u, kUPolls);
    }
    return;
  }

  const uint32_t tmem = T.tmem;
  if (warp == 1) {
    // ---- scales to the ring, then the unit's eight MMAs ----
    long long i = 0;
    for (long long u = u0; u < u1; ++u, ++i) {
      const int s = (int)(i % NS), d = (int)(i % kUDBufs);
      // every lane waits (each then sees the stage's bytes), the warp decides together
      bool ok = mbar_wait_bounded(smem_u32(&T.full[s]), (uint32_t)(i / NS) & 1u, kUPolls);
      if (ok && i >= kUDBufs)
        ok = mbar_wait_bounded(smem_u32(&T.dempty[d]), (uint32_t)(i / kUDBufs - 1) & 1u, kUPolls);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(p.status, kUTimeout);
        break;
      }
      const uint4* src = reinterpret_cast<const uint4*>(sbase + (size_t)s * kUStage + kUA + kUB);
#pragma unroll
      for (int q = 0; q < 4; ++q) T.scales[d][lane * 4 + q] = src[lane * 4 + q];
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&T.dfull[d]));
        tc_fence_after();
        const uint32_t a0 = stage0 + (uint32_t)s * kUStage, b0 = a0 + kUA;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = smem_desc(a0 + (kk >> 2) * kUHalf + (kk & 3) * 32, 16, 1024, 2);
          const uint64_t bd = smem_desc(b0 + kk * 256, 128, kUImg, 0);
          tc_mma(tmem + (uint32_t)(d * kUDCols + 16 * kk), ad, bd);
        }
        tc_commit(smem_u32(&T.empty[s]));
        tc_commit(smem_u32(&T.dfull[d]));
      }
      __syncwarp();
    }
    // every MMA has finished before the columns are released
    if (lane == 0) {
      tc_commit(smem_u32(&T.drain));
      mbar_wait_bounded(smem_u32(&T.drain), 0u, kUPolls);
    }
    __syncwarp();
    tc_fence_before();
    named_bar_sync(2, 32 + kUEpi);
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kUTmemCols) : "memory");
    return;
  }

  // ---- epilogue warps: row R of every tile, K half kh of every unit ----
  pdl_wait();
  const int R = 32 * (warp & 3) + lane, kh = (warp - 2) >> 2;
  const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const int E = __ldg(p.xexp);
  float y = 0.0f;
  bool dead = false;
  int tile = (int)(u0 / nks), ks = (int)(u0 % nks);
  bool piece_whole = ks == 0;
  long long i = 0;
  for (long long u = u0; u < u1; ++u, ++i) {
    const int d = (int)(i % kUDBufs);
    if (!dead) {
      const bool ok = mbar_wait_bounded(smem_u32(&T.dfull[d]), (uint32_t)(i / kUDBufs) & 1u, kUPolls);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(p.status, kUTimeout);
        dead = true;
      }
    }
    uint32_t r[32];
    uint2 sc = make_uint2(0u, 0u);
    if (!dead) {
      tc_fence_after();
      const uint4 s4 = T.scales[d][R];
      sc = kh == 0 ? make_uint2(s4.x, s4.y) : make_uint2(s4.z, s4.w);
#pragma unroll
      for (int k = 0; k < 4; ++k) tc_ld8(tq + (uint32_t)(d * kUDCols + 16 * (4 * kh + k)), &r[8 * k]);
      tc_wait_ld(r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&T.dempty[d]));
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) r[k] = 0u;
    }
    const uint32_t sw[2] = {sc.x, sc.y};
#pragma unroll
    for (int k = 0; k < 4; ++k) {   // MMA 4 kh + k: blocks 8 kh + 2k and 8 kh + 2k + 1
      const uint32_t f = e4m3x2_to_f16x2((sw[k >> 1] >> (16 * (k & 1))) & 0xFFFFu);
      const float s0 = __half2float(__ushort_as_half((unsigned short)(f & 0xFFFFu)));
      const float s1 = __half2float(__ushort_as_half((unsigned short)(f >> 16)));
      float v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = __uint_as_float(r[8 * k + c]);
      const float t0 = __fmaf_rn(0x1p-10f, __fadd_rn(v[2], v[3]), __fadd_rn(v[0], v[1]));
      const float t1 = __fmaf_rn(0x1p-10f, __fadd_rn(v[6], v[7]), __fadd_rn(v[4], v[5]));
      y = __fmaf_rn(s0, t0, y);
      y = __fmaf_rn(s1, t1, y);
    }
    // ---- end of a tile piece ----
    const bool last_of_tile = ks == nks - 1;
    const int cur_tile = tile;
    if (++ks == nks) { ks = 0; ++tile; }
    if (!last_of_tile && u + 1 < u1) continue;
    const bool whole = piece_whole && last_of_tile;
    piece_whole = true;
    // the two K halves of the row, added in that order
    if (kh == 1) T.red[R] = y;
    named_bar_sync(3, kUEpi);
    float v = y;
    if (kh == 0) v = __fadd_rn(y, T.red[R]);
    named_bar_sync(3, kUEpi);
    y = 0.0f;
    if (kh == 1) continue;
    if (!whole) {
      p.partials[(size_t)(cur_tile + blockIdx.x) * kURows + R] = v;
      named_bar_sync(1, 128);   // deposits, then an acquire-release count
      const long long c0 = u_owner((long long)cur_tile * nks, U, G);
      const long long c1 = u_owner((long long)(cur_tile + 1) * nks - 1, U, G);
      if (warp == 2 && lane == 0) T.flag = atom_add_acq_rel_gpu(p.counters + cur_tile, 1u);
      named_bar_sync(1, 128);
      const uint32_t prev = T.flag;
      if (prev != (uint32_t)(c1 - c0)) continue;
      float a = 0.0f;
      for (long long cc = c0; cc <= c1; ++cc)
        a += cc == blockIdx.x ? v : __ldcg(p.partials + (size_t)(cur_tile + cc) * kURows + R);
      v = a;
      if (warp == 2 && lane == 0) p.counters[cur_tile] = 0u;
    }
    ustore<EPI>(p, T, cur_tile, R, v, E);
  }
  tc_fence_before();
  named_bar_sync(2, 32 + kUEpi);
}

template <int EPI>
cudaError_t launch_umma_one(const UParams& p, cudaStream_t st, bool pdl) {
  const int smem = p.n_stages * kUStage + (int)sizeof(UTail) + 1024;
  static std::atomic<unsigned long long> attr{0};
  {
    const cudaError_t e = set_smem_once(attr, gemv_umma_kernel<EPI>, kUNumStages * kUStage + (int)sizeof(UTail) + 1024);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_ctas);
  cfg.blockDim = dim3(kUThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_umma_kernel<EPI>, p);
}

}  // namespace

bool gemv_umma_eligible(int fmt, const GemvParams& g) {
  if (fmt != kFmtNVFP4 || g.N != 1 || g.slots.n_slots != nullptr || !tensor_maps_available()) return false;
  const char* sel = getenv("BWS_PRODUCT_KERNEL");   // opt-in: the mma.sync kernel streams faster
  if (sel == nullptr || strcmp(sel, "tcgen05") != 0) return false;
  if (g.d_in % 256 != 0 || g.n_mats < 1) return false;
  // the activation image takes the two f16 band rows of the token's block
  if (g.x.hi == nullptr || reinterpret_cast<const char*>(g.x.lo) - reinterpret_cast<const char*>(g.x.hi) !=
                               4 * (ptrdiff_t)g.d_in_pad)
    return false;
  for (int i = 0; i < g.n_mats; ++i) {
    if (((uintptr_t)g.mats[i].codes & 31) != 0 || ((uintptr_t)g.mats[i].scales & 15) != 0) return false;
  }
  return true;
}

// Runs the one-token NVFP4 product described by g on the tensor cores; the
// activations were prepared as the E4M3 band image (prep layout
// kLayoutImage) in g.x.hi. Scratch: g.counters (g.n_tiles words, zero) and
// g.partials, as for the other TMA kernels.
cudaError_t launch_gemv_umma(int epi, const GemvParams& g, uint32_t* status, cudaStream_t st, bool pdl) {
  UParams p;
  memset(&p, 0, sizeof(p));
  p.n_mats = g.n_mats;
  int tile = 0, row = 0;
  for (int i = 0; i < g.n_mats; ++i) {
    const GemvMat& M = g.mats[i];
    if (!encode_fp4_2d(&p.mats[i].codes, M.codes, (uint64_t)g.d_in, (uint64_t)M.d_out, kBoxRows))
      return cudaErrorInvalidValue;
    if (!encode_2d(&p.mats[i].scales, M.scales, (uint64_t)g.d_in / 16, (uint64_t)M.d_out, 16, kBoxRows, false))
      return cudaErrorInvalidValue;
    p.mats[i].scale32 = M.scale32;
    p.mats[i].d_out = M.d_out;
    p.mats[i].out_row_off = epi == kEpiSwiGLU ? 0 : row;
    p.mats[i].tile_begin = tile;
    row += M.d_out;
    tile += (M.d_out + kURows - 1) / kURows;
  }
  p.nks = g.d_in / 256;
  p.n_tiles = gemv_tma_tiles(epi, g.mats, g.n_mats);
  p.n_units = (long long)p.n_tiles * p.nks;
  const long long ctas = num_sms();   // one CTA per SM
  p.n_ctas = (int)(p.n_units < ctas ? p.n_units : ctas);
  p.img = reinterpret_cast<const uint8_t*>(g.x.hi);
  p.xexp = g.x.exp;
  p.out = g.out;
  p.out_ld = g.out_ld;
  p.partials = g.partials;
  p.counters = g.counters;
  p.status = status;
  if (p.n_tiles > g.n_tiles ||
      ((long long)p.n_tiles + p.n_ctas) * kURows * (long long)sizeof(float) >
          ((long long)g.n_tiles + gemv_max_warps()) * kSlotFloats * (long long)sizeof(float))
    return cudaErrorInvalidValue;
  p.n_stages = kUNumStages;
  if (p.n_ctas <= 0) return cudaSuccess;
  if (epi == kEpiStoreBF16) return launch_umma_one<kEpiStoreBF16>(p, st, pdl);
  if (epi == kEpiResidF32) return launch_umma_one<kEpiResidF32>(p, st, pdl);
  if (epi == kEpiSwiGLU) return launch_umma_one<kEpiSwiGLU>(p, st, pdl);
  if (epi == kEpiStoreF32) return launch_umma_one<kEpiStoreF32>(p, st, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace bws
