// Shared device helpers of the weight-stream kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define BWS_DEV __device__ __forceinline__

namespace bws {

// ---- programmatic dependent launch ---------------------------------------
// A kernel calls pdl_launch_dependents() early so the next kernel in the
// stream may be scheduled while it runs, and pdl_wait() before it reads
// anything an earlier kernel wrote (it returns once the preceding grid has
// completed and its writes are visible).
BWS_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
BWS_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- loads ----------------------------------------------------------------
// Weights are read exactly once per step: stream them past L1.
BWS_DEV uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
BWS_DEV uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
BWS_DEV uint32_t ld_stream_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
BWS_DEV uint32_t ld_stream_u8(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
// Activations are small and shared by every warp: keep them in L1.
BWS_DEV uint4 ld_act_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// L2 prefetch of a 16-byte aligned range whose size is a multiple of 16.
BWS_DEV void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}
// Coherent (L1-bypassing) load of data another SM wrote in this grid.
// Atomic add with acquire-release semantics at GPU scope; returns the old value.
BWS_DEV uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// 32 bytes (eight floats, 32-byte aligned) through L2 in one request.
BWS_DEV void ld_cg_f8(const float* p, float4& a, float4& b) {
  asm volatile("ld.global.cg.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(a.x), "=f"(a.y), "=f"(a.z), "=f"(a.w), "=f"(b.x), "=f"(b.y), "=f"(b.z), "=f"(b.w)
               : "l"(p));
}
BWS_DEV float4 ld_cg_f4(const float4* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

// ---- async global -> shared copies (per thread, 16 bytes, bypassing L1) ---
BWS_DEV void cp_async16(uint32_t smem_addr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr), "l"(g) : "memory");
}
// 8 bytes global -> shared, asynchronously; src_bytes 0 writes zeros and reads nothing.
BWS_DEV void cp_async8_zfill(uint32_t smem_addr, const void* g, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" :: "r"(smem_addr), "l"(g), "r"(src_bytes) : "memory");
}
// cp_async8_zfill with an L2 policy (see l2_evict_first).
BWS_DEV void cp_async8_zfill_hint(uint32_t smem_addr, const void* g, uint32_t src_bytes, uint64_t pol) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2, %3;"
               :: "r"(smem_addr), "l"(g), "r"(src_bytes), "l"(pol) : "memory");
}
// One arrival on the mbarrier once every earlier cp.async of this thread has
// landed (counted in the barrier's expected arrivals: no pending increment).
BWS_DEV void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}
BWS_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
BWS_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }
BWS_DEV uint4 lds_v4(uint32_t smem_addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr));
  return v;
}

// ---- mbarrier and TMA (shared::cta, no clusters) ----------------------------
BWS_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
BWS_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
BWS_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
BWS_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
BWS_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
BWS_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete, at most max_polls
// polls (each try_wait itself blocks for a hardware-defined while). Returns
// false if the wait ran out.
BWS_DEV bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t max_polls) {
  for (uint32_t i = 0; i < max_polls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// 2D tiled TMA load of box (x = inner coordinate in elements, y = row) into
// shared memory, completing on mbarrier bar.
BWS_DEV void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}
// An L2 policy for data read once per step (streamed weights): its lines are
// the first to be replaced, so the stream does not push out the small data
// that every kernel reads back soon (activations, partial sums, code).
BWS_DEV uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// tma_load_2d with an L2 policy.
BWS_DEV void tma_load_2d_hint(uint32_t dst, const void* tmap, int x, int y, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(pol) : "memory");
}
// tma_load_3d (below) with an L2 policy.
BWS_DEV void tma_load_3d_hint(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol) : "memory");
}
// 3D tiled TMA load of box (x, y, z) into shared memory, completing on bar.
BWS_DEV void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar) : "memory");
}
// 1D bulk copy global -> shared (16-byte aligned, size % 16 == 0).
BWS_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// L2 prefetch of a 2D tiled box (no shared memory, no completion).
BWS_DEV void tma_prefetch_2d(const void* tmap, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" :: "l"(tmap), "r"(x), "r"(y)
               : "memory");
}
BWS_DEV void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}
BWS_DEV void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}
BWS_DEV uint32_t lds_u8(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
BWS_DEV uint32_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// ---- conversions (hardware, exact for these inputs) ------------------------
// Two E2M1 codes in one byte -> f16x2. Every E2M1 value is exact in f16.
BWS_DEV uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low8) {
  uint32_t r;
  asm("{ .reg .b8 b; cvt.u8.u32 b, %1; cvt.rn.f16x2.e2m1x2 %0, b; }" : "=r"(r) : "r"(byte_in_low8));
  return r;
}
// Two E4M3 codes in 16 bits -> f16x2. Every E4M3 value is exact in f16.
BWS_DEV uint32_t e4m3x2_to_f16x2(uint32_t two_bytes_in_low16) {
  uint32_t r;
  asm("{ .reg .b16 h; cvt.u16.u32 h, %1; cvt.rn.f16x2.e4m3x2 %0, h; }" : "=r"(r) : "r"(two_bytes_in_low16));
  return r;
}
// Unpack the 4 bytes of a word, and convert each byte's two E2M1 codes.
BWS_DEV void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      "  mov.b32 {b0, b1, b2, b3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "  cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "  cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(w));
}
BWS_DEV void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& r0, uint32_t& r1) {
  asm("{ .reg .b16 h0, h1;\n"
      "  mov.b32 {h0, h1}, %2;\n"
      "  cvt.rn.f16x2.e4m3x2 %0, h0;\n"
      "  cvt.rn.f16x2.e4m3x2 %1, h1; }"
      : "=r"(r0), "=r"(r1) : "r"(w));
}
// Encoders with round-to-nearest-even and saturation to the largest finite
// value. The first source operand lands in the upper part of the result.
BWS_DEV uint32_t f32x2_to_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{ .reg .b8 b; cvt.rn.satfinite.e2m1x2.f32 b, %1, %2; cvt.u32.u8 %0, b; }"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
BWS_DEV uint32_t f32x2_to_e4m3x2(float hi, float lo) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
BWS_DEV float e4m3_to_f32(uint32_t code) {
  uint32_t h = e4m3x2_to_f16x2(code & 0xFF);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFF)));
}

BWS_DEV uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Broadcast the low / high f16 of a pair to both halves.
BWS_DEV uint32_t bcast_lo(uint32_t x) { return __byte_perm(x, 0, 0x1010); }
BWS_DEV uint32_t bcast_hi(uint32_t x) { return __byte_perm(x, 0, 0x3232); }

// D += A * B, A 16x16 f16 (row), B 16x8 f16 (col), D 16x8 f32.
BWS_DEV void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                           uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Exact power of two as FP32 (e in [-149, 127]); 0 below.
BWS_DEV float exp2i(int e) {
  if (e >= -126) return __int_as_float((e + 127) << 23);
  if (e >= -149) return __int_as_float(1 << (e + 149));
  return 0.0f;
}
// x * 2^e exactly (up to the final rounding of an out-of-range result).
BWS_DEV float ldexp_exact(float x, int e) {
  int a = e > 127 ? 127 : (e < -126 ? -126 : e);
  int b = e - a;
  b = b > 127 ? 127 : (b < -126 ? -126 : b);
  return __fmul_rn(__fmul_rn(x, exp2i(a)), exp2i(b));
}
// floor(log2 |x|) for finite x != 0, exact for subnormals.
BWS_DEV int floor_log2_abs(float x) {
  uint32_t b = __float_as_uint(x) & 0x7FFFFFFFu;
  int e = (int)(b >> 23);
  if (e > 0) return e - 127;
  return (31 - __clz((int)b)) - 149;
}

// Polls a flag until it is non-zero (acquire, GPU scope); false after
// max_polls reads.
BWS_DEV bool poll_acquire(const uint32_t* f, uint32_t max_polls) {
  for (uint32_t i = 0; i < max_polls; ++i) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v != 0u) return true;
    __nanosleep(32);
  }
  return false;
}
BWS_DEV void store_release(uint32_t* f, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(f), "r"(v) : "memory");
}

BWS_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
BWS_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace bws
