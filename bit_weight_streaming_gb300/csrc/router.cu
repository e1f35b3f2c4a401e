// MoE router: z = W_r x over the routed experts, then each token's top-k
// experts and their combine weights ([LingMoE] section 3: each MoE layer
// sends every token to 8 of its 512 routed experts, plus the shared one).
//
// The pages name the routing but not its arithmetic. Reading used here: the
// router is a BF16 [E][d] matrix applied to the layer's normalised input m
// (the BF16 row the experts also read), with FP32 accumulation; a token's
// experts are the k largest logits (equal logits: the lower expert id first);
// their combine weights are the softmax of those k logits, i.e. the full
// softmax renormalised over the chosen experts.
//
// One kernel: CTA b computes the logits of experts [8b, 8b + 8) for every
// token, one warp per expert. Each warp copies its router row into shared
// memory before griddepcontrol.wait (the rows do not depend on the kernels
// before), so the copy overlaps the input's producer; after the wait the CTA
// copies x into shared memory in one round, and the dot products read only
// shared memory. The last CTA to finish
// (an acquire-release count) reads all logits back from L2 and chooses each
// token's experts, one warp per token, by k rounds of a warp-wide maximum of
// the logits' order-preserving bit patterns, then of the lowest expert id
// holding that maximum. In the decode stack it also writes the layer's slot table and raises
// the table's ready flag for the expert kernels.
#include "bws_abi_util.h"
#include "bws_common.cuh"
#include "bws_internal.h"
#include "moe_route.cuh"

namespace bws {
namespace {

constexpr int kRouterRows = 8;       // experts per CTA, one warp each
constexpr int kRouterThreads = 32 * kRouterRows;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// The logit a key (argmax_key) was made from.
__device__ __forceinline__ float key_value(unsigned long long key) {
  const uint32_t b = (uint32_t)(key >> 32);
  return __uint_as_float((b & 0x80000000u) ? (b & 0x7FFFFFFFu) : ~b);
}

__global__ void __launch_bounds__(kRouterThreads) router_kernel(RouterParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_last;
  __shared__ float s_z[kMaxTokens][kMaxTopk];
  __shared__ int s_id[kMaxTokens][kMaxTopk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterRows + warp;
  const int n16 = p.d / 8;   // 16-byte chunks of a row
  uint16_t* row = reinterpret_cast<uint16_t*>(smem) + (size_t)warp * p.d;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem) + (size_t)kRouterRows * p.d;   // x [N][d]
  if (e < p.E) {
    const uint16_t* src = p.W + (size_t)e * p.d;
    for (int c = lane; c < n16; c += 32) cp_async16(smem_u32(row + (size_t)c * 8), src + (size_t)c * 8);
  }
  cp_async_commit();
  pdl_launch_dependents();
  pdl_wait();   // x is the previous kernel's output: one round of copies into shared memory
  for (int i = threadIdx.x; i < p.N * n16; i += blockDim.x) cp_async16(smem_u32(xs + (size_t)i * 8), p.x + (size_t)i * 8);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (e < p.E) {
    // two independent FMA chains per token (even and odd K positions)
    float acc0[kMaxTokens], acc1[kMaxTokens];
#pragma unroll
    for (int n = 0; n < kMaxTokens; ++n) acc0[n] = acc1[n] = 0.0f;
#pragma unroll 2
    for (int c = lane; c < n16; c += 32) {
      const uint4 w = lds_v4(smem_u32(row + (size_t)c * 8));
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int n = 0; n < kMaxTokens; ++n) {
        if (n < p.N) {
          const uint4 xv = lds_v4(smem_u32(xs + (size_t)n * p.d + (size_t)c * 8));
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          float a0 = acc0[n], a1 = acc1[n];
#pragma unroll
          for (int i = 0; i < 4; ++i) {   // BF16 x BF16 products are exact in FP32
            a0 = fmaf(bf16_lo(wv[i]), bf16_lo(xw[i]), a0);
            a1 = fmaf(bf16_hi(wv[i]), bf16_hi(xw[i]), a1);
          }
          acc0[n] = a0;
          acc1[n] = a1;
        }
      }
    }
#pragma unroll
    for (int n = 0; n < kMaxTokens; ++n) {
      if (n < p.N) {
        const float s = warp_sum(acc0[n] + acc1[n]);
        if (lane == 0) p.z[(size_t)n * p.E + e] = s;
      }
    }
  }
  __syncthreads();   // the CTA's logits are written; thread 0's release below covers them
  if (threadIdx.x == 0) s_last = atom_add_acq_rel_gpu(p.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;

  // the last CTA: every token's top-k over the logits in L2, one warp per
  // token. Each logit becomes its order-preserving 32-bit pattern; a lane
  // keeps the best of its experts (i = lane mod 32, the lowest i among equal
  // patterns), and each round takes the warp's largest pattern, then the
  // lowest expert id holding it, and the lane that held it rescans.
  uint32_t* vb = reinterpret_cast<uint32_t*>(smem);   // [N][E], rows no longer needed
  for (int i = threadIdx.x; i < p.N * p.E; i += blockDim.x) {
    float v = __ldcg(p.z + i);
    if (v != v) v = -INFINITY;   // a NaN logit ranks last
    vb[i] = (uint32_t)(argmax_key(v, 0) >> 32);   // > 0 for every value: 0 marks a taken expert
  }
  __syncthreads();
  if (warp < p.N) {
    uint32_t* vt = vb + (size_t)warp * p.E;
    uint32_t bv = 0u;
    int bi = -1;
    auto rescan = [&]() {
      bv = 0u;
      bi = -1;
      for (int i = lane; i < p.E; i += 32)
        if (vt[i] > bv) {
          bv = vt[i];
          bi = i;
        }
    };
    rescan();
    for (int j = 0; j < p.topk; ++j) {
      const uint32_t vmax = __reduce_max_sync(0xffffffffu, bv);
      const int id = (int)__reduce_min_sync(0xffffffffu, (bv == vmax && bi >= 0) ? (uint32_t)bi : 0xffffffffu);
      if (lane == 0) {
        s_id[warp][j] = id;
        s_z[warp][j] = key_value((unsigned long long)vmax << 32);
      }
      if ((id & 31) == lane) {   // the owner takes it out and finds its next best
        vt[id] = 0u;
        rescan();
      }
    }
    __syncwarp();
    // softmax over the chosen logits; the first is the largest
    float ex = 0.0f;
    if (lane < p.topk) ex = expf(s_z[warp][lane] - s_z[warp][0]);
    const float sum = warp_sum(ex);
    if (lane < p.topk) {
      p.ids[warp * p.topk + lane] = s_id[warp][lane];
      p.route_w[warp * p.topk + lane] = __fdiv_rn(ex, sum);
    }
  }
  if (p.has_route) {
    __syncthreads();   // the ids and weights above are written
    moe_route_body(p.route);
  }
}

}  // namespace

size_t router_smem_bytes(int N, int E, int d) {
  const size_t rows = (size_t)(kRouterRows + N) * d * 2;   // the CTA's router rows, then x
  const size_t keys = (size_t)N * E * 4;
  return rows > keys ? rows : keys;
}

int router_ctas(int E) { return (E + kRouterRows - 1) / kRouterRows; }

cudaError_t launch_router(const RouterParams& p, cudaStream_t st, bool pdl) {
  const size_t smem = router_smem_bytes(p.N, p.E, p.d);
  if (smem > (size_t)kRouterSmemMax) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr{0};
  const cudaError_t e = set_smem_once(attr, router_kernel, kRouterSmemMax);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)router_ctas(p.E));
  cfg.blockDim = dim3(kRouterThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, router_kernel, p);
}

}  // namespace bws

namespace {

int check_router(const void* W, const void* x, int N, int E, int d, int topk, const char* name) {
  using namespace bws;
  if (!W || !x) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (N < 1 || N > kMaxTokens) return fail(BWS_ERR_INVALID_ARG, "%s: N = %d must be in [1, %d]", name, N, kMaxTokens);
  if (E < 1 || E > kRouterMaxExperts)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: n_experts = %d must be in [1, %d]", name, E, kRouterMaxExperts);
  if (topk < 1 || topk > kMaxTopk || topk > E)
    return fail(BWS_ERR_INVALID_ARG, "%s: topk = %d must be in [1, min(%d, n_experts)]", name, topk, kMaxTopk);
  if (d < 8 || d % 8 || d > kRouterMaxD)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: d = %d must be a multiple of 8 in [8, %d]", name, d, kRouterMaxD);
  if (!aligned(W, 16) || !aligned(x, 16)) return fail(BWS_ERR_MISALIGNED, "%s: W and x must be 16-byte aligned", name);
  return BWS_OK;
}

}  // namespace

extern "C" {

size_t bws_moe_router_workspace_size(int N, int n_experts) {
  if (N < 1 || N > bws::kMaxTokens || n_experts < 1 || n_experts > bws::kRouterMaxExperts) return 0;
  return 256 + bws::align256(sizeof(float) * (size_t)N * n_experts);
}

int bws_moe_router_topk(const uint16_t* W_router, const uint16_t* x, int N, int n_experts, int d, int topk,
                        float* logits, int32_t* ids, float* route_w, void* workspace, size_t workspace_bytes,
                        void* stream) {
  using namespace bws;
  const char* name = "bws_moe_router_topk";
  int rc = check_router(W_router, x, N, n_experts, d, topk, name);
  if (rc) return rc;
  if (!ids || !route_w) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned(ids, 4) || !aligned(route_w, 4) || (logits && !aligned(logits, 4)))
    return fail(BWS_ERR_MISALIGNED, "%s: ids, route_w and logits must be 4-byte aligned", name);
  const size_t need = bws_moe_router_workspace_size(N, n_experts);
  if (!workspace || workspace_bytes < need)
    return fail(BWS_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, need, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(BWS_ERR_MISALIGNED, "%s: workspace must be 256-byte aligned", name);
  cudaStream_t st = as_stream(stream);
  char* w = static_cast<char*>(workspace);
  RouterParams p = {};
  p.W = W_router;
  p.x = x;
  p.N = N;
  p.E = n_experts;
  p.d = d;
  p.topk = topk;
  p.z = logits != nullptr ? logits : reinterpret_cast<float*>(w + 256);
  p.counter = reinterpret_cast<uint32_t*>(w);
  p.ids = ids;
  p.route_w = route_w;
  cudaError_t e = cudaMemsetAsync(p.counter, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = launch_router(p, st, false);
  return cuda_status(e, name);
}

}  // extern "C"
