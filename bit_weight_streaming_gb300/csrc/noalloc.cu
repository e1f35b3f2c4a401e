// NVFP4 GEMV for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory on the device: code that
// runs while a framework holds every byte of the device in its own pool,
// plugins invoked from a runtime that forbids allocation during a step, or
// latency-critical paths that must not call into an allocator. This entry
// point runs the same activation-prep and product kernels as bws_nvfp4_gemv,
// but its scratch lives in one statically sized device array defined in this
// file, which every GPU that loads the library keeps until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/bws.h"
#include "bws_abi_util.h"
#include "bws_internal.h"

namespace {

constexpr size_t kScratchBytes = (size_t)8 << 20;   // 8 MiB, see include/bws.h
constexpr int kMaxContexts = 64;

// The scratch. In host code this name is only a stand-in for the device
// array; its device address is looked up with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// A __device__ array's address belongs to the context that loaded the
// module: after cudaDeviceReset, or with another driver-API context current
// on the same device, the address looked up before is stale. The lookups are
// therefore cached per context, keyed on the context's process-unique id.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

std::mutex g_mu;
unsigned long long g_ctx_id[kMaxContexts] = {};
void* g_scratch_addr[kMaxContexts] = {};
int g_n_ctx = 0;

// Device address of the scratch in the current context, looked up the first
// time a context calls (with that context current).
int scratch_address(void** out) {
  const char* name = "bws_nvfp4_gemv_noalloc";
  cudaError_t e = cudaSuccess;
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return bws::fail(BWS_ERR_CUDA, "%s: driver context queries unavailable", name);
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS) return bws::fail(BWS_ERR_CUDA, "%s: cuCtxGetCurrent failed", name);
  if (ctx == nullptr) {
    // no context yet on this thread: the runtime's lookup makes the device's
    // primary context current
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return bws::cuda_status(e, "bws_nvfp4_gemv_noalloc: cudaGetSymbolAddress");
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return bws::fail(BWS_ERR_CUDA, "%s: no current CUDA context", name);
  }
  if (get_id(ctx, &id) != CUDA_SUCCESS) return bws::fail(BWS_ERR_CUDA, "%s: cuCtxGetId failed", name);
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_n_ctx; ++i) {
    if (g_ctx_id[i] == id) {
      *out = g_scratch_addr[i];
      return BWS_OK;
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return bws::cuda_status(e, "bws_nvfp4_gemv_noalloc: cudaGetSymbolAddress");
  // a full table recycles its entries in turn (a context past the 64th seen)
  static int next_recycled = 0;
  int slot = g_n_ctx;
  if (g_n_ctx < kMaxContexts) {
    ++g_n_ctx;
  } else {
    slot = next_recycled;
    next_recycled = (next_recycled + 1) % kMaxContexts;
  }
  g_ctx_id[slot] = id;
  g_scratch_addr[slot] = p;
  *out = p;
  return BWS_OK;
}

}  // namespace

extern "C" int bws_nvfp4_gemv_noalloc(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                                      const uint16_t* x, int N, int d_out, int d_in, uint16_t* y, void* stream) {
  if (N == 0 || d_out == 0) return bws_nvfp4_gemv(codes, scales, tensor_scale, x, N, d_out, d_in, y, nullptr, 0, stream);
  if (N > 0 && N <= bws::kMaxTokens && d_out > 0 && d_in >= 32 && d_in % 32 == 0) {
    const int n_tiles = (d_out + bws::kTileRows - 1) / bws::kTileRows;
    const size_t need = bws::gemv_workspace_layout(N, d_in, n_tiles, bws::gemv_max_warps()).total;
    if (need > kScratchBytes)
      return bws::fail(BWS_ERR_WORKSPACE,
                       "bws_nvfp4_gemv_noalloc: N=%d, d_out=%d, d_in=%d needs %zu bytes of scratch, more than "
                       "the %zu-byte static scratch; use bws_nvfp4_gemv with a workspace",
                       N, d_out, d_in, need, kScratchBytes);
  }
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != BWS_OK) return rc;
  // The product kernels clear what must start at zero (the tile counters are
  // zeroed by the activation prep of every call); everything else in the
  // scratch is written before it is read.
  return bws_nvfp4_gemv(codes, scales, tensor_scale, x, N, d_out, d_in, y, ws, kScratchBytes, stream);
}
