// NVFP4 GEMV for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory on the device: code that
// runs while a framework holds every byte of the device in its own pool,
// plugins invoked from a runtime that forbids allocation during a step, or
// latency-critical paths that must not call into an allocator. This entry
// point runs the same activation-prep and product kernels as bws_nvfp4_gemv,
// but its scratch lives in one statically sized device array defined in this
// file, which every GPU that loads the library keeps until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/bws.h"
#include "bws_abi_util.h"
#include "bws_internal.h"

namespace {

constexpr size_t kScratchBytes = (size_t)8 << 20;   // 8 MiB, see include/bws.h
constexpr int kMaxDevices = 64;

// The scratch. In host code this name is only a stand-in for the device
// array; its device address is looked up with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return bws::cuda_status(e, "bws_nvfp4_gemv_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return bws::fail(BWS_ERR_INVALID_ARG, "bws_nvfp4_gemv_noalloc: device %d beyond the %d supported", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return bws::cuda_status(e, "bws_nvfp4_gemv_noalloc: cudaGetSymbolAddress");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
