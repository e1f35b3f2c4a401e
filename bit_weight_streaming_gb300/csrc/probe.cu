// Measurement kernels: an HBM read probe and an L2 flush.
#include "bws_common.cuh"
#include "bws_internal.h"

namespace bws {

// Streaming read of every 16-byte word, XOR-folded so the loads cannot be
// dropped; one atomic per CTA.
__global__ void __launch_bounds__(512) hbm_read_probe_kernel(const uint4* __restrict__ src, size_t n16,
                                                             uint32_t* __restrict__ out) {
  uint32_t acc = 0;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ld_stream_v4(src + i);
    const uint4 b = ld_stream_v4(src + i + stride);
    const uint4 c = ld_stream_v4(src + i + 2 * stride);
    const uint4 d = ld_stream_v4(src + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
  }
  for (; i < n16; i += stride) {
    const uint4 a = ld_stream_v4(src + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if ((threadIdx.x & 31) == 0) atomicXor(out, acc);
}

__global__ void __launch_bounds__(512) l2_flush_kernel(uint4* __restrict__ buf, size_t n16, uint32_t salt) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    buf[i] = make_uint4(salt, (uint32_t)i, salt, (uint32_t)(i >> 32));
}

cudaError_t launch_hbm_read_probe(const void* src, size_t n_bytes, uint32_t* out, cudaStream_t st) {
  hbm_read_probe_kernel<<<num_sms() * 4, 512, 0, st>>>(reinterpret_cast<const uint4*>(src), n_bytes / 16, out);
  return cudaGetLastError();
}

// Writes the first half of buf, then streams through the second half: the
// write evicts whatever the cache held, and the read evicts the dirty lines
// that write left, so the next kernel starts with a cold L2 holding only
// clean lines and pays no write-back.
cudaError_t launch_l2_flush(void* buf, size_t n_bytes, cudaStream_t st) {
  static uint32_t salt = 1;
  const size_t half16 = n_bytes / 32;
  l2_flush_kernel<<<num_sms() * 4, 512, 0, st>>>(reinterpret_cast<uint4*>(buf), half16, salt++);
  // the checksum of the read lands in the (already overwritten) first word
  hbm_read_probe_kernel<<<num_sms() * 4, 512, 0, st>>>(reinterpret_cast<const uint4*>(buf) + half16,
                                                         half16, reinterpret_cast<uint32_t*>(buf));
  return cudaGetLastError();
}

// One CTA runs the library's bounded flag wait (the acquire poll the MoE
// expert kernels use on their routing table's ready flag) on flag with a
// poll limit; when the limit runs out it sets the timeout bit in status[1]
// and returns, as every bounded wait in the library does.
__global__ void __launch_bounds__(32) wait_flag_kernel(const uint32_t* flag, uint32_t max_polls, uint32_t* hdr) {
  if (threadIdx.x != 0) return;
  hdr[0] = 0u;   // no token flags to collect
  if (!poll_acquire(flag, max_polls)) atomicOr(hdr + 1, 0x100u);
}

cudaError_t launch_wait_flag(const uint32_t* flag, uint32_t max_polls, uint32_t* hdr, cudaStream_t st) {
  wait_flag_kernel<<<1, 32, 0, st>>>(flag, max_polls, hdr);
  return cudaGetLastError();
}

// tokens[n]: the row of the largest argmax key of token n (keys the product
// kernel's epilogue combined), or row_token[row] when a map is given; -1 if
// no output was seen.
__global__ void __launch_bounds__(32) argmax_finish_kernel(const unsigned long long* keys, int N,
                                                           const int32_t* row_token, int32_t* tokens) {
  pdl_launch_dependents();
  pdl_wait();
  const int n = threadIdx.x;
  if (n >= N) return;
  const unsigned long long k = keys[n];
  const int row = k == 0ull ? -1 : argmax_row(k);
  tokens[n] = (row >= 0 && row_token != nullptr) ? row_token[row] : row;
}

cudaError_t launch_argmax_finish(const unsigned long long* keys, int N, const int32_t* row_token, int32_t* tokens,
                                 cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, argmax_finish_kernel, keys, N, row_token, tokens);
}

}  // namespace bws
