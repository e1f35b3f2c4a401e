// Quantizers: NVFP4 (E2M1 + E4M3 per 16 + FP32 tensor scale), MXFP4 (E2M1 +
// E8M0 per 32) and row-wise FP8 E4M3. Set-up work, run once per tensor.
//
// Every rounding decision is an IEEE FP32 operation with round-to-nearest-even
// (__fdiv_rn / __fmul_rn, no contraction) followed by the hardware encoders
// cvt.rn.satfinite.{e2m1x2,e4m3x2}.f32, so codes are reproducible bit for bit.
#include "bws_common.cuh"
#include "bws_internal.h"

namespace bws {

// ---- NVFP4 ------------------------------------------------------------------

// Pass 1: amax(|W|) over the whole tensor. Non-negative floats order like
// their bit patterns, so an integer atomicMax gives an exact, order-free max.
__global__ void __launch_bounds__(256) abs_max_kernel(const float4* __restrict__ W, size_t n4,
                                                      uint32_t* __restrict__ amax_bits) {
  float m = 0.0f;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    float4 v = W[i];
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  m = warp_max(m);
  __shared__ float sm[8];
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? sm[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(v));
  }
}

__global__ void zero_u32_kernel(uint32_t* p, int n) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0u;
}

BWS_DEV float nvfp4_tensor_scale_from_amax(float amax) {
  float s = __fdiv_rn(amax, 2688.0f);  // 6 * 448
  return s > 0.0f ? s : 1.0f;
}

// Pass 2: one thread per 16-weight block.
__global__ void __launch_bounds__(256) nvfp4_quantize_kernel(const float* __restrict__ W,
                                                             long long n_blocks,
                                                             const uint32_t* __restrict__ amax_bits,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales,
                                                             float* __restrict__ tensor_scale) {
  const float s_t = nvfp4_tensor_scale_from_amax(__uint_as_float(*amax_bits));
  long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b == 0) *tensor_scale = s_t;
  if (b >= n_blocks) return;
  const float4* src = reinterpret_cast<const float4*>(W + b * 16);
  float w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 v = src[i];
    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(w[i]));
  const float sb = __fdiv_rn(__fdiv_rn(amax, 6.0f), s_t);
  const uint32_t code_b = f32x2_to_e4m3x2(0.0f, sb) & 0xFF;
  const float d_b = __fmul_rn(e4m3_to_f32(code_b), s_t);
  uint32_t packed[2] = {0u, 0u};
  if (d_b > 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = f32x2_to_e2m1x2(__fdiv_rn(w[2 * i + 1], d_b), __fdiv_rn(w[2 * i], d_b));
      packed[i >> 2] |= (byte & 0xFF) << (8 * (i & 3));
    }
  }
  *reinterpret_cast<uint2*>(codes + b * 8) = make_uint2(packed[0], packed[1]);
  scales[b] = (uint8_t)code_b;
}

// ---- MXFP4 ------------------------------------------------------------------

// One thread per 32-weight block.
__global__ void __launch_bounds__(256) mxfp4_quantize_kernel(const float* __restrict__ W,
                                                             long long n_blocks,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales) {
  long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= n_blocks) return;
  const float4* src = reinterpret_cast<const float4*>(W + b * 32);
  float w[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 v = src[i];
    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(w[i]));
  uint32_t packed[4] = {0u, 0u, 0u, 0u};
  int e = -127;
  if (amax > 0.0f) {
    e = floor_log2_abs(amax) - 2;  // 2 = largest exponent of E2M1 (6 = 1.5 * 2^2)
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    const float inv = exp2i(-e);   // exact: -e in [-127, 127]
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t byte = f32x2_to_e2m1x2(__fmul_rn(w[2 * i + 1], inv), __fmul_rn(w[2 * i], inv));
      packed[i >> 2] |= (byte & 0xFF) << (8 * (i & 3));
    }
  }
  *reinterpret_cast<uint4*>(codes + b * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  scales[b] = (uint8_t)(e + 127);
}

// ---- FP8 row-wise -------------------------------------------------------------

// One CTA per row.
__global__ void __launch_bounds__(256) fp8_rowwise_quantize_kernel(const float* __restrict__ W, int cols,
                                                                   uint8_t* __restrict__ codes,
                                                                   float* __restrict__ row_scale) {
  const size_t row = blockIdx.x;
  const float* w = W + row * (size_t)cols;
  float m = 0.0f;
  for (int j = threadIdx.x; j < cols; j += blockDim.x) m = fmaxf(m, fabsf(w[j]));
  m = warp_max(m);
  __shared__ float sm[8];
  __shared__ float s_row;
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? sm[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) {
      s_row = __fdiv_rn(v, 448.0f);
      row_scale[row] = s_row;
    }
  }
  __syncthreads();
  const float s = s_row;
  uint8_t* c = codes + row * (size_t)cols;
  for (int j = 2 * threadIdx.x; j < cols; j += 2 * blockDim.x) {
    uint32_t two = 0u;
    if (s > 0.0f) two = f32x2_to_e4m3x2(__fdiv_rn(w[j + 1], s), __fdiv_rn(w[j], s));
    *reinterpret_cast<uint16_t*>(c + j) = (uint16_t)two;
  }
}

// ---- launchers -----------------------------------------------------------------

cudaError_t launch_nvfp4_quantize(const float* W, int d_out, int d_in, uint8_t* codes,
                                  uint8_t* scales, float* tensor_scale, void* ws, cudaStream_t st) {
  uint32_t* amax = reinterpret_cast<uint32_t*>(ws);
  zero_u32_kernel<<<1, 32, 0, st>>>(amax, 1);
  const size_t n = (size_t)d_out * d_in;
  const size_t n4 = n / 4;
  int grid = (int)((n4 + 255) / 256);
  if (grid > 152 * 8) grid = 152 * 8;
  if (grid < 1) grid = 1;
  abs_max_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float4*>(W), n4, amax);
  const long long nb = (long long)n / 16;
  nvfp4_quantize_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, st>>>(W, nb, amax, codes, scales,
                                                                     tensor_scale);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_quantize(const float* W, int rows, int d_in, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t st) {
  const long long nb = (long long)rows * d_in / 32;
  mxfp4_quantize_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, st>>>(W, nb, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_fp8_rowwise_quantize(const float* W, int rows, int cols, uint8_t* codes,
                                        float* row_scale, cudaStream_t st) {
  fp8_rowwise_quantize_kernel<<<rows, 256, 0, st>>>(W, cols, codes, row_scale);
  return cudaGetLastError();
}

}  // namespace bws
