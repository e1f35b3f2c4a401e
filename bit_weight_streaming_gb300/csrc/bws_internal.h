// Internal launch interface between the C ABI (abi.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bws {

constexpr int kFmtNVFP4 = 1;
constexpr int kFmtMXFP4 = 2;
constexpr int kFmtFP8 = 3;

// Epilogues of a weight-stream product.
constexpr int kEpiStoreBF16 = 0;   // y bf16 [N][out_ld]
constexpr int kEpiStoreF32 = 1;    // y fp32 [N][out_ld]
constexpr int kEpiResidF32 = 2;    // r fp32 [N][out_ld] += y
constexpr int kEpiSwiGLU = 3;      // h bf16 = SiLU(gate) * up, mats[0]=gate, mats[1]=up

constexpr int kMaxMats = 4;
constexpr int kMaxTokens = 8;
constexpr int kSegK = 128;          // k values per work unit
constexpr int kWarpsPerCta = 8;
constexpr int kTileRows = 32;       // two m16 sub-tiles per work unit
constexpr int kSlotFloats = 32 * 8; // one warp's partial sums for one tile

struct GemvMat {
  const uint8_t* codes;
  const uint8_t* scales;   // NVFP4 E4M3 [d_out][d_in/16]; MXFP4 E8M0 [d_out][d_in/32]
  const float* scale32;    // NVFP4 tensor scale [1]; FP8 row scales [d_out]
  int d_out;
  int out_row_off;         // row offset of this matrix in the output
  int tile_begin;          // first tile of this matrix
};

// Activations as the product kernels read them: per token t, f16 values
// x * 2^(14 - E_t) ("hi band") and, for elements below 2^-14 after that
// scaling, x * 2^(43 - E_t) ("lo band"); E_t = floor(log2 max|x_t|).
struct XPrep {
  const uint16_t* hi;      // f16 [N][d_in_pad]
  const uint16_t* lo;      // f16 [N][d_in_pad]
  const int* exp;          // [N]
  const uint32_t* flags;   // [N] bws_status_bits
};

struct GemvParams {
  GemvMat mats[kMaxMats];
  int n_mats;
  int N, d_in, d_in_pad, nseg;
  int n_tiles;
  long long n_units;
  long long n_warps;       // warps that share the units (<= n_units)
  XPrep x;
  void* out;
  int out_ld;
  float* partials;         // [(n_tiles + n_warps) * kSlotFloats]
  uint32_t* counters;      // [n_tiles], zero on entry, left zero on exit
  int prefetch_units;       // units pulled into L2 before waiting on the inputs
  int prefetch_ahead;       // rolling L2 prefetch distance in units (0 = off)
};

// Workspace layout of one product call (all offsets 256-byte aligned).
struct GemvWorkspace {
  size_t off_hdr, off_exp, off_flags, off_hi, off_lo, off_counters, off_partials, total;
};
GemvWorkspace gemv_workspace_layout(int N, int d_in, int n_tiles, long long max_warps);
int num_sms();
long long gemv_max_warps();

cudaError_t launch_prep_x(const uint16_t* x, int N, int d_in, int d_in_pad, uint16_t* xhi,
                          uint16_t* xlo, int* xexp, uint32_t* xflags, uint32_t* hdr,
                          uint32_t* zero_ptr, int zero_words, cudaStream_t st, bool pdl);
cudaError_t launch_gemv(int fmt, int epi, const GemvParams& p, cudaStream_t st, bool pdl);

cudaError_t launch_nvfp4_quantize(const float* W, int d_out, int d_in, uint8_t* codes,
                                  uint8_t* scales, float* tensor_scale, void* ws, cudaStream_t st);
cudaError_t launch_mxfp4_quantize(const float* W, int rows, int d_in, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t st);
cudaError_t launch_fp8_rowwise_quantize(const float* W, int rows, int cols, uint8_t* codes,
                                        float* row_scale, cudaStream_t st);

cudaError_t launch_hbm_read_probe(const void* src, size_t n_bytes, uint32_t* out, cudaStream_t st);
cudaError_t launch_l2_flush(void* buf, size_t n_bytes, cudaStream_t st);

}  // namespace bws
