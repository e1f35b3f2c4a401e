// C ABI of the weight-stream library: argument checks, workspace layout and
// launches. See include/bws.h for the contract of every entry point.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "../../include/bws.h"
#include "bws_abi_util.h"
#include "bws_internal.h"

namespace {
thread_local char g_err[512] = "";
}

namespace bws {

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) {
    g_err[0] = 0;
    return BWS_OK;
  }
  return fail(BWS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void clear_error() { g_err[0] = 0; }

}  // namespace bws

using namespace bws;

namespace {

int check_tokens(int N) {
  if (N < 1 || N > kMaxTokens) return fail(BWS_ERR_INVALID_ARG, "N = %d must be in [1, %d]", N, kMaxTokens);
  return BWS_OK;
}


// The activation layout a prepare-only call writes: the one the product of an
// aligned matrix of this shape reads (the pointers below are never
// dereferenced, only tested for alignment).
int generic_layout(int fmt, const GemvParams& shape) {
  GemvParams g = shape;
  g.n_mats = 1;
  g.mats[0].codes = reinterpret_cast<const uint8_t*>(256);
  g.mats[0].scales = reinterpret_cast<const uint8_t*>(256);
  return product_layout(fmt, g);
}

constexpr int kPhaseBoth = 0, kPhasePrepare = 1, kPhaseProduct = 2;

// Shared body of every product call: prep the activations, then the product
// (phase: both, the prep alone, or the product on activations an earlier
// prepare-only call left in the workspace).
int run_product(int fmt, int epi, GemvParams& p, const uint16_t* x, int N, int d_in, void* ws,
                size_t ws_bytes, void* out, int out_ld, cudaStream_t st, const char* name, int phase = kPhaseBoth,
                const int32_t* row_token = nullptr, int32_t* tokens = nullptr) {
  p.N = N;
  p.d_in = d_in;
  p.nseg = nseg_of(d_in);
  p.d_in_pad = p.nseg * kSegK;
  p.n_units = (long long)p.n_tiles * p.nseg;
  const long long maxw = gemv_max_warps();
  p.n_warps = p.n_units < maxw ? p.n_units : maxw;
  const GemvWorkspace L = gemv_workspace_layout(N, d_in, p.n_tiles, maxw);
  if (ws == nullptr || ws_bytes < L.total)
    return fail(BWS_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", name, L.total, ws_bytes);
  if (!aligned(ws, 256)) return fail(BWS_ERR_MISALIGNED, "%s: workspace must be 256-byte aligned", name);
  char* w = static_cast<char*>(ws);
  PrepParams q = {};
  q.mode = kPrepCopy;
  q.x = x;
  q.ld = d_in;
  q.N = N;
  q.d_in = d_in;
  q.d_in_pad = p.d_in_pad;
  q.hi = reinterpret_cast<uint16_t*>(w + L.off_hi);
  q.lo = reinterpret_cast<uint16_t*>(w + L.off_lo);
  q.exp = reinterpret_cast<int*>(w + L.off_exp);
  q.flags = reinterpret_cast<uint32_t*>(w + L.off_flags);
  q.hdr = reinterpret_cast<uint32_t*>(w + L.off_hdr);
  q.status_clear = q.hdr + 1;
  q.zero_ptr = reinterpret_cast<uint32_t*>(w + L.off_counters);
  q.zero_words = p.n_tiles;
  if (tokens != nullptr) {   // greedy argmax: the keys after the tile counters, zeroed with them
    p.amax_key = reinterpret_cast<unsigned long long*>(q.zero_ptr + argmax_key_word(p.n_tiles));
    p.no_store = out == nullptr;
    q.zero_words = argmax_key_word(p.n_tiles) + 2 * N;
  }
  p.x.hi = q.hi;
  p.x.lo = q.lo;
  p.x.exp = q.exp;
  p.x.flags = q.flags;
  p.x.shared = 1;
  p.counters = q.zero_ptr;
  p.partials = reinterpret_cast<float*>(w + L.off_partials);
  p.out = out;
  p.out_ld = out_ld;
  p.out_slot_stride = 0;
  p.prefetch_units = fmt == kFmtFP8 ? 4 : 8;
  if (phase == kPhasePrepare) {
    q.interleave = generic_layout(fmt, p);
    return cuda_status(launch_prep(q, st, true), name);
  }
  q.interleave = product_layout(fmt, p);   // the layout its product reads
  if (phase == kPhaseProduct) {
    if (q.interleave != generic_layout(fmt, p))
      return fail(BWS_ERR_MISALIGNED,
                  "%s: the prepared activations are laid out for 16-byte aligned codes and scales "
                  "(32-byte codes for the tensor-core kernel); this matrix is not",
                  name);
    return cuda_status(launch_product(fmt, epi, p, q.hdr + 1, st, true), name);
  }
  if (tokens != nullptr && !(gemv_tma_eligible(fmt, p) && !gemv_umma_eligible(fmt, p)))
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: the fused argmax needs the TMA product kernel (d %% 128 == 0, "
                "16-byte aligned weights)", name);
  cudaError_t e = launch_prep(q, st, true);
  if (e != cudaSuccess) return cuda_status(e, name);
  e = launch_product(fmt, epi, p, q.hdr + 1, st, true);
  if (e == cudaSuccess && tokens != nullptr) e = launch_argmax_finish(p.amax_key, N, row_token, tokens, st, true);
  return cuda_status(e, name);
}

int tiles_rows32(int d_out) { return (d_out + kTileRows - 1) / kTileRows; }

}  // namespace

extern "C" {

int bws_version(void) { return 100; }

const char* bws_last_error(void) { return g_err; }

size_t bws_nvfp4_quantize_workspace_size(int d_out, int d_in) {
  (void)d_out;
  (void)d_in;
  return 256;
}

int bws_nvfp4_quantize(const float* W, int d_out, int d_in, uint8_t* codes, uint8_t* scales,
                       float* tensor_scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (!W || !codes || !scales || !tensor_scale || !workspace)
    return fail(BWS_ERR_INVALID_ARG, "bws_nvfp4_quantize: null pointer");
  if (d_out < 1 || d_in < 16 || d_in % 16 != 0)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "bws_nvfp4_quantize: d_out=%d d_in=%d (d_in %% 16 == 0 needed)", d_out, d_in);
  if (workspace_bytes < 4) return fail(BWS_ERR_WORKSPACE, "bws_nvfp4_quantize: workspace too small");
  if (!aligned(W, 16) || !aligned(codes, 8) || !aligned(workspace, 4))
    return fail(BWS_ERR_MISALIGNED, "bws_nvfp4_quantize: W 16-byte and codes 8-byte alignment needed");
  return cuda_status(launch_nvfp4_quantize(W, d_out, d_in, codes, scales, tensor_scale, workspace,
                                           as_stream(stream)), "bws_nvfp4_quantize");
}

int bws_mxfp4_quantize(const float* W, int rows, int d_in, uint8_t* codes, uint8_t* scales, void* stream) {
  if (!W || !codes || !scales) return fail(BWS_ERR_INVALID_ARG, "bws_mxfp4_quantize: null pointer");
  if (rows < 1 || d_in < 32 || d_in % 32 != 0)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "bws_mxfp4_quantize: rows=%d d_in=%d (d_in %% 32 == 0 needed)", rows, d_in);
  if (!aligned(W, 16) || !aligned(codes, 16))
    return fail(BWS_ERR_MISALIGNED, "bws_mxfp4_quantize: W and codes 16-byte alignment needed");
  return cuda_status(launch_mxfp4_quantize(W, rows, d_in, codes, scales, as_stream(stream)),
                     "bws_mxfp4_quantize");
}

int bws_fp8_rowwise_quantize(const float* W, int rows, int cols, uint8_t* codes, float* row_scale,
                             void* stream) {
  if (!W || !codes || !row_scale) return fail(BWS_ERR_INVALID_ARG, "bws_fp8_rowwise_quantize: null pointer");
  if (rows < 1 || cols < 2 || cols % 2 != 0)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "bws_fp8_rowwise_quantize: rows=%d cols=%d (even cols needed)", rows, cols);
  if (!aligned(W, 4) || !aligned(codes, 2))
    return fail(BWS_ERR_MISALIGNED, "bws_fp8_rowwise_quantize: misaligned pointer");
  return cuda_status(launch_fp8_rowwise_quantize(W, rows, cols, codes, row_scale, as_stream(stream)),
                     "bws_fp8_rowwise_quantize");
}

size_t bws_gemv_workspace_size(int N, int d_out_total, int d_in) {
  if (N < 1 || N > kMaxTokens || d_out_total < 1 || d_in < 1) return 0;
  const int n_tiles = (d_out_total + 15) / 16 + kMaxMats;
  return gemv_workspace_layout(N, d_in, n_tiles, gemv_max_warps()).total;
}

// Returns BWS_OK to proceed, or a status; *noop is set when there is nothing
// to compute (N == 0 or d_out == 0).
static int check_product_common(const char* name, const void* codes, const void* x, const void* y, int N,
                                int d_out, int d_in, bool* noop) {
  *noop = false;
  if (N < 0 || N > kMaxTokens) return check_tokens(N);
  if (d_out < 0 || d_in < 0) return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: negative dimension", name);
  if (N == 0 || d_out == 0) {
    *noop = true;
    g_err[0] = 0;
    return BWS_OK;
  }
  if (!codes || !x || !y) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (d_in < 32 || d_in % 32 != 0)
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "%s: d_out=%d d_in=%d (d_in %% 32 == 0 needed)", name, d_out, d_in);
  if (!aligned(codes, 16) || !aligned(x, 16))
    return fail(BWS_ERR_MISALIGNED, "%s: codes and x must be 16-byte aligned", name);
  return BWS_OK;
}

int bws_nvfp4_gemv(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale, const uint16_t* x,
                   int N, int d_out, int d_in, uint16_t* y, void* workspace, size_t workspace_bytes,
                   void* stream) {
  const char* name = "bws_nvfp4_gemv";
  bool noop;
  int rc = check_product_common(name, codes, x, y, N, d_out, d_in, &noop);
  if (rc || noop) return rc;
  if (!scales || !tensor_scale) return fail(BWS_ERR_INVALID_ARG, "%s: null scales", name);
  if (!aligned(scales, 2) || !aligned(tensor_scale, 4) || !aligned(y, 2))
    return fail(BWS_ERR_MISALIGNED, "%s: scales 2-byte, tensor_scale 4-byte, y 2-byte alignment needed", name);
  GemvParams p = {};
  p.n_mats = 1;
  p.mats[0] = {codes, scales, tensor_scale, d_out, 0, 0};
  p.n_tiles = tiles_rows32(d_out);
  return run_product(kFmtNVFP4, kEpiStoreBF16, p, x, N, d_in, workspace, workspace_bytes, y, d_out,
                     as_stream(stream), name);
}

int bws_nvfp4_prepare(const uint16_t* x, int N, int d_in, int d_out_max, void* workspace, size_t workspace_bytes,
                      void* stream) {
  const char* name = "bws_nvfp4_prepare";
  bool noop;
  const uint8_t* dummy = reinterpret_cast<const uint8_t*>(x);   // only the shape checks read it
  int rc = check_product_common(name, dummy, x, x, N, d_out_max, d_in, &noop);
  if (rc || noop) return rc;
  GemvParams p = {};
  p.n_tiles = tiles_rows32(d_out_max);
  return run_product(kFmtNVFP4, kEpiStoreBF16, p, x, N, d_in, workspace, workspace_bytes, nullptr, 0,
                     as_stream(stream), name, kPhasePrepare);
}

int bws_nvfp4_gemv_prepared(const uint8_t* codes, const uint8_t* scales, const float* tensor_scale, int N,
                            int d_out, int d_in, uint16_t* y, void* workspace, size_t workspace_bytes,
                            void* stream) {
  const char* name = "bws_nvfp4_gemv_prepared";
  bool noop;
  int rc = check_product_common(name, codes, codes, y, N, d_out, d_in, &noop);
  if (rc || noop) return rc;
  if (!scales || !tensor_scale) return fail(BWS_ERR_INVALID_ARG, "%s: null scales", name);
  if (!aligned(scales, 2) || !aligned(tensor_scale, 4) || !aligned(y, 2))
    return fail(BWS_ERR_MISALIGNED, "%s: scales 2-byte, tensor_scale 4-byte, y 2-byte alignment needed", name);
  GemvParams p = {};
  p.n_mats = 1;
  p.mats[0] = {codes, scales, tensor_scale, d_out, 0, 0};
  p.n_tiles = tiles_rows32(d_out);
  return run_product(kFmtNVFP4, kEpiStoreBF16, p, nullptr, N, d_in, workspace, workspace_bytes, y, d_out,
                     as_stream(stream), name, kPhaseProduct);
}

int bws_nvfp4_gate_up_silu(const uint8_t* gate_codes, const uint8_t* gate_scales, const float* gate_ts,
                           const uint8_t* up_codes, const uint8_t* up_scales, const float* up_ts,
                           const uint16_t* x, int N, int d_inter, int d_in, uint16_t* h, void* workspace,
                           size_t workspace_bytes, void* stream) {
  const char* name = "bws_nvfp4_gate_up_silu";
  bool noop;
  int rc = check_product_common(name, gate_codes, x, h, N, d_inter, d_in, &noop);
  if (rc || noop) return rc;
  if (!up_codes || !gate_scales || !up_scales || !gate_ts || !up_ts)
    return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned(up_codes, 16) || !aligned(gate_scales, 2) || !aligned(up_scales, 2) || !aligned(gate_ts, 4) ||
      !aligned(up_ts, 4) || !aligned(h, 2))
    return fail(BWS_ERR_MISALIGNED, "%s: misaligned pointer", name);
  GemvParams p = {};
  p.n_mats = 2;
  p.mats[0] = {gate_codes, gate_scales, gate_ts, d_inter, 0, 0};
  p.mats[1] = {up_codes, up_scales, up_ts, d_inter, 0, 0};
  p.n_tiles = (d_inter + 15) / 16;
  return run_product(kFmtNVFP4, kEpiSwiGLU, p, x, N, d_in, workspace, workspace_bytes, h, d_inter,
                     as_stream(stream), name);
}

int bws_fp8_lmhead_gemv(const uint8_t* W, const float* row_scale, const uint16_t* x, int N, int V, int d,
                        float* logits, void* workspace, size_t workspace_bytes, void* stream) {
  const char* name = "bws_fp8_lmhead_gemv";
  bool noop;
  int rc = check_product_common(name, W, x, logits, N, V, d, &noop);
  if (rc || noop) return rc;
  if (!row_scale) return fail(BWS_ERR_INVALID_ARG, "%s: null row_scale", name);
  if (!aligned(row_scale, 4) || !aligned(logits, 4))
    return fail(BWS_ERR_MISALIGNED, "%s: row_scale and logits 4-byte alignment needed", name);
  GemvParams p = {};
  p.n_mats = 1;
  p.mats[0] = {W, nullptr, row_scale, V, 0, 0};
  p.n_tiles = tiles_rows32(V);
  return run_product(kFmtFP8, kEpiStoreF32, p, x, N, d, workspace, workspace_bytes, logits, V,
                     as_stream(stream), name);
}

int bws_fp8_lmhead_argmax(const uint8_t* W, const float* row_scale, const uint16_t* x, int N, int V, int d,
                          float* logits, const int32_t* row_token, int32_t* token, void* workspace,
                          size_t workspace_bytes, void* stream) {
  const char* name = "bws_fp8_lmhead_argmax";
  bool noop;
  int rc = check_product_common(name, W, x, token, N, V, d, &noop);
  if (rc || noop) return rc;
  if (!row_scale) return fail(BWS_ERR_INVALID_ARG, "%s: null row_scale", name);
  if (!aligned(row_scale, 4) || !aligned(token, 4) || (logits && !aligned(logits, 4)) ||
      (row_token && !aligned(row_token, 4)))
    return fail(BWS_ERR_MISALIGNED, "%s: row_scale, logits, row_token and token 4-byte alignment needed", name);
  GemvParams p = {};
  p.n_mats = 1;
  p.mats[0] = {W, nullptr, row_scale, V, 0, 0};
  p.n_tiles = tiles_rows32(V);
  return run_product(kFmtFP8, kEpiStoreF32, p, x, N, d, workspace, workspace_bytes, logits, V, as_stream(stream),
                     name, kPhaseBoth, row_token, token);
}

int bws_status_word(const void* workspace, uint32_t* status, void* stream) {
  if (!workspace || !status) return fail(BWS_ERR_INVALID_ARG, "bws_status_word: null pointer");
  const GemvWorkspace L = gemv_workspace_layout(1, 32, 1, 1);
  uint32_t hdr2[2] = {0, 0}, flags[kMaxTokens] = {0};
  cudaStream_t st = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(hdr2, static_cast<const char*>(workspace) + L.off_hdr, 8,
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(flags, static_cast<const char*>(workspace) + L.off_flags, sizeof(flags),
                        cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e, "bws_status_word");
  uint32_t s = hdr2[1];
  for (uint32_t i = 0; i < hdr2[0] && i < (uint32_t)kMaxTokens; ++i) s |= flags[i];
  *status = s;
  if (s & BWS_STATUS_WAIT_TIMEOUT)
    return fail(BWS_ERR_TIMEOUT, "bws_status_word: a bounded device wait ran out (status 0x%x)", s);
  g_err[0] = 0;
  return BWS_OK;
}

int bws_debug_wait_flag(const uint32_t* flag, uint32_t max_polls, void* workspace, size_t workspace_bytes,
                        void* stream) {
  const char* name = "bws_debug_wait_flag";
  if (!flag || !workspace) return fail(BWS_ERR_INVALID_ARG, "%s: null pointer", name);
  if (max_polls == 0 || max_polls > (1u << 24))
    return fail(BWS_ERR_INVALID_ARG, "%s: max_polls must be in [1, 2^24]", name);
  const GemvWorkspace L = gemv_workspace_layout(1, 32, 1, 1);
  if (workspace_bytes < L.off_hdr + 8 || !aligned(workspace, 256) || !aligned(flag, 4))
    return fail(BWS_ERR_WORKSPACE, "%s: workspace of %zu bytes (256-byte aligned) and a 4-byte aligned flag needed",
                name, L.off_hdr + 8);
  uint32_t* hdr = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + L.off_hdr);
  cudaStream_t st = as_stream(stream);
  cudaError_t e = cudaMemsetAsync(hdr, 0, 8, st);
  if (e == cudaSuccess) e = launch_wait_flag(flag, max_polls, hdr, st);
  return cuda_status(e, name);
}

int bws_hbm_read_probe(const void* src, size_t n_bytes, uint32_t* out, void* stream) {
  if (!src || !out) return fail(BWS_ERR_INVALID_ARG, "bws_hbm_read_probe: null pointer");
  if (n_bytes == 0 || n_bytes % 16 != 0 || !aligned(src, 16))
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "bws_hbm_read_probe: n_bytes %% 16 == 0 and 16-byte alignment needed");
  return cuda_status(launch_hbm_read_probe(src, n_bytes, out, as_stream(stream)), "bws_hbm_read_probe");
}

int bws_l2_flush(void* buf, size_t n_bytes, void* stream) {
  if (!buf) return fail(BWS_ERR_INVALID_ARG, "bws_l2_flush: null pointer");
  if (n_bytes % 16 != 0 || !aligned(buf, 16))
    return fail(BWS_ERR_UNSUPPORTED_SHAPE, "bws_l2_flush: n_bytes %% 16 == 0 and 16-byte alignment needed");
  return cuda_status(launch_l2_flush(buf, n_bytes, as_stream(stream)), "bws_l2_flush");
}

}  // extern "C"
