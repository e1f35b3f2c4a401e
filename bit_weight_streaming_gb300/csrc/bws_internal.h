// Internal launch interface between the C ABI (abi.cu, stack.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
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
constexpr int kEpiSwiGLU = 3;      // h bf16 = SiLU(gate) * up

constexpr int kMaxMats = 4;
constexpr int kMaxTokens = 8;
constexpr int kMaxTopk = 8;
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

// Expert ("slot") mode: the matrices of a product are experts picked on the
// device. Slot s uses expert slot_expert[s] (-1: the shared expert). Tiles are
// numbered slot-major; the number of live slots is read from n_slots.
struct SlotMode {
  const int* n_slots;          // device [1]; nullptr: plain mode
  const int* slot_expert;      // device [max_slots]
  const uint8_t* codes;        // routed expert e starts at codes + e * codes_stride
  size_t codes_stride;
  const uint8_t* scales;
  size_t scales_stride;
  const uint8_t* shared_codes;
  const uint8_t* shared_scales;
  int rows;                    // rows of one matrix (one half for SwiGLU)
  int up_row_off;              // SwiGLU: first row of the up half in the expert tensor
  int tiles_per_slot;
  int max_slots;
  int n_experts;
  const uint32_t* ready;       // optional: non-zero once the slot table is written (MoeRoute::ready):
                               // the TMA expert kernel then reads it, and primes its first
                               // weight stages, before waiting for the kernels before
};

// Activations as the product kernels read them. Row (slot, tok) holds, for
// token tok of slot s, f16 values x * 2^(14 - E) ("hi band") and, for elements
// below 2^-14 after that scaling, x * 2^(43 - E) ("lo band"), with
// E = floor(log2 max|x|) of that row. Each slot block has N + 1 rows, the
// last all zero (read by the MMA columns of absent tokens).
struct XPrep {
  const uint16_t* hi;      // f16 [slots][N + 1][d_in_pad]
  const uint16_t* lo;
  const int* exp;          // [slots][N]
  const uint32_t* flags;   // [slots][N] bws_status_bits
  int shared;              // 1: every slot reads slot 0's activations
};

struct GemvParams {
  GemvMat mats[kMaxMats];
  int n_mats;
  SlotMode slots;
  int N, d_in, d_in_pad, nseg;
  int n_tiles;             // plain mode: all tiles; slot mode: tiles_per_slot * max_slots
  long long n_units;       // plain mode only
  long long n_warps;       // plain mode: warps sharing the units; slot mode: warps launched
  XPrep x;
  void* out;
  int out_ld;
  size_t out_slot_stride;  // elements between slots' outputs
  float* partials;         // [(n_tiles + warps) * kSlotFloats]
  uint32_t* counters;      // [n_tiles], zero on entry, left zero on exit
  int prefetch_units;      // units pulled into L2 before waiting on the inputs
  size_t partials_bytes;   // slot mode: size of the partials scratch (0: the plain-mode size)
  int split_light;         // TMA kernel: the last split_light CTAs start late (they wait for the
                           // slots the prep before holds): give them a lighter share (SplitK)
  int deposit;             // TMA kernel: tile pieces leave their raw sums in partials for the
                           // next prep to finish (PrepParams::fin_*), nothing else is stored
  unsigned long long* amax_key;   // TMA kernel, kEpiStoreF32, optional: per token the largest
                           // argmax_key(value, row) of the outputs (zero on entry)
  int no_store;            // with amax_key: the outputs themselves are not stored
};

// Greedy argmax over a product's outputs: the key orders by value (FP32 bits
// mapped to an order-preserving u32), then by lower row index, so the
// largest key over all outputs is the largest value with the lowest index
// among equal ones, whatever order the keys are combined in.
__host__ __device__ inline unsigned long long argmax_key(float v, int row) {
  uint32_t b;
  memcpy(&b, &v, 4);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)b << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)row);
}
__host__ __device__ inline int argmax_row(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}
// Word offset of the argmax keys after n_tiles tile counters (8-byte aligned).
inline int argmax_key_word(int n_tiles) { return (n_tiles + 1) & ~1; }
// tokens[n] = row (or row_token[row]) of keys[n], n < N.
cudaError_t launch_argmax_finish(const unsigned long long* keys, int N, const int32_t* row_token, int32_t* tokens,
                                 cudaStream_t st, bool pdl);

// MoE helpers.
struct MoeRoute {
  const int32_t* ids;      // [N][topk]
  const float* route_w;    // [N][topk]
  int N, topk, n_experts;
  int has_shared;
  int max_slots;
  int* n_slots;            // out [1]
  int* slot_expert;        // out [max_slots]
  float* cw;               // out [max_slots][N] combine weights
  uint32_t* status;        // out [1]: bit 4 set if an id was out of range
  int* tok_slots;          // optional out [N][topk]: each token's routed slots in ascending order
                           // (-1 for an id out of range), so that a combine reads only them
  uint32_t* ready;         // optional: set to 1 (release) once the table is written; the routing
                           // then runs without waiting for the kernels before (it reads only
                           // ids and weights), so the experts' kernels can read the table early
};
// MoE router (router.cu): z = W x for the E routed experts, then each
// token's top-k experts (largest logits, lower id first on equal logits) and
// their softmax-renormalised combine weights.
struct RouterParams {
  const uint16_t* W;       // bf16 [E][d], 16-byte aligned
  const uint16_t* x;       // bf16 [N][d], 16-byte aligned
  int N, E, d, topk;       // d % 8 == 0
  float* z;                // out [N][E] FP32 logits
  uint32_t* counter;       // zero on entry; counts the CTAs that finished
  int32_t* ids;            // out [N][topk], largest logit first
  float* route_w;          // out [N][topk]
  int has_route;           // also write the slot table of route (ids / route_w = the outputs above)
  MoeRoute route;
};
constexpr int kRouterMaxD = 7168;
constexpr int kRouterMaxExperts = 2048;
constexpr int kRouterSmemMax = 16 * 2 * kRouterMaxD;   // 8 rows and 8 tokens of x at the largest d (224 KB)
size_t router_smem_bytes(int N, int E, int d);
int router_ctas(int E);
cudaError_t launch_router(const RouterParams& p, cudaStream_t st, bool pdl);

// A stream-K split of n_units units over n_ctas CTAs into contiguous ranges:
// CTA c takes units [splitk_begin(c), splitk_begin(c + 1)). The CTAs from lf
// on get num/den of the others' share (uniform: lf = n_ctas, num = den = 1).
struct SplitK {
  long long n_units;
  int n_ctas, lf, num, den;
};
__host__ __device__ inline long long splitk_weight(const SplitK& s, long long c) {
  return c <= s.lf ? c * s.den : (long long)s.lf * s.den + (c - s.lf) * s.num;
}
__host__ __device__ inline long long splitk_begin(const SplitK& s, long long c) {
  return s.n_units * splitk_weight(s, c) / splitk_weight(s, s.n_ctas);
}
// The CTA whose range holds unit u: the last c with splitk_begin(c) <= u,
// i.e. with weight W(c) <= ((u + 1) W(n_ctas) - 1) / n_units.
// (Divisions in 32 bits where the operands fit: a 64-bit division is a long
// dependent chain on the GPU.)
__host__ __device__ inline int splitk_owner(const SplitK& s, long long u) {
  const long long x = (u + 1) * splitk_weight(s, s.n_ctas) - 1;
  const uint32_t t = x <= 0xFFFFFFFFLL ? (uint32_t)x / (uint32_t)s.n_units : (uint32_t)(x / s.n_units);
  const uint32_t w_lf = (uint32_t)s.lf * (uint32_t)s.den;
  const uint32_t c = t < w_lf ? t / (uint32_t)s.den : (uint32_t)s.lf + (t - w_lf) / (uint32_t)s.num;
  return (int)(c < (uint32_t)s.n_ctas - 1 ? c : (uint32_t)s.n_ctas - 1);
}

// Input of the activation prep kernel.
constexpr int kPrepCopy = 0;      // x bf16 -> bands
constexpr int kPrepRmsNorm = 1;   // r fp32 -> BF16(RMSNorm(r)) -> bands
struct PrepParams {
  int mode;
  const uint16_t* x;       // kPrepCopy: row (slot, tok) at x + slot * x_slot_stride + tok * ld
  int ld;
  size_t x_slot_stride;
  float* r;                // kPrepRmsNorm: residual [N][d_in]
  const uint16_t* x0;      // kPrepRmsNorm, optional: r = x0 first
  float eps;
  int N, d_in, d_in_pad;
  const int* n_slots;      // device; nullptr: one slot
  int max_slots;
  uint16_t* hi;
  uint16_t* lo;
  int* exp;
  uint32_t* flags;
  uint32_t* hdr;           // [0] = N (status reads), may be null
  uint32_t* status_clear;  // two words zeroed by the prep (the call's status words), may be null
  uint32_t* zero_ptr;      // counters of the next product, zeroed
  int zero_words;
  int interleave;          // 0: linear rows; kLayoutImage: the tensor-core kernel's E4M3 band
                           // image (one token); else the unit size in k (256 NVFP4, 128 FP8)
                           // of the TMA kernel's layout (see gemv_tma.cu)
  // kPrepRmsNorm, optional (comb_ys != nullptr): the previous MoE layer's
  // combine first, r[tok] += sum over live slots s, in slot order, of
  // comb_cw[s][tok] * comb_ys[s][tok][:]
  const float* comb_ys;
  const float* comb_cw;
  const int* comb_n_slots;
  int comb_max_slots;      // the layer's most slots (the arrays' extent)
  // optional: each token's routed slots, ascending (MoeRoute::tok_slots); the
  // combine then reads the shared slot and these only, in slot order
  const int* comb_tok_slots;
  int comb_topk, comb_has_shared;
  // optional: one extra CTA computes an MoE layer's slot table (one-CTA rows only)
  int has_route;
  MoeRoute route;
  // optional (fin_partials != nullptr): the input rows are the previous
  // product's outputs, finished here from the raw sums its CTAs deposited
  // (GemvParams::deposit): for each row, its tile's deposits added in CTA
  // order, scaled, then the product's store (kEpiResidF32: r += y, in
  // kPrepRmsNorm; kEpiStoreBF16: bf16(y), kEpiSwiGLU: bf16(SiLU(g) * u), in
  // kPrepCopy, also written back to x)
  const float* fin_partials;
  SplitK fin_split;        // the product's stream-K split and units per tile (TmaGeom)
  int fin_nks;
  int fin_epi, fin_fmt, fin_n_mats;
  int fin_row_off[kMaxMats], fin_tile_begin[kMaxMats];   // the matrices' first output row and tile
  const float* fin_scale[kMaxMats];
  const int* fin_xexp;     // exponents of the product's input rows [N]
  // optional (one-slot rows, not the tensor-core image): the BF16 row formed,
  // written to tap_x [N][d_in] (verification tap of the decode step)
  uint16_t* tap_x;
};

// Workspace of one product call (all offsets 256-byte aligned).
struct GemvWorkspace {
  size_t off_hdr, off_exp, off_flags, off_hi, off_lo, off_counters, off_partials, total;
};
GemvWorkspace gemv_workspace_layout(int N, int d_in, int n_tiles, long long max_warps, int slots = 1);
size_t align256(size_t v);
// Devices the per-device caches below cover (ordinals 0..kMaxDevices-1).
constexpr int kMaxDevices = 64;
// The current device's ordinal (0 if it cannot be read or is out of range).
int current_device();
// SM count of the current device (cached per device).
int num_sms();
// Sets a kernel's dynamic shared-memory limit once per device: attribute
// settings are per device, so a second GPU needs its own call.
template <typename K>
cudaError_t set_smem_once(std::atomic<unsigned long long>& done, K kernel, int bytes) {
  const unsigned long long bit = 1ull << current_device();
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}
long long gemv_max_warps();

cudaError_t launch_prep(const PrepParams& q, cudaStream_t st, bool pdl);
// Whether a prep can finish the deposits of a product into rows of d values.
bool prep_can_finish(int d);
// CTAs a prep of rows of d values runs per row (a cluster), finishing or not.
int prep_ctas_per_row(int d, bool fin);
cudaError_t launch_gemv(int fmt, int epi, const GemvParams& p, cudaStream_t st, bool pdl);
// The TMA-fed product kernel (gemv_tma.cu) for plain-mode NVFP4 (d_in % 256
// == 0) and FP8 (d_in % 128 == 0) products with 16-byte aligned tensors.
bool gemv_tma_eligible(int fmt, const GemvParams& p);
// Tiles of 128 rows (SwiGLU: 64 gate + 64 up rows) of the TMA kernels.
int gemv_tma_tiles(int epi, const GemvMat* mats, int n_mats);
// The TMA kernel's stream-K split of a product: n_tiles tiles of nks units.
struct TmaGeom {
  int n_tiles, nks;
  SplitK split;
};
TmaGeom gemv_tma_geometry(int fmt, int epi, const GemvParams& g);
// Whether g's partials scratch holds the deposits (GemvParams::deposit) of
// the TMA kernel's split: one [N][128] float slot per (tile, CTA) piece.
bool gemv_tma_deposit_fits(const TmaGeom& t, const GemvParams& g);
// Activation layout the TMA kernel reads for this format (PrepParams::interleave).
inline int tma_interleave(int fmt) { return fmt == kFmtFP8 ? 128 : 256; }
// PrepParams::interleave for the tensor-core kernel: one token's E4M3 band
// image (gemv_umma.cu), written over the token's two f16 band rows.
constexpr int kLayoutImage = -1;
// The tensor-core product (gemv_umma.cu): one-token NVFP4, d_in % 256 == 0,
// codes 32-byte and scales 16-byte aligned, taken when the environment sets
// BWS_PRODUCT_KERNEL=tcgen05 (opt-in: it streams slower than the mma.sync
// kernel, see gemv_umma.cu).
bool gemv_umma_eligible(int fmt, const GemvParams& p);
cudaError_t launch_gemv_umma(int epi, const GemvParams& p, uint32_t* status, cudaStream_t st, bool pdl);
// The activation layout the product of p reads (PrepParams::interleave).
inline int product_layout(int fmt, const GemvParams& p) {
  if (gemv_umma_eligible(fmt, p)) return kLayoutImage;
  return gemv_tma_eligible(fmt, p) ? tma_interleave(fmt) : 0;
}
cudaError_t launch_gemv_tma(int fmt, int epi, const GemvParams& p, uint32_t* status, cudaStream_t st, bool pdl);
// The TMA-fed MXFP4 expert kernel (gemv_tma_moe.cu) for slot-mode products
// with d_in % 256 == 0 and 16-byte aligned expert tensors and strides; its
// activations are prepared with the 256-weight TMA layout.
bool moe_tma_shape_ok(const uint8_t* codes, size_t codes_stride, const uint8_t* shared_codes, const uint8_t* scales,
                      size_t scales_stride, const uint8_t* shared_scales, int d_in, int N);
bool moe_tma_eligible(int epi, const GemvParams& p);
// Partial-sum scratch (bytes) the TMA expert kernel needs for max_slots slots of rows rows.
size_t moe_tma_partials_bytes(int epi, int rows, int max_slots);
int moe_tma_tiles_per_slot(int epi, int rows);
cudaError_t launch_gemv_tma_moe(int epi, const GemvParams& p, uint32_t* status, cudaStream_t st, bool pdl);
// Product with the best kernel for its shape.
inline cudaError_t launch_product(int fmt, int epi, const GemvParams& p, uint32_t* status, cudaStream_t st,
                                  bool pdl) {
  if (gemv_umma_eligible(fmt, p)) return launch_gemv_umma(epi, p, status, st, pdl);
  return gemv_tma_eligible(fmt, p) ? launch_gemv_tma(fmt, epi, p, status, st, pdl) : launch_gemv(fmt, epi, p, st, pdl);
}

cudaError_t launch_moe_route(const MoeRoute& m, cudaStream_t st, bool pdl);
// y[tok][i] (+)= sum over live slots s of cw[s][tok] * ys[s][tok][i]
cudaError_t launch_moe_combine(const float* ys, const float* cw, const int* n_slots, int N, int d,
                               void* out, int out_mode /* kEpiStoreBF16 or kEpiResidF32 */, cudaStream_t st,
                               bool pdl);

cudaError_t launch_nvfp4_quantize(const float* W, int d_out, int d_in, uint8_t* codes,
                                  uint8_t* scales, float* tensor_scale, void* ws, cudaStream_t st);
cudaError_t launch_mxfp4_quantize(const float* W, int rows, int d_in, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t st);
cudaError_t launch_fp8_rowwise_quantize(const float* W, int rows, int cols, uint8_t* codes,
                                        float* row_scale, cudaStream_t st);

cudaError_t launch_hbm_read_probe(const void* src, size_t n_bytes, uint32_t* out, cudaStream_t st);
cudaError_t launch_l2_flush(void* buf, size_t n_bytes, cudaStream_t st);
cudaError_t launch_wait_flag(const uint32_t* flag, uint32_t max_polls, uint32_t* hdr, cudaStream_t st);

}  // namespace bws
