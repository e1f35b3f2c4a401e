/*
 * bws.h -- C ABI of the decode-step weight stream (GB300 / sm_103a).
 *
 * The library streams block-scaled 4-bit (NVFP4, MXFP4) and 8-bit (FP8 E4M3)
 * weights against BF16 activations with FP32 accumulation: the batch-1 and
 * speculative-verify (N <= 8 token) decode step whose time is set by the
 * bytes of weights read ([Spark27B] "Decode speed is bytes divided by
 * bandwidth"; [LingMoE] sections 4 and 5).
 *
 * Page names used in the citations below:
 *   [Spark27B] mdjawad.com, DGX Spark post on Qwen3.8-27B NVFP4 decoding
 *   [LingMoE]  magicnetworld.com, reading of NVIDIA's "3 Ways to Boost MoE
 *              Inference on NVIDIA DGX Spark" (Ling-3.0-flash)
 *
 * Conventions for every entry point
 *   - Tensor pointers are DEVICE pointers unless a parameter says "host".
 *     The caller owns every buffer; the library never allocates device memory
 *     on these paths and never frees a caller pointer.
 *   - BF16 data is passed as its 16-bit patterns (uint16_t).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *     asynchronous on that stream; argument checks are synchronous.
 *   - Matrices are row-major. NVFP4 / MXFP4 codes are packed two per byte,
 *     element 2k in the low nibble; an E2M1 code is sign:1 exp:2 mant:1.
 *   - Scratch memory ("workspace") is passed by the caller; the size needed is
 *     returned by the matching *_workspace_size() function. Its contents need
 *     no initialisation and are overwritten by every call. Two calls that use
 *     the same workspace must not run concurrently.
 *   - Return value: BWS_OK or a BWS_ERR_* code; bws_last_error() returns a
 *     thread-local message for the last failing call on this host thread.
 *     Invalid arguments are reported before anything is enqueued.
 */
#ifndef BWS_H
#define BWS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum bws_status {
  BWS_OK = 0,
  BWS_ERR_INVALID_ARG = 1,      /* null pointer, N out of range, bad enum  */
  BWS_ERR_UNSUPPORTED_SHAPE = 2,/* a dimension the kernels do not support  */
  BWS_ERR_MISALIGNED = 3,       /* a pointer below its required alignment  */
  BWS_ERR_FORMAT = 4,           /* wrong or inconsistent format tag        */
  BWS_ERR_CUDA = 5,             /* a CUDA runtime call failed              */
  BWS_ERR_TIMEOUT = 6,          /* a bounded device wait ran out           */
  BWS_ERR_WORKSPACE = 7         /* workspace smaller than required         */
};

/* Weight formats of a matrix (the ABI carries the tag explicitly so that a
 * tensor can never be read in a format it was not written in: [LingMoE]
 * section 11 describes FP8 weights silently read as BF16). */
enum bws_format {
  BWS_FMT_NVFP4 = 1,   /* E2M1 codes, E4M3 scale per 16 along d_in, FP32 tensor scale */
  BWS_FMT_MXFP4 = 2,   /* E2M1 codes, E8M0 scale per 32 along d_in                    */
  BWS_FMT_FP8_ROW = 3  /* E4M3 codes, FP32 scale per row                              */
};

/* Bits of the device status word (bws_status_word). */
enum bws_status_bits {
  BWS_STATUS_X_TWO_BANDS = 1u,  /* an activation needed the second f16 band  */
  BWS_STATUS_X_FLUSHED = 2u,    /* an activation below 2^-57 of its token's
                                   largest magnitude was treated as zero     */
  BWS_STATUS_X_ROUNDED = 8u,    /* one-token NVFP4 products on the tensor
                                   cores: an activation below 2^-19 of its
                                   token's largest magnitude was rounded to a
                                   multiple of 2^-26 of that magnitude       */
  BWS_STATUS_WAIT_TIMEOUT = 0x100u /* a bounded device wait ran out: the
                                   results of that call are not valid        */
};

/* Library version (major*10000 + minor*100 + patch). */
int bws_version(void);

/* Message describing the last error on the calling host thread ("" if none). */
const char* bws_last_error(void);

/* ------------------------------------------------------------------------ */
/* Quantizers (set-up work: they run once per weight tensor, not per step)  */
/* ------------------------------------------------------------------------ */

/* NVFP4 quantization ([Spark27B] "Fewer bytes per weight: NVFP4": E2M1
 * elements, one E4M3 scale per 16 consecutive weights chosen so the block's
 * largest magnitude maps to 6, one FP32 scale per tensor bringing the block
 * scales into E4M3's range).
 *   W        fp32 [d_out][d_in], 16-byte aligned
 *   codes    u8   [d_out][d_in/2]   out
 *   scales   u8   [d_out][d_in/16]  out (E4M3 codes)
 *   tensor_scale  fp32 [1]          out: s_t = amax(|W|) / (6*448), 1 if that is 0
 * Per block b, in FP32 with round-to-nearest-even:
 *   code_b = E4M3(amax_b / 6 / s_t), d_b = dec(code_b) * s_t,
 *   q = E2M1(w / d_b) (zero codes where d_b == 0); both encoders saturate.
 * d_in % 16 == 0, d_out >= 1. Workspace: bws_nvfp4_quantize_workspace_size(). */
size_t bws_nvfp4_quantize_workspace_size(int d_out, int d_in);
int bws_nvfp4_quantize(const float* W, int d_out, int d_in, uint8_t* codes,
                       uint8_t* scales, float* tensor_scale, void* workspace,
                       size_t workspace_bytes, void* stream);

/* MXFP4 quantization ([LingMoE] section 17: 4-bit micro-scaling floats whose
 * small blocks share a scale; block size 32, E8M0 scale and clipping follow
 * the OCP MX definition): e = clamp(floor(log2 amax_b) - 2, -127, 127),
 * scale code e + 127, q = E2M1(w * 2^-e) saturating; a zero block gets code 0
 * and zero codes.
 *   W fp32 [rows][d_in]; codes u8 [rows][d_in/2]; scales u8 [rows][d_in/32].
 * d_in % 32 == 0. */
int bws_mxfp4_quantize(const float* W, int rows, int d_in, uint8_t* codes,
                       uint8_t* scales, void* stream);

/* Row-wise FP8 E4M3 quantization of an output layer ([LingMoE] section 7:
 * the BF16 head is quantized to FP8 when the model loads):
 * s_r = amax_r / 448, code = E4M3(w / s_r) saturating; s_r = 0 and zero codes
 * for a row whose s_r is 0.
 *   W fp32 [rows][cols]; codes u8 [rows][cols]; row_scale fp32 [rows]. */
int bws_fp8_rowwise_quantize(const float* W, int rows, int cols, uint8_t* codes,
                             float* row_scale, void* stream);

/* ------------------------------------------------------------------------ */
/* Weight-stream products                                                    */
/* ------------------------------------------------------------------------ */

/* Workspace bytes for one product call over a weight tensor with d_out_total
 * output rows (all matrices of the call together) and d_in columns, N tokens. */
size_t bws_gemv_workspace_size(int N, int d_out_total, int d_in);

/* NVFP4 GEMV / skinny GEMM: y[n][i] = s_t * sum_j dec(s_b(i,j)) * q_ij * x[n][j]
 * for N = 1..8 token rows (N = 1 is the plain decode step, N = K+1 the
 * speculative verify pass of [Spark27B] "More tokens per weight read").
 * Products are exact and accumulate in FP32; y is rounded to BF16.
 *   codes/scales/tensor_scale as written by bws_nvfp4_quantize
 *   x  bf16 [N][d_in]; y bf16 [N][d_out]
 * d_in % 32 == 0; codes, scales, x, y 16-byte aligned. N == 0 or d_out == 0
 * is a no-op that returns BWS_OK. */
int bws_nvfp4_gemv(const uint8_t* codes, const uint8_t* scales,
                   const float* tensor_scale, const uint16_t* x, int N,
                   int d_out, int d_in, uint16_t* y, void* workspace,
                   size_t workspace_bytes, void* stream);

/* bws_nvfp4_gemv in two phases, for several products of one input (the
 * query, key and value projections of a token, or the gate and up halves
 * called separately): bws_nvfp4_prepare writes the activations x bf16
 * [N][d_in] into the workspace, sized with bws_gemv_workspace_size(N,
 * d_out_max, d_in), in the layout the product kernel of a matrix with
 * 16-byte aligned codes and scales reads; every bws_nvfp4_gemv_prepared
 * call with the same N and d_in and d_out <= d_out_max then runs only the
 * product on them (same results as bws_nvfp4_gemv). The workspace holds the
 * prepared activations until the next prepare or bws_nvfp4_gemv call on it;
 * its status word (bws_status_word) is cleared by the prepare and collects
 * the products'. A matrix whose codes or scales are not 16-byte aligned
 * (d_in % 256 == 0) is rejected with BWS_ERR_MISALIGNED: its kernel reads
 * another layout. Same shape constraints as bws_nvfp4_gemv. */
int bws_nvfp4_prepare(const uint16_t* x, int N, int d_in, int d_out_max,
                      void* workspace, size_t workspace_bytes, void* stream);
int bws_nvfp4_gemv_prepared(const uint8_t* codes, const uint8_t* scales,
                            const float* tensor_scale, int N, int d_out,
                            int d_in, uint16_t* y, void* workspace,
                            size_t workspace_bytes, void* stream);

/* bws_nvfp4_gemv for callers that cannot allocate device memory (a caller
 * whose framework owns the whole device pool, a plugin called from a runtime
 * that forbids allocation during a step, a latency-critical path that must
 * not enter an allocator). The pages have no counterpart: this is a property
 * of the library, not of the method. Same arguments and results as
 * bws_nvfp4_gemv, without the workspace: the call uses an 8 MiB scratch array
 * that the library defines as static device memory, which every GPU that
 * loads the library holds until the process exits.
 *   - Sizes whose scratch exceeds 8 MiB (about N * d_in * 8 bytes plus
 *     (d_out/32 + 16 * SMs) KiB) are rejected with BWS_ERR_WORKSPACE and a
 *     message; the call allocates nothing (no cudaMalloc, no allocating
 *     library routine).
 *   - The first call in a CUDA context looks up the scratch's device address
 *     (once per context, with that context current: a device that was reset,
 *     or another driver-API context made current on it, gets a lookup of its
 *     own); make that first call before any stream capture.
 *   - All calls on a device share the one scratch array and it keeps the last
 *     call's contents: calls that overlap on the GPU (different streams, or
 *     host threads without ordering) race with each other. Order them. */
int bws_nvfp4_gemv_noalloc(const uint8_t* codes, const uint8_t* scales,
                           const float* tensor_scale, const uint16_t* x, int N,
                           int d_out, int d_in, uint16_t* y, void* stream);

/* Fused MLP front half: h[n][i] = BF16( SiLU(g) * u ) with g = W_gate x,
 * u = W_up x, both NVFP4 [d_inter][d_in], computed in FP32 and never written
 * out ([Spark27B] flow figure: gate, up, SiLU, then down). SiLU(g) =
 * g / (1 + exp(-g)).  h bf16 [N][d_inter]. Same constraints as bws_nvfp4_gemv. */
int bws_nvfp4_gate_up_silu(const uint8_t* gate_codes, const uint8_t* gate_scales,
                           const float* gate_tensor_scale,
                           const uint8_t* up_codes, const uint8_t* up_scales,
                           const float* up_tensor_scale, const uint16_t* x,
                           int N, int d_inter, int d_in, uint16_t* h,
                           void* workspace, size_t workspace_bytes, void* stream);

/* FP8 output layer: logits[n][v] = s_v * sum_j dec(W[v][j]) * x[n][j], FP32
 * out ([Spark27B]: the 248,320 x 5,120 output layer is read in full every
 * step; [LingMoE] section 7).
 *   W u8 [V][d] E4M3; row_scale fp32 [V]; x bf16 [N][d]; logits fp32 [N][V].
 * d % 32 == 0. */
int bws_fp8_lmhead_gemv(const uint8_t* W, const float* row_scale,
                        const uint16_t* x, int N, int V, int d, float* logits,
                        void* workspace, size_t workspace_bytes, void* stream);

/* The FP8 output layer with the greedy choice of the next token fused into
 * its epilogue ([Spark27B] "MTP": the whole 248,320-row output layer is read
 * only to pick one token; "Shaving the step": a reduced-vocabulary draft head
 * of the 100,032 most used rows). For each token row n, token[n] = the row
 * of the largest logit (ties: the lowest row), mapped through row_token when
 * given (a reduced head's row -> vocabulary id), -1 if V == 0. The logits of
 * bws_fp8_lmhead_gemv are also stored when `logits` is not NULL. Every CTA
 * keeps the best (value, lowest row) per token over the tiles it stores and
 * one 64-bit atomic max per CTA and token combines them: the result does not
 * depend on the order the CTAs finish in.
 *   W, row_scale, x, N, V, d: as bws_fp8_lmhead_gemv (d % 128 == 0, W
 *   16-byte aligned: the TMA kernel carries the fused epilogue, else
 *   BWS_ERR_UNSUPPORTED_SHAPE); row_token int32 [V] or NULL; token int32 [N].
 * Workspace: bws_gemv_workspace_size(N, V, d). */
int bws_fp8_lmhead_argmax(const uint8_t* W, const float* row_scale,
                          const uint16_t* x, int N, int V, int d, float* logits,
                          const int32_t* row_token, int32_t* token, void* workspace,
                          size_t workspace_bytes, void* stream);

/* One MXFP4 mixture-of-experts layer ([LingMoE] sections 3, 4 and 8: each
 * token is routed to top-k of n_experts routed experts plus one shared
 * expert; only the activated experts' weights are read; N tokens of a
 * verify pass widen the set of distinct experts).
 * Expert e's weights: gate_up rows [0, inter) are the gate, rows
 * [inter, 2*inter) the up projection, both [.][hidden]; down is
 * [hidden][inter]. Expert e's tensors start at base + e * stride bytes. */
typedef struct bws_moe_layer {
  int n_experts;           /* routed experts (e.g. 512)                      */
  int hidden;              /* model width (e.g. 2560), % 32 == 0             */
  int inter;               /* expert intermediate width (e.g. 768), % 32 == 0*/
  const uint8_t* gate_up_codes;  size_t gate_up_codes_stride;  /* [2*inter][hidden/2] */
  const uint8_t* gate_up_scales; size_t gate_up_scales_stride; /* [2*inter][hidden/32] */
  const uint8_t* down_codes;     size_t down_codes_stride;     /* [hidden][inter/2]    */
  const uint8_t* down_scales;    size_t down_scales_stride;    /* [hidden][inter/32]   */
  /* shared expert (weight 1), same shapes; NULL codes = no shared expert */
  const uint8_t* shared_gate_up_codes; const uint8_t* shared_gate_up_scales;
  const uint8_t* shared_down_codes;    const uint8_t* shared_down_scales;
} bws_moe_layer;

/* y[n] = shared(x[n]) + sum_k route_w[n][k] * expert_{ids[n][k]}(x[n]) with
 * expert(x) = W_down BF16(SiLU(W_gate x) * W_up x); FP32 accumulation, y BF16.
 *   L host pointer to the layer descriptor (copied during the call)
 *   ids int32 [N][topk] device, distinct per token, in [0, n_experts)
 *   route_w fp32 [N][topk] device; x bf16 [N][hidden]; y bf16 [N][hidden]
 * N in [1, 8], topk in [1, 8]. Ids are read on the device; an id out of range
 * is skipped and flagged in the status word (see bws_mxfp4_moe_inspect). */
size_t bws_mxfp4_moe_workspace_size(const bws_moe_layer* L, int N, int topk);
int bws_mxfp4_moe_gemv(const bws_moe_layer* L, const int32_t* ids,
                       const float* route_w, int N, int topk, const uint16_t* x,
                       uint16_t* y, void* workspace, size_t workspace_bytes,
                       void* stream);

/* W4A8: MXFP4 weights times MXFP8 activations on the tensor cores
 * ([LingMoE] section 3: the MoE baseline runs W4A8, 4-bit MXFP4 weights with
 * 8-bit activations; the pages do not give the activation quantizer, which is
 * read from the OCP MX rule).
 *
 * bws_mxfp8_quantize: x bf16 [N][d] (device, finite) -> codes u8 [N][d] E4M3
 * and scales u8 [N][d/32] E8M0, per block of 32 values along the row:
 *   e = clamp(floor(log2 amax) - 8, -127, 127), scale code e + 127,
 *   code_j = E4M3(x_j * 2^-e), nearest even, saturating at 448, sign kept;
 * an all-zero block gets scale code 0 and zero codes. N >= 0 (0: no-op),
 * d % 32 == 0. One kernel on the stream, no workspace.
 *
 * bws_mxfp4_w4a8_gemv: y[n][i] = sum_j w_ij * xq[n][j], w the MXFP4 weights
 * (codes and scales as bws_mxfp4_quantize writes them) and xq the MXFP8
 * quantization of x above; FP32 accumulation, y rounded to BF16.
 *   codes u8 [d_out][d_in/2] (32-byte aligned), scales u8 [d_out][d_in/32]
 *   (8-byte aligned), x bf16 [N][d_in], y bf16 [N][d_out]: device pointers
 *   N in [1, 8], d_in % 256 == 0; N == 0 or d_out == 0 is a no-op.
 *   Workspace: bws_w4a8_workspace_size(N, d_out, d_in) bytes, 256-byte
 *   aligned (0 for sizes out of range); its status word (bws_status_word)
 *   reports a bounded wait that ran out. Two kernels on the stream: the
 *   activation quantizer, then the product (one CTA per SM). */
int bws_mxfp8_quantize(const uint16_t* x, int N, int d, uint8_t* codes,
                       uint8_t* scales, void* stream);
size_t bws_w4a8_workspace_size(int N, int d_out, int d_in);
int bws_mxfp4_w4a8_gemv(const uint8_t* codes, const uint8_t* scales,
                        const uint16_t* x, int N, int d_out, int d_in,
                        uint16_t* y, void* workspace, size_t workspace_bytes,
                        void* stream);

/* MoE router ([LingMoE] section 3: each MoE layer sends every token to 8 of
 * its 512 routed experts, plus one shared expert). The pages name the routing
 * but not its arithmetic; this library reads it as
 *   z[n][e] = sum_j W[e][j] * x[n][j]   (BF16 operands, FP32 accumulation)
 *   ids[n][0..topk) = the topk largest z[n][.], largest first; on equal
 *                     logits the lower expert id ranks first; NaN ranks last
 *   route_w[n][i]   = exp(z_i - z_0) / sum_j exp(z_j - z_0) over the chosen
 *                     (the softmax over all experts renormalised over them)
 *   W_router bf16 [n_experts][d], x bf16 [N][d]: device, 16-byte aligned
 *   logits fp32 [N][n_experts] device or NULL (then kept in the workspace)
 *   ids int32 [N][topk], route_w fp32 [N][topk]: device outputs
 * N in [1, 8], n_experts in [1, 2048], topk in [1, min(8, n_experts)],
 * d % 8 == 0 and d <= 7168. Workspace: bws_moe_router_workspace_size(N,
 * n_experts) bytes, 256-byte aligned (returns 0 for sizes out of range).
 * One kernel on the stream; the ids feed bws_mxfp4_moe_gemv directly. */
size_t bws_moe_router_workspace_size(int N, int n_experts);
int bws_moe_router_topk(const uint16_t* W_router, const uint16_t* x, int N,
                        int n_experts, int d, int topk, float* logits,
                        int32_t* ids, float* route_w, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Verification tap: copies to HOST memory, from the workspace of the last
 * bws_mxfp4_moe_gemv call with the same (L, N, topk), the number of live
 * expert slots, the expert of every slot (-1 = shared expert; shared first,
 * then the distinct routed experts in ascending id order), the SwiGLU
 * activations h bf16 [N*topk + has_shared][N][inter] in slot order (rows of
 * slots >= *n_slots are stale) and the status word (bit 4: an id was out of
 * range). Synchronises the stream. */
int bws_mxfp4_moe_inspect(const void* workspace, const bws_moe_layer* L, int N,
                          int topk, int* n_slots, int32_t* slot_expert,
                          uint16_t* h, uint32_t* status, void* stream);

/* ------------------------------------------------------------------------ */
/* Whole decode step                                                         */
/* ------------------------------------------------------------------------ */

/* One weight matrix of a layer stack, in the layout its quantizer writes. */
typedef struct bws_matrix {
  int format;              /* enum bws_format                                  */
  int d_out, d_in;         /* d_in % 32 == 0                                   */
  const uint8_t* codes;    /* 16-byte aligned                                  */
  const uint8_t* scales;   /* NVFP4: E4M3 [d_out][d_in/16]; MXFP4: E8M0 [d_out][d_in/32]; FP8: NULL */
  const float* scale32;    /* NVFP4: tensor scale [1]; FP8: row scales [d_out]; MXFP4: NULL */
} bws_matrix;

enum bws_layer_kind {
  BWS_LAYER_MIXER_MLP = 1, /* token mixer (weight-free op) + SwiGLU MLP        */
  BWS_LAYER_MLP = 2,       /* SwiGLU MLP only                                  */
  BWS_LAYER_MOE = 3        /* MXFP4 mixture of experts                         */
};

/* One layer. [Spark27B] "Decode speed is bytes divided by bandwidth": each
 * layer is a token-mixing block then the MLP, and the mixing operation itself
 * (attention over the cache, or the Gated DeltaNet state update) reads no
 * weights. Its stand-in here takes the first mixer_out.d_in entries of the
 * concatenated input projections. */
typedef struct bws_layer {
  int kind;                      /* enum bws_layer_kind                        */
  int n_mixer_in;                /* MIXER_MLP: 1..4 input projections          */
  bws_matrix mixer_in[4];        /* MIXER_MLP: same format and d_in = hidden   */
  bws_matrix mixer_out;          /* MIXER_MLP: [hidden][d_v]                   */
  bws_matrix gate, up, down;     /* MIXER_MLP, MLP: gate/up [inter][hidden], down [hidden][inter] */
  bws_moe_layer moe;             /* MOE                                         */
  const int32_t* ids;            /* MOE: device [N][topk]                       */
  const float* route_w;          /* MOE: device [N][topk]                       */
  int topk;                      /* MOE                                         */
  const uint16_t* router;        /* MOE, optional: bf16 [n_experts][hidden], 16-byte aligned. When set,
                                    the step routes the layer itself (bws_moe_router_topk on the layer's
                                    normalised input, then the experts) and WRITES the chosen ids and
                                    weights to ids / route_w, which must then be writable device buffers.
                                    NULL: ids / route_w are inputs, read on the device every step. */
} bws_layer;

typedef struct bws_stack {
  int hidden;                    /* residual width, % 32 == 0                  */
  int n_layers;
  const bws_layer* layers;       /* host array [n_layers], read at plan creation */
  bws_matrix head;               /* output layer [vocab][hidden], FP8 row-scaled */
  float rms_eps;                 /* weightless RMSNorm epsilon (e.g. 1e-6)     */
} bws_stack;

/* A validated stack with its launch sequence. Create once, run many times;
 * the plan copies the descriptors. A dense stack (layers MIXER_MLP or MLP,
 * every layer matrix NVFP4 with d_in % 256 == 0, an NVFP4 or FP8 output layer
 * with hidden % 128 == 0, 16-byte aligned tensors) can run as one persistent
 * cooperative kernel after a small init kernel (opt-in for now: set the
 * environment variable BWS_STEP_KERNEL=1 before creating the plan); for it
 * the plan builds, on
 * the device current at creation, a table of TMA descriptors in a small
 * device allocation it owns (about 600 B per matrix) and frees on destroy.
 * Any other stack runs as a chain of per-product kernels and the plan owns no
 * device memory. Create, run and destroy the plan with the same device
 * current. */
typedef struct bws_stack_plan bws_stack_plan;

int bws_decode_step_plan_create(const bws_stack* S, int N, bws_stack_plan** plan);
void bws_decode_step_plan_destroy(bws_stack_plan* plan);
size_t bws_decode_step_workspace_size(const bws_stack_plan* plan);

/* Runs the whole decode step for the plan's N tokens:
 *   r = x0
 *   MIXER_MLP: a = BF16(RMSNorm(r)); u = BF16([W_in1 a, W_in2 a, ...]);
 *              r += W_out u[:d_v]; then the MLP
 *   MLP:       m = BF16(RMSNorm(r)); r += W_down BF16(SiLU(W_gate m) * W_up m)
 *   MOE:       m = BF16(RMSNorm(r)); r += MoE(m)
 *   logits = head(BF16(RMSNorm(r)))
 * RMSNorm is weightless: r / sqrt(mean(r^2) + eps). The residual r is FP32.
 *   x0 bf16 [N][hidden]; logits fp32 [N][vocab].
 * With a non-default stream the first call records the step as a CUDA graph
 * and later calls with the same (x0, logits, workspace, stream) replay it; on
 * the legacy default stream the kernels are launched directly. */
int bws_decode_step_stream(bws_stack_plan* plan, const uint16_t* x0, float* logits,
                           void* workspace, size_t workspace_bytes, void* stream);

/* The decode step with greedy decoding fused into the output layer (see
 * bws_fp8_lmhead_argmax): tokens int32 [N] receives each token row's
 * next-token choice; logits (fp32 [N][vocab]) are stored too unless NULL;
 * row_token (int32 [vocab] or NULL) maps output rows to vocabulary ids.
 * Graph recording and replay as bws_decode_step_stream (keyed also on
 * tokens and row_token). The kernel chain only (not the persistent kernel). */
int bws_decode_step_greedy(bws_stack_plan* plan, const uint16_t* x0, float* logits,
                           const int32_t* row_token, int32_t* tokens,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Number of kernels one decode step launches (2 for the persistent kernel). */
int bws_decode_step_kernel_count(const bws_stack_plan* plan);

/* Verification tap of the kernel chain (not the persistent kernel): runs the
 * same step as bws_decode_step_stream, launched directly on the stream (no
 * graph), and also copies into `tap` (device, 256-byte aligned,
 * bws_decode_step_tap_size bytes) what each stage of the layer recipe
 * received or produced, as the GPU formed it, so that every stage can be
 * checked on its own against its definition from its actual input. Records
 * follow in launch order, each starting on a 256-byte boundary:
 *   MIXER_MLP layer: a bf16 [N][hidden] (BF16(RMSNorm(r))), r fp32
 *     [N][hidden] (the residual a normalised), v bf16 [N][d_v] (the first
 *     d_v outputs of the mixer input projections, the mixer-out input), then
 *     the MLP records below;
 *   MIXER_MLP and MLP layers: m bf16 [N][hidden], r fp32 [N][hidden] (the
 *     residual m normalised), h bf16 [N][inter] (the down projection input);
 *   MOE layer: m, r as above; with a router, its logits fp32
 *     [N][n_experts], then the ids int32 [N][topk] and weights fp32
 *     [N][topk] it chose; then the slot count int32 [1], the slot experts
 *     int32 [S] (-1: the shared expert), the combine weights fp32 [S][N], h
 *     bf16 [S][N][inter] per slot and the slots' outputs fp32 [S][N][hidden]
 *     (S = N * topk + 1 with a shared expert, else N * topk; slots past the
 *     count hold stale values);
 *   the output layer: x bf16 [N][hidden] and the r it normalised.
 * The logits go to `logits` as with bws_decode_step_stream. */
size_t bws_decode_step_tap_size(const bws_stack_plan* plan);
int bws_decode_step_tap(bws_stack_plan* plan, const uint16_t* x0, float* logits,
                        void* workspace, size_t workspace_bytes, void* tap,
                        size_t tap_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Status and measurement                                                    */
/* ------------------------------------------------------------------------ */

/* Copies the device status word of a workspace (an OR of bws_status_bits set
 * by the calls that used it) into *status (host); synchronises the stream.
 * Returns BWS_ERR_TIMEOUT (with *status filled in) when a bounded device wait
 * of those calls ran out, else BWS_OK. */
int bws_status_word(const void* workspace, uint32_t* status, void* stream);

/* Failure-path check of the bounded device waits (no counterpart on the
 * pages): one CTA polls *flag (device, acquire loads, a short sleep between
 * polls) until it is non-zero, at most max_polls times (1..2^24), with the
 * same wait the MoE expert kernels run on their routing table's ready flag.
 * A flag that stays zero makes the wait run out: the kernel sets
 * BWS_STATUS_WAIT_TIMEOUT in the workspace's status word and returns, so
 * bws_status_word then reports BWS_ERR_TIMEOUT. Nothing hangs and the context
 * stays usable. workspace: 256-byte aligned, bws_gemv_workspace_size(1, 1, 32)
 * bytes suffice. */
int bws_debug_wait_flag(const uint32_t* flag, uint32_t max_polls, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Read-only streaming sum over n_bytes (% 16 == 0) of src; writes one u32
 * checksum to out. Used to measure the achievable HBM read bandwidth. */
int bws_hbm_read_probe(const void* src, size_t n_bytes, uint32_t* out, void* stream);

/* Leaves L2 cold and clean for the next kernel: writes the first half of buf,
 * then streams through the second half (n_bytes should be >= 4 x L2). */
int bws_l2_flush(void* buf, size_t n_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* BWS_H */
