// Host-side helpers shared by the C ABI translation units.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/bws.h"
#include "bws_internal.h"

namespace bws {

// MoE layer pieces used by the decode stream (moe.cu).
size_t moe_workspace_bytes(const bws_moe_layer* L, int N, int topk);
void moe_counter_span(const bws_moe_layer* L, int N, int topk, size_t* offset, int* words);
int check_moe_layer(const bws_moe_layer* L, int N, int topk, const char* name);
int enqueue_moe(const bws_moe_layer* L, const int32_t* ids, const float* route_w, int N, int topk,
                const uint16_t* x, void* y, int out_mode, void* ws, cudaStream_t st, const XPrep* x_prepped,
                const char* name);
// The decode stream's view of an MoE workspace: route buffer `buffer` (0 or
// 1) with the routing parameters of a layer, the slot outputs ys and the tile
// counters the prep before the experts zeroes.
struct MoeStackView {
  MoeRoute route;
  float* ys;
  uint16_t* h;             // SwiGLU activations of the slots [max_slots][N][inter]
  uint32_t* counters;
  int n_counters;
};
MoeStackView moe_stack_view(const bws_moe_layer* L, const int32_t* ids, const float* route_w, int N, int topk,
                            void* ws, int buffer);
// Activation layout the layer's gate/up kernel reads (PrepParams::interleave).
int moe_x_layout(const bws_moe_layer* L, int N);
// gate/up, prep h and down for the slots of a slot table (activations xp).
// ready: optional flag of the slot table (SlotMode::ready).
int enqueue_moe_experts(const bws_moe_layer* L, int N, int topk, const int* n_slots, const int* slot_expert,
                        const XPrep& xp, char* w, cudaStream_t st, const char* name,
                        const uint32_t* ready = nullptr);

// Records a message for bws_last_error() and returns code.
int fail(int code, const char* fmt, ...);
// BWS_OK for cudaSuccess (clearing the message), else BWS_ERR_CUDA.
int cuda_status(cudaError_t e, const char* what);
void clear_error();

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline int nseg_of(int d_in) { return (d_in + 127) / 128; }

}  // namespace bws
