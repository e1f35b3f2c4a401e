// Host interface of the persistent decode-step kernel (step.cu), used by the
// decode-step plan (stack.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/bws.h"

namespace bws {

struct StepProgram;

// The program of a dense stack (layers of kind MIXER_MLP or MLP, every matrix
// NVFP4 with d_in % 256 == 0, output layer NVFP4 or FP8 with hidden % 128 ==
// 0, hidden % 128 == 0), built on the current device: tensor maps and the
// product table are copied to a small device allocation owned by the
// program. nullptr if the stack does not qualify (the plan then uses the
// per-product kernel chain) or the device cannot run it.
StepProgram* step_program_create(int N, int hidden, float eps, const bws_layer* layers, int n_layers,
                                 const bws_matrix& head);
void step_program_destroy(StepProgram* program);
// Workspace bytes the program's step needs (256-byte aligned base).
size_t step_program_workspace(const StepProgram* program);
// CTAs of the persistent kernel.
int step_program_grid(const StepProgram* program);
// Byte offset in the workspace of the optional trace (-1: none) and the
// number of products.
long long step_program_trace(const StepProgram* program, int* n_prods);
// Enqueues one step: an init kernel, then the persistent kernel (2 launches).
cudaError_t step_program_enqueue(const StepProgram* program, const uint16_t* x0, float* logits, void* ws,
                                 cudaStream_t st);

}  // namespace bws
