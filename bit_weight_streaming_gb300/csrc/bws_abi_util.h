// Host-side helpers shared by the C ABI translation units.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace bws {

// Records a message for bws_last_error() and returns code.
int fail(int code, const char* fmt, ...);
// BWS_OK for cudaSuccess (clearing the message), else BWS_ERR_CUDA.
int cuda_status(cudaError_t e, const char* what);
void clear_error();

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline int nseg_of(int d_in) { return (d_in + 127) / 128; }

}  // namespace bws
