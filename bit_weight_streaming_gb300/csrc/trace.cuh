// Opt-in timestamp trace (measurement aid, compiled in only with -DBWS_TRACE):
// kernels append one record per CTA with global-timer readings at the points
// they choose; bws_trace_read_<unit>() copies a translation unit's records to
// the host and clears them. Without BWS_TRACE nothing here is compiled.
#pragma once
#ifdef BWS_TRACE
#include <cuda_runtime.h>

#include <cstdint>

namespace bws {

constexpr unsigned kTraceCap = 1u << 17;   // records per translation unit

struct TraceRec {
  unsigned long long kind;   // kernel kind and variant
  unsigned long long cta;    // blockIdx.x | smid << 32
  unsigned long long t[6];   // global-timer readings (ns)
};

static __device__ TraceRec g_trace[kTraceCap];
static __device__ unsigned int g_trace_n;

__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void trace_put(unsigned kind, const unsigned long long (&t)[6]) {
  const unsigned i = atomicAdd(&g_trace_n, 1u);
  if (i >= kTraceCap) return;
  unsigned s;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
  TraceRec& r = g_trace[i];
  r.kind = kind;
  r.cta = blockIdx.x | ((unsigned long long)s << 32);
#pragma unroll
  for (int k = 0; k < 6; ++k) r.t[k] = t[k];
}

// Host: copies up to cap records into host memory and clears the trace;
// returns the number copied (-1 on a CUDA error).
static inline int trace_read(void* host, int cap) {
  unsigned n = 0;
  if (cudaMemcpyFromSymbol(&n, g_trace_n, sizeof(n)) != cudaSuccess) return -1;
  if (n > kTraceCap) n = kTraceCap;
  if ((int)n > cap) n = (unsigned)cap;
  if (n && cudaMemcpyFromSymbol(host, g_trace, n * sizeof(TraceRec)) != cudaSuccess) return -1;
  const unsigned z = 0;
  if (cudaMemcpyToSymbol(g_trace_n, &z, sizeof(z)) != cudaSuccess) return -1;
  return (int)n;
}

}  // namespace bws
#endif
