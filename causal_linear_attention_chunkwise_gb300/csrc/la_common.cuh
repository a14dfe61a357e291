// la_common.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace la {

// Kernel ids and wait sites recorded in the device error word.
enum : unsigned int {
  KID_PREFILL_TC_STATE = 1,
  KID_PREFILL_TC_OUT = 2,
  KID_SELFTEST = 3,
  KID_NONCAUSAL = 4,
};

__device__ __forceinline__ void record_device_error(unsigned int *word, unsigned int kernel,
                                                    unsigned int site) {
  if (word) atomicCAS(word, 0u, (kernel & 0xffu) | ((site & 0xffu) << 8) | 0x10000u);
}

// phi: 0 identity, 1 elu(x) + 1 (alpha = 1): x + 1 for x > 0, exp(x) otherwise.
__device__ __forceinline__ float feature_map(int phi, float x) {
  if (phi == 1) return x > 0.f ? x + 1.f : __expf(x);
  return x;
}

// Precise variant for the fp32 path (expf keeps the fp32 error well inside 1e-5).
__device__ __forceinline__ float feature_map_precise(int phi, float x) {
  if (phi == 1) return x > 0.f ? x + 1.f : expf(x);
  return x;
}

// log(alpha) = -softplus(g) = -(max(g, 0) + log1p(exp(-|g|))), overflow-free.
__device__ __forceinline__ float neg_softplus(float g) {
  return -(fmaxf(g, 0.f) + log1pf(expf(-fabsf(g))));
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

}  // namespace la

// Opt-in event trace for kernel development.  Built with -DLA_TRACE, kernels
// record clock64() stamps of pipeline events for one chosen CTA into
// la::g_trace[event][chunk] (relative to the CTA's start), which the using
// translation unit defines; otherwise every LA_TRACE_EVENT compiles to nothing.
namespace la {
constexpr int kTraceEvents = 16, kTraceChunks = 64;
}  // namespace la
#ifdef LA_TRACE
#define LA_TRACE_EVENT(on, t0, ev, c)                                          \
  do {                                                                         \
    if ((on) && (c) < ::la::kTraceChunks)                                      \
      ::la::g_trace[(ev)][(c)] = clock64() - (t0);                             \
  } while (0)
#else
#define LA_TRACE_EVENT(on, t0, ev, c) \
  do {                                \
  } while (0)
#endif
