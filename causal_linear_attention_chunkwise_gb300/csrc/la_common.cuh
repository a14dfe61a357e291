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
  KID_CHANNEL_GATE_TC = 5,
  KID_DELTA_TC = 6,
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

// 16 bytes of T, unpacked to fp32.
template <typename T> struct Pack16;
template <> struct Pack16<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4 &u, float *f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};
template <> struct Pack16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4 &u, float *f) {
    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(b[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
};

// Copy nrows rows of `width` elements (row r at src + r * src_stride) to
// dst[r * dst_stride + c] as op(x) in fp32, in 16-byte vectors.  Every load a
// thread makes is issued before its first store, so the rows arrive in one
// memory round trip rather than one per loop iteration.  Needs: src 16-byte
// aligned; width a power of two, and width and src_stride multiples of
// 16 bytes / sizeof(T); nrows * width / Pack16<T>::N <= MAXV * nthreads.
template <typename T, int MAXV, typename Op>
__device__ __forceinline__ void stage_slab(const T *__restrict__ src, size_t src_stride,
                                           int nrows, int width, float *dst, int dst_stride,
                                           Op op, int tid, int nthreads) {
  using P = Pack16<T>;
  const int vpr = width / P::N;  // vectors per row, a power of two
  const int shv = __ffs(vpr) - 1;
  const int nvec = nrows * vpr;
  uint4 buf[MAXV];
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int vi = tid + i * nthreads;
    if (vi < nvec)
      buf[i] = *reinterpret_cast<const uint4 *>(src + (size_t)(vi >> shv) * src_stride +
                                                (vi & (vpr - 1)) * P::N);
  }
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int vi = tid + i * nthreads;
    if (vi < nvec) {
      float f[P::N];
      P::unpack(buf[i], f);
      float *d = dst + (vi >> shv) * dst_stride + (vi & (vpr - 1)) * P::N;
#pragma unroll
      for (int u = 0; u < P::N; ++u) d[u] = op(f[u]);
    }
  }
}

}  // namespace la

// Opt-in event trace for kernel development.  Built with -DLA_TRACE, kernels
// record clock64() stamps of pipeline events for one chosen CTA (relative to
// the CTA's start) into a shared-memory table [event][chunk], which the CTA
// copies to global memory as it exits: a global store per event would hold up
// the next barrier its thread reaches (a barrier waits for the participating
// threads' earlier memory accesses), and so distort the timeline it records.
// Otherwise every trace macro compiles to nothing and the table takes no room.
// A kernel short of shared memory keeps fewer chunks (kTraceChunks / shrink).
namespace la {
constexpr int kTraceEvents = 16, kTraceChunks = 64;
#ifdef LA_TRACE
constexpr uint32_t trace_smem_bytes(int shrink = 1) {
  return kTraceEvents * (kTraceChunks / shrink) * 4;
}
#else
constexpr uint32_t trace_smem_bytes(int = 1) { return 0; }
#endif
}  // namespace la
#ifdef LA_TRACE
// Declares the kernel's table of kTraceChunks / shrink chunks at smem_ptr and
// clears it (before a block barrier).
#define LA_TRACE_TABLE(smem_ptr, shrink)                                           \
  constexpr int la_trc_n = ::la::kTraceChunks / (shrink);                          \
  uint32_t *la_trc = reinterpret_cast<uint32_t *>(smem_ptr);                       \
  for (int i_ = threadIdx.x; i_ < ::la::kTraceEvents * la_trc_n; i_ += blockDim.x) \
    la_trc[i_] = 0u
#define LA_TRACE_EVENT(on, t0, ev, c)                                              \
  do {                                                                             \
    if ((on) && (c) < la_trc_n)                                                    \
      la_trc[(ev) * la_trc_n + (c)] = (uint32_t)(clock64() - (t0));                \
  } while (0)
// Copies the table to long long dst[kTraceEvents][kTraceChunks] (after a block
// barrier); chunks past the table's stay as they were.
#define LA_TRACE_FLUSH(on, dst)                                                    \
  do {                                                                             \
    if (on)                                                                        \
      for (int i_ = threadIdx.x; i_ < ::la::kTraceEvents * la_trc_n; i_ += blockDim.x) \
        (dst)[(i_ / la_trc_n) * ::la::kTraceChunks + i_ % la_trc_n] = (long long)la_trc[i_]; \
  } while (0)
#else
#define LA_TRACE_TABLE(smem_ptr, shrink) \
  do {                                   \
  } while (0)
#define LA_TRACE_EVENT(on, t0, ev, c) \
  do {                                \
  } while (0)
#define LA_TRACE_FLUSH(on, dst) \
  do {                          \
  } while (0)
#endif
