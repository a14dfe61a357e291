// la_decode.cu -- one recurrent decode step over B*H fp32 states, in place.
//
//     S <- alpha S + phi(k) v^T ;  o = phi(q)^T S        (update, then read)
//
// ("CS336 lecture 4, code 1: linear attention", gated_linear_attention_recurrent;
// "adv13 - Linear Attention / SSM" section 3.2; "Linear / sparse attention
// tutorial" section 8.1: a decode step touches only the fixed-size state.)
//
// The step is a pure stream over the states: 4 * d_k * d_v bytes read and the
// same written per (b, h), a few flops per element.  One CTA per (b, h) with
// DV / 16 warps; warp w owns value columns [16w, 16w + 16).  Lane l owns the
// float4 column group (l & 3) and rows (l >> 2) + 8m, so each warp load covers
// eight 64-byte row segments (full 32-byte sectors).  All of a thread's state
// loads are issued before any use, with streaming cache hints since a state is
// touched once per step.  The reduction o_j = sum_i phi(q_i) S_ij runs over
// the lanes that share a column group, with warp shuffles (xor 4, 8, 16).
#include <cuda_bf16.h>

#include "../../include/la_gb300.h"
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(DV * 2)
decode_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              int phi, const float *__restrict__ log_alpha, float *__restrict__ S,
              T *__restrict__ o) {
  static_assert(DV % 16 == 0 && DK % 8 == 0, "tile shape");
  constexpr int RPL = DK / 8;  // rows per lane
  __shared__ float qf[DK], kf[DK], vv[DV];
  const size_t bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int col = warp * 16 + (lane & 3) * 4;
  const int r0 = lane >> 2;

  float4 *Sb = reinterpret_cast<float4 *>(S + bh * DK * DV);
  float4 s[RPL];
#pragma unroll
  for (int m = 0; m < RPL; ++m) s[m] = __ldcs(&Sb[((r0 + 8 * m) * DV + col) >> 2]);

  for (int i = tid; i < DK; i += DV * 2) {
    qf[i] = feature_map(phi, to_f32(q[bh * DK + i]));
    kf[i] = feature_map(phi, to_f32(k[bh * DK + i]));
  }
  for (int i = tid; i < DV; i += DV * 2) vv[i] = to_f32(v[bh * DV + i]);
  const float a = log_alpha ? __expf(log_alpha[bh]) : 1.f;
  __syncthreads();

  const float4 vj = make_float4(vv[col], vv[col + 1], vv[col + 2], vv[col + 3]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int m = 0; m < RPL; ++m) {
    const int r = r0 + 8 * m;
    const float kr = kf[r], qr = qf[r];
    float4 x = s[m];
    x.x = fmaf(kr, vj.x, a * x.x);
    x.y = fmaf(kr, vj.y, a * x.y);
    x.z = fmaf(kr, vj.z, a * x.z);
    x.w = fmaf(kr, vj.w, a * x.w);
    __stcs(&Sb[(r * DV + col) >> 2], x);
    acc.x = fmaf(qr, x.x, acc.x);
    acc.y = fmaf(qr, x.y, acc.y);
    acc.z = fmaf(qr, x.z, acc.z);
    acc.w = fmaf(qr, x.w, acc.w);
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
  }
  if (r0 == 0) {
    T *ob = o + bh * DV + col;
    ob[0] = from_f32<T>(acc.x);
    ob[1] = from_f32<T>(acc.y);
    ob[2] = from_f32<T>(acc.z);
    ob[3] = from_f32<T>(acc.w);
  }
}

template <typename T, int D>
cudaError_t launch_d(const DecodeArgs &a) {
  const unsigned grid = (unsigned)((size_t)a.B * a.H);
  decode_kernel<T, D, D><<<grid, D * 2, 0, a.stream>>>(
      static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v),
      a.phi, a.log_alpha, a.S, static_cast<T *>(a.o));
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const DecodeArgs &a) {
  switch (a.dk) {
    case 16: return launch_d<T, 16>(a);
    case 32: return launch_d<T, 32>(a);
    case 64: return launch_d<T, 64>(a);
    case 128: return launch_d<T, 128>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_supported(int dk, int dv) {
  return dk == dv && (dk == 16 || dk == 32 || dk == 64 || dk == 128);
}

cudaError_t launch_decode(const DecodeArgs &a) {
  if (!decode_supported(a.dk, a.dv)) return cudaErrorInvalidValue;
  if (a.dtype == LA_F32) return launch_t<float>(a);
  return launch_t<__nv_bfloat16>(a);
}

}  // namespace la
