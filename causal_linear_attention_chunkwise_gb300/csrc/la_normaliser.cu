// la_normaliser.cu -- the denominator of normalised linear attention and the
// division by it, after the numerator phi(q_t)^T S_t has been written to O by
// the prefill kernels ("Linear / sparse attention tutorial" Q11 and section
// 2.2):
//
//     z_t = a_t z_{t-1} + phi(k_t),   den_t = phi(q_t)^T z_t,   o_t <- o_t / den_t
//
// z is a d_k-vector per sequence, so this is a scan of O(d_k) work per token
// (against O(d_k d_v) for the numerator).  A sequence is cut into blocks of
// kBlock tokens, and two kernels run over (block, sequence):
//   1. block totals: with zeta = 0 at the block start, zeta <- a_t zeta + phi(k_t)
//      over the block gives its contribution to z at the block end, and the
//      sum of its log decays gives the factor e^{A_m} that the block applies to
//      the z coming into it.  Block 0 also copies z0 into the workspace, so
//      that z_final may overwrite z0.
//   2. apply: each block folds the totals of the blocks before it into its
//      incoming z (z <- e^{A_i} z + zeta_i, from z0), walks its tokens again to
//      form every den_t, and divides its rows of O in place.  The last block
//      writes z_final.
// One thread per key channel carries z; tokens are staged through shared
// memory kTok at a time, and four threads per token sum phi(q_t) .* z_t over the
// channels.  The grid is (sequence, block).
#include <cuda_bf16.h>
#include <cstdint>
#include <cstring>

#include "../../include/la_gb300.h"
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kBlock = 256;  // tokens per block
constexpr int kTok = 32;     // tokens staged at a time
constexpr int kThreadsN = 128;
constexpr int kMaxDk = 128;

// Elements of T in one 16-byte vector, unpacked to fp32 and packed back.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4 &u, float *f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 pack(const float *f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b;
      memcpy(&b, &w[i], 4);
      const float2 x = __bfloat1622float2(b);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
  __device__ static uint4 pack(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      memcpy(&w[i], &b, 4);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Stage rows [row0, row0 + nt) of a [*, dk] tensor into dst[t * dkp + c] as
// phi(x) in fp32, with every 16-byte load of the pass issued before any use
// and 16-byte shared stores (dst and dkp are multiples of 4 floats).
// phi uses the fast exponential: its relative error (a few 1e-7) stays far
// below the fp32 tolerance of 1e-5, and the precise one made staging the
// larger part of the kernels' instructions.
// Rows start on 16-byte boundaries: the tensor does, and dk * sizeof(T) is a
// multiple of 16 for every supported d_k (a power of two, 16 .. 128).
template <typename T>
__device__ __forceinline__ void stage_rows(const T *__restrict__ src, size_t row0, int nt, int dk,
                                           int dkp, int phi, float *dst, int tid) {
  using V = Vec16<T>;
  constexpr int kMaxVec = kTok * kMaxDk / V::N / kThreadsN;  // per thread, at most
  const int nvec = nt * dk / V::N;
  const int sh = __ffs(dk) - 1;  // dk = 2^sh
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src + row0 * dk);
  uint4 buf[kMaxVec];
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int vi = tid + i * kThreadsN;
    if (vi < nvec) buf[i] = s4[vi];
  }
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int vi = tid + i * kThreadsN;
    if (vi < nvec) {
      float f[V::N];
      V::unpack(buf[i], f);
      const int e = vi * V::N;  // a vector never spans two rows
      float *d = dst + (e >> sh) * dkp + (e & (dk - 1));
#pragma unroll
      for (int u = 0; u < V::N; u += 4)
        *reinterpret_cast<float4 *>(d + u) =
            make_float4(feature_map(phi, f[u]), feature_map(phi, f[u + 1]),
                        feature_map(phi, f[u + 2]), feature_map(phi, f[u + 3]));
    }
  }
}

__device__ __forceinline__ float log_decay_of(int kind, const float *__restrict__ decay, int h,
                                              size_t bhL, int t) {
  switch (kind) {
    case LA_DECAY_HEAD: return decay[h];
    case LA_DECAY_TOKEN: return decay[bhL + t];
    case LA_DECAY_GATE_LOGIT: return neg_softplus(decay[bhL + t]);
    default: return 0.f;
  }
}

// Workspace layout (floats): totals [BH][nblk][dk], block log decays
// [BH][nblk], incoming z0 [BH][dk].
struct NormWs {
  float *tot, *logA, *z0;
};

__host__ __device__ inline NormWs norm_ws(void *base, size_t bh, int nblk, int dk) {
  float *f = static_cast<float *>(base);
  NormWs w;
  w.tot = f;
  w.logA = f + bh * nblk * dk;
  w.z0 = w.logA + bh * nblk;
  return w;
}

template <typename T>
__global__ void __launch_bounds__(kThreadsN, 4)
norm_block_totals_kernel(const T *__restrict__ k, int H, int L, int dk, int nblk, int phi,
                         int decay_kind, const float *__restrict__ decay,
                         const float *__restrict__ z0, void *ws) {
  __shared__ __align__(16) float kf[kTok][kMaxDk + 4];  // phi(k) of the staged tokens
  __shared__ float el[kTok];              // e^{lambda_t}
  __shared__ float ll[kTok];              // lambda_t
  const int tid = threadIdx.x;
  const int bh = blockIdx.x, m = blockIdx.y, h = bh % H;
  const size_t bhL = (size_t)bh * L;
  const int tb = m * kBlock;
  const int nb = min(kBlock, L - tb);
  const NormWs w = norm_ws(ws, (size_t)gridDim.x, nblk, dk);

  float zeta = 0.f;  // channel tid's total over the tokens so far
  float lsum = 0.f;  // sum of the log decays (thread 0)
  for (int t0 = 0; t0 < nb; t0 += kTok) {
    const int nt = min(kTok, nb - t0);
    const size_t row0 = bhL + tb + t0;
    __syncthreads();  // the previous pass is done with the staging buffers
    stage_rows(k, row0, nt, dk, kMaxDk + 4, phi, &kf[0][0], tid);
    for (int t = tid; t < nt; t += kThreadsN) {
      ll[t] = log_decay_of(decay_kind, decay, h, bhL, tb + t0 + t);
      el[t] = expf(ll[t]);
    }
    __syncthreads();
    if (tid < dk)
      for (int t = 0; t < nt; ++t) zeta = fmaf(el[t], zeta, kf[t][tid]);
    if (tid == 0)
      for (int t = 0; t < nt; ++t) lsum += ll[t];
  }
  if (tid < dk) {
    w.tot[((size_t)bh * nblk + m) * dk + tid] = zeta;
    if (m == 0) w.z0[(size_t)bh * dk + tid] = z0 ? z0[(size_t)bh * dk + tid] : 0.f;
  }
  if (tid == 0) w.logA[(size_t)bh * nblk + m] = lsum;
}

template <typename T>
__global__ void __launch_bounds__(kThreadsN, 4)
norm_apply_kernel(const T *__restrict__ q, const T *__restrict__ k, int H, int L, int dk,
                  int dv, int nblk, int phi, int decay_kind, const float *__restrict__ decay,
                  const void *ws, T *O, float *z_final) {
  extern __shared__ float sm[];
  // Rows padded to dk + 4 floats: 16-byte stores when staging, and the four
  // threads of a token in the den sum (rows t, t + 1, ...) land in distinct banks.
  const int dkp = dk + 4;
  float *qf = sm;                // [kTok][dkp]  phi(q)
  float *kf = qf + kTok * dkp;   // [kTok][dkp]  phi(k)
  float *pr = kf + kTok * dkp;   // [kTok][dkp]  phi(q) .* z
  float *el = pr + kTok * dkp;   // [kTok]       e^{lambda_t}
  float *den = el + kTok;        // [kTok]       1 / den_t
  float *ea = den + kTok;        // [kThreadsN]  e^{A_i} of earlier blocks, in groups

  const int tid = threadIdx.x;
  const int bh = blockIdx.x, m = blockIdx.y, h = bh % H;
  const size_t bhL = (size_t)bh * L;
  const int tb = m * kBlock;
  const int nb = min(kBlock, L - tb);
  const NormWs w = norm_ws(const_cast<void *>(ws), (size_t)gridDim.x, nblk, dk);

  float z = tid < dk ? w.z0[(size_t)bh * dk + tid] : 0.f;  // z coming into this block
  for (int i0 = 0; i0 < m; i0 += kThreadsN) {  // fold the earlier blocks, in groups
    const int ni = min(kThreadsN, m - i0);
    __syncthreads();
    if (tid < ni) ea[tid] = expf(w.logA[(size_t)bh * nblk + i0 + tid]);
    __syncthreads();
    if (tid < dk) {
      const float *tot = w.tot + ((size_t)bh * nblk + i0) * dk + tid;
#pragma unroll 8
      for (int i = 0; i < ni; ++i) z = fmaf(ea[i], z, tot[(size_t)i * dk]);
    }
  }
  for (int t0 = 0; t0 < nb; t0 += kTok) {
    const int nt = min(kTok, nb - t0);
    const size_t row0 = bhL + tb + t0;  // first token of this pass
    __syncthreads();  // the previous pass is done with the staging buffers
    stage_rows(q, row0, nt, dk, dkp, phi, qf, tid);
    stage_rows(k, row0, nt, dk, dkp, phi, kf, tid);
    for (int t = tid; t < nt; t += kThreadsN)
      el[t] = expf(log_decay_of(decay_kind, decay, h, bhL, tb + t0 + t));
    __syncthreads();
    if (tid < dk) {
      for (int t = 0; t < nt; ++t) {
        z = fmaf(el[t], z, kf[t * dkp + tid]);
        pr[t * dkp + tid] = qf[t * dkp + tid] * z;
      }
    }
    __syncthreads();
    {  // den_t: four threads per token, each a quarter of the channels
      const int t = tid >> 2, part = tid & 3;
      float s = 0.f;
      if (t < nt)
        for (int c = part; c < dk; c += 4) s += pr[t * dkp + c];
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (t < nt && part == 0) den[t] = 1.f / s;  // one division per token
    }
    __syncthreads();
    {  // o_t <- o_t / den_t, in 16-byte vectors (rows of d_v elements start aligned)
      using V = Vec16<T>;
      uint4 *o4 = reinterpret_cast<uint4 *>(O + row0 * dv);
      const int shv = __ffs(dv) - 1;  // dv = 2^shv
      for (int vi = tid; vi < nt * dv / V::N; vi += kThreadsN) {
        float f[V::N];
        V::unpack(o4[vi], f);
        const float r = den[(vi * V::N) >> shv];  // 1 / den_t; a vector never spans two rows
#pragma unroll
        for (int u = 0; u < V::N; ++u) f[u] *= r;
        o4[vi] = V::pack(f);
      }
    }
  }
  if (z_final && m == nblk - 1 && tid < dk) z_final[(size_t)bh * dk + tid] = z;
}

}  // namespace

size_t normaliser_workspace_bytes(int B, int H, int L, int dk) {
  if (B <= 0 || H <= 0 || L <= 0) return 0;
  const size_t bh = (size_t)B * H;
  const size_t nblk = (size_t)(L + kBlock - 1) / kBlock;
  return sizeof(float) * (bh * nblk * dk + bh * nblk + bh * dk);
}

cudaError_t launch_normaliser(const NormaliserArgs &a) {
  if (a.dk <= 0 || a.dk > kThreadsN || a.L <= 0) return cudaErrorInvalidValue;
  const int nblk = (a.L + kBlock - 1) / kBlock;
  const unsigned bh = (unsigned)((size_t)a.B * a.H);
  dim3 grid(bh, (unsigned)nblk);
  const size_t smem = sizeof(float) * ((size_t)3 * kTok * (a.dk + 4) + 2 * kTok + kThreadsN);
  cudaError_t e = cudaFuncSetAttribute(norm_apply_kernel<float>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(norm_apply_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.dtype == LA_F32) {
    norm_block_totals_kernel<float><<<grid, kThreadsN, 0, a.stream>>>(
        static_cast<const float *>(a.k), a.H, a.L, a.dk, nblk, a.phi, a.decay_kind, a.decay,
        a.z0, a.workspace);
    norm_apply_kernel<float><<<grid, kThreadsN, smem, a.stream>>>(
        static_cast<const float *>(a.q), static_cast<const float *>(a.k), a.H, a.L, a.dk, a.dv,
        nblk, a.phi, a.decay_kind, a.decay, a.workspace, static_cast<float *>(a.O), a.z_final);
  } else {
    norm_block_totals_kernel<__nv_bfloat16><<<grid, kThreadsN, 0, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.k), a.H, a.L, a.dk, nblk, a.phi, a.decay_kind,
        a.decay, a.z0, a.workspace);
    norm_apply_kernel<__nv_bfloat16><<<grid, kThreadsN, smem, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k), a.H,
        a.L, a.dk, a.dv, nblk, a.phi, a.decay_kind, a.decay, a.workspace,
        static_cast<__nv_bfloat16 *>(a.O), a.z_final);
  }
  return cudaGetLastError();
}

}  // namespace la
