// la_variants.cu -- CUDA-core kernels for three forms of the state recurrence
// beyond the plain one (fp32 arithmetic, fp32 or bf16 inputs):
//
//   normalised    o_t = phi(q_t)^T S_t / phi(q_t)^T z_t,  z_t = a_t z_{t-1} + phi(k_t)
//                 ("Linear / sparse attention tutorial" Q11 and section 2.2: z is
//                 the state of one extra value column of ones, so it decays with S)
//   channel gate  S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T, alpha_t in (0,1]^{d_k}
//                 ("Linear / sparse attention tutorial" Q21, GLA)
//   delta rule    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
//                 ("Linear / Sparse Attention - minimal runnable implementation",
//                 delta_rule_recurrent, with the state transposed to [d_k, d_v];
//                 "Linear / sparse attention tutorial" Q21 for the gate alpha_t)
//
// with o_t = phi(q_t)^T S_t (update before read) in all three.
//
// The first two are chunkwise, like the SIMT prefill kernel: per chunk of
// n <= C tokens the intra-chunk scores are formed exactly with their decay
// (every exponent is a difference Lam_i - Lam_j with i >= j, so it is <= 0 for
// log decays <= 0), the inter-chunk read uses the state of the previous chunk
// and the state is then advanced by the whole chunk.  The normalised form adds
// the denominator as the same two parts with v = 1: the decayed row sums of
// the scores plus e^{Lam_i} phi(q_i).z.  The channel gate has one cumulative
// log decay per key channel, so its score for (i, j) is
// sum_c q_ic k_jc e^{Lam_ic - Lam_jc}; once the scores are formed the decays
// are folded into q (e^{Lam_ic}) and k (e^{Lam_end,c - Lam_jc}) in place.
//
// The delta rule runs token by token: each step erases along k before it
// writes, and every column of S is independent of the others
// (S[:, c] <- a S[:, c] + k (beta (v_c - a k^T S[:, c]))), so a CTA owns 32
// value columns, a warp 4 of them, and a lane rows lane + 32 m of those
// columns in registers.  The two dot products of a step are warp reductions.
#include <cuda_bf16.h>

#include "../../include/la_gb300.h"
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunk = 64;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float log_decay_at(int kind, const float *__restrict__ decay, int h,
                                              size_t bhL, int t) {
  switch (kind) {
    case LA_DECAY_HEAD: return decay[h];
    case LA_DECAY_TOKEN: return decay[bhL + t];
    case LA_DECAY_GATE_LOGIT: return neg_softplus(decay[bhL + t]);
    default: return 0.f;
  }
}

// lam[i] = sum of the log decays of tokens s0 .. s0 + i (one warp, lanes 0..31).
__device__ __forceinline__ void chunk_log_prefix(float *lam, int n, int kind,
                                                 const float *__restrict__ decay, int h,
                                                 size_t bhL, int s0, int lane) {
  float carry = 0.f;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    float x = i < n ? log_decay_at(kind, decay, h, bhL, s0 + i) : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(kFull, x, off);
      if (lane >= off) x += y;
    }
    if (i < n) lam[i] = carry + x;
    carry += __shfl_sync(kFull, x, 31);
  }
}

// ---------------------------------------------------------------------------
// Normalised form.  One CTA per (b, h) holds the whole state S (d_k x d_v) and
// z (d_k) in shared memory, so S0/S_final and z0/z_final may alias.
template <typename T>
__global__ void __launch_bounds__(kThreads)
normalised_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                  int H, int L, int dk, int dv, int C, int phi, int decay_kind,
                  const float *__restrict__ decay, const float *S0, const float *z0,
                  T *__restrict__ O, float *S_final, float *z_final) {
  extern __shared__ float smem[];
  float *qs = smem;         // [C][dk]  phi(q)
  float *ks = qs + C * dk;  // [C][dk]  phi(k)
  float *vs = ks + C * dk;  // [C][dv]
  float *P = vs + C * dv;   // [C][C]   masked, decayed scores
  float *S = P + C * C;     // [dk][dv]
  float *z = S + dk * dv;   // [dk]
  float *lam = z + dk;      // [C]      inclusive log-decay prefix
  float *den = lam + C;     // [C]      denominators
  float *eq = den + C;      // [C]      e^{Lam_i}: weight of the inter-chunk read of row i
  float *ek = eq + C;       // [C]      e^{Lam_end - Lam_j}: weight of key j in the update

  const int tid = threadIdx.x;
  const int bh = blockIdx.x;
  const int h = bh % H;
  const size_t bhL = (size_t)bh * L;

  for (int x = tid; x < dk * dv; x += kThreads) S[x] = S0 ? S0[(size_t)bh * dk * dv + x] : 0.f;
  for (int r = tid; r < dk; r += kThreads) z[r] = z0 ? z0[(size_t)bh * dk + r] : 0.f;

  for (int s0 = 0; s0 < L; s0 += C) {
    const int n = min(C, L - s0);
    __syncthreads();  // the previous chunk's readers are done
    for (int x = tid; x < n * dk; x += kThreads) {
      qs[x] = feature_map_precise(phi, to_f32(q[(bhL + s0) * dk + x]));
      ks[x] = feature_map_precise(phi, to_f32(k[(bhL + s0) * dk + x]));
    }
    for (int x = tid; x < n * dv; x += kThreads) vs[x] = to_f32(v[(bhL + s0) * dv + x]);
    if (tid < 32) chunk_log_prefix(lam, n, decay_kind, decay, h, bhL, s0, tid);
    __syncthreads();
    for (int x = tid; x < n * n; x += kThreads) {
      const int i = x / n, j = x % n;
      float p = 0.f;
      if (j <= i) {
        float dot = 0.f;
        for (int c = 0; c < dk; ++c) dot = fmaf(qs[i * dk + c], ks[j * dk + c], dot);
        p = dot * expf(lam[i] - lam[j]);
      }
      P[i * C + j] = p;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {  // phi(q_i)^T z_i, in its two parts
      float inter = 0.f;
      for (int r = 0; r < dk; ++r) inter = fmaf(qs[i * dk + r], z[r], inter);
      float intra = 0.f;
      for (int j = 0; j <= i; ++j) intra += P[i * C + j];
      eq[i] = expf(lam[i]);
      ek[i] = expf(lam[n - 1] - lam[i]);
      den[i] = fmaf(eq[i], inter, intra);
    }
    __syncthreads();
    for (int x = tid; x < n * dv; x += kThreads) {
      const int i = x / dv, c = x % dv;
      float inter = 0.f;
      for (int r = 0; r < dk; ++r) inter = fmaf(qs[i * dk + r], S[r * dv + c], inter);
      float intra = 0.f;
      for (int j = 0; j <= i; ++j) intra = fmaf(P[i * C + j], vs[j * dv + c], intra);
      O[(bhL + s0 + i) * dv + c] = from_f32<T>(fmaf(eq[i], inter, intra) / den[i]);
    }
    __syncthreads();  // every read of S and z for this chunk's output is done
    const float eend = eq[n - 1];
    for (int x = tid; x < dk * dv; x += kThreads) {
      const int r = x / dv, c = x % dv;
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(ek[j] * ks[j * dk + r], vs[j * dv + c], acc);
      S[x] = fmaf(eend, S[x], acc);
    }
    for (int r = tid; r < dk; r += kThreads) {
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(ek[j], ks[j * dk + r], acc);
      z[r] = fmaf(eend, z[r], acc);
    }
  }
  __syncthreads();
  if (S_final)
    for (int x = tid; x < dk * dv; x += kThreads) S_final[(size_t)bh * dk * dv + x] = S[x];
  if (z_final)
    for (int r = tid; r < dk; r += kThreads) z_final[(size_t)bh * dk + r] = z[r];
}

// ---------------------------------------------------------------------------
// Per-channel gate.  One CTA per (b, h) and slice of dvt value columns, with
// its slice of S (d_k x dvt) in shared memory; log_alpha is [B,H,L,d_k].
template <typename T>
__global__ void __launch_bounds__(kThreads)
channel_gate_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    int L, int dk, int dv, int C, int dvt, int phi,
                    const float *__restrict__ log_alpha, const float *S0, T *__restrict__ O,
                    float *S_final) {
  extern __shared__ float smem[];
  float *qs = smem;          // [C][dk]  phi(q), then e^{Lam_i} phi(q_i)
  float *ks = qs + C * dk;   // [C][dk]  phi(k), then e^{Lam_end - Lam_j} phi(k_j)
  float *lam = ks + C * dk;  // [C][dk]  per-channel inclusive log-decay prefix
  float *vs = lam + C * dk;  // [C][dvt]
  float *P = vs + C * dvt;   // [C][C]
  float *S = P + C * C;      // [dk][dvt]

  const int tid = threadIdx.x;
  const int bh = blockIdx.x;
  const int j0 = blockIdx.y * dvt;
  const int nv = min(dvt, dv - j0);
  const size_t bhL = (size_t)bh * L;

  for (int x = tid; x < dk * nv; x += kThreads) {
    const int r = x / nv, c = x % nv;
    S[r * dvt + c] = S0 ? S0[((size_t)bh * dk + r) * dv + j0 + c] : 0.f;
  }

  for (int s0 = 0; s0 < L; s0 += C) {
    const int n = min(C, L - s0);
    __syncthreads();
    for (int x = tid; x < n * dk; x += kThreads) {
      qs[x] = feature_map_precise(phi, to_f32(q[(bhL + s0) * dk + x]));
      ks[x] = feature_map_precise(phi, to_f32(k[(bhL + s0) * dk + x]));
    }
    for (int x = tid; x < n * nv; x += kThreads) {
      const int t = x / nv, c = x % nv;
      vs[t * dvt + c] = to_f32(v[(bhL + s0 + t) * dv + j0 + c]);
    }
    for (int r = tid; r < dk; r += kThreads) {  // one channel per thread, in token order
      float acc = 0.f;
      for (int t = 0; t < n; ++t) {
        acc += log_alpha[(bhL + s0 + t) * dk + r];
        lam[t * dk + r] = acc;
      }
    }
    __syncthreads();
    for (int x = tid; x < n * n; x += kThreads) {
      const int i = x / n, j = x % n;
      float p = 0.f;
      if (j <= i)
        for (int c = 0; c < dk; ++c)
          p = fmaf(qs[i * dk + c] * ks[j * dk + c], expf(lam[i * dk + c] - lam[j * dk + c]), p);
      P[i * C + j] = p;
    }
    __syncthreads();
    for (int x = tid; x < n * dk; x += kThreads) {  // fold the decays into q and k
      const int r = x % dk;
      qs[x] *= expf(lam[x]);
      ks[x] *= expf(lam[(n - 1) * dk + r] - lam[x]);
    }
    __syncthreads();
    for (int x = tid; x < n * nv; x += kThreads) {
      const int i = x / nv, c = x % nv;
      float acc = 0.f;
      for (int r = 0; r < dk; ++r) acc = fmaf(qs[i * dk + r], S[r * dvt + c], acc);
      for (int j = 0; j <= i; ++j) acc = fmaf(P[i * C + j], vs[j * dvt + c], acc);
      O[(bhL + s0 + i) * dv + j0 + c] = from_f32<T>(acc);
    }
    __syncthreads();
    for (int x = tid; x < dk * nv; x += kThreads) {
      const int r = x / nv, c = x % nv;
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(ks[j * dk + r], vs[j * dvt + c], acc);
      S[r * dvt + c] = fmaf(expf(lam[(n - 1) * dk + r]), S[r * dvt + c], acc);
    }
  }
  __syncthreads();
  if (S_final) {
    for (int x = tid; x < dk * nv; x += kThreads) {
      const int r = x / nv, c = x % nv;
      S_final[((size_t)bh * dk + r) * dv + j0 + c] = S[r * dvt + c];
    }
  }
}

// ---------------------------------------------------------------------------
// Delta rule, token by token.  CTA (b, h, slice of 32 value columns); warp w
// owns slice columns 4w .. 4w+3; lane l owns rows l + 32 m.  Tokens are staged
// through shared memory kTok at a time.
constexpr int kTok = 32;
constexpr int kDeltaCols = 32;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
  return x;
}

template <typename T, int DK>
__global__ void __launch_bounds__(kThreads)
delta_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, int L,
             int dv, int phi, const float *__restrict__ beta, const float *__restrict__ log_alpha,
             const float *S0, T *__restrict__ O, float *S_final) {
  constexpr int MR = (DK + 31) / 32;  // rows per lane
  __shared__ float qf[kTok][DK], kf[kTok][DK], vv[kTok][kDeltaCols], bt[kTok], at[kTok];

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int bh = blockIdx.x;
  const int j0 = blockIdx.y * kDeltaCols;
  const int nv = min(kDeltaCols, dv - j0);
  const int cb = warp * 4;  // first slice column of this warp
  const size_t bhL = (size_t)bh * L;

  float s[MR][4];
#pragma unroll
  for (int m = 0; m < MR; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int r = lane + 32 * m;
      s[m][c] = (S0 && r < DK && cb + c < nv) ? S0[((size_t)bh * DK + r) * dv + j0 + cb + c]
                                              : 0.f;
    }

  for (int t0 = 0; t0 < L; t0 += kTok) {
    const int nt = min(kTok, L - t0);
    __syncthreads();  // every warp is done with the previous tokens
    for (int x = tid; x < nt * DK; x += kThreads) {
      qf[x / DK][x % DK] = feature_map_precise(phi, to_f32(q[(bhL + t0) * DK + x]));
      kf[x / DK][x % DK] = feature_map_precise(phi, to_f32(k[(bhL + t0) * DK + x]));
    }
    for (int x = tid; x < nt * kDeltaCols; x += kThreads) {
      const int t = x / kDeltaCols, c = x % kDeltaCols;
      vv[t][c] = c < nv ? to_f32(v[(bhL + t0 + t) * dv + j0 + c]) : 0.f;
    }
    for (int t = tid; t < nt; t += kThreads) {
      bt[t] = beta[bhL + t0 + t];
      at[t] = log_alpha ? expf(log_alpha[bhL + t0 + t]) : 1.f;
    }
    __syncthreads();
    for (int t = 0; t < nt; ++t) {
      float kr[MR], qr[MR];
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        const int r = lane + 32 * m;
        kr[m] = r < DK ? kf[t][r] : 0.f;
        qr[m] = r < DK ? qf[t][r] : 0.f;
      }
      const float a = at[t], b = bt[t];
      float o[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float u = 0.f;  // (k^T S)_c
#pragma unroll
        for (int m = 0; m < MR; ++m) u = fmaf(kr[m], s[m][c], u);
        u = warp_sum(u);
        const float w = b * (vv[t][cb + c] - a * u);  // what is written along k
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          s[m][c] = fmaf(kr[m], w, a * s[m][c]);
          acc = fmaf(qr[m], s[m][c], acc);
        }
        o[c] = warp_sum(acc);
      }
      if (lane < 4 && cb + lane < nv) {
        const float mine = lane == 0 ? o[0] : lane == 1 ? o[1] : lane == 2 ? o[2] : o[3];
        O[(bhL + t0 + t) * dv + j0 + cb + lane] = from_f32<T>(mine);
      }
    }
  }
  if (S_final) {
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int r = lane + 32 * m;
        if (r < DK && cb + c < nv) S_final[((size_t)bh * DK + r) * dv + j0 + cb + c] = s[m][c];
      }
  }
}

template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t smem) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <typename T>
cudaError_t launch_normalised_t(const VariantArgs &a) {
  const int C = a.chunk;
  const size_t smem = sizeof(float) * ((size_t)2 * C * a.dk + (size_t)C * a.dv + (size_t)C * C +
                                       (size_t)a.dk * a.dv + a.dk + 4 * C);
  auto kern = normalised_kernel<T>;
  cudaError_t e = allow_smem(kern, smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(a.B * a.H), kThreads, smem, a.stream>>>(
      static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v),
      a.H, a.L, a.dk, a.dv, C, a.phi, a.decay_kind, a.decay, a.S0, a.z0, static_cast<T *>(a.O),
      a.S_final, a.z_final);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_channel_gate_t(const VariantArgs &a) {
  const int C = a.chunk;
  const int dvt = a.dv < 32 ? a.dv : 32;
  const size_t smem = sizeof(float) * ((size_t)3 * C * a.dk + (size_t)C * dvt + (size_t)C * C +
                                       (size_t)a.dk * dvt);
  auto kern = channel_gate_kernel<T>;
  cudaError_t e = allow_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(a.B * a.H), (unsigned)((a.dv + dvt - 1) / dvt));
  kern<<<grid, kThreads, smem, a.stream>>>(
      static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v),
      a.L, a.dk, a.dv, C, dvt, a.phi, a.decay, a.S0, static_cast<T *>(a.O), a.S_final);
  return cudaGetLastError();
}

template <typename T, int DK>
cudaError_t launch_delta_d(const VariantArgs &a) {
  dim3 grid((unsigned)(a.B * a.H), (unsigned)((a.dv + kDeltaCols - 1) / kDeltaCols));
  delta_kernel<T, DK><<<grid, kThreads, 0, a.stream>>>(
      static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v),
      a.L, a.dv, a.phi, a.beta, a.decay, a.S0, static_cast<T *>(a.O), a.S_final);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_delta_t(const VariantArgs &a) {
  switch (a.dk) {
    case 16: return launch_delta_d<T, 16>(a);
    case 32: return launch_delta_d<T, 32>(a);
    case 64: return launch_delta_d<T, 64>(a);
    case 128: return launch_delta_d<T, 128>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_variant(const VariantArgs &a) {
  if (a.dk > 128 || a.dv > 128 || a.dk <= 0 || a.dv <= 0) return cudaErrorInvalidValue;
  if (a.form != VARIANT_DELTA && (a.chunk < 1 || a.chunk > kMaxChunk))
    return cudaErrorInvalidValue;
  const bool f32 = a.dtype == LA_F32;
  switch (a.form) {
    case VARIANT_NORMALISED:
      return f32 ? launch_normalised_t<float>(a) : launch_normalised_t<__nv_bfloat16>(a);
    case VARIANT_CHANNEL_GATE:
      return f32 ? launch_channel_gate_t<float>(a) : launch_channel_gate_t<__nv_bfloat16>(a);
    case VARIANT_DELTA:
      return f32 ? launch_delta_t<float>(a) : launch_delta_t<__nv_bfloat16>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace la
