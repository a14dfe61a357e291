// la_prefill_simt.cu -- chunkwise causal linear attention on the CUDA cores.
//
// The fp32 path (inputs and arithmetic in fp32; the tensor cores' tf32 would
// not meet a 1e-5 relative error) and the general path for shapes the
// tensor-core kernels do not take (any 1 <= C <= 64, d <= 128).
//
// One CTA owns one (b, h) sequence and a slice of DVT value columns; it walks
// the chunks in order with its slice of S (d_k x DVT, fp32) in shared memory.
// Per chunk of n <= C tokens ("Linear / Sparse Attention - minimal runnable
// implementation", linear_attn_chunkwise; gate factors as in the "Linear /
// sparse attention tutorial" section 6.2, expanded over one chunk):
//   Lam_i = sum of the chunk's log decays up to token i (inclusive)
//   P_ij  = exp(Lam_i - Lam_j) phi(q_i).phi(k_j)  for j <= i, else 0
//   O_i   = sum_j P_ij v_j + exp(Lam_i) phi(q_i)^T S
//   S    <- exp(Lam_{n-1}) S + sum_j exp(Lam_{n-1} - Lam_j) phi(k_j) v_j^T
// Exponents are differences with i >= j, so they are <= 0 and cannot overflow.
#include <cuda_bf16.h>

#include "../../include/la_gb300.h"
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunk = 64;

__device__ __forceinline__ float token_log_decay(int kind, const float *__restrict__ decay,
                                                 int h, size_t bhL, int t) {
  switch (kind) {
    case LA_DECAY_HEAD: return decay[h];
    case LA_DECAY_TOKEN: return decay[bhL + t];
    case LA_DECAY_GATE_LOGIT: return neg_softplus(decay[bhL + t]);
    default: return 0.f;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
prefill_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    int H, int L, int dk, int dv, int C, int dvt, int phi, int decay_kind,
                    const float *__restrict__ decay, const float *S0, T *__restrict__ O,
                    float *S_final) {
  extern __shared__ float smem[];
  // q and k rows are padded to dk + 1 floats: the score loop reads one k row
  // per lane, and an unpadded stride of dk (a multiple of 16) would put all
  // of a warp's reads in one or two shared-memory banks.
  const int dkp = dk + 1;
  float *qs = smem;                   // [C][dkp]  phi(q) of the chunk
  float *ks = qs + C * dkp;           // [C][dkp]  phi(k)
  float *vs = ks + C * dkp;           // [C][dvt]  value slice
  float *P = vs + C * dvt;            // [C][C]    masked, decayed scores
  float *S = P + C * C;               // [dk][dvt] state slice
  float *lam = S + dk * dvt;          // [C]       inclusive log-decay prefix
  float *eq = lam + C;                // [C]       e^{Lam_i}, weight of row i's inter read
  float *ek = eq + C;                 // [C]       e^{Lam_end - Lam_j}, weight of key j

  const int tid = threadIdx.x;
  const int bh = blockIdx.x;
  const int h = bh % H;
  const int j0 = blockIdx.y * dvt;
  const int nv = min(dvt, dv - j0);
  const size_t bhL = (size_t)bh * L;

  for (int x = tid; x < dk * nv; x += kThreads) {
    int r = x / nv, c = x % nv;
    S[r * dvt + c] = S0 ? S0[((size_t)bh * dk + r) * dv + j0 + c] : 0.f;
  }

  for (int s0 = 0; s0 < L; s0 += C) {
    const int n = min(C, L - s0);
    __syncthreads();  // previous chunk's readers of qs/ks/vs/S are done
    for (int x = tid; x < n * dk; x += kThreads) {
      const int t = x / dk, r = x % dk;
      qs[t * dkp + r] = feature_map_precise(phi, to_f32(q[(bhL + s0) * dk + x]));
      ks[t * dkp + r] = feature_map_precise(phi, to_f32(k[(bhL + s0) * dk + x]));
    }
    for (int x = tid; x < n * nv; x += kThreads) {
      int t = x / nv, c = x % nv;
      vs[t * dvt + c] = to_f32(v[(bhL + s0 + t) * dv + j0 + c]);
    }
    if (tid < 32) {  // inclusive prefix of the chunk's log decays (warp scan)
      float carry = 0.f;
      for (int base = 0; base < n; base += 32) {
        int i = base + tid;
        float x = i < n ? token_log_decay(decay_kind, decay, h, bhL, s0 + i) : 0.f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          float y = __shfl_up_sync(0xffffffffu, x, off);
          if (tid >= off) x += y;
        }
        if (i < n) lam[i] = carry + x;
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
    }
    __syncthreads();
    for (int x = tid; x < n * n; x += kThreads) {
      int i = x / n, j = x % n;
      float p = 0.f;
      if (j <= i) {
        float dot = 0.f;
        for (int c = 0; c < dk; ++c) dot = fmaf(qs[i * dkp + c], ks[j * dkp + c], dot);
        p = dot * expf(lam[i] - lam[j]);
      }
      P[i * C + j] = p;
    }
    for (int i = tid; i < n; i += kThreads) {
      eq[i] = expf(lam[i]);
      ek[i] = expf(lam[n - 1] - lam[i]);
    }
    __syncthreads();
    for (int x = tid; x < n * nv; x += kThreads) {
      int i = x / nv, c = x % nv;
      float inter = 0.f;
      for (int r = 0; r < dk; ++r) inter = fmaf(qs[i * dkp + r], S[r * dvt + c], inter);
      float intra = 0.f;
      for (int j = 0; j <= i; ++j) intra = fmaf(P[i * C + j], vs[j * dvt + c], intra);
      O[(bhL + s0 + i) * dv + j0 + c] = from_f32<T>(fmaf(eq[i], inter, intra));
    }
    __syncthreads();  // all reads of S for this chunk's output are done
    const float eend = eq[n - 1];
    for (int x = tid; x < dk * nv; x += kThreads) {
      int r = x / nv, c = x % nv;
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(ek[j] * ks[j * dkp + r], vs[j * dvt + c], acc);
      S[r * dvt + c] = fmaf(eend, S[r * dvt + c], acc);
    }
  }
  __syncthreads();
  if (S_final) {
    for (int x = tid; x < dk * nv; x += kThreads) {
      int r = x / nv, c = x % nv;
      S_final[((size_t)bh * dk + r) * dv + j0 + c] = S[r * dvt + c];
    }
  }
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a) {
  const int C = a.chunk;
  if (C < 1 || C > kMaxChunk || a.dk > 128 || a.dv > 128) return cudaErrorInvalidValue;
  const int dvt = a.dv < 32 ? a.dv : 32;
  const size_t smem =
      sizeof(float) * ((size_t)2 * C * (a.dk + 1) + (size_t)C * dvt + (size_t)C * C +
                       (size_t)a.dk * dvt + 3 * C);
  dim3 grid((unsigned)(a.B * a.H), (unsigned)((a.dv + dvt - 1) / dvt));
  if (a.dtype == LA_F32) {
    auto kern = prefill_simt_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, a.stream>>>(
        static_cast<const float *>(a.q), static_cast<const float *>(a.k),
        static_cast<const float *>(a.v), a.H, a.L, a.dk, a.dv, C, dvt, a.phi, a.decay_kind,
        a.decay, a.S0, static_cast<float *>(a.O), a.S_final);
  } else {
    auto kern = prefill_simt_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
        static_cast<const __nv_bfloat16 *>(a.v), a.H, a.L, a.dk, a.dv, C, dvt, a.phi,
        a.decay_kind, a.decay, a.S0, static_cast<__nv_bfloat16 *>(a.O), a.S_final);
  }
  return cudaGetLastError();
}

}  // namespace la
