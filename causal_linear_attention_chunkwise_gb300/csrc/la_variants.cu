// la_variants.cu -- CUDA-core kernels for two further forms of the state
// recurrence (fp32 arithmetic, fp32 or bf16 inputs):
//
//   channel gate  S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T, alpha_t in (0,1]^{d_k}
//                 ("Linear / sparse attention tutorial" Q21, GLA)
//   delta rule    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
//                 ("Linear / Sparse Attention - minimal runnable implementation",
//                 delta_rule_recurrent, with the state transposed to [d_k, d_v];
//                 "Linear / sparse attention tutorial" Q21 for the gate alpha_t)
//
// with o_t = phi(q_t)^T S_t (update before read) in both.
//
// The channel gate is chunkwise, like the SIMT prefill kernel: per chunk of
// n <= C tokens the intra-chunk scores are formed exactly with their decay
// (every exponent is a difference Lam_i - Lam_j with i >= j, so it is <= 0 for
// log decays <= 0), the inter-chunk read uses the state of the previous chunk
// and the state is then advanced by the whole chunk.  With one cumulative log
// decay per key channel, the score for (i, j) is sum_c q_ic k_jc
// e^{Lam_ic - Lam_jc}.  When every cumulative log decay of the chunk lies in
// [-80, 80] the factors split: q~_i = e^{Lam_i} q_i, k~_j = e^{-Lam_j} k_j and
// the score is the plain dot product q~_i . k~_j (the state then advances as
// S <- e^{Lam_end} (S + k~^T V)).  Otherwise each score term takes its own
// factor, and the decays are folded into q (e^{Lam_ic}) and k
// (e^{Lam_end,c - Lam_jc}) once the scores are formed.
//
// The delta rule runs token by token: each step erases along k before it
// writes, and every column of S is independent of the others
// (S[:, c] <- a S[:, c] + k (beta (v_c - a k^T S[:, c]))).
#include <cuda_bf16.h>

#include "../../include/la_gb300.h"
#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunk = 64;
constexpr float kSplitMax = 80.f;  // e^{80} * e^{80} stays inside the fp32 range
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Per-channel gate.  One CTA per (b, h) and slice of dvt value columns, with
// its slice of S (d_k x dvt) in shared memory; log_alpha is [B,H,L,d_k].
// Rows of q, k and the log-decay prefix are padded to dk + 1 floats: the score
// loop reads one k row per lane, and a stride of dk (a multiple of 16) would put
// a warp's reads in one or two shared-memory banks.
template <typename T>
__global__ void __launch_bounds__(kThreads)
channel_gate_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    int L, int dk, int dv, int C, int dvt, int phi,
                    const float *__restrict__ log_alpha, const float *S0, T *__restrict__ O,
                    float *S_final) {
  extern __shared__ float smem[];
  const int dkp = dk + 1;
  float *qs = smem;           // [C][dkp]  phi(q), then e^{Lam_i} phi(q_i)
  float *ks = qs + C * dkp;   // [C][dkp]  phi(k), then e^{Lam_end - Lam_j} phi(k_j)
  float *lam = ks + C * dkp;  // [C][dkp]  per-channel inclusive log-decay prefix
  float *vs = lam + C * dkp;  // [C][dvt]
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
    const auto phi_of = [phi](float x) { return feature_map_precise(phi, x); };
    const auto same = [](float x) { return x; };
    stage_slab<T, 8>(q + (bhL + s0) * dk, dk, n, dk, qs, dkp, phi_of, tid, kThreads);
    stage_slab<T, 8>(k + (bhL + s0) * dk, dk, n, dk, ks, dkp, phi_of, tid, kThreads);
    stage_slab<T, 2>(v + (bhL + s0) * dv + j0, dv, n, nv, vs, dvt, same, tid, kThreads);
    stage_slab<float, 8>(log_alpha + (bhL + s0) * dk, dk, n, dk, lam, dkp, same, tid, kThreads);
    __syncthreads();
    int wide = 0;  // a cumulative log decay of this chunk outside [-kSplitMax, kSplitMax]
    for (int r = tid; r < dk; r += kThreads) {  // one channel per thread, in token order
      float acc = 0.f;
      for (int t = 0; t < n; ++t) {
        acc += lam[t * dkp + r];
        lam[t * dkp + r] = acc;
        wide |= !(fabsf(acc) <= kSplitMax);
      }
    }
    if (!__syncthreads_or(wide)) {
      // Split form: q~_i = e^{Lam_i} q_i and k~_j = e^{-Lam_j} k_j, every factor in
      // [e^{-kSplitMax}, e^{kSplitMax}], so P_ij = q~_i . k~_j needs no exponential.
      for (int x = tid; x < n * dk; x += kThreads) {
        const int y = (x / dk) * dkp + x % dk;
        const float l = lam[y];
        qs[y] *= expf(l);
        ks[y] *= expf(-l);
      }
      __syncthreads();
      for (int x = tid; x < n * n; x += kThreads) {
        const int i = x / n, j = x % n;
        float p = 0.f;
        if (j <= i)
          for (int c = 0; c < dk; ++c) p = fmaf(qs[i * dkp + c], ks[j * dkp + c], p);
        P[i * C + j] = p;
      }
      __syncthreads();
      for (int x = tid; x < n * nv; x += kThreads) {
        const int i = x / nv, c = x % nv;
        float acc = 0.f;
        for (int r = 0; r < dk; ++r) acc = fmaf(qs[i * dkp + r], S[r * dvt + c], acc);
        for (int j = 0; j <= i; ++j) acc = fmaf(P[i * C + j], vs[j * dvt + c], acc);
        O[(bhL + s0 + i) * dv + j0 + c] = from_f32<T>(acc);
      }
      __syncthreads();
      for (int x = tid; x < dk * nv; x += kThreads) {  // S <- e^{Lam_end} (S + k~^T V)
        const int r = x / nv, c = x % nv;
        float acc = 0.f;
        for (int j = 0; j < n; ++j) acc = fmaf(ks[j * dkp + r], vs[j * dvt + c], acc);
        S[r * dvt + c] = expf(lam[(n - 1) * dkp + r]) * (S[r * dvt + c] + acc);
      }
      continue;
    }
    // Exact form for chunks with strong decay: every score term takes its own factor.
    for (int x = tid; x < n * n; x += kThreads) {
      const int i = x / n, j = x % n;
      float p = 0.f;
      if (j <= i)
        for (int c = 0; c < dk; ++c)
          p = fmaf(qs[i * dkp + c] * ks[j * dkp + c], expf(lam[i * dkp + c] - lam[j * dkp + c]),
                   p);
      P[i * C + j] = p;
    }
    __syncthreads();
    for (int x = tid; x < n * dk; x += kThreads) {  // fold the decays into q and k
      const int y = (x / dk) * dkp + x % dk;
      qs[y] *= expf(lam[y]);
      ks[y] *= expf(lam[(n - 1) * dkp + x % dk] - lam[y]);
    }
    __syncthreads();
    for (int x = tid; x < n * nv; x += kThreads) {
      const int i = x / nv, c = x % nv;
      float acc = 0.f;
      for (int r = 0; r < dk; ++r) acc = fmaf(qs[i * dkp + r], S[r * dvt + c], acc);
      for (int j = 0; j <= i; ++j) acc = fmaf(P[i * C + j], vs[j * dvt + c], acc);
      O[(bhL + s0 + i) * dv + j0 + c] = from_f32<T>(acc);
    }
    __syncthreads();
    for (int x = tid; x < dk * nv; x += kThreads) {
      const int r = x / nv, c = x % nv;
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(ks[j * dkp + r], vs[j * dvt + c], acc);
      S[r * dvt + c] = fmaf(expf(lam[(n - 1) * dkp + r]), S[r * dvt + c], acc);
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
// owns slice columns 4w .. 4w+3.  Lane 8 cl + g holds column 4w + cl, rows
// VW g + 8 VW i + e (i < RPL / VW, e < VW) of it in registers: RPL = d_k / 8
// rows, read from shared memory as VW-wide vectors (a warp's read of one
// vector index covers 8 VW consecutive floats, once per column: no bank
// conflicts).  The two dot products of a step are reductions over the 8 lanes
// of a column (xor 1, 2, 4).  Tokens are staged through shared memory kTok at
// a time, and each step's k and q are loaded while the previous step runs.
constexpr int kTok = 32;
constexpr int kDeltaCols = 32;

__device__ __forceinline__ float group8_sum(float x) {
  x += __shfl_xor_sync(kFull, x, 1);
  x += __shfl_xor_sync(kFull, x, 2);
  x += __shfl_xor_sync(kFull, x, 4);
  return x;
}

template <int VW>
__device__ __forceinline__ void load_rows(float *dst, const float *row, int g, int ni) {
  // dst[VW i + e] = row[VW g + 8 VW i + e]
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i >= ni) break;
    const float *p = row + VW * g + 8 * VW * i;
    if constexpr (VW == 4) {
      const float4 x = *reinterpret_cast<const float4 *>(p);
      dst[4 * i] = x.x; dst[4 * i + 1] = x.y; dst[4 * i + 2] = x.z; dst[4 * i + 3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2 *>(p);
      dst[2 * i] = x.x; dst[2 * i + 1] = x.y;
    }
  }
}

template <typename T, int DK>
__global__ void __launch_bounds__(kThreads)
delta_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, int L,
             int dv, int phi, const float *__restrict__ beta, const float *__restrict__ log_alpha,
             const float *S0, T *__restrict__ O, float *S_final) {
  static_assert(DK % 16 == 0 && DK <= 128, "d_k");
  constexpr int RPL = DK / 8;                // rows per lane
  constexpr int VW = RPL < 4 ? RPL : 4;      // vector width of a row read
  constexpr int NI = RPL / VW;               // vectors per lane
  __shared__ __align__(16) float qf[kTok][DK];
  __shared__ __align__(16) float kf[kTok][DK];
  __shared__ float vv[kTok][kDeltaCols], bt[kTok], at[kTok];

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane & 7, cl = lane >> 3;
  const int bh = blockIdx.x;
  const int j0 = blockIdx.y * kDeltaCols;
  const int nv = min(kDeltaCols, dv - j0);
  const int c = warp * 4 + cl;  // this lane's slice column
  const bool live = c < nv;
  const size_t bhL = (size_t)bh * L;
  auto row_of = [&](int m) { return VW * g + 8 * VW * (m / VW) + m % VW; };

  float s[RPL];
#pragma unroll
  for (int m = 0; m < RPL; ++m)
    s[m] = (S0 && live) ? S0[((size_t)bh * DK + row_of(m)) * dv + j0 + c] : 0.f;

  for (int t0 = 0; t0 < L; t0 += kTok) {
    const int nt = min(kTok, L - t0);
    __syncthreads();  // every warp is done with the previous tokens
    const auto phi_of = [phi](float x) { return feature_map_precise(phi, x); };
    const auto same = [](float x) { return x; };
    stage_slab<T, 4>(q + (bhL + t0) * DK, DK, nt, DK, &qf[0][0], DK, phi_of, tid, kThreads);
    stage_slab<T, 4>(k + (bhL + t0) * DK, DK, nt, DK, &kf[0][0], DK, phi_of, tid, kThreads);
    stage_slab<T, 1>(v + (bhL + t0) * dv + j0, dv, nt, nv, &vv[0][0], kDeltaCols, same, tid,
                     kThreads);
    for (int x = tid; x < nt * kDeltaCols; x += kThreads)  // columns past d_v read as 0
      if (x % kDeltaCols >= nv) vv[x / kDeltaCols][x % kDeltaCols] = 0.f;
    for (int t = tid; t < nt; t += kThreads) {
      bt[t] = beta[bhL + t0 + t];
      at[t] = log_alpha ? expf(log_alpha[bhL + t0 + t]) : 1.f;
    }
    __syncthreads();
    float kr[RPL], qr[RPL];
    load_rows<VW>(kr, kf[0], g, NI);
    load_rows<VW>(qr, qf[0], g, NI);
    float a = at[0], b = bt[0], vc = vv[0][c];
    for (int t = 0; t < nt; ++t) {
      float kn[RPL], qn[RPL];  // the next step's rows and scalars, loaded ahead
      const int tn = t + 1 < nt ? t + 1 : t;
      load_rows<VW>(kn, kf[tn], g, NI);
      load_rows<VW>(qn, qf[tn], g, NI);
      const float an = at[tn], bn = bt[tn], vn = vv[tn][c];
      float u0 = 0.f, u1 = 0.f;  // (k^T S)_c, two partial sums
#pragma unroll
      for (int m = 0; m < RPL; m += 2) {
        u0 = fmaf(kr[m], s[m], u0);
        u1 = fmaf(kr[m + 1], s[m + 1], u1);
      }
      const float u = group8_sum(u0 + u1);
      const float w = b * (vc - a * u);  // what is written along k
      float o0 = 0.f, o1 = 0.f;
#pragma unroll
      for (int m = 0; m < RPL; m += 2) {
        s[m] = fmaf(kr[m], w, a * s[m]);
        s[m + 1] = fmaf(kr[m + 1], w, a * s[m + 1]);
        o0 = fmaf(qr[m], s[m], o0);
        o1 = fmaf(qr[m + 1], s[m + 1], o1);
      }
      const float o = group8_sum(o0 + o1);
      if (g == 0 && live) O[(bhL + t0 + t) * dv + j0 + c] = from_f32<T>(o);
#pragma unroll
      for (int m = 0; m < RPL; ++m) {
        kr[m] = kn[m];
        qr[m] = qn[m];
      }
      a = an;
      b = bn;
      vc = vn;
    }
  }
  if (S_final && live) {
#pragma unroll
    for (int m = 0; m < RPL; ++m) S_final[((size_t)bh * DK + row_of(m)) * dv + j0 + c] = s[m];
  }
}

template <typename Kern>
cudaError_t allow_smem(Kern kern, size_t smem) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <typename T>
cudaError_t launch_channel_gate_t(const VariantArgs &a) {
  const int C = a.chunk;
  const int dvt = a.dv < 32 ? a.dv : 32;
  const size_t smem = sizeof(float) * ((size_t)3 * C * (a.dk + 1) + (size_t)C * dvt +
                                       (size_t)C * C + (size_t)a.dk * dvt);
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
    case VARIANT_CHANNEL_GATE:
      if (channel_gate_tc_supported(a)) return launch_channel_gate_tc(a);
      return f32 ? launch_channel_gate_t<float>(a) : launch_channel_gate_t<__nv_bfloat16>(a);
    case VARIANT_DELTA:
      if (delta_tc_supported(a)) return launch_delta_tc(a);
      return f32 ? launch_delta_t<float>(a) : launch_delta_t<__nv_bfloat16>(a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace la
