// la_delta_tc.cu -- the (gated) delta rule on the 5th-gen tensor cores, a chunk
// of 64 tokens at a time: bf16 q, k, v with fp32 accumulation, d_k = d_v = D in
// {64, 128}.
//
// The rule ("Linear / Sparse Attention - minimal runnable implementation",
// delta_rule_recurrent; "Linear / sparse attention tutorial" section 5 and
// Q21, the gated form), with S kept as [d_k, d_v] like every other state here:
//   S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
//   o_t = phi(q_t)^T S_t,   k_t = phi(k_t) as given.
// Writing u_t = beta_t (v_t - alpha_t S_{t-1}^T k_t) turns it into
// S_t = alpha_t S_{t-1} + k_t u_t^T, and unrolling it over a chunk (Lam the
// inclusive prefix of log alpha from the chunk start, Gam_tj = e^{Lam_t - Lam_j})
// gives the unit lower-triangular system (I + A) U = diag(beta) V -
// diag(beta e^{Lam}) K S_in with A_tj = beta_t Gam_tj (k_t . k_j) for j < t.
// So with T = (I + A)^{-1} (the WY form; the tutorial's section 5.3):
//   W  = T diag(beta e^{Lam}) K,  U0 = T diag(beta) V,  U = U0 - W S_in,
//   O  = diag(e^{Lam}) Q S_in + P U,       P_tj = Gam_tj (q_t . k_j), j <= t,
//   S' = e^{Lam_end} S_in + Kt^T U,        Kt_j = e^{Lam_end - Lam_j} k_j.
// Substituting U, everything that does not involve S_in is formed off the
// state chain, once per chunk:
//   M  = -Kt^T W      (d_k x d_k),   Qe = diag(e^{Lam}) Q - P W   (64 x d_k),
// and the chain itself is
//   S' = e^{Lam_end} S_in + Kt^T U0 + M S_in,     O = P U0 + Qe S_in.
// The state stays fp32 in TMEM; only the products with S_in see its bf16 copy.
//
// Per chunk (one CTA per (b, h) sequence):
//   PREP   phi on q, k; Lam, beta; V <- diag(beta) V; Kb = diag(beta e^Lam) K;
//          after K K^T: K <- Kt in place
//   MMA    G = K K^T, P' = Q K^T                     (M 64, N 64, K D)
//   SOLVE  A and P from G, P'; T = (I + A)^{-1} by 16 x 16 blocks (CUDA cores, fp32)
//   MMA    W = T Kb, U0 = T V                        (M 64, N D, K 64)
//   EPI    W, U0 -> bf16
//   MMA    Kt^T W, P W, O = P U0                     (M D / 64, N D, K 64)
//   EPI    M = -Kt^T W -> bf16, Qe = e^Lam Q - P W -> bf16 (in place of Q)
//   MMA    chain: S += Kt^T U0, S += M S_in, O += Qe S_in
//   ST     S_in for the next chunk: bf16 copy, TMEM S *= e^{Lam_end}
//   EPI    O -> bf16 -> TMA store
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "../../include/la_gb300.h"
#include "la_common.cuh"
#include "la_internal.h"
#include "la_ptx.cuh"
#include "la_tc_sync.cuh"
#include "la_tma_host.h"

#ifdef LA_TRACE
namespace la {
namespace {
__device__ long long g_trace[kTraceEvents][kTraceChunks];
}
}  // namespace la
extern "C" int la_trace_read_delta(long long *out) {
  return (int)cudaMemcpyFromSymbol(out, la::g_trace, sizeof(la::g_trace));
}
#endif

namespace la {
namespace {
using namespace tc;

// Warp roles: 0 TMA, 1 MMA, 2..3 PREP (64 threads), 4..11 SOLVE (256 threads),
// 12..15 EPI, 16..19 ST.  The TMEM warpgroups start at a multiple of four warps.
constexpr int kThreads = 640;
constexpr int W_TMA = 0, W_MMA = 1, W_PREP = 2, W_SOLVE = 4, W_EPI = 12, W_ST = 16;
constexpr int kPrepThreads = (W_SOLVE - W_PREP) * 32;
constexpr int kSolveThreads = (W_EPI - W_SOLVE) * 32;
constexpr uint32_t BAR_PREP = 1, BAR_SOLVE = 2, BAR_EPI = 3, BAR_ST = 4;
constexpr int kAS = 65;  // fp32 row stride of the solve's A and T (conflict-free columns)

// The MMA issuer's bounded wait.  It polls the phase without a suspend-time
// hint: a suspended issuer resumed up to ~1 us after the phase it waited for
// had completed, and each of its waits is on the chunk's critical path.
static __device__ __noinline__ bool issuer_wait_slow(uint64_t *bar, uint32_t parity, Ctl *ctl,
                                                     unsigned int *err, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < kSpinCap; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*(volatile uint32_t *)&ctl->abort) return false;
      if (global_timer_ns() - t0 > kWaitNs) break;
    }
  }
  atomicExch(&ctl->abort, 1u);
  record_device_error(err, KID_DELTA_TC, site);
  return false;
}

template <int D>
struct DtSmem {
  static constexpr bool SMALL = D == 64;
  static constexpr int NST = SMALL ? 3 : 1;   // q | k | v stages (and Kb tiles)
  static constexpr bool GSEP = SMALL;         // G, P' in their own TMEM columns
  static constexpr uint32_t TILE = 64 * D * 2;
  static constexpr uint32_t STAGE = 3 * TILE;
  static constexpr uint32_t MBOX = D * 128;   // one 64-column box of a [D][D] bf16 matrix
  static constexpr uint32_t OFF_KB = NST * STAGE;
  static constexpr uint32_t OFF_T = OFF_KB + NST * TILE;      // [64][64] bf16, K-major
  static constexpr uint32_t OFF_P = OFF_T + 8192;             // [64][64] bf16, K-major
  static constexpr uint32_t OFF_W = OFF_P + 8192;             // [64][D] bf16 (MN-major B)
  static constexpr uint32_t OFF_U = OFF_W + TILE;             // [64][D] bf16
  static constexpr uint32_t OFF_M = OFF_U + TILE;             // [D][D] bf16, K-major
  static constexpr uint32_t OFF_S = OFF_M + D * D * 2;        // [D][D] bf16, MN-major
  // O staging: its own tile at D = 64; at D = 128 it shares the W tile (W of a
  // chunk is read before its O is stored; the next W waits for that store).
  static constexpr uint32_t OFF_O = SMALL ? OFF_S + D * D * 2 : OFF_W;
  static constexpr uint32_t OFF_A = SMALL ? OFF_O + TILE : OFF_S + D * D * 2;  // fp32 [64][kAS]
  static constexpr uint32_t OFF_TF = OFF_A + 64 * kAS * 4;     // fp32 [64][kAS]
  static constexpr uint32_t OFF_PS = OFF_TF + 64 * kAS * 4;    // [64][64] bf16 P staging
  static constexpr uint32_t OFF_R = OFF_PS + 8192;             // fp32 [3][16][17]
  static constexpr uint32_t OFF_LAM = OFF_R + 3 * 16 * 17 * 4; // [NST][64] Lam
  static constexpr uint32_t OFF_BETA = OFF_LAM + NST * 64 * 4; // [NST][64] beta
  static constexpr uint32_t OFF_SCR = OFF_BETA + NST * 64 * 4; // 16 floats
  static constexpr uint32_t OFF_BAR = OFF_SCR + 64;
  static constexpr int NBAR = 4 * NST + 11;
  static constexpr uint32_t OFF_CTL = OFF_BAR + 8 * NBAR;
  static constexpr uint32_t OFF_TRC = OFF_CTL + 64;  // trace builds
  static constexpr uint32_t BYTES = OFF_TRC + trace_smem_bytes();
  static_assert(STAGE % 1024 == 0 && OFF_KB % 1024 == 0 && OFF_T % 1024 == 0 &&
                    OFF_P % 1024 == 0 && OFF_W % 1024 == 0 && OFF_U % 1024 == 0 &&
                    OFF_M % 1024 == 0 && OFF_S % 1024 == 0 && OFF_O % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  static_assert(BYTES <= 232448, "exceeds the per-block shared memory limit");
  // TMEM columns: S (D), O (D), X (W, then Kt^T W: D), Y (U0, then P W: D),
  // and G | P' (128), which shares X's columns at D = 128.
  static constexpr uint32_t T_S = 0, T_O = D, T_X = 2 * D, T_Y = 3 * D;
  static constexpr uint32_t T_G = GSEP ? 4 * D : T_X;
  static constexpr uint32_t T_COLS = 512;
  static_assert((GSEP ? T_G + 128 : T_Y + D) <= T_COLS, "TMEM budget");
};

struct DtParams {
  int H, L, BH, n_chunks;
  const float *beta;       // [BH][L]
  const float *log_alpha;  // [BH][L] or null
  const float *S0;
  float *S_final;
  unsigned int *err;
};

// dst <- src * fac(row) over one [64][D] bf16 tile (same swizzled layout).
template <int D, typename Fac>
__device__ __forceinline__ void scaled_copy(const unsigned char *src, unsigned char *dst, Fac fac,
                                            int t, int n) {
  constexpr int kChunks = 64 * D * 2 / 16;
  for (int x = t; x < kChunks; x += n) {
    const uint4 u = *reinterpret_cast<const uint4 *>(src + (size_t)x * 16);
    const float f = fac((x & 511) >> 3);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_bf16(__uint_as_float(w[e] << 16) * f, __uint_as_float(w[e] & 0xffff0000u) * f);
    *reinterpret_cast<uint4 *>(dst + (size_t)x * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int D, bool PHI, bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
delta_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                DtParams p) {
  using SM = DtSmem<D>;
  constexpr int NST = SM::NST;
  constexpr bool GSEP = SM::GSEP;
  extern __shared__ __align__(1024) unsigned char smem[];
  float *lam = reinterpret_cast<float *>(smem + SM::OFF_LAM);
  float *bet = reinterpret_cast<float *>(smem + SM::OFF_BETA);
  float *scr = reinterpret_cast<float *>(smem + SM::OFF_SCR);
  float *As = reinterpret_cast<float *>(smem + SM::OFF_A);
  float *Ts = reinterpret_cast<float *>(smem + SM::OFF_TF);
  float *Rs = reinterpret_cast<float *>(smem + SM::OFF_R);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::OFF_BAR);
  uint64_t *empty = full + NST;
  uint64_t *prep_a = empty + NST;   // [NST] phi, Lam, beta, V scaled, Kb
  uint64_t *prep_b = prep_a + NST;  // [NST] K <- Kt in place
  uint64_t *t_ready = prep_b + NST; // T and P tiles written
  uint64_t *g_full = t_ready + 1;   // G, P' in TMEM
  uint64_t *wu_full = g_full + 1;   // W, U0 in TMEM
  uint64_t *wu_ready = wu_full + 1; // W, U0 tiles written
  uint64_t *m_full = wu_ready + 1;  // Kt^T W, P W in TMEM; O = P U0 issued
  uint64_t *m_ready = m_full + 1;   // M and Qe tiles written
  uint64_t *s_ready = m_ready + 1;  // bf16 S_in copy written, TMEM S scaled
  uint64_t *s_done = s_ready + 1;   // the chain's MMAs (and all before) done
  uint64_t *o_free = s_done + 1;    // O read out of TMEM
  uint64_t *drain = o_free + 1;
  uint64_t *g_free = drain + 1;     // (GSEP) A and P built: G, P' TMEM may be overwritten
  Ctl *ctl = reinterpret_cast<Ctl *>(smem + SM::OFF_CTL);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, nc = p.n_chunks;
  const size_t bhL = (size_t)bh * p.L;
  const bool trace_on = blockIdx.x == 0;
  const long long t0 = clock64();
  (void)trace_on;
  (void)t0;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&prep_a[s], 1);
      mbar_init(&prep_b[s], 1);
    }
    mbar_init(t_ready, 1);
    mbar_init(g_full, 1);
    mbar_init(wu_full, 1);
    mbar_init(wu_ready, 1);
    mbar_init(m_full, 1);
    mbar_init(m_ready, 1);
    mbar_init(s_ready, 1);
    mbar_init(s_done, 1);
    mbar_init(o_free, 1);
    mbar_init(drain, 1);
    mbar_init(g_free, 1);
    ctl->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(&ctl->tmem_base, SM::T_COLS);
    tmem_relinquish();
  }
  LA_TRACE_TABLE(smem + SM::OFF_TRC, 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == W_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
      int issued = 0;
      for (int c = 0; c < nc; ++c) {
        const int s = c % NST;
        if (c >= NST && !wait1(&empty[s], ((c / NST) - 1) & 1, ctl, p.err, KID_DELTA_TC, 1)) break;
        unsigned char *stg = smem + s * SM::STAGE;
        mbar_arrive_expect_tx(&full[s], SM::STAGE);
        for (int b = 0; b < D / BOX; ++b) {
          tma_load_3d(stg + b * BOX_BYTES, &tmQ, &full[s], b * BOX, c * CH, bh);
          tma_load_3d(stg + SM::TILE + b * BOX_BYTES, &tmK, &full[s], b * BOX, c * CH, bh);
          tma_load_3d(stg + 2 * SM::TILE + b * BOX_BYTES, &tmV, &full[s], b * BOX, c * CH, bh);
        }
        issued = c + 1;
      }
      if (*(volatile uint32_t *)&ctl->abort)
        for (int c = max(0, issued - NST); c < issued; ++c) drain_wait(&full[c % NST], (c / NST) & 1);
      for (int c = max(0, nc - NST); c < nc; ++c) drain_wait(&empty[c % NST], (c / NST) & 1);
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nc > 0) {
      constexpr uint32_t id_g = idesc_bf16_f32(64, 64, false, false);
      constexpr uint32_t id_tx = idesc_bf16_f32(64, D, false, true);   // T Kb, T V, P W, P U0, Qe S
      constexpr uint32_t id_kt = idesc_bf16_f32(D, D, true, true);     // Kt^T W, Kt^T U0
      constexpr uint32_t id_ms = idesc_bf16_f32(D, D, false, true);    // M S
      constexpr uint32_t HI = smem_desc_sw128_hi(1024);
      const uint32_t sbase = smem_u32(smem);
      const uint32_t dKM = smem_desc_sw128_lo(sbase, 16);
      const uint32_t dMN = smem_desc_sw128_lo(sbase, BOX_BYTES);
      const uint32_t dMS = smem_desc_sw128_lo(sbase, SM::MBOX);
      auto at = [](uint32_t d, uint32_t off) { return d + (off >> 4); };
      auto w = [&](uint64_t *bar, uint32_t par, uint32_t site) {
        return mbar_test(bar, par) || issuer_wait_slow(bar, par, ctl, p.err, site);
      };
      // G = K K^T and P' = Q K^T of chunk c.
      auto issue_g = [&](int c) {
        const uint32_t qo = (c % NST) * SM::STAGE, ko = qo + SM::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * BOX_BYTES + 32 * (kk % 4);
          mma_bf16_w(tmem + SM::T_G, at(dKM, ko + off), at(dKM, ko + off), HI, id_g, kk > 0);
          mma_bf16_w(tmem + SM::T_G + 64, at(dKM, qo + off), at(dKM, ko + off), HI, id_g, kk > 0);
        }
        mma_commit(g_full);
        LA_TRACE_EVENT(trace_on, t0, 1, c);
      };
      bool ok = w(&prep_a[0], 0, 2);
      if (ok) {
        tc_fence_after();
        issue_g(0);
      }
      // GSEP: G, P' of chunk g_next may go once the solve has read chunk
      // g_next - 1's out of TMEM and chunk g_next's prep is done.  The issue is
      // tried without blocking once this chunk's M, Qe MMAs are out (the solve
      // of the next chunk has usually built by then), and otherwise made with
      // blocking waits before this chunk's W, U0.
      int g_next = 1;
      auto try_g = [&](bool block) -> bool {
        if (!GSEP || g_next >= nc) return true;
        const int k = g_next;
        if (block) {
          if (!w(g_free, (k - 1) & 1, 5)) return false;
          if (!w(&prep_a[k % NST], (k / NST) & 1, 5)) return false;
        } else if (!mbar_test(g_free, (k - 1) & 1) || !mbar_test(&prep_a[k % NST], (k / NST) & 1)) {
          return true;
        }
        tc_fence_after();
        issue_g(k);
        ++g_next;
        return true;
      };
      for (int c = 0; ok && c < nc; ++c) {
        const int s = c % NST;
        const uint32_t qo = s * SM::STAGE, ko = qo + SM::TILE, vo = qo + 2 * SM::TILE;
        const uint32_t kbo = SM::OFF_KB + s * SM::TILE;
        const uint32_t to = SM::OFF_T, po = SM::OFF_P;
        // GSEP: the next chunk's G, P' as soon as the solve has read this
        // chunk's out of TMEM, so that the solve can start it right after this one.
        while (ok && GSEP && g_next <= c + 1 && g_next < nc) ok = try_g(true);
        if (!ok) break;
        // W = T Kb, U0 = T V (X and Y are free once the previous chunk's M, Qe are out).
        if (!(ok = w(t_ready, c & 1, 3))) break;
        if (c >= 1 && !(ok = w(m_ready, (c - 1) & 1, 4))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < CH / 16; ++kk) {
          mma_bf16_w(tmem + SM::T_X, at(dKM, to + 32 * kk), at(dMN, kbo + 2048 * kk), HI, id_tx, kk > 0);
          mma_bf16_w(tmem + SM::T_Y, at(dKM, to + 32 * kk), at(dMN, vo + 2048 * kk), HI, id_tx, kk > 0);
        }
        mma_commit(wu_full);
        LA_TRACE_EVENT(trace_on, t0, 5, c);
        // Kt^T W -> X, P W -> Y, O = P U0 (O is free once the previous chunk's O is out).
        if (!(ok = w(wu_ready, c & 1, 6))) break;
        if (!(ok = w(&prep_b[s], (c / NST) & 1, 7))) break;
        if (c >= 1 && !(ok = w(o_free, (c - 1) & 1, 8))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < CH / 16; ++kk) {
          mma_bf16_w(tmem + SM::T_X, at(dMN, ko + 2048 * kk), at(dMN, SM::OFF_W + 2048 * kk), HI,
                     id_kt, kk > 0);
          mma_bf16_w(tmem + SM::T_Y, at(dKM, po + 32 * kk), at(dMN, SM::OFF_W + 2048 * kk), HI,
                     id_tx, kk > 0);
          mma_bf16_w(tmem + SM::T_O, at(dKM, po + 32 * kk), at(dMN, SM::OFF_U + 2048 * kk), HI,
                     id_tx, kk > 0);
        }
        mma_commit(m_full);
        LA_TRACE_EVENT(trace_on, t0, 7, c);
        try_g(false);
        // The state chain.
        if (!(ok = w(m_ready, c & 1, 9))) break;
        if (!(ok = w(s_ready, c & 1, 10))) break;
        try_g(false);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < CH / 16; ++kk)  // S += Kt^T U0
          mma_bf16_w(tmem + SM::T_S, at(dMN, ko + 2048 * kk), at(dMN, SM::OFF_U + 2048 * kk), HI,
                     id_kt, 1u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // S += M S_in, O += Qe S_in
          mma_bf16_w(tmem + SM::T_S, at(dKM, SM::OFF_M + (kk / 4) * SM::MBOX + 32 * (kk % 4)),
                     at(dMS, SM::OFF_S + 2048 * kk), HI, id_ms, 1u);
          mma_bf16_w(tmem + SM::T_O, at(dKM, qo + (kk / 4) * BOX_BYTES + 32 * (kk % 4)),
                     at(dMS, SM::OFF_S + 2048 * kk), HI, id_tx, 1u);
        }
        mma_commit(s_done);
        mma_commit(&empty[s]);
        LA_TRACE_EVENT(trace_on, t0, 9, c);
        try_g(false);
        if (!GSEP && c + 1 < nc) {
          if (!(ok = w(&prep_a[(c + 1) % NST], ((c + 1) / NST) & 1, 11))) break;
          if (!(ok = w(m_ready, c & 1, 12))) break;
          tc_fence_after();
          issue_g(c + 1);
        }
      }
      mma_commit(drain);
      drain_wait(drain, 0);
    }
  } else if (warp >= W_PREP && warp < W_SOLVE) {
    // ------------------------------------------------------------ PREP
    const int t = tid - W_PREP * 32;
    auto gwait = [&](uint64_t *bar, uint32_t par, uint32_t site) {
      return wait_grp<kPrepThreads>(bar, par, ctl, p.err, KID_DELTA_TC, site, BAR_PREP, t);
    };
    bool ok = true;
    for (int c = 0; ok && c < nc; ++c) {
      const int s = c % NST;
      unsigned char *qt = smem + s * SM::STAGE, *kt = qt + SM::TILE, *vt = kt + SM::TILE;
      unsigned char *kb = smem + SM::OFF_KB + s * SM::TILE;
      if (!(ok = gwait(&full[s], (c / NST) & 1, 13))) break;
      if (t < 64) {  // inclusive prefix of log alpha (warps 2, 3), beta
        const int tok = c * CH + t;
        float x = 0.f, b = 0.f;
        if (tok < p.L) {
          b = p.beta[bhL + tok];
          if (GATED) x = p.log_alpha[bhL + tok];
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, off);
          if (lane >= off) x += y;
        }
        if (t == 31) scr[0] = x;
        lam[s * 64 + t] = x;
        bet[s * 64 + t] = b;
      }
      named_bar_sync(BAR_PREP, kPrepThreads);
      if (t >= 32 && t < 64) lam[s * 64 + t] += scr[0];
      named_bar_sync(BAR_PREP, kPrepThreads);
      const float *lm = lam + s * 64, *bt = bet + s * 64;
      if constexpr (PHI) tile_pass<D, 2, true, false>(qt, [](int, int) { return 1.f; }, t, kPrepThreads);
      if (!PHI) (void)qt;
      tile_pass<D, 1, false, true>(vt, [bt](int, int r) { return bt[r]; }, t, kPrepThreads);
      fence_proxy_async_smem();  // phi(k) is read back below by the other threads
      named_bar_sync(BAR_PREP, kPrepThreads);
      scaled_copy<D>(kt, kb, [lm, bt](int r) { return bt[r] * __expf(lm[r]); }, t, kPrepThreads);
      fence_proxy_async_smem();
      named_bar_sync(BAR_PREP, kPrepThreads);
      if (t == 0) mbar_arrive(&prep_a[s]);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 0, c);
      // Once K K^T and Q K^T have read phi(K): K <- Kt in place.
      if (!(ok = gwait(g_full, c & 1, 14))) break;
      const float le = lm[63];
      tile_pass<D, 1, false, true>(kt, [lm, le](int, int r) { return __expf(le - lm[r]); }, t,
                                   kPrepThreads);
      fence_proxy_async_smem();
      named_bar_sync(BAR_PREP, kPrepThreads);
      if (t == 0) mbar_arrive(&prep_b[s]);
    }
  } else if (warp >= W_SOLVE && warp < W_EPI) {
    // ------------------------------------------------------------ SOLVE: T = (I + A)^{-1}, P
    // Warps 4..7 build A from G, warps 8..11 build P from P' (each warpgroup
    // reaches every TMEM lane quarter); all 256 threads then invert I + A.
    const int t = tid - W_SOLVE * 32;
    const int quarter = warp & 3;
    const bool p_side = warp >= W_SOLVE + 4;
    const int row = acc_row<64>(quarter, lane);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    auto swait = [&](uint64_t *bar, uint32_t par, uint32_t site) {
      return wait_grp<kSolveThreads>(bar, par, ctl, p.err, KID_DELTA_TC, site, BAR_SOLVE, t);
    };
    bool ok = true;
    for (int c = 0; ok && c < nc; ++c) {
      const int s = c % NST;
      if (!(ok = swait(&prep_a[s], (c / NST) & 1, 15))) break;
      if (!(ok = swait(g_full, c & 1, 16))) break;
      LA_TRACE_EVENT(trace_on && t == 0, t0, 2, c);
      tc_fence_after();
      const float *lm = lam + s * 64, *bt = bet + s * 64;
      // A (fp32) from G, or P (bf16) from P' into a staging tile (the P tile
      // itself may still be read by the previous chunk's MMAs).  The M = 64
      // accumulators keep their rows in 16 lanes of each warp quarter; a
      // 16x256b load spreads them over all 32 threads: rows ra and ra + 8,
      // columns 8 q + c2 and + 1 for q = 0..7.
      unsigned char *ps = smem + SM::OFF_PS;
      {
        const int ra = 16 * quarter + (lane >> 2), c2 = 2 * (lane & 3);
        uint32_t g[32];
        __syncwarp();
        tmem_ld_16x256b_x8(tmem + lane_off + SM::T_G + (p_side ? 64 : 0), g);
        tmem_ld_wait();
        const float la = lm[ra], lb = lm[ra + 8], ba = bt[ra], bb = bt[ra + 8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = 8 * q + c2;
          const float l0 = lm[j], l1 = lm[j + 1];
          // decay between the rows' tokens and keys j, j + 1 (keys up to the row)
          const float fa0 = j <= ra ? __expf(la - l0) : 0.f;
          const float fa1 = j + 1 <= ra ? __expf(la - l1) : 0.f;
          const float fb0 = j <= ra + 8 ? __expf(lb - l0) : 0.f;
          const float fb1 = j + 1 <= ra + 8 ? __expf(lb - l1) : 0.f;
          const float ga0 = __uint_as_float(g[4 * q]), ga1 = __uint_as_float(g[4 * q + 1]);
          const float gb0 = __uint_as_float(g[4 * q + 2]), gb1 = __uint_as_float(g[4 * q + 3]);
          if (p_side) {
            const uint32_t sw = (uint32_t)((q ^ (ra & 7)) << 4) + (uint32_t)(c2 << 1);
            // rows ra and ra + 8 share (row & 7), so one swizzle serves both
            *reinterpret_cast<uint32_t *>(ps + ra * 128 + sw) = pack_bf16(fa0 * ga0, fa1 * ga1);
            *reinterpret_cast<uint32_t *>(ps + (ra + 8) * 128 + sw) = pack_bf16(fb0 * gb0, fb1 * gb1);
          } else {  // strictly below the diagonal
            As[ra * kAS + j] = j < ra ? ba * fa0 * ga0 : 0.f;
            As[ra * kAS + j + 1] = j + 1 < ra ? ba * fa1 * ga1 : 0.f;
            As[(ra + 8) * kAS + j] = j < ra + 8 ? bb * fb0 * gb0 : 0.f;
            As[(ra + 8) * kAS + j + 1] = j + 1 < ra + 8 ? bb * fb1 * gb1 : 0.f;
          }
        }
      }
      tc_fence_before();
      named_bar_sync(BAR_SOLVE, kSolveThreads);
      if (SM::GSEP && t == 0) mbar_arrive(g_free);  // G, P' read out of TMEM
      LA_TRACE_EVENT(trace_on && t == 0, t0, 13, c);
      // Diagonal 16 x 16 blocks by forward substitution, one column per thread
      // (zero above the diagonal), right-looking: once x_j is final, every
      // later row's sum takes its term at once, so the dependent chain is the
      // 16 steps of j, not the 120 products.
      if (t < 64) {
        const int I = t >> 4, col = t & 15, r0 = 16 * I;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = i == col ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < 15; ++j) {
          float a[16];
#pragma unroll
          for (int i = j + 1; i < 16; ++i) a[i] = As[(r0 + i) * kAS + r0 + j];
          const float xj = j >= col ? x[j] : 0.f;
#pragma unroll
          for (int i = j + 1; i < 16; ++i) x[i] -= a[i] * xj;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Ts[(r0 + i) * kAS + r0 + col] = i >= col ? x[i] : 0.f;
      }
      named_bar_sync(BAR_SOLVE, kSolveThreads);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 14, c);
      // Below the diagonal, by distance d = I - J:
      //   R = sum_{K=J}^{I-1} A_IK T_KJ,   T_IJ = -T_II R.
      // 64 threads per block; each takes four rows of one column.  The column
      // vector is loaded once per block of 16 and each row's 16 values
      // before their products, so the loads overlap.
#pragma unroll 1
      for (int d = 1; d <= 3; ++d) {
        const int b = t >> 6, tt = t & 63, ri = tt >> 4, j = tt & 15;
        const bool act = b < 4 - d;
        const int I = d + b, J = I - d, i0 = 16 * I + 4 * ri;
        if (act) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
          for (int K = J; K < I; ++K) {
            float tv[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) tv[m] = Ts[(16 * K + m) * kAS + 16 * J + j];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              float av[16];
#pragma unroll
              for (int m = 0; m < 16; ++m) av[m] = As[(i0 + r) * kAS + 16 * K + m];
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int m = 0; m < 16; m += 2) {
                s0 += av[m] * tv[m];
                s1 += av[m + 1] * tv[m + 1];
              }
              acc[r] += s0 + s1;
            }
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) Rs[b * 272 + (4 * ri + r) * 17 + j] = acc[r];
        }
        named_bar_sync(BAR_SOLVE, kSolveThreads);
        if (act) {
          float rv[16];
#pragma unroll
          for (int m = 0; m < 16; ++m) rv[m] = Rs[b * 272 + m * 17 + j];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            float tv[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) tv[m] = Ts[(i0 + r) * kAS + 16 * I + m];  // zero above the diagonal
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; m += 2) {
              s0 += tv[m] * rv[m];
              s1 += tv[m + 1] * rv[m + 1];
            }
            Ts[(i0 + r) * kAS + 16 * J + j] = -(s0 + s1);
          }
        }
        named_bar_sync(BAR_SOLVE, kSolveThreads);
        if (d < 3) LA_TRACE_EVENT(trace_on && t == 0, t0, 10 + d, c);
      }
      LA_TRACE_EVENT(trace_on && t == 0, t0, 3, c);
      // The T and P tiles were last read by the previous chunk's MMAs.
      if (c >= 1 && !(ok = swait(m_full, (c - 1) & 1, 17))) break;
      LA_TRACE_EVENT(trace_on && t == 0, t0, 15, c);
      {  // P staging -> P tile: the same swizzled layout, 16 bytes x2 per thread
        const uint4 *src = reinterpret_cast<const uint4 *>(smem + SM::OFF_PS);
        uint4 *dst = reinterpret_cast<uint4 *>(smem + SM::OFF_P);
        dst[t] = src[t];
        dst[t + kSolveThreads] = src[t + kSolveThreads];
      }
      {  // T -> bf16, K-major rows; 16-byte chunk x2 per thread; zero above the block diagonal
        unsigned char *tt = smem + SM::OFF_T;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int x = t + kSolveThreads * u, r = x >> 3, ch = x & 7, j0 = 8 * ch;
          uint32_t w4[4] = {0u, 0u, 0u, 0u};
          if ((j0 >> 4) <= (r >> 4)) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w4[e] = pack_bf16(Ts[r * kAS + j0 + 2 * e], Ts[r * kAS + j0 + 2 * e + 1]);
          }
          *reinterpret_cast<uint4 *>(tt + r * 128 + ((ch ^ (r & 7)) << 4)) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(BAR_SOLVE, kSolveThreads);
      if (t == 0) mbar_arrive(t_ready);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 4, c);
    }
  } else if (warp >= W_EPI && warp < W_ST) {
    // ------------------------------------------------------------ EPI
    const int t = tid - W_EPI * 32;
    const int quarter = warp & 3;
    const int row = acc_row<64>(quarter, lane);     // token row of an M = 64 product
    const int mrow = acc_row<D>(quarter, lane);     // row of an M = D product
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    auto ewait = [&](uint64_t *bar, uint32_t par, uint32_t site) {
      return wait_wg(bar, par, ctl, p.err, KID_DELTA_TC, site, BAR_EPI);
    };
    // 32 fp32 columns of TMEM row -> 16 bf16 pairs * sc into a swizzled tile.
    auto put32 = [&](unsigned char *base, uint32_t blk, int r, int col, const uint32_t (&v)[32],
                     float sc) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          pk[j] = pack_bf16(__uint_as_float(v[16 * h + 2 * j]) * sc,
                            __uint_as_float(v[16 * h + 2 * j + 1]) * sc);
        st_row16(base, blk, r, col + 16 * h, pk);
      }
    };
    bool ok = true;
    for (int c = 0; ok && c < nc; ++c) {
      const int s = c % NST;
      // W, U0 -> bf16 tiles (U0's tile was last read by the previous chain).
      if (!(ok = ewait(wu_full, c & 1, 18))) break;
      if (c >= 1 && !(ok = ewait(s_done, (c - 1) & 1, 19))) break;
      if (!SM::SMALL && t == 0) tma_store_wait_read<0>();  // O staging shares the W tile
      __syncwarp();
      named_bar_sync(BAR_EPI, 128);
      tc_fence_after();
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        uint32_t r[32], u[32];
        __syncwarp();
        tmem_ld32(tmem + lane_off + SM::T_X + col, r);
        tmem_ld32(tmem + lane_off + SM::T_Y + col, u);
        tmem_ld_wait();
        if (row >= 0) {
          put32(smem + SM::OFF_W, BOX_BYTES, row, col, r, 1.f);
          put32(smem + SM::OFF_U, BOX_BYTES, row, col, u, 1.f);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_EPI, 128);
      if (t == 0) mbar_arrive(wu_ready);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 6, c);
      // M = -Kt^T W -> bf16 (K-major rows), Qe = e^{Lam} Q - P W in place of Q.
      if (!(ok = ewait(m_full, c & 1, 20))) break;
      tc_fence_after();
      const float *lm = lam + s * 64;
      unsigned char *qt = smem + s * SM::STAGE;
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        uint32_t r[32], u[32];
        __syncwarp();
        tmem_ld32(tmem + lane_off + SM::T_X + col, r);
        tmem_ld32(tmem + lane_off + SM::T_Y + col, u);
        tmem_ld_wait();
        if (mrow >= 0) put32(smem + SM::OFF_M, SM::MBOX, mrow, col, r, -1.f);
        if (row >= 0) {
          const float el = __expf(lm[row]);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int cc = col + 2 * j;
            const uint32_t qw = *reinterpret_cast<const uint32_t *>(
                qt + (cc >> 6) * BOX_BYTES + sw128_offset(row, cc & 63));
            pk[j] = pack_bf16(__uint_as_float(qw << 16) * el - __uint_as_float(u[2 * j]),
                              __uint_as_float(qw & 0xffff0000u) * el - __uint_as_float(u[2 * j + 1]));
          }
          st_row16(qt, BOX_BYTES, row, col, pk);
          st_row16(qt, BOX_BYTES, row, col + 16, pk + 8);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_EPI, 128);
      if (t == 0) mbar_arrive(m_ready);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 8, c);
      // O -> bf16 -> TMA store.
      if (!(ok = ewait(s_done, c & 1, 21))) break;
      tc_fence_after();
      if (SM::SMALL && t == 0) tma_store_wait_read<0>();
      __syncwarp();
      named_bar_sync(BAR_EPI, 128);
      unsigned char *o_sm = smem + SM::OFF_O;
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(tmem + lane_off + SM::T_O + col, r);
        tmem_ld_wait();
        if (row >= 0) put32(o_sm, BOX_BYTES, row, col, r, 1.f);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_EPI, 128);
      if (t == 0) {
        mbar_arrive(o_free);
        for (int bb = 0; bb < D / BOX; ++bb)
          tma_store_3d(&tmO, o_sm + bb * BOX_BYTES, bb * BOX, c * CH, bh);
        tma_store_commit();
      }
    }
    if (t == 0) tma_store_wait_all();
  } else if (warp >= W_ST) {
    // ------------------------------------------------------------ ST: the state chain
    const int t = tid - W_ST * 32;
    const int quarter = warp & 3;
    const int srow = acc_row<D>(quarter, lane);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    auto swait = [&](uint64_t *bar, uint32_t par, uint32_t site) {
      return wait_wg(bar, par, ctl, p.err, KID_DELTA_TC, site, BAR_ST);
    };
#pragma unroll 1
    for (int col = 0; col < D; col += 32) {  // S0 (or zeros) into TMEM
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
      if (srow >= 0 && p.S0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.S0 + ((size_t)bh * D + srow) * D + col);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 f = src[j];
          r[4 * j] = __float_as_uint(f.x);
          r[4 * j + 1] = __float_as_uint(f.y);
          r[4 * j + 2] = __float_as_uint(f.z);
          r[4 * j + 3] = __float_as_uint(f.w);
        }
      }
      __syncwarp();
      tmem_st32(tmem + lane_off + SM::T_S + col, r);
    }
    tmem_st_wait();
    bool ok = true;
    for (int c = 0; ok && c < nc; ++c) {
      const int s = c % NST;
      if (!(ok = swait(&prep_a[s], (c / NST) & 1, 22))) break;
      if (c >= 1 && !(ok = swait(s_done, (c - 1) & 1, 23))) break;
      tc_fence_after();
      const float e = GATED ? __expf(lam[s * 64 + 63]) : 1.f;
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(tmem + lane_off + SM::T_S + col, r);
        tmem_ld_wait();
        if (srow >= 0) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              pk[j] = pack_bf16(__uint_as_float(r[16 * h + 2 * j]), __uint_as_float(r[16 * h + 2 * j + 1]));
            st_row16(smem + SM::OFF_S, SM::MBOX, srow, col + 16 * h, pk);
          }
        }
        if (GATED) {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * e);
          __syncwarp();
          tmem_st32(tmem + lane_off + SM::T_S + col, r);
        }
      }
      if (GATED) tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_ST, 128);
      if (t == 0) mbar_arrive(s_ready);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 10, c);
    }
    if (ok && nc > 0 && swait(s_done, (nc - 1) & 1, 24) && p.S_final) {
      tc_fence_after();
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(tmem + lane_off + SM::T_S + col, r);
        tmem_ld_wait();
        if (srow >= 0) {
          float4 *dst = reinterpret_cast<float4 *>(p.S_final + ((size_t)bh * D + srow) * D + col);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) {
    __syncwarp();
    tmem_dealloc(tmem, SM::T_COLS);
  }
  LA_TRACE_FLUSH(trace_on, &g_trace[0][0]);
}

template <int D, bool PHI, bool GATED>
cudaError_t launch_dt(const VariantArgs &a) {
  using SM = DtSmem<D>;
  const int BH = a.B * a.H;
  DtParams p{};
  p.H = a.H;
  p.L = a.L;
  p.BH = BH;
  p.n_chunks = (a.L + CH - 1) / CH;
  p.beta = a.beta;
  p.log_alpha = a.decay;
  p.S0 = a.S0;
  p.S_final = a.S_final;
  p.err = device_error_word();
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_bf16_3d(&tq, a.q, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&tk, a.k, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&tv, a.v, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&to, a.O, D, a.L, BH, BOX, BOX))
    return cudaErrorInvalidValue;
  auto kern = delta_tc_kernel<D, PHI, GATED>;
  static int smem_set[64];
  cudaError_t e = set_smem_once(kern, SM::BYTES, smem_set);
  if (e != cudaSuccess) return e;
  kern<<<BH, kThreads, SM::BYTES, a.stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

}  // namespace

// The rule as the pages state it: phi = identity on keys the caller has
// normalised.  Under elu + 1 the keys are long (|phi(k)|^2 ~ 1.3 d_k) and O
// cancels heavily; bf16 operands then miss the 2e-2 row tolerance by up to 3x
// (a CPU emulation of this pipeline), so that case keeps the fp32 CUDA-core
// kernel.
bool delta_tc_supported(const VariantArgs &a) {
  return a.form == VARIANT_DELTA && a.dtype == LA_BF16 && a.phi == LA_PHI_IDENTITY &&
         a.dk == a.dv && (a.dk == 64 || a.dk == 128);
}

cudaError_t launch_delta_tc(const VariantArgs &a) {
  const bool gated = a.decay != nullptr;
  if (a.dk == 128) return gated ? launch_dt<128, false, true>(a) : launch_dt<128, false, false>(a);
  return gated ? launch_dt<64, false, true>(a) : launch_dt<64, false, false>(a);
}

}  // namespace la
