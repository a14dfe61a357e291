// la_channel_gate_tc.cu -- the per-channel (GLA) gate on the 5th-gen tensor
// cores: bf16 q, k, v with fp32 accumulation, chunk C = 64, d_k = d_v = D in
// {64, 128}.
//
// The recurrence ("Linear / sparse attention tutorial" section 2.4 and Q21):
//   S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T,   o_t = phi(q_t)^T S_t,
// with one gate per key channel c (a row of S), given as log alpha_{t,c} <= 0.
// Over a chunk, Lam_{i,c} = sum_{r <= i} log alpha_{r,c} (inclusive prefix
// from the chunk start) expands it to
//   o_i   = sum_c q_ic e^{Lam_ic} S_c[c,:] + sum_{j <= i} P_ij v_j,
//   P_ij  = sum_c q_ic k_jc e^{Lam_ic - Lam_jc},
//   S_c+1 = diag(e^{Lam_end}) S_c + sum_j (k_j * e^{Lam_end - Lam_j}) v_j^T.
// The decay sits inside P's channel sum, so it cannot be applied to P after
// the product.  A chunk each of whose parts (8 or 16 tokens) falls by at most
// its share of kChunkSpanMax takes one reference m_c per channel (the middle
// of Lam_c's range):  P_ij = (q_i e^{Lam_i - m}) . (k_j e^{m - Lam_j}), every
// factor within e^{40}, one MMA P^T = Ko Qo^T (M 64 keys, N 64 queries), and
// Qo doubles as the inter term's operand against diag(e^m) S_c.  Other chunks
// form four query blocks of 16 (the secondary chunking of gated linear
// attention): block I takes the reference
// r_I = Lam at its first token, and its scores against every key j up to its
// own last token are one product of scaled operands,
//   P[I, j] = (q_i * e^{Lam_i - r_I}) . (k_j * e^{r_I - Lam_j}),
// where both factors are <= 1 for keys of earlier blocks, and the key factor
// of the block's own keys is at most e^{span} (span = r_I - Lam at the block's
// last token).  So each query block needs its own scaled copy of the keys,
// K^(I) (rows 0 .. 16 I + 15), and the scores are four MMAs
// P^T[:, 16 I ..] = K^(I) Qh_I^T (M = 64 keys, N = 16 queries).  A block whose
// span exceeds kDiagSpanMax in some channel (a decay stronger than e^-5 per
// token on average) would overflow those factors: its key factors are capped,
// and its 16 x 16 diagonal scores are recomputed exactly on the CUDA cores.
//
// Per chunk the MMAs are (D = d_k = d_v; blocked form, the one-reference
// form in brackets):
//   P^T_I = K^(I) Qh_I^T                 M 64, N 16, K D   (x4)  [Ko Qo^T, N 64]
//   O     = Qt S_c,  Qt_i = q_i e^{Lam_i} M 64, N D,  K D   [Qo diag(e^m) S_c]
//   S    += Kt^T V,  Kt_j = k_j e^{Lam_end - Lam_j}   M D, N D, K 64
//   O    += P V                          M 64, N D,  K 64
// and the state chain (a warpgroup) copies S_c (row c scaled by e^{m_c} in
// the one-reference form) to bf16 for the inter term and multiplies row c of
// S by e^{Lam_end,c} in TMEM before the update adds to it.  One CTA carries
// one segment of a (b, h) sequence; with a workspace, a state pass first forms
// the earlier segments' own states, which each segment folds into its
// incoming state.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
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
extern "C" int la_trace_read_cg(long long *out) {
  return (int)cudaMemcpyFromSymbol(out, la::g_trace, sizeof(la::g_trace));
}
#endif

namespace la {
namespace {
using namespace tc;

// Largest within-block decay span (in log space) whose key factors e^{span}
// stay far from fp32 and bf16 overflow in the factored scores.
constexpr float kDiagSpanMax = 80.f;
// Largest fall of Lam through a chunk (per key channel) for which the chunk
// takes one reference point per channel instead of one per 16-token block:
// its query and key factors then stay within e^{40}.  A chunk takes it when
// every part of it (8 or 16 tokens) falls by at most its share of that.
constexpr float kChunkSpanMax = 80.f;

// Warp roles: 0 TMA, 1 MMA, 2..11 PREP (320 threads), 12..15 EPI (P and O
// epilogues), 16..19 ST (the state chain).  The two TMEM warpgroups start at a
// multiple of four warps, so warp w reaches TMEM lanes 32 (w % 4) ..
constexpr int kThreads = 640;
constexpr int W_TMA = 0, W_MMA = 1, W_PREP = 2, W_EPI = 12, W_ST = 16;
constexpr int kPrepThreads = (W_EPI - W_PREP) * 32;
constexpr uint32_t BAR_PREP = 1, BAR_EPI = 2, BAR_ST = 3;

template <int D>
struct CgSmem {
  // d = 64 has room for two log decay tiles, loaded by TMA ahead of PREP (LAPF).
  static constexpr int NST = D == 64 ? 4 : 2;   // q | k | v stages
  static constexpr bool LAPF = D == 64;
  static constexpr int NX = D == 64 ? 2 : 1;    // X buffers: Qt and K^(I) (blocks), or Ko
  static constexpr int NP = D == 64 ? 2 : 1;    // bf16 P tiles
  static constexpr int NO = 1;                  // O staging tile (d = 64: room for a fourth stage)
  static constexpr uint32_t TILE = 64 * D * 2;  // [64 tokens][D] bf16 in D/64 boxes of 8 KB
  static constexpr uint32_t STAGE = 3 * TILE;
  // K^(I) region: K^(0) rows 0..15, K^(1) 16..47, K^(2) 48..95, K^(3)
  // 96..159; each MMA reads 64 rows from its copy's first (rows past a copy's
  // keys are masked out of P), the last copy's exactly.  The one-reference
  // form keeps its Ko in rows 0..63.
  static constexpr int KROWS = 160;
  static constexpr uint32_t KBOX = KROWS * 128;  // one 64-channel box of the region
  static constexpr uint32_t XBUF = TILE + (D / 64) * KBOX;  // Qt, then the K^(I) region (Ko: rows 0..63)
  static constexpr uint32_t S_BLOCK = D * 128;              // [D][64] bf16 block of S
  static constexpr uint32_t OFF_X = NST * STAGE;
  static constexpr uint32_t OFF_P = OFF_X + NX * XBUF;      // [64 keys][64 queries] bf16
  static constexpr uint32_t OFF_S = OFF_P + NP * 8192;
  static constexpr uint32_t OFF_O = OFF_S + (D / 64) * S_BLOCK;
  static constexpr uint32_t OFF_DEC = OFF_O + NO * TILE;    // [NST][D] e^{Lam_end,c}
  // PREP items are (block, channel pair, part): parts of 8 tokens at d = 64, whole
  // 16-token blocks at d = 128, so that either has 256 items.
  static constexpr int PARTS = D == 64 ? 2 : 1;
  static constexpr uint32_t OFF_TOT = OFF_DEC + NST * D * 4;  // [4 PARTS][D] part sums
  static constexpr uint32_t OFF_FIRST = OFF_TOT + 4 * PARTS * D * 4;  // [4][D] first log decays
  static constexpr uint32_t LA_TILE = 64 * D * 4;          // [64 tokens][D] fp32 log decays
  static constexpr uint32_t OFF_LA = OFF_FIRST + 4 * D * 4;  // LAPF: [2] log decay tiles
  static constexpr uint32_t OFF_EX = OFF_LA + (LAPF ? 2 * LA_TILE : 0);  // [16][16] exact diagonal scores
  static constexpr uint32_t OFF_FLAG = OFF_EX + 256 * 4;    // [NST] span exceeded
  static constexpr uint32_t OFF_MODE = OFF_FLAG + 16;       // [NST] one reference (1) or blocks (0)
  static constexpr uint32_t OFF_EM = OFF_MODE + 16;         // [NST][D] e^{m}: the state's row scale
  static constexpr uint32_t OFF_BAR = OFF_EM + NST * D * 4;
  static constexpr int NBAR = 3 * NST + NX + 2 + NP + 2 + 2 + 2 + 1 + 4;
  static constexpr uint32_t OFF_CTL = OFF_BAR + 8 * NBAR;
  static constexpr int kTraceShrink = D == 64 ? 1 : 16;  // trace builds: chunks kept
  static constexpr uint32_t OFF_TRC = OFF_CTL + 64;
  static constexpr uint32_t BYTES = OFF_TRC + trace_smem_bytes(kTraceShrink);
  static_assert(STAGE % 1024 == 0 && OFF_X % 1024 == 0 && XBUF % 1024 == 0 &&
                    OFF_P % 1024 == 0 && OFF_S % 1024 == 0 && OFF_O % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  static_assert(BYTES <= 232448, "exceeds the per-block shared memory limit");
  // TMEM columns: P^T x2 (64 each), O x2 (D each), S (D).
  static constexpr uint32_t T_P = 0, T_O = 128, T_S = 128 + 2 * D, T_COLS = 512;
  static_assert(T_S + D <= T_COLS, "TMEM budget");
};

// First row of K^(I) in the K^(I) region.
__host__ __device__ constexpr int k_row0(int I) { return I == 0 ? 0 : I == 1 ? 16 : I == 2 ? 48 : 96; }

struct CgParams {
  int H, L, BH, n_chunks;
  // Segments of a sequence (one without a workspace): the first has
  // first_chunks chunks, the others seg_chunks each (the last may have fewer).
  int first_chunks, seg_chunks, n_seg;
  // The state pass cuts every segment but the last into state_parts pieces,
  // one block each; a sequence has n_slot = (n_seg - 1) state_parts + 1
  // workspace slots (the last for a copy of S0).
  int state_parts, n_slot;
  const float *log_alpha;  // [BH][L][D]
  const __nv_bfloat16 *q, *k;
  const float *S0;
  float *S_final;
  float *ws_state;         // [BH][n_slot][D][D]: slot j < n_slot-1 = piece j's own state;
                           // slot n_slot-1 = a copy of S0 when S_final is S0
  float *ws_logdec;        // [BH][n_slot][D]: piece j's total log decay per key channel
  unsigned int *err;
};

// First chunk and chunk count of segment seg.
__device__ __forceinline__ void seg_range(const CgParams &p, int seg, int &c0, int &n) {
  c0 = seg == 0 ? 0 : p.first_chunks + (seg - 1) * p.seg_chunks;
  n = min(seg == 0 ? p.first_chunks : p.seg_chunks, p.n_chunks - c0);
}

// First chunk and chunk count of state-pass piece j (part j % state_parts of
// segment j / state_parts, the parts as even as whole chunks allow).
__device__ __forceinline__ void piece_range(const CgParams &p, int j, int &c0, int &n) {
  int s0, sn;
  seg_range(p, j / p.state_parts, s0, sn);
  const int part = j % p.state_parts, base = sn / p.state_parts, rem = sn % p.state_parts;
  c0 = s0 + part * base + min(part, rem);
  n = base + (part < rem ? 1 : 0);
}

// Byte offset of element (row, col) in a bf16 tile of 128-byte swizzled rows
// whose 64-column boxes are `box` bytes apart.
__device__ __forceinline__ uint32_t tile_off(int row, int col, uint32_t box) {
  return (uint32_t)(col >> 6) * box + sw128_offset((uint32_t)row, (uint32_t)(col & 63));
}

__device__ __forceinline__ void st_bf16(unsigned char *p, float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  *reinterpret_cast<__nv_bfloat16 *>(p) = b;
}

__device__ __forceinline__ float log_alpha_at(const CgParams &p, size_t bhL, int tok, int ch,
                                              int D) {
  return tok < p.L ? p.log_alpha[(bhL + tok) * D + ch] : 0.f;  // padding decays nothing
}

// Exact scores of the four 16 x 16 diagonal blocks of chunk c, written over
// the factored ones in the bf16 P tile (row = key, column = query): for a
// chunk whose within-block decay span exceeds kDiagSpanMax somewhere.  Rare:
// one thread per channel forms its terms q_ic k_jc e^{Lam_ic - Lam_jc} and
// adds them into a shared [16][16] table.  Called by the 128 EPI threads.
template <int D, bool PHI>
__device__ __noinline__ void exact_diagonal(const CgParams &p, int bh, int tok0, unsigned char *pt,
                                            float *ex, int t) {
  const size_t bhL = (size_t)bh * p.L;
  for (int I = 0; I < 4; ++I) {
    for (int x = t; x < 256; x += 128) ex[x] = 0.f;
    named_bar_sync(BAR_EPI, 128);
    if (t < D) {
      float lam[16], qv[16], kv[16];
      float run = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int tok = tok0 + 16 * I + i;
        run += log_alpha_at(p, bhL, tok, t, D);
        lam[i] = run;
        float a = 0.f, b = 0.f;
        if (tok < p.L) {
          a = __bfloat162float(p.q[(bhL + tok) * D + t]);
          b = __bfloat162float(p.k[(bhL + tok) * D + t]);
        }
        qv[i] = PHI ? elu1_fast(a) : a;
        kv[i] = PHI ? elu1_fast(b) : b;
      }
      for (int i = 0; i < 16; ++i)
        for (int j = 0; j <= i; ++j)
          atomicAdd(&ex[i * 16 + j], qv[i] * kv[j] * __expf(lam[i] - lam[j]));
    }
    named_bar_sync(BAR_EPI, 128);
    for (int x = t; x < 256; x += 128) {
      const int i = x >> 4, j = x & 15;
      if (j <= i)
        st_bf16(pt + sw128_offset(16 * I + j, 16 * I + i), ex[x]);
    }
    named_bar_sync(BAR_EPI, 128);
  }
}

template <int D, bool PHI>
__global__ void __launch_bounds__(kThreads, 1)
channel_gate_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmO,
                       const __grid_constant__ CUtensorMap tmA, CgParams p) {
  using SM = CgSmem<D>;
  constexpr int NST = SM::NST, NX = SM::NX, NP = SM::NP, NO = SM::NO;
  extern __shared__ __align__(1024) unsigned char smem[];
  float *dec = reinterpret_cast<float *>(smem + SM::OFF_DEC);
  float *hsum = reinterpret_cast<float *>(smem + SM::OFF_TOT);
  float *first = reinterpret_cast<float *>(smem + SM::OFF_FIRST);
  float *ex = reinterpret_cast<float *>(smem + SM::OFF_EX);
  volatile uint32_t *flag = reinterpret_cast<volatile uint32_t *>(smem + SM::OFF_FLAG);
  volatile uint32_t *mode = reinterpret_cast<volatile uint32_t *>(smem + SM::OFF_MODE);
  float *emv = reinterpret_cast<float *>(smem + SM::OFF_EM);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::OFF_BAR);
  uint64_t *empty = full + NST;
  uint64_t *prep = empty + NST;     // [NST] scaled operands, factors and flag ready
  uint64_t *xfree = prep + NST;     // [NX] the MMAs reading an X buffer are done
  uint64_t *p_full = xfree + NX;    // [2] P^T in TMEM
  uint64_t *p_ready = p_full + 2;   // [NP] bf16 P in shared memory
  uint64_t *o_full = p_ready + NP;  // [2] O complete in TMEM
  uint64_t *o_free = o_full + 2;    // [2] O TMEM buffer read
  uint64_t *s_ready = o_free + 2;   // bf16 S_c in smem, TMEM S = diag(e^{Lam_end}) S_c
  uint64_t *s_done = s_ready + 1;   // the update of chunk c (and every MMA before it) done
  uint64_t *drain = s_done + 1;
  uint64_t *la_full = drain + 1;    // LAPF: [2] log decay tile landed
  uint64_t *la_empty = la_full + 2; // LAPF: [2] log decay tile read by PREP
  Ctl *ctl = reinterpret_cast<Ctl *>(smem + SM::OFF_CTL);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Grid (B*H, segments): a CTA runs one segment of a sequence from its
  // incoming state.
  const int bh = blockIdx.x, seg = blockIdx.y;
  int cbase, nc;
  seg_range(p, seg, cbase, nc);
  const size_t bhL = (size_t)bh * p.L;
  // The incoming state: S0 folded with the earlier segments' own states (their
  // per-channel decays applied), for a segment after the first.  S0 is read
  // from the state pass's copy of it when S_final is the same buffer, so that
  // the last segment cannot overwrite it before another reads it.
  const bool alias0 = p.n_seg > 1 && p.S0 && p.S0 == p.S_final;
  const float *slots = p.n_seg > 1 ? p.ws_state + (size_t)bh * p.n_slot * D * D : nullptr;
  const float *S_base = alias0 ? slots + (size_t)(p.n_slot - 1) * D * D
                               : (p.S0 ? p.S0 + (size_t)bh * D * D : nullptr);
  const bool needs_pass = p.n_seg > 1 && (seg > 0 || alias0);
  const bool last_seg = seg == p.n_seg - 1;
  const bool trace_on = blockIdx.x == 0 && blockIdx.y == 0;
  const long long t0 = clock64();
  (void)trace_on;
  (void)t0;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&prep[s], 1);
      flag[s] = 0;
    }
    for (int i = 0; i < NX; ++i) mbar_init(&xfree[i], 1);
    for (int i = 0; i < NP; ++i) mbar_init(&p_ready[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 1);
    }
    mbar_init(s_ready, 1);
    mbar_init(s_done, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&la_full[i], 1);
      mbar_init(&la_empty[i], 1);
    }
    ctl->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(&ctl->tmem_base, SM::T_COLS);
    tmem_relinquish();
  }
  LA_TRACE_TABLE(smem + SM::OFF_TRC, SM::kTraceShrink);
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
      if constexpr (SM::LAPF) tma_prefetch_desc(&tmA);
      int issued = 0, la_issued = 0;
      for (int c = 0; c < nc; ++c) {
        const int s = c % NST;
        if constexpr (SM::LAPF) {  // the chunk's log decays, once PREP has read the buffer's last
          const int lb = c & 1;
          if (c >= 2 && !wait1(&la_empty[lb], ((c >> 1) - 1) & 1, ctl, p.err, KID_CHANNEL_GATE_TC, 2))
            break;
          mbar_arrive_expect_tx(&la_full[lb], SM::LA_TILE);
          tma_load_3d(smem + SM::OFF_LA + lb * SM::LA_TILE, &tmA, &la_full[lb], 0, (cbase + c) * CH, bh);
          la_issued = c + 1;
        }
        if (c >= NST && !wait1(&empty[s], ((c / NST) - 1) & 1, ctl, p.err, KID_CHANNEL_GATE_TC, 1))
          break;
        unsigned char *stg = smem + s * SM::STAGE;
        mbar_arrive_expect_tx(&full[s], SM::STAGE);
        const int tok = (cbase + c) * CH;
        for (int b = 0; b < D / BOX; ++b) {
          tma_load_3d(stg + b * BOX_BYTES, &tmQ, &full[s], b * BOX, tok, bh);
          tma_load_3d(stg + SM::TILE + b * BOX_BYTES, &tmK, &full[s], b * BOX, tok, bh);
          tma_load_3d(stg + 2 * SM::TILE + b * BOX_BYTES, &tmV, &full[s], b * BOX, tok, bh);
        }
        issued = c + 1;
        LA_TRACE_EVENT(trace_on, t0, 0, c);
      }
      if (*(volatile uint32_t *)&ctl->abort) {
        for (int c = max(0, issued - NST); c < issued; ++c) drain_wait(&full[c % NST], (c / NST) & 1);
        for (int c = max(0, la_issued - 2); c < la_issued; ++c) drain_wait(&la_full[c & 1], (c >> 1) & 1);
      }
      for (int c = max(0, nc - NST); c < nc; ++c) drain_wait(&empty[c % NST], (c / NST) & 1);
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nc > 0) {
      constexpr uint32_t id_p = idesc_bf16_f32(64, 16, false, false);
      constexpr uint32_t id_p64 = idesc_bf16_f32(64, 64, false, false);
      constexpr uint32_t id_qs = idesc_bf16_f32(64, D, false, true);
      constexpr uint32_t id_kv = idesc_bf16_f32(D, D, true, true);
      constexpr uint32_t id_pv = idesc_bf16_f32(64, D, true, true);
      constexpr uint32_t HI = smem_desc_sw128_hi(1024);
      const uint32_t sbase = smem_u32(smem);
      const uint32_t dKM = smem_desc_sw128_lo(sbase, 16);           // K-major rows
      const uint32_t dMN = smem_desc_sw128_lo(sbase, BOX_BYTES);    // MN-major, 8 KB blocks
      const uint32_t dMS = smem_desc_sw128_lo(sbase, SM::S_BLOCK);  // MN-major state blocks
      auto at = [](uint32_t d, uint32_t off) { return d + (off >> 4); };
      // P^T of chunk c: one MMA over the one-reference operands, or four, one
      // per query block.  one_ref keeps each chunk's form (bit c % 32) for its
      // chain step, which reads Qo from the stage in the one-reference form.
      uint32_t one_ref = 0;
      auto issue_p = [&](int c) {
        const uint32_t qo = (c % NST) * SM::STAGE;
        const uint32_t xo = SM::OFF_X + (c % NX) * SM::XBUF + SM::TILE;
        if (mode[c % NST]) {
          one_ref |= 1u << (c & 31);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_w(tmem + SM::T_P + 64 * (c & 1),
                       at(dKM, xo + (kk / 4) * SM::KBOX + 32 * (kk % 4)),
                       at(dKM, qo + (kk / 4) * BOX_BYTES + 32 * (kk % 4)), HI, id_p64, kk > 0);
          mma_commit(&p_full[c & 1]);
          return;
        }
        one_ref &= ~(1u << (c & 31));
        for (int I = 0; I < 4; ++I) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_w(tmem + SM::T_P + 64 * (c & 1) + 16 * I,
                       at(dKM, xo + (kk / 4) * SM::KBOX + k_row0(I) * 128 + 32 * (kk % 4)),
                       at(dKM, qo + (kk / 4) * BOX_BYTES + 16 * I * 128 + 32 * (kk % 4)), HI, id_p,
                       kk > 0);
        }
        mma_commit(&p_full[c & 1]);
      };
      // Three streams of MMA work, each in chunk order, issued as their inputs
      // become ready (non-blocking tests), so that no stream waits behind
      // another's inputs; the oldest work is tested first (P V releases a
      // stage for the next loads):
      //   P^T of chunk kp: its operands prepared; its TMEM buffer was read by
      //     the P epilogue of chunk kp - 2, whose P V has been issued;
      //   chain step kc (O = Qt S_c, or Qo diag(e^m) S_c, S += Kt^T V): after P^T of kc, so that
      //     the commit freeing the X buffer covers it; O's buffer read;
      //   P V of chunk km: after its chain step (which starts O).
      int kp = 0, kc = 0, km = 0;
      bool ok = true;
      uint64_t idle_since = 0;
      uint32_t idle = 0;
      while (ok && km < nc) {
        bool did = false;
        if (km < kc && mbar_test(&p_ready[km % NP], (km / NP) & 1)) {
          tc_fence_after();
          const int s = km % NST;
          const uint32_t vo = s * SM::STAGE + 2 * SM::TILE, po = SM::OFF_P + 8192 * (km % NP);
          const uint32_t o_t = tmem + SM::T_O + D * (km & 1);
#pragma unroll
          for (int kk = 0; kk < CH / 16; ++kk)  // O += P V
            mma_bf16_w(o_t, at(dMN, po + 2048 * kk), at(dMN, vo + 2048 * kk), HI, id_pv, 1u);
          mma_commit(&o_full[km & 1]);
          mma_commit(&empty[s]);
          LA_TRACE_EVENT(trace_on, t0, 5, km);
          ++km;
          did = true;
        }
        if (kc < kp && mbar_test(s_ready, kc & 1) &&
            (kc < 2 || mbar_test(&o_free[kc & 1], ((kc >> 1) - 1) & 1))) {
          tc_fence_after();
          const int s = kc % NST, xb = kc % NX;
          const uint32_t ko = s * SM::STAGE + SM::TILE, vo = ko + SM::TILE;
          const uint32_t xo = (one_ref >> (kc & 31)) & 1u ? s * SM::STAGE : SM::OFF_X + xb * SM::XBUF;
          const uint32_t o_t = tmem + SM::T_O + D * (kc & 1);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)  // O = Qt S_c
            mma_bf16_w(o_t, at(dKM, xo + (kk / 4) * BOX_BYTES + 32 * (kk % 4)),
                       at(dMS, SM::OFF_S + 2048 * kk), HI, id_qs, kk > 0);
#pragma unroll
          for (int kk = 0; kk < CH / 16; ++kk)  // S += Kt^T V
            mma_bf16_w(tmem + SM::T_S, at(dMN, ko + 2048 * kk), at(dMN, vo + 2048 * kk), HI,
                       id_kv, 1u);
          mma_commit(s_done);
          mma_commit(&xfree[xb]);
          LA_TRACE_EVENT(trace_on, t0, 4, kc);
          ++kc;
          did = true;
        }
        if (kp < nc && kp <= km + 1 && mbar_test(&prep[kp % NST], (kp / NST) & 1)) {
          tc_fence_after();
          issue_p(kp);
          LA_TRACE_EVENT(trace_on, t0, 3, kp);
          ++kp;
          did = true;
        }
        if (did) {
          idle = 0;
          idle_since = 0;
        } else if (++idle == 256) {  // spin (a sleep delays the reaction to a barrier
                                        // by far more than asked); bounded: give up after the limit
          idle = 0;
          const uint64_t now = global_timer_ns();
          if (idle_since == 0) {
            idle_since = now;
          } else if (now - idle_since > kWaitNs || *(volatile uint32_t *)&ctl->abort) {
            if (!*(volatile uint32_t *)&ctl->abort) {
              atomicExch(&ctl->abort, 1u);
              record_device_error(p.err, KID_CHANNEL_GATE_TC, 3);
            }
            ok = false;
          }
        }
      }
      // Every issued MMA finishes before TMEM is released (on the normal path
      // the consumers have already observed them).
      mma_commit(drain);
      drain_wait(drain, 0);
    }
  } else if (warp >= W_PREP && warp < W_EPI) {
    // ------------------------------------------------------------ PREP
    const int t = tid - W_PREP * 32;
    // Items (block I, channel pair cp, part hh): TPI tokens of two adjacent
    // channels, so that every shared-memory access moves a bf16 pair and the
    // swizzled address is formed once per row for both; one item per thread,
    // the same in every chunk.  Consecutive threads take consecutive pairs
    // (coalesced log decay loads, one tile row per warp).  An item's log
    // decays, loaded for the part sums, stay in registers for its pass.
    constexpr int PARTS = SM::PARTS, TPI = 16 / PARTS;
    constexpr int NPAIR = D / 2, NITEM = 4 * PARTS * NPAIR;
    static_assert(NITEM <= kPrepThreads, "one item per PREP thread");
    const bool has_item = t < NITEM;
    const int cp = t % NPAIR, hh = (t / NPAIR) % PARTS, c0 = 2 * cp;
    // Blocks in the order 0, 1, 3, 2: the warps of blocks 0 and 3 (and of 1
    // and 2) share a scheduler, which evens out the K^(J) copies (3 - I a
    // token).  Threads without an item keep an unused I in range.
    int I = (t / (PARTS * NPAIR)) & 3;
    I ^= I >> 1;
    auto load_item = [&](int tok0, float2 (&a)[TPI]) {
#pragma unroll
      for (int i = 0; i < TPI; ++i) {
        const int tok = tok0 + 16 * I + TPI * hh + i;
        a[i] = tok < p.L ? *reinterpret_cast<const float2 *>(p.log_alpha + (bhL + tok) * D + c0)
                         : make_float2(0.f, 0.f);  // padding decays nothing
      }
    };
    // LAPF: the chunk's log decays come as a TMA tile (zero past L: padding
    // decays nothing), which every thread waits for itself.
    auto read_item = [&](const float *labuf, float2 (&a)[TPI]) {
#pragma unroll
      for (int i = 0; i < TPI; ++i)
        a[i] = *reinterpret_cast<const float2 *>(labuf + (16 * I + TPI * hh + i) * D + c0);
    };
    float2 ai[TPI];
    bool ok = true;
    for (int c = 0; ok && c < nc; ++c) {
      const int s = c % NST, xb = c % NX;
      const int tok0 = (cbase + c) * CH;
      // Part sums and blocks' first log decays: they do not need the stage, so
      // their loads go out while the chunk's tiles are arriving.
      bool la_ok = true;
      if constexpr (SM::LAPF)
        la_ok = wait1(&la_full[c & 1], (c >> 1) & 1, ctl, p.err, KID_CHANNEL_GATE_TC, 6);
      // The one-reference form needs Lam falling through the chunk (log decays
      // <= 0) by at most kChunkSpanMax; each thread tests its own part against
      // its share, so the choice rides on the barrier that publishes the sums.
      bool need_blocks = false;
      if (has_item && la_ok) {
        if constexpr (SM::LAPF)
          read_item(reinterpret_cast<const float *>(smem + SM::OFF_LA + (c & 1) * SM::LA_TILE), ai);
        else
          load_item(tok0, ai);
        float2 sum = make_float2(0.f, 0.f);
        bool rising = false;  // a log decay above zero in the item
#pragma unroll
        for (int i = 0; i < TPI; ++i) {
          sum.x += ai[i].x;
          sum.y += ai[i].y;
          rising = rising || fmaxf(ai[i].x, ai[i].y) > 0.f;
        }
        need_blocks = rising || fmaxf(-sum.x, -sum.y) > kChunkSpanMax / (4 * PARTS);
        *reinterpret_cast<float2 *>(hsum + (PARTS * I + hh) * D + c0) = sum;
        if (hh == 0) *reinterpret_cast<float2 *>(first + I * D + c0) = ai[0];
      }
      // One barrier publishes the part sums, the stage's arrival (its flag
      // reset: the P epilogue of the stage's last chunk is past), the wait for
      // this chunk's X buffer, every thread's wait for its log decays and
      // whether any part needs the blocked form.
      bool fok = true;
      if (t == 0) {
        fok = wait1(&full[s], (c / NST) & 1, ctl, p.err, KID_CHANNEL_GATE_TC, 7);
        if (fok) flag[s] = 0;
        if (fok && c >= NX) fok = wait1(&xfree[xb], ((c / NX) - 1) & 1, ctl, p.err, KID_CHANNEL_GATE_TC, 8);
      }
      __syncwarp();
      const bool blocked = bar_red_or(BAR_PREP, kPrepThreads, need_blocks || !(fok && la_ok));
      if (blocked && *(volatile uint32_t *)&ctl->abort) {  // a wait gave up (it set abort)
        ok = false;
        break;
      }
      LA_TRACE_EVENT(trace_on && t == 0, t0, 1, c);
      // Per channel of the pair: base = the blocks before I, lend = the whole
      // chunk, rnext[J] = r of a later query block J (the blocks before it
      // plus its first token's own log decay), r = the block's first Lam.
      auto block_sums = [&](float2 &base, float2 &lend, float2 (&rnext)[4]) {
        base = make_float2(0.f, 0.f);
        lend = base;
#pragma unroll
        for (int J = 0; J < 4; ++J) {
          float2 tj = make_float2(0.f, 0.f);
#pragma unroll
          for (int h = 0; h < PARTS; ++h) {
            const float2 x = *reinterpret_cast<const float2 *>(hsum + (PARTS * J + h) * D + c0);
            tj.x += x.x;
            tj.y += x.y;
          }
          rnext[J] = lend;
          if (J < I) {
            base.x += tj.x;
            base.y += tj.y;
          }
          lend.x += tj.x;
          lend.y += tj.y;
        }
      };
      LA_TRACE_EVENT(trace_on && t == 0, t0, 9, c);
      if (t == 0) mode[s] = blocked ? 0u : 1u;
      unsigned char *qt = smem + s * SM::STAGE, *kt = qt + SM::TILE;
      unsigned char *xq = smem + SM::OFF_X + xb * SM::XBUF, *xk = xq + SM::TILE;
      // q and k of two channels as bf16 pairs; phi = elu + 1 in packed bf16
      // arithmetic (half the instructions of fp32, one more rounding).
      auto load_qk = [&](uint32_t off, float &qx, float &qy, float &kx, float &ky) {
        uint32_t qw = *reinterpret_cast<const uint32_t *>(qt + off);
        uint32_t kw = *reinterpret_cast<const uint32_t *>(kt + off);
        if (PHI) {
          qw = elu1_bf16x2(qw);
          kw = elu1_bf16x2(kw);
        }
        qx = __uint_as_float(qw << 16), qy = __uint_as_float(qw & 0xffff0000u);
        kx = __uint_as_float(kw << 16), ky = __uint_as_float(kw & 0xffff0000u);
      };
      float2 base, lend, rnext[4];
      block_sums(base, lend, rnext);
      float2 run = base;
      if (hh) {  // the block's first part
        const float2 h0 = *reinterpret_cast<const float2 *>(hsum + (PARTS * I) * D + c0);
        run.x += h0.x;
        run.y += h0.y;
      }
      if (has_item && I == 3 && hh == 0)
        *reinterpret_cast<float2 *>(dec + s * D + c0) = make_float2(__expf(lend.x), __expf(lend.y));
      if (has_item && !blocked) {
        // One reference per channel for the whole chunk, m = the middle of its
        // Lam range: Qo = q e^{Lam_t - m} (it also stands for Qt, the state
        // being stored as diag(e^m) S_c), Ko = k e^{m - Lam_t}, both within
        // e^{kChunkSpanMax / 2}, P^T = Ko Qo^T in one MMA, Kt = Ko e^{lend - m}.
        const float2 l0 = *reinterpret_cast<const float2 *>(first + c0);
        const float2 m = make_float2(0.5f * (l0.x + lend.x), 0.5f * (l0.y + lend.y));
        const float2 eK = make_float2(__expf(lend.x - m.x), __expf(lend.y - m.y));
        if (I == 0 && hh == 0)
          *reinterpret_cast<float2 *>(emv + s * D + c0) = make_float2(__expf(m.x), __expf(m.y));
        // LAPF: the log decays are read again from the tile (kept until the
        // pass ends), so that the loop need not be unrolled to index
        // registers: short code keeps the instruction cache warm.
        const float *la_it = reinterpret_cast<const float *>(smem + SM::OFF_LA + (c & 1) * SM::LA_TILE) +
                             (16 * I + TPI * hh) * D + c0;
        // Two tokens a step, their loads ahead of their stores (a load after
        // a shared-memory store waits for it: the addresses may alias).
#pragma unroll(SM::LAPF ? 1 : TPI / 2)
        for (int i = 0; i < TPI; i += 2) {
          float2 a[2];
          uint32_t qw[2], kw[2], off[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if constexpr (SM::LAPF)
              a[u] = *reinterpret_cast<const float2 *>(la_it + (i + u) * D);
            else
              a[u] = ai[i + u];
            off[u] = tile_off(16 * I + TPI * hh + i + u, c0, BOX_BYTES);
            qw[u] = *reinterpret_cast<const uint32_t *>(qt + off[u]);
            kw[u] = *reinterpret_cast<const uint32_t *>(kt + off[u]);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            run.x += a[u].x;
            run.y += a[u].y;
            if (PHI) {
              qw[u] = elu1_bf16x2(qw[u]);
              kw[u] = elu1_bf16x2(kw[u]);
            }
            const float qx = __uint_as_float(qw[u] << 16), qy = __uint_as_float(qw[u] & 0xffff0000u);
            const float kx = __uint_as_float(kw[u] << 16), ky = __uint_as_float(kw[u] & 0xffff0000u);
            const float dx = run.x - m.x, dy = run.y - m.y;
            const float kox = kx * __expf(-dx), koy = ky * __expf(-dy);
            *reinterpret_cast<uint32_t *>(qt + off[u]) = pack_bf16(qx * __expf(dx), qy * __expf(dy));  // Qo
            *reinterpret_cast<uint32_t *>(xk + tile_off(16 * I + TPI * hh + i + u, c0, SM::KBOX)) =
                pack_bf16(kox, koy);                                                                // Ko
            *reinterpret_cast<uint32_t *>(kt + off[u]) = pack_bf16(kox * eK.x, koy * eK.y);         // Kt
          }
        }
      } else if (has_item) {
        if (I == 0 && hh == 0) *reinterpret_cast<float2 *>(emv + s * D + c0) = make_float2(1.f, 1.f);
#pragma unroll
        for (int J = 0; J < 4; ++J) {
          if (J > I) {
            const float2 f = *reinterpret_cast<const float2 *>(first + J * D + c0);
            rnext[J].x += f.x;
            rnext[J].y += f.y;
          }
        }
        const float2 fI = *reinterpret_cast<const float2 *>(first + I * D + c0);
        const float2 r = make_float2(base.x + fI.x, base.y + fI.y);
        const float erx = __expf(r.x), ery = __expf(r.y);
        // Every key factor e^{x - Lam_t} (x = lend or a later block's r) is
        // e^{x - r} e^{r - Lam_t}: the first factor is the item's, so a token
        // takes one exponential for all its key copies and one for its query,
        // as long as |r - Lam_t| and x - r stay within kDiagSpanMax (always,
        // for log decays <= 0 and blocks whose span is within it).  An item
        // past that takes every factor directly, in a loop kept short so that
        // the rare case adds little code.
        const float2 eL = make_float2(__expf(lend.x - r.x), __expf(lend.y - r.y));
        float2 eJ[4];
        bool item_fast = fmaxf(lend.x - r.x, lend.y - r.y) <= kDiagSpanMax;
#pragma unroll
        for (int J = 0; J < 4; ++J) {
          if (J > I) {
            eJ[J] = make_float2(__expf(rnext[J].x - r.x), __expf(rnext[J].y - r.y));
            item_fast = item_fast && fmaxf(rnext[J].x - r.x, rnext[J].y - r.y) <= kDiagSpanMax;
          }
        }
        {
          float2 rr = run;
          float mx = 0.f;
#pragma unroll
          for (int i = 0; i < TPI; ++i) {
            rr.x += ai[i].x;
            rr.y += ai[i].y;
            mx = fmaxf(mx, fmaxf(fabsf(r.x - rr.x), fabsf(r.y - rr.y)));
          }
          item_fast = item_fast && mx <= kDiagSpanMax;
        }
        if (item_fast) {
#pragma unroll
          for (int i = 0; i < TPI; ++i) {
            run.x += ai[i].x;
            run.y += ai[i].y;
            const int row = 16 * I + TPI * hh + i;
            const uint32_t off = tile_off(row, c0, BOX_BYTES);
            float qx, qy, kx, ky;
            load_qk(off, qx, qy, kx, ky);
            const float dx = r.x - run.x, dy = r.y - run.y;  // the block's span so far
            const float qhx = qx * __expf(-dx), qhy = qy * __expf(-dy);                 // <= 1
            *reinterpret_cast<uint32_t *>(qt + off) = pack_bf16(qhx, qhy);              // Qh
            *reinterpret_cast<uint32_t *>(xq + off) = pack_bf16(qhx * erx, qhy * ery);  // Qt
            const float kux = kx * __expf(dx), kuy = ky * __expf(dy);
            *reinterpret_cast<uint32_t *>(xk + tile_off(k_row0(I) + row, c0, SM::KBOX)) =  // K^(I)
                pack_bf16(kux, kuy);
            *reinterpret_cast<uint32_t *>(kt + off) = pack_bf16(kux * eL.x, kuy * eL.y);    // Kt
#pragma unroll
            for (int J = 0; J < 4; ++J)                                                  // K^(J), J > I
              if (J > I)
                *reinterpret_cast<uint32_t *>(xk + tile_off(k_row0(J) + row, c0, SM::KBOX)) =
                    pack_bf16(kux * eJ[J].x, kuy * eJ[J].y);
          }
        } else {
#pragma unroll 1
          for (int i = 0; i < TPI; ++i) {
            const int row = 16 * I + TPI * hh + i, tok = tok0 + row;
            const float2 a = tok < p.L
                                 ? *reinterpret_cast<const float2 *>(p.log_alpha + (bhL + tok) * D + c0)
                                 : make_float2(0.f, 0.f);
            run.x += a.x;
            run.y += a.y;
            const uint32_t off = tile_off(row, c0, BOX_BYTES);
            float qx, qy, kx, ky;
            load_qk(off, qx, qy, kx, ky);
            const float qhx = qx * __expf(run.x - r.x), qhy = qy * __expf(run.y - r.y);
            *reinterpret_cast<uint32_t *>(qt + off) = pack_bf16(qhx, qhy);              // Qh
            *reinterpret_cast<uint32_t *>(xq + off) = pack_bf16(qhx * erx, qhy * ery);  // Qt
            *reinterpret_cast<uint32_t *>(kt + off) =                                   // Kt
                pack_bf16(kx * __expf(lend.x - run.x), ky * __expf(lend.y - run.y));
            *reinterpret_cast<uint32_t *>(xk + tile_off(k_row0(I) + row, c0, SM::KBOX)) =  // K^(I)
                pack_bf16(kx * __expf(fminf(r.x - run.x, kDiagSpanMax)),
                          ky * __expf(fminf(r.y - run.y, kDiagSpanMax)));
#pragma unroll
            for (int J = 0; J < 4; ++J)                                                // K^(J), J > I
              if (J > I)
                *reinterpret_cast<uint32_t *>(xk + tile_off(k_row0(J) + row, c0, SM::KBOX)) =
                    pack_bf16(kx * __expf(rnext[J].x - run.x), ky * __expf(rnext[J].y - run.y));
          }
        }
        // The block's largest span sits at its last token (its last part).
        if (hh == PARTS - 1 && fmaxf(r.x - run.x, r.y - run.y) > kDiagSpanMax) flag[s] = 1u;
      }
      fence_proxy_async_smem();
      named_bar_sync(BAR_PREP, kPrepThreads);
      if (t == 0) {
        mbar_arrive(&prep[s]);
        if constexpr (SM::LAPF) mbar_arrive(&la_empty[c & 1]);  // the tile may be refilled
      }
      LA_TRACE_EVENT(trace_on && t == 0, t0, 2, c);
    }
  } else if (warp >= W_EPI && warp < W_ST) {
    // ------------------------------------------------------------ EPI: P and O epilogues
    const int t = tid - W_EPI * 32;
    const int quarter = warp & 3;
    const int row = acc_row<64>(quarter, lane);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    auto ewait = [&](uint64_t *bar, uint32_t par, uint32_t site) {
      return wait_wg(bar, par, ctl, p.err, KID_CHANNEL_GATE_TC, site, BAR_EPI);
    };
    auto p_epilogue = [&](int c) -> bool {
      const int s = c % NST;
      if (!ewait(&p_full[c & 1], (c >> 1) & 1, 9)) return false;
      if (!ewait(&prep[s], (c / NST) & 1, 10)) return false;
      if (NP == 1 && c >= 1 && !ewait(&o_full[(c - 1) & 1], ((c - 1) >> 1) & 1, 11)) return false;
      tc_fence_after();
      unsigned char *pt = smem + SM::OFF_P + 8192 * (c % NP);
      uint32_t r[2][32];
      __syncwarp();
      tmem_ld32(tmem + lane_off + SM::T_P + 64 * (c & 1), r[0]);
      tmem_ld32(tmem + lane_off + SM::T_P + 64 * (c & 1) + 32, r[1]);
      tmem_ld_wait();
      if (row >= 0) {  // row = key j; column = query i; causal: keep i >= j
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = 32 * h + 8 * q8 + 2 * e;
              w4[e] = pack_bf16(i >= row ? __uint_as_float(r[h][8 * q8 + 2 * e]) : 0.f,
                                i + 1 >= row ? __uint_as_float(r[h][8 * q8 + 2 * e + 1]) : 0.f);
            }
            const int chunk16 = 4 * h + q8;
            *reinterpret_cast<uint4 *>(pt + row * 128 + ((chunk16 ^ (row & 7)) << 4)) =
                make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      if (flag[s]) {
        named_bar_sync(BAR_EPI, 128);
        exact_diagonal<D, PHI>(p, bh, (cbase + c) * CH, pt, ex, t);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_EPI, 128);
      if (t == 0) mbar_arrive(&p_ready[c % NP]);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 6, c);
      return true;
    };
    auto o_epilogue = [&](int c) -> bool {
      const int b = c & 1;
      if (!ewait(&o_full[b], (c >> 1) & 1, 12)) return false;
      tc_fence_after();
      if (t == 0) {
        if (NO == 2) tma_store_wait_read<1>();
        else tma_store_wait_read<0>();
      }
      __syncwarp();
      named_bar_sync(BAR_EPI, 128);
      unsigned char *o_sm = smem + SM::OFF_O + (c % NO) * SM::TILE;
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(tmem + lane_off + SM::T_O + D * b + col, r);
        tmem_ld_wait();
        if (row >= 0) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              pk[j] = pack_bf16(__uint_as_float(r[16 * h + 2 * j]), __uint_as_float(r[16 * h + 2 * j + 1]));
            st_row16(o_sm, BOX_BYTES, row, col + 16 * h, pk);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_EPI, 128);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 7, c);
      if (t == 0) {
        mbar_arrive(&o_free[b]);
        for (int bb = 0; bb < D / BOX; ++bb)
          tma_store_3d(&tmO, o_sm + bb * BOX_BYTES, bb * BOX, (cbase + c) * CH, bh);
        tma_store_commit();
      }
      return true;
    };
    bool ok = true;
    for (int c = 0; ok && c < nc; ++c) {
      ok = p_epilogue(c);
      if (ok && c >= 1) ok = o_epilogue(c - 1);
    }
    if (ok && nc > 0) o_epilogue(nc - 1);
    if (t == 0) tma_store_wait_all();
  } else if (warp >= W_ST) {
    // ------------------------------------------------------------ ST: the state chain
    const int t = tid - W_ST * 32;
    const int quarter = warp & 3;
    const int srow = acc_row<D>(quarter, lane);  // key channel
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    auto swait = [&](uint64_t *bar, uint32_t par, uint32_t site) {
      return wait_wg(bar, par, ctl, p.err, KID_CHANNEL_GATE_TC, site, BAR_ST);
    };
    // The incoming state (or zeros) into TMEM.  With segments this kernel is a
    // programmatic dependent of the state pass, and only this warpgroup reads
    // its results, so only it waits, and only where it needs them: first
    // segments run alongside the state pass.
    if (needs_pass) pdl_wait_previous();
    const float *ld_row = p.n_seg > 1 ? p.ws_logdec + (size_t)bh * p.n_slot * D + srow : nullptr;
#pragma unroll 1
    for (int col = 0; col < D; col += 32) {
      float acc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = 0.f;
      if (srow >= 0 && S_base) {
        const float4 *src = reinterpret_cast<const float4 *>(S_base + (size_t)srow * D + col);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 f = src[j];
          acc[4 * j] = f.x;
          acc[4 * j + 1] = f.y;
          acc[4 * j + 2] = f.z;
          acc[4 * j + 3] = f.w;
        }
      }
      if (srow >= 0) {
        for (int j2 = 0; j2 < seg * p.state_parts; ++j2) {  // S <- diag(e^{A_j}) S + dS_j, pieces in order
          const float e = __expf(ld_row[(size_t)j2 * D]);
          const float4 *src =
              reinterpret_cast<const float4 *>(slots + ((size_t)j2 * D + srow) * D + col);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 f = src[j];
            acc[4 * j] = fmaf(e, acc[4 * j], f.x);
            acc[4 * j + 1] = fmaf(e, acc[4 * j + 1], f.y);
            acc[4 * j + 2] = fmaf(e, acc[4 * j + 2], f.z);
            acc[4 * j + 3] = fmaf(e, acc[4 * j + 3], f.w);
          }
        }
      }
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(acc[j]);
      __syncwarp();
      tmem_st32(tmem + lane_off + SM::T_S + col, r);
    }
    tmem_st_wait();
    bool ok = true;
    for (int c = 0; ok && c < nc; ++c) {
      const int s = c % NST;
      if (!(ok = swait(&prep[s], (c / NST) & 1, 13))) break;
      if (c >= 1 && !(ok = swait(s_done, (c - 1) & 1, 14))) break;
      tc_fence_after();
      const float e = srow >= 0 ? dec[s * D + srow] : 1.f;
      const float em = srow >= 0 ? emv[s * D + srow] : 1.f;  // diag(e^m) S_c for Qo
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
              pk[j] = pack_bf16(em * __uint_as_float(r[16 * h + 2 * j]),
                                em * __uint_as_float(r[16 * h + 2 * j + 1]));
            st_row16(smem + SM::OFF_S, SM::S_BLOCK, srow, col + 16 * h, pk);
          }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * e);
        __syncwarp();
        tmem_st32(tmem + lane_off + SM::T_S + col, r);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_ST, 128);
      if (t == 0) mbar_arrive(s_ready);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 8, c);
    }
    if (ok && nc > 0 && last_seg && swait(s_done, (nc - 1) & 1, 15) && p.S_final) {
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

// ================================================================ segment states
// Per (b,h, segment s < NS-1): the segment's own state
//   dS_s = sum_t diag(w_t) phi(k_t) v_t^T,   w_t[i] = exp(sum_{r > t in s} log alpha_r[i]),
// the decay from each token to the segment end per key channel, and the
// segment's total log decay per channel.  The chunks go last first, so each
// chunk's weights are its in-chunk suffix sums plus a carry (the log decay of
// the later chunks): no state chain, every MMA accumulates into TMEM.
template <int D>
struct CgStateSmem {
  // Stages to cover the loads' latency (the pass's own work per chunk is
  // short); at d = 64 a block runs two pieces of a segment.
  static constexpr int NST = 3;
  static constexpr uint32_t TILE = 64 * D * 2;           // K or V, bf16, swizzled boxes
  static constexpr uint32_t LAT = 64 * D * 4;            // log alpha, fp32 [64][D]
  static constexpr uint32_t STAGE = 2 * TILE + LAT;      // K | V | log alpha
  static constexpr uint32_t OFF_OCT = NST * STAGE;       // [8][D] octet sums of the chunk
  static constexpr uint32_t OFF_CARRY = OFF_OCT + 8 * D * 4;  // [2][D] log decay after the chunk
  static constexpr uint32_t OFF_BAR = OFF_CARRY + 2 * D * 4;
  static constexpr uint32_t OFF_CTL = OFF_BAR + 8 * (3 * NST + 1);
  static constexpr uint32_t BYTES = OFF_CTL + 64;
  static constexpr uint32_t PIECE = (BYTES + 1023) / 1024 * 1024;  // one piece's region
  static_assert(STAGE % 1024 == 0 && TILE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert((D == 64 ? 2 : 1) * PIECE <= 232448, "exceeds the per-block shared memory limit");
};

constexpr int kThreadsCgState = 384;  // warps 0 TMA, 1 MMA, 2-3 idle, 4-11 transform (256)
constexpr int W_XF = 4, kXfThreads = 256;
constexpr uint32_t BAR_XF = 5;

// PB pieces per block, each with its own copy of the pipeline (warps 12 pc ..
// 12 pc + 11), shared memory region and TMEM columns: the pieces of one
// segment then share an SM for certain.
template <int D, bool PHI, int PB>
__global__ void __launch_bounds__(kThreadsCgState * PB, 1)
cg_segment_state_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmA, CgParams p) {
  using SM = CgStateSmem<D>;
  constexpr int NST = SM::NST;
  extern __shared__ __align__(1024) unsigned char smem_all[];
  const int pc = (int)threadIdx.x / kThreadsCgState;  // this thread's piece in the block
  unsigned char *smem = smem_all + pc * SM::PIECE;
  Ctl *ctl0 = reinterpret_cast<Ctl *>(smem_all + SM::OFF_CTL);  // holds the TMEM base
  const uint32_t bar_xf = BAR_XF + 2 * pc;
  float *oct = reinterpret_cast<float *>(smem + SM::OFF_OCT);
  float *carry = reinterpret_cast<float *>(smem + SM::OFF_CARRY);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::OFF_BAR);
  uint64_t *empty = full + NST;
  uint64_t *ready = empty + NST;  // K rows weighted
  uint64_t *done = ready + NST;   // every MMA finished
  Ctl *ctl = reinterpret_cast<Ctl *>(smem + SM::OFF_CTL);
  const int tid = (int)threadIdx.x - pc * kThreadsCgState, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();  // the output kernel may start; its later segments wait
  const int piece = blockIdx.x * PB + pc, bh = blockIdx.y;
  if (piece == 0 && p.S0 && p.S0 == p.S_final) {  // S0 aside, for when S_final overwrites it
    const float4 *src = reinterpret_cast<const float4 *>(p.S0 + (size_t)bh * D * D);
    float4 *dst = reinterpret_cast<float4 *>(p.ws_state + ((size_t)bh * p.n_slot + p.n_slot - 1) * D * D);
    for (int i = tid; i < D * D / 4; i += kThreadsCgState) dst[i] = src[i];
  }
  int cbase, nc;  // at least one chunk (the plan's parts are never empty)
  piece_range(p, piece, cbase, nc);
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&ready[s], 1);
    }
    mbar_init(done, 1);
    ctl->abort = 0;
    fence_mbarrier_init();
  }
  for (int i = tid; i < D; i += kThreadsCgState) carry[i] = 0.f;
  if (pc == 0 && warp == 1) {
    tmem_alloc(&ctl0->tmem_base, PB * D);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl0->tmem_base + pc * D;
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmA);
      int issued = 0;
      for (int c = 0; c < nc; ++c) {
        const int s = c % NST;
        if (c >= NST && !wait1(&empty[s], ((c / NST) - 1) & 1, ctl, p.err, KID_CHANNEL_GATE_TC, 30))
          break;
        unsigned char *st = smem + s * SM::STAGE;
        mbar_arrive_expect_tx(&full[s], SM::STAGE);
        const int tok = (cbase + nc - 1 - c) * CH;  // chunks last first
        for (int b = 0; b < D / BOX; ++b) {
          tma_load_3d(st + b * BOX_BYTES, &tmK, &full[s], b * BOX, tok, bh);
          tma_load_3d(st + SM::TILE + b * BOX_BYTES, &tmV, &full[s], b * BOX, tok, bh);
        }
        tma_load_3d(st + 2 * SM::TILE, &tmA, &full[s], 0, tok, bh);
        issued = c + 1;
      }
      if (*(volatile uint32_t *)&ctl->abort)
        for (int c = max(0, issued - NST); c < issued; ++c) drain_wait(&full[c % NST], (c / NST) & 1);
      for (int c = max(0, nc - NST); c < nc; ++c) drain_wait(&empty[c % NST], (c / NST) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(D, D, true, true);
      for (int c = 0; c < nc; ++c) {
        const int s = c % NST;
        if (!wait1(&ready[s], (c / NST) & 1, ctl, p.err, KID_CHANNEL_GATE_TC, 31)) break;
        tc_fence_after();
        const uint32_t kt = smem_u32(smem + s * SM::STAGE), vt = kt + SM::TILE;
#pragma unroll
        for (int kk = 0; kk < CH / 16; ++kk)  // S += K~^T V over the chunk's 64 tokens
          mma_bf16(tmem, smem_desc_sw128(kt + 2048 * kk, BOX_BYTES, 1024),
                   smem_desc_sw128(vt + 2048 * kk, BOX_BYTES, 1024), idesc, (c | kk) != 0);
        mma_commit(&empty[s]);
      }
      mma_commit(done);
      drain_wait(done, 0);
    }
  } else if (warp >= W_XF) {
    const int t = tid - W_XF * 32;  // 0..255
    // Items (channel pair cp, octet q of 8 tokens): D/2 x 8 of them, NIT a
    // thread.  An item's log decays, read for the octet sums, stay in
    // registers for its weights.
    constexpr int NPAIR = D / 2, NITEM = NPAIR * 8, NIT = NITEM / kXfThreads;
    static_assert(NITEM % kXfThreads == 0, "whole items per thread");
    float2 av[NIT][8];
    bool ok = true;
    for (int c = 0; ok && c < nc; ++c) {
      const int s = c % NST;
      if (!(ok = wait_grp<kXfThreads>(&full[s], (c / NST) & 1, ctl, p.err, KID_CHANNEL_GATE_TC, 32,
                                      bar_xf, t)))
        break;
      unsigned char *kt = smem + s * SM::STAGE;
      const float *la = reinterpret_cast<const float *>(kt + 2 * SM::TILE);
      const float *cin = carry + (c & 1) * D;
      float *cout = carry + ((c + 1) & 1) * D;
#pragma unroll
      for (int j = 0; j < NIT; ++j) {  // octet sums
        const int it = t + j * kXfThreads, cp = it % NPAIR, q = it / NPAIR;
        float2 sum = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          av[j][i] = *reinterpret_cast<const float2 *>(la + (8 * q + i) * D + 2 * cp);
          sum.x += av[j][i].x;
          sum.y += av[j][i].y;
        }
        *reinterpret_cast<float2 *>(oct + q * D + 2 * cp) = sum;
      }
      named_bar_sync(bar_xf, kXfThreads);
#pragma unroll
      for (int j = 0; j < NIT; ++j) {  // weights, K rows in place
        const int it = t + j * kXfThreads, cp = it % NPAIR, q = it / NPAIR, c0 = 2 * cp;
        float2 run = *reinterpret_cast<const float2 *>(cin + c0);  // decay after the chunk
        float2 tot = make_float2(0.f, 0.f);
#pragma unroll
        for (int q2 = 0; q2 < 8; ++q2) {
          const float2 o = *reinterpret_cast<const float2 *>(oct + q2 * D + c0);
          tot.x += o.x;
          tot.y += o.y;
          if (q2 > q) {
            run.x += o.x;
            run.y += o.y;
          }
        }
        if (q == 0) {
          const float2 cc = *reinterpret_cast<const float2 *>(cin + c0);
          *reinterpret_cast<float2 *>(cout + c0) = make_float2(cc.x + tot.x, cc.y + tot.y);
        }
        const uint32_t cbox = (uint32_t)c0 >> 6, cin64 = (uint32_t)c0 & 63u;
        uint32_t kw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          kw[i] = *reinterpret_cast<const uint32_t *>(kt + cbox * BOX_BYTES +
                                                      sw128_offset((uint32_t)(8 * q + i), cin64));
#pragma unroll
        for (int i = 7; i >= 0; --i) {  // token 8 q + i: the decay of the tokens after it
          const uint32_t off = cbox * BOX_BYTES + sw128_offset((uint32_t)(8 * q + i), cin64);
          const uint32_t w = PHI ? elu1_bf16x2(kw[i]) : kw[i];  // as the output pass forms its keys
          const float kx = __uint_as_float(w << 16), ky = __uint_as_float(w & 0xffff0000u);
          *reinterpret_cast<uint32_t *>(kt + off) = pack_bf16(kx * __expf(run.x), ky * __expf(run.y));
          run.x += av[j][i].x;
          run.y += av[j][i].y;
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(bar_xf, kXfThreads);
      if (t == 0) mbar_arrive(&ready[s]);
    }
    // The accumulated state (warps 4-7: lane quarters 0-3) into slot s+1, and
    // the segment's total log decay per key channel.
    if (t < 128 && wait_wg(done, 0, ctl, p.err, KID_CHANNEL_GATE_TC, 33, bar_xf + 1)) {
      tc_fence_after();
      const int quarter = warp & 3;
      const int row = acc_row<D>(quarter, lane);
      const size_t slot = (size_t)bh * p.n_slot + piece;  // the piece's own state
      float *dst = p.ws_state + slot * D * D;
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        __syncwarp();
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + col, r);
        tmem_ld_wait();
        if (row >= 0) {
          float4 *o = reinterpret_cast<float4 *>(dst + (size_t)row * D + col);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            o[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                               __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
      }
      if (ok)
        for (int i = t; i < D; i += 128)
          p.ws_logdec[((size_t)bh * p.n_slot + piece) * D + i] = carry[(nc & 1) * D + i];
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (pc == 0 && warp == 1) {
    __syncwarp();
    tmem_dealloc(ctl0->tmem_base, PB * D);
  }
}

// Segments per sequence: enough (sequence, segment) blocks to fill the SMs
// once, at least 8 chunks per segment, and only with a workspace.  The first
// segments start at once, alongside the state pass; the others wait for the
// state pass.  So the first segment is the longer one, by the state pass's
// cost per chunk relative to the output pass's (share, measured): f chunks of
// output take as long as f chunks of state pass plus a later segment's g,
// i.e. g = (1 - share) f.  At d = 64 the state pass cuts each segment into
// two pieces run side by side, which lowers its share.  Measured best: 0.4 at
// d = 64 with two segments, 0.25 with more (the later segments also fold
// more states), 0.3 at d = 128.
constexpr double kStateShare64Two = 0.4, kStateShare64 = 0.25, kStateShare128 = 0.3;
struct CgPlan {
  int n_chunks, first_chunks, seg_chunks, n_seg, state_parts, n_slot;
};
CgPlan cg_plan(int B, int H, int L, int D) {
  const int nc = (L + CH - 1) / CH, BH = B * H;
  const int ns = std::max(1, std::min(sm_count() / std::max(1, BH), nc / 8));
  if (ns <= 1) return CgPlan{nc, nc, nc, 1, 1, 1};
  const double share = D == 64 ? (ns == 2 ? kStateShare64Two : kStateShare64) : kStateShare128;
  const double f = nc / (1.0 + (1.0 - share) * (ns - 1));
  const int first = std::max(1, std::min(nc - 1, (int)std::lround(f)));
  const int g = (nc - first + ns - 2) / (ns - 1);
  const int n_seg = 1 + (nc - first + g - 1) / g;
  // Every state-passed segment (all but the last) has first or g chunks.
  const int parts = D == 64 && first >= 2 && (n_seg <= 2 || g >= 2) ? 2 : 1;
  return CgPlan{nc, first, g, n_seg, parts, (n_seg - 1) * parts + 1};
}

size_t cg_ws_bytes(int B, int H, int L, int D) {
  const CgPlan pl = cg_plan(B, H, L, D);
  if (pl.n_seg <= 1) return 0;
  const size_t bh = (size_t)B * H, slots = bh * pl.n_slot;
  return slots * D * D * sizeof(float) + slots * D * sizeof(float);
}

template <int D, bool PHI>
cudaError_t launch_cg(const VariantArgs &a) {
  using SM = CgSmem<D>;
  const int BH = a.B * a.H;
  CgParams p{};
  p.H = a.H;
  p.L = a.L;
  p.BH = BH;
  const CgPlan pl = cg_plan(a.B, a.H, a.L, D);
  const bool segs = pl.n_seg > 1 && a.workspace && a.ws_bytes >= cg_ws_bytes(a.B, a.H, a.L, D);
  p.n_chunks = pl.n_chunks;
  p.first_chunks = segs ? pl.first_chunks : pl.n_chunks;
  p.seg_chunks = segs ? pl.seg_chunks : pl.n_chunks;
  p.n_seg = segs ? pl.n_seg : 1;
  p.state_parts = segs ? pl.state_parts : 1;
  p.n_slot = segs ? pl.n_slot : 1;
  if (segs) {
    p.ws_state = static_cast<float *>(a.workspace);
    p.ws_logdec = p.ws_state + (size_t)BH * pl.n_slot * D * D;
  }
  p.log_alpha = a.decay;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.k = static_cast<const __nv_bfloat16 *>(a.k);
  p.S0 = a.S0;
  p.S_final = a.S_final;
  p.err = device_error_word();
  CUtensorMap tq, tk, tv, to, ta;
  if (!make_tmap_bf16_3d(&tq, a.q, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&tk, a.k, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&tv, a.v, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&to, a.O, D, a.L, BH, BOX, BOX) ||
      !make_tmap_f32_3d(&ta, a.decay, D, a.L, BH, D, CH))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (segs) {  // the segments' own states first, a block per segment
    using SS = CgStateSmem<D>;
    if constexpr (D == 64) {
      if (pl.state_parts == 2) {
        auto ks = cg_segment_state_kernel<D, PHI, 2>;
        static int smem_set_state2[64];
        if ((e = set_smem_once(ks, 2 * SS::PIECE, smem_set_state2)) != cudaSuccess) return e;
        ks<<<dim3(pl.n_seg - 1, BH), 2 * kThreadsCgState, 2 * SS::PIECE, a.stream>>>(tk, tv, ta, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
    }
    if (pl.state_parts == 1) {
      auto ks = cg_segment_state_kernel<D, PHI, 1>;
      static int smem_set_state[64];
      if ((e = set_smem_once(ks, SS::PIECE, smem_set_state)) != cudaSuccess) return e;
      ks<<<dim3(pl.n_seg - 1, BH), kThreadsCgState, SS::PIECE, a.stream>>>(tk, tv, ta, p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  auto kern = channel_gate_tc_kernel<D, PHI>;
  static int smem_set[64];
  if ((e = set_smem_once(kern, SM::BYTES, smem_set)) != cudaSuccess) return e;
  if (segs)
    e = launch_pdl(kern, dim3(BH, p.n_seg), kThreads, SM::BYTES, a.stream, tq, tk, tv, to, ta, p);
  else
    kern<<<dim3(BH, p.n_seg), kThreads, SM::BYTES, a.stream>>>(tq, tk, tv, to, ta, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool channel_gate_tc_supported(const VariantArgs &a) {
  return a.form == VARIANT_CHANNEL_GATE && a.dtype == LA_BF16 && a.chunk == CH && a.dk == a.dv &&
         (a.dk == 64 || a.dk == 128);
}

size_t channel_gate_tc_workspace_bytes(int B, int H, int L, int d) {
  if (B <= 0 || H <= 0 || L <= 0 || (d != 64 && d != 128)) return 0;
  return cg_ws_bytes(B, H, L, d);
}

cudaError_t launch_channel_gate_tc(const VariantArgs &a) {
  const bool phi = a.phi != LA_PHI_IDENTITY;
  if (a.dk == 128) return phi ? launch_cg<128, true>(a) : launch_cg<128, false>(a);
  return phi ? launch_cg<64, true>(a) : launch_cg<64, false>(a);
}

}  // namespace la
