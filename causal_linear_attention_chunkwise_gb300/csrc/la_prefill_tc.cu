// la_prefill_tc.cu -- chunkwise causal linear attention prefill on the 5th-gen
// tensor cores (tcgen05 MMAs into TMEM, TMA-staged tiles), bf16 inputs with
// fp32 accumulation, chunk C = 64, d_k = d_v = D in {64, 128}.
//
// The chunkwise form ("Linear / Sparse Attention - minimal runnable
// implementation", linear_attn_chunkwise; "Linear / sparse attention tutorial"
// section 6.2) for chunk c with incoming state S_c, within-chunk inclusive
// log-decay prefix Lam_i and chunk total A_c = Lam_{n-1}:
//
//   P     = phi(Q_c) phi(K_c)^T                                  (MMA1, 64x64)
//   P_ij <- P_ij exp(Lam_i - Lam_j) if j <= i else 0             (registers)
//   O_c   = P V_c                                                (MMA2)
//         + Qt_c S_c,       Qt_i = exp(Lam_i) phi(q_i)           (MMA3)
//   S_c+1 = exp(A_c) S_c + Kt_c^T V_c,  Kt_j = exp(A_c - Lam_j) phi(k_j)  (MMA4)
//
// Gate factors are the expansion of S_t = a_t S_{t-1} + phi(k_t) v_t^T over one
// chunk ("CS336 lecture 4, code 1: linear attention",
// gated_linear_attention_recurrent / _parallel); every exponent is a
// difference with i >= j or a chunk-local sum <= 0, so nothing overflows.
//
// Parallelism over the sequence.  A sequence of NC chunks is cut into NS
// segments of G chunks.  Three kernels, launched back to back on one stream:
//   segment_state_kernel  per (b, h, segment s < NS-1): the segment's own
//       state  dS_s = sum_t exp(Lam_end - Lam_t) phi(k_t) v_t^T  (one long
//       K = tokens GEMM, weights relative to the segment end, so no rescaling
//       between chunks) and its total log decay A_s;
//   state_scan_kernel     per (b, h), elementwise over the state:
//       S_in[0] = S0 (or 0),  S_in[s+1] = exp(A_s) S_in[s] + dS_s;
//   chunk_output_kernel   per (b, h, segment): the chunk loop above from
//       S_in[s]; the last segment also writes S_final.
// With NS = 1 only the output kernel runs.  The associative combination of
// (decay, state) pairs across segments is the same state passing the chunk
// loop performs across chunks.  The scan and the output kernel are
// programmatic dependent launches: each may start while the kernel before it
// runs, and waits for it (griddepcontrol.wait) before reading what it wrote.
//
// The non-causal form O = phi(Q) (phi(K)^T V) ("adv13 - Linear Attention /
// SSM" section 4.3) reuses the segment-state kernel over every chunk, then
// runs noncausal_output_kernel.  At d = 64 its blocks sum a sequence's
// segment states themselves; at d = 128 (four times the bytes per state) the
// scan sums them into one extra slot first.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/la_gb300.h"
#include "la_common.cuh"
#include "la_internal.h"
#include "la_ptx.cuh"
#include "la_tc_sync.cuh"
#include "la_tma_host.h"

#ifdef LA_TRACE
namespace la {
__device__ long long g_trace[kTraceEvents][kTraceChunks];
// Global-timer stamps per CTA of the three prefill kernels: [kernel][cta][slot].
__device__ unsigned long long g_cta[3][1024][3];
}
extern "C" int la_trace_read(long long *out) {
  return (int)cudaMemcpyFromSymbol(out, la::g_trace, sizeof(la::g_trace));
}
extern "C" int la_cta_read(unsigned long long *out) {
  return (int)cudaMemcpyFromSymbol(out, la::g_cta, sizeof(la::g_cta));
}
// Per-chunk events of the segment-state kernel's CTA (0, 0): [event][chunk].
namespace la {
__device__ long long g_strace[kTraceEvents][kTraceChunks];
}
extern "C" int la_strace_read(long long *out) {
  return (int)cudaMemcpyFromSymbol(out, la::g_strace, sizeof(la::g_strace));
}
#define LA_CTA_STAMP(kern, slot)                                                             \
  do {                                                                                     \
    const unsigned cta_ = blockIdx.x + gridDim.x * blockIdx.y;                             \
    if (cta_ < 1024) ::la::g_cta[(kern)][cta_][(slot)] = ::la::global_timer_ns();           \
  } while (0)
#else
#define LA_CTA_STAMP(kern, slot) \
  do {                           \
  } while (0)
#endif

namespace la {
namespace {
using namespace tc;

constexpr int kMaxSegChunks = 32;       // G <= 32 (2048 tokens per segment)

// Warp roles (both tcgen05 kernels).
constexpr int W_TMA = 0, W_MMA = 1, WG1 = 4, WG2 = 8;
constexpr uint32_t BAR_WG2 = 2;

// ---------------------------------------------------------------- math helpers
// A token's log decay in two steps: the stored input of a token (a gate logit for
// LA_DECAY_GATE_LOGIT; 0 beyond the sequence, where the log decay is 0
// for every kind), then its log decay.
__device__ __forceinline__ float token_decay_raw(int kind, const float *__restrict__ decay, int h,
                                                 size_t bhL, int tok, int L) {
  if (tok >= L) return kind == LA_DECAY_GATE_LOGIT ? -INFINITY : 0.f;
  return kind == LA_DECAY_HEAD ? decay[h] : decay[bhL + tok];
}
__device__ __forceinline__ float token_log_decay(int kind, float raw) {
  return kind == LA_DECAY_GATE_LOGIT ? neg_softplus(raw) : raw;
}

// ---------------------------------------------------------------- parameters
struct TcParams {
  int H, L, BH;
  int n_chunks;     // chunks per sequence (NC)
  int seg_chunks;   // G
  int n_seg;        // NS
  int phi, decay_kind;
  const float *decay;
  const float *S0;  // read directly only when NS == 1
  float *S_final;
  float *ws_state;  // [BH][NS][D][srow]: slot s = incoming state of segment s
  float *ws_logdec; // [BH][NS]: total log decay of segment s (s < NS-1)
  unsigned int *err;
  // The normalised form (d = 64): state rows carry z in column D (srow = D + 16),
  // and the output is divided by the denominator riding in O's column D.
  int srow;           // floats per state row in the workspace slots (D, or D + 16)
  const float *z0;    // [BH][D] or null (= zeros)
  float *z_final;     // [BH][D] or null
};

// ================================================================ shared pieces

// ================================================================ segment state
// Shared memory: NST stages of {K tile, V tile}; the segment's suffix log
// decays; per-stage row weights; barriers.
template <int D, bool NORM = false, bool DEEP = false>
struct StateSmem {
  // The two transform groups take alternate chunks, so the stage count must
  // be even: stage s is then always used by group s % 2, and every phase of
  // its barriers is waited on, in order, by that one group.  (With an odd
  // count a group could wait on a stage whose previous phase belongs to the
  // other group and has not completed yet; the parity test would then pass
  // early.)  Two stages for D = 128 (three blocks fit on an SM) and six for
  // D = 64 (two blocks).
  // DEEP (D = 128): both groups transform every chunk together, so any count
  // works, and three stages put 96 KB of K and V in flight per block, at two
  // blocks per SM: more of the load latency hidden, when the pass fits in one
  // wave of two blocks per SM.
  static_assert(!DEEP || D == 128, "the deep form is the d = 128 one");
  static constexpr bool ALT = !DEEP;
  static constexpr int NST = DEEP ? 3 : D == 128 ? 2 : 6;
  static_assert(!ALT || NST % 2 == 0, "stages must alternate between the two transform groups");
  static constexpr uint32_t TILE = 64 * D * 2;
  static constexpr uint32_t STAGE = 2 * TILE;
  // NORM: one constant block of ones (column 0) after the stages, read as the
  // second 64-column block of every V operand: the state gains column D = z.
  static constexpr uint32_t OFF_ONES = NST * STAGE;
  static constexpr uint32_t OFF_SUF = OFF_ONES + (NORM ? 8192 : 0);      // floats [G*64]
  static constexpr uint32_t OFF_BAR = OFF_SUF + kMaxSegChunks * CH * 4;
  static constexpr uint32_t OFF_CTL = OFF_BAR + 8 * (3 * NST + 1);
  static constexpr uint32_t OFF_SCR = OFF_CTL + 64;                       // 8 floats
  static constexpr uint32_t OFF_TRC = OFF_SCR + 64;                       // trace builds
  static constexpr uint32_t BYTES = OFF_TRC + trace_smem_bytes();
};

constexpr int kThreadsState = 384;  // warps 0..11: TMA, MMA, -, -, XG0 (4..7), XG1 (8..11)
constexpr uint32_t BAR_XG0 = 1, BAR_XG1 = 2, BAR_XG = 3;

template <int D, bool PHI, bool DECAY, bool NORM = false, bool DEEP = false>
__global__ void __launch_bounds__(kThreadsState, 2)  // two CTAs per SM
segment_state_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, TcParams p) {
  using SM = StateSmem<D, NORM, DEEP>;
  static_assert(!NORM || D == 64, "the normalised form rides the d = 64 kernels");
  constexpr int ZW = NORM ? 16 : 0;
  constexpr uint32_t kTmemCols = NORM ? 128 : D;
  constexpr int NST = SM::NST;
  extern __shared__ __align__(1024) unsigned char smem[];
  float *suf = reinterpret_cast<float *>(smem + SM::OFF_SUF);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::OFF_BAR);
  uint64_t *empty = full + NST;
  uint64_t *ready = empty + NST;   // K tile transformed
  uint64_t *done = ready + NST;    // all MMAs finished
  Ctl *ctl = reinterpret_cast<Ctl *>(smem + SM::OFF_CTL);
  float *scr = reinterpret_cast<float *>(smem + SM::OFF_SCR);
  pdl_launch_dependents();  // the scan may be scheduled now; it waits for this grid
  if (threadIdx.x == 0) LA_CTA_STAMP(0, 0);
  const bool st_on = blockIdx.x == 0 && blockIdx.y == 0;
  const long long st_t0 = clock64();
  (void)st_on;
  (void)st_t0;
  LA_TRACE_TABLE(smem + SM::OFF_TRC, 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x, bh = blockIdx.y, h = bh % p.H;
  const int c0 = seg * p.seg_chunks;
  const int nc = min(p.seg_chunks, p.n_chunks - c0);
  const int tok0 = c0 * CH;
  const size_t bhL = (size_t)bh * p.L;

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
  if (warp == W_MMA) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if constexpr (NORM) {  // the ones block: column 0 = 1, columns 1..15 = 0 (of 16 read)
    if (tid < 64) {
      unsigned char *ob = smem + SM::OFF_ONES + tid * 128;
      *reinterpret_cast<uint4 *>(ob + ((0 ^ (tid & 7)) << 4)) = make_uint4(pack_bf16(1.f, 0.f), 0u, 0u, 0u);
      *reinterpret_cast<uint4 *>(ob + ((1 ^ (tid & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == W_TMA) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int issued = 0;
      for (int c = 0; c < nc; ++c) {
        const int s = c % NST;
        if (c >= NST &&
            !wait1(&empty[s], ((c / NST) - 1) & 1, ctl, p.err, KID_PREFILL_TC_STATE, 1))
          break;
        if (c >= NST) LA_TRACE_EVENT(st_on, st_t0, 4, c - NST);
        unsigned char *st = smem + s * SM::STAGE;
        mbar_arrive_expect_tx(&full[s], SM::STAGE);
        // The segment's chunks last first: when the pass ends, the K and V
        // tiles still in L2 are those of the segments' first chunks, which
        // the output kernel's first blocks read first.
        const int tok = tok0 + (nc - 1 - c) * CH;
        for (int b = 0; b < D / BOX; ++b) {
          if (!LA_CHK(b * BOX + BOX <= D && tok < p.L && bh < p.BH, KID_PREFILL_TC_STATE, 1))
            continue;
          tma_load_3d(st + b * BOX_BYTES, &tmK, &full[s], b * BOX, tok, bh);
          tma_load_3d(st + SM::TILE + b * BOX_BYTES, &tmV, &full[s], b * BOX, tok, bh);
        }
        LA_TRACE_EVENT(st_on, st_t0, 0, c);
        issued = c + 1;
      }
      if (*(volatile uint32_t *)&ctl->abort)
        for (int c = max(0, issued - NST); c < issued; ++c) drain_wait(&full[c % NST], (c / NST) & 1);
      // Producer tail: wait for the last stage releases (tcgen05.commit arrivals).
      for (int c = max(0, nc - NST); c < nc; ++c) drain_wait(&empty[c % NST], (c / NST) & 1);
    }
  } else if (warp == W_MMA) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(D, D + ZW, true, true);
      for (int c = 0; c < nc; ++c) {
        const int s = c % NST;
        if (!wait1(&ready[s], (c / NST) & 1, ctl, p.err, KID_PREFILL_TC_STATE, 2)) break;
        tc_fence_after();
        LA_TRACE_EVENT(st_on, st_t0, 3, c);
        const uint32_t kt = smem_u32(smem + s * SM::STAGE);
        const uint32_t vt = kt + SM::TILE;
        // V's second 64-column block: its next box (d = 128), or the ones
        // block (NORM), LBO bytes on.
        const uint32_t v_lbo = NORM ? smem_u32(smem + SM::OFF_ONES) - vt : BOX_BYTES;
#pragma unroll
        for (int kk = 0; kk < CH / 16; ++kk)
          mma_bf16(tmem, smem_desc_sw128(kt + 2048 * kk, BOX_BYTES, 1024),
                   smem_desc_sw128(vt + 2048 * kk, v_lbo, 1024), idesc, (c | kk) != 0);
        mma_commit(&empty[s]);
      }
      mma_commit(done);
      drain_wait(done, 0);  // every issued MMA has finished before TMEM is released
    }
  } else if (warp >= WG1) {
    const int g = (warp - WG1) >> 2;           // transform group 0 or 1
    const int t = tid - WG1 * 32 - 128 * g;    // 0..127 within the group
    const uint32_t gbar = g ? BAR_XG1 : BAR_XG0;
    // Token weights of the segment: suf[i] = exp(sum_{r > i} lambda_r), the
    // decay from token i to the segment end; A_s = sum of all lambda.  Both
    // groups (256 threads) take PER consecutive tokens each: all of a
    // thread's decay inputs are loaded before any is used, so the prologue
    // costs one memory round trip, then a suffix scan over threads.
    const int ntok = nc * CH;
    constexpr bool scale = DECAY;
    float seg_total = 0.f;
    if (scale) {
      constexpr int PER = kMaxSegChunks * CH / 256;
      const int t2 = tid - WG1 * 32, wid = t2 >> 5;  // 0..255, warp 0..7
      float raw[PER], sfx[PER];
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int i = t2 * PER + j;
        raw[j] = i < ntok ? token_decay_raw(p.decay_kind, p.decay, h, bhL, tok0 + i, p.L) : 0.f;
      }
      float run = 0.f;  // this thread's tokens after token j
#pragma unroll
      for (int j = PER - 1; j >= 0; --j) {
        sfx[j] = run;
        if (t2 * PER + j < ntok) run += token_log_decay(p.decay_kind, raw[j]);
      }
      float x = run;  // sum over this lane and the later lanes of the warp
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32) x += y;
      }
      if (lane == 0) scr[wid] = x;
      named_bar_sync(BAR_XG, 256);
      float later = x - run, total = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < 8; ++w2) {
        total += scr[w2];
        if (w2 > wid) later += scr[w2];
      }
#pragma unroll
      for (int j = 0; j < PER; ++j)  // the token's weight itself (<= 1)
        if (t2 * PER + j < ntok) suf[t2 * PER + j] = __expf(sfx[j] + later);
      seg_total = total;
    }
    named_bar_sync(BAR_XG, 256);  // suffix sums visible to both groups
    constexpr bool phi = PHI;
    // ALT: group g takes chunks g, g + 2, ...; otherwise both groups (256
    // threads, one barrier) take every chunk.
    constexpr int NT = SM::ALT ? 128 : 256;
    const int tx = SM::ALT ? t : tid - WG1 * 32;
    const uint32_t xbar = SM::ALT ? gbar : BAR_XG;
    for (int c = SM::ALT ? g : 0; c < nc; c += SM::ALT ? 2 : 1) {
      const int s = c % NST;
      if (!wait_grp<NT>(&full[s], (c / NST) & 1, ctl, p.err, KID_PREFILL_TC_STATE, 3, xbar, tx)) break;
      LA_TRACE_EVENT(st_on && tx == 0, st_t0, 1, c);
      unsigned char *kt = smem + s * SM::STAGE;
      LA_TRACE_EVENT(st_on && tx == 0, st_t0, 5, c);
      const float *w = suf + (nc - 1 - c) * CH;  // the chunk's tokens (chunks last first)
      if constexpr (phi || scale)
        tile_pass<D, 1, phi, scale>(kt, [w](int, int r) { return w[r]; }, tx, NT);
      LA_TRACE_EVENT(st_on && tx == 0, st_t0, 6, c);
      fence_proxy_async_smem();
      LA_TRACE_EVENT(st_on && (tx & 31) == 0 && tx < 128, st_t0, 8 + (tx >> 5), c);
      named_bar_sync(xbar, NT);
      if (tx == 0) mbar_arrive(&ready[s]);
      LA_TRACE_EVENT(st_on && tx == 0, st_t0, 2, c);
    }
    // Read the accumulated state out of TMEM (group 0) into segment slot s+1.
    if (g == 0 && wait_wg(done, 0, ctl, p.err, KID_PREFILL_TC_STATE, 4, BAR_XG0)) {
      tc_fence_after();
      const int quarter = warp & 3;
      const int row = acc_row<D>(quarter, lane);
      if (!LA_CHK(seg + 1 < p.n_seg && bh < p.BH, KID_PREFILL_TC_STATE, 4)) seg_total = 0.f;
      float *dst = p.ws_state + (((size_t)bh * p.n_seg + min(seg + 1, p.n_seg - 1)) * D) * p.srow;
      if constexpr (NORM) {  // z: state column D (the 15 after it are zero)
        __syncwarp();
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + D, r);
        tmem_ld_wait();
        if (row >= 0) {
          float4 *o = reinterpret_cast<float4 *>(dst + (size_t)row * p.srow + D);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            o[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                               __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
      }
#pragma unroll 1
      for (int col = 0; col < D; col += 32) {
        __syncwarp();
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + col, r);
        tmem_ld_wait();
        if (row >= 0) {
          float4 *o = reinterpret_cast<float4 *>(dst + (size_t)row * p.srow + col);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            o[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                               __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
      }
      if (t == 0) p.ws_logdec[(size_t)bh * p.n_seg + seg] = seg_total;
    }
  }
  __syncwarp();  // lanes that skipped a lane-0 role loop wait for lane 0
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  LA_TRACE_FLUSH(st_on, &g_strace[0][0]);
  if (threadIdx.x == 0) LA_CTA_STAMP(0, 2);
}

// ================================================================ state scan
// slot 0 <- S0 (or 0); slot s+1 <- exp(A_s) slot s + slot s+1, for s < NS-1.
__global__ void __launch_bounds__(256, 2)
state_scan_kernel(int D, int srow, int n_seg, const float *S0, const float *z0,
                  float *__restrict__ ws_state, const float *__restrict__ ws_logdec) {
  // Launched as a programmatic dependent of the segment-state kernel: let the
  // output kernel's CTAs start, then wait until the segment states are written.
  pdl_launch_dependents();
  if (threadIdx.x == 0) LA_CTA_STAMP(1, 0);
  pdl_wait_previous();
  if (threadIdx.x == 0) LA_CTA_STAMP(1, 1);
  const int bh = blockIdx.y;
  // A slot is D rows of srow floats: the state, then (srow > D) z in column D.
  const size_t n4 = (size_t)D * srow / 4;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const int r4 = srow / 4, row = (int)(i / r4), c4 = (int)(i % r4);
  float4 *slots = reinterpret_cast<float4 *>(ws_state) + (size_t)bh * n_seg * n4;
  const float *logdec = ws_logdec + (size_t)bh * n_seg;
  float4 cur = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c4 < D / 4) {
    if (S0) cur = reinterpret_cast<const float4 *>(S0)[((size_t)bh * D + row) * (D / 4) + c4];
  } else if (c4 == D / 4 && z0) {
    cur.x = z0[(size_t)bh * D + row];
  }
  slots[i] = cur;
  // Segments in batches of 20: every load of a batch is issued before the
  // first use, so a batch costs one memory round trip (one batch for up to 21
  // segments).
  constexpr int kB = 20;
  for (int s0 = 0; s0 + 1 < n_seg; s0 += kB) {
    float4 d[kB];
    float a[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      if (s0 + j + 1 < n_seg) {
        d[j] = slots[(size_t)(s0 + j + 1) * n4 + i];
        a[j] = logdec[s0 + j];
      }
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      if (s0 + j + 1 < n_seg) {
        const float e = __expf(a[j]);
        cur.x = fmaf(e, cur.x, d[j].x);
        cur.y = fmaf(e, cur.y, d[j].y);
        cur.z = fmaf(e, cur.z, d[j].z);
        cur.w = fmaf(e, cur.w, d[j].w);
        slots[(size_t)(s0 + j + 1) * n4 + i] = cur;
      }
    }
  }
}

// ================================================================ chunk output
// d = 64: each output CTA carries two independent state chains, the states of
//   two segments of one (b, h) sequence, each with its own hand-over (MMA into
//   TMEM, then the TMEM -> bf16 copy), so that one chain's hand-over overlaps
//   the other chain's work.  Their chunks are interleaved into one sequence
//   of virtual chunks k = 0, 1, ...: while both have chunks left they
//   alternate.
// d = 128: one segment per CTA and one 128-column chain, computed transposed
//   so that every product has M = 128: S^T += V^T K, O^T = S^T Q^T (A, the
//   bf16 copy of S^T, read from TMEM) and O^T += V^T P^T.  The state hand-over
//   then stays in TMEM.
template <int DK, bool NORM = false>
struct OutSmem {
  static constexpr bool PAIRS = DK == 64;                       // two segments per CTA
  static constexpr int NCHAIN = PAIRS ? 2 : 1;                  // state chains
  static constexpr int CW = PAIRS ? 64 : DK / NCHAIN;           // state columns per chain
  // The normalised form carries one more value column (ones: the denominator
  // in O, z in the state), as a second 16-column block of every value-side
  // operand; ZW = 16 extra columns (one used, the rest zero).
  static constexpr int ZW = NORM ? 16 : 0;
  static constexpr int CWT = CW + ZW;                           // TMEM columns per chain
  static_assert(!NORM || PAIRS, "the normalised form rides the d = 64 kernel");
  // d = 128 keeps the output and the state transposed in TMEM (see the kernel):
  // its bf16 state copy lives in TMEM, not in shared memory.
  static constexpr bool TRANS = DK == 128 && NCHAIN == 1;
  // d = 128 takes a fourth input stage in the room of a second P tile and a
  // second O staging tile: the deeper prefetch is worth more than either.
  static constexpr int NST = PAIRS ? (NORM ? 4 : 5) : 4;
  static constexpr int NPB = TRANS ? 1 : 2;                // P tiles in shared memory
  static constexpr int NOB = TRANS ? 1 : 2;                // O store staging tiles
  static constexpr uint32_t TILE = 64 * DK * 2;            // Q, K, V or O tile of one chunk
  static constexpr uint32_t STAGE = (NORM ? 4 : 3) * TILE; // Q | K | V (| ones block)
  static constexpr uint32_t OFF_P = NST * STAGE;           // NPB x [64][64] bf16
  static constexpr uint32_t S_BLOCK = DK * 128;            // [DK][64] bf16, MN-major
  static constexpr uint32_t S_BYTES =                      // one chain's bf16 state (and z)
      TRANS ? 0 : S_BLOCK * (CW / 64 + (NORM ? 1 : 0));
  static constexpr uint32_t OFF_S = OFF_P + NPB * 8192;
  static constexpr uint32_t OFF_O = OFF_S + NCHAIN * S_BYTES;  // NOB x O tile store staging
  static constexpr uint32_t OFF_OFR = OFF_O + NOB * TILE;  // [2][64] output token factors (TRANS)
  static constexpr uint32_t OFF_LAM = OFF_OFR + 2 * 64 * 4;  // [NST][64] inclusive prefix
  static constexpr uint32_t OFF_VF = OFF_LAM + NST * 64 * 4;   // [NST][64] exp(A/2 - Lam_j)
  static constexpr uint32_t OFF_OF = OFF_VF + NST * 64 * 4;    // [NST][64] exp(Lam_i - A/2)
  static constexpr uint32_t OFF_RAW = OFF_OF + NST * 64 * 4;  // [4][64] decay inputs
  static constexpr uint32_t OFF_SPLIT = OFF_RAW + 4 * 64 * 4;  // [NST] split decay used
  static constexpr uint32_t OFF_SCR = OFF_SPLIT + 16 * 4;      // 16 floats
  static constexpr uint32_t OFF_BAR = OFF_SCR + 16 * 4;
  static constexpr int NBAR = 4 * NST + 4 * 2 + 2 * 2 + 1;
  static constexpr uint32_t OFF_CTL = OFF_BAR + 8 * NBAR;
  static constexpr uint32_t OFF_TRC = OFF_CTL + 64;  // trace builds
  static constexpr uint32_t BYTES = OFF_TRC + trace_smem_bytes();
  static_assert(STAGE % 1024 == 0 && OFF_P % 1024 == 0 && OFF_S % 1024 == 0 &&
                    OFF_O % 1024 == 0 && S_BYTES % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  static_assert(BYTES <= 232448, "exceeds the per-block shared memory limit");
  // TMEM columns: P and O by virtual chunk parity, S by chain (CWT columns each).
  // TRANS: O^T buffers of 64 columns (lanes = value columns), S^T fp32 (128
  // columns), and two bf16 copies of S^T as MMA A operands (64 columns each).
  static constexpr uint32_t T_P = 0, T_O = 128, T_OW = TRANS ? 64 : DK + ZW;
  static constexpr uint32_t T_S = 128 + 2 * T_OW, T_SB = T_S + 128, T_COLS = 512;
  static_assert(T_S + NCHAIN * CWT <= T_COLS && (!TRANS || T_SB + 128 <= T_COLS), "TMEM budget");
};

// Warps: 0 TMA, 1 MMA, 2-7 PREP (192 threads), 8-11 WG2, 12-15 WG3.
constexpr int W_PREP = 2, kPrepThreads = 192;
constexpr int WG3 = 12;
constexpr uint32_t BAR_PREP = 1, BAR_WG3 = 3;
// d = 64 without decay or z: a fifth warpgroup (warps 16-19, WG4) takes the O
// epilogue from WG2, whose two epilogues otherwise set the chunk period.  The
// other forms use more registers than 640 threads leave (at most 102 each).
template <int DK, bool DECAY, bool NORM>
constexpr bool kOutWG4 = DK == 64 && !DECAY && !NORM;
template <int DK, bool DECAY, bool NORM>
constexpr int kThreadsOut = kOutWG4<DK, DECAY, NORM> ? 640 : 512;
constexpr int WG4 = 16;
constexpr uint32_t BAR_WG4 = 4;

// Decay of a chunk with total log decay A, reference r = A/2.  Split form:
// the decay between tokens i >= j, exp(Lam_i - Lam_j) = exp(Lam_i - r) *
// exp(r - Lam_j), has its token-j factor folded into the rows of V in shared
// memory and its token-i factor applied to the output rows in registers:
//   V'_j = exp(r - Lam_j) v_j,   O'_i = sum_{j<=i} (q_i . k_j) V'_j + q_i (e^r S_c),
//   O_i  = exp(Lam_i - r) O'_i,  e^r S_c + K^T V' = exp(r - A) S_c+1 in TMEM.
// P = QK^T stays the product of the unscaled operands (so the rounding to
// bf16 comes after q . k cancels), and Q and K need no second pass.  With
// A >= this bound every factor lies in [e^-40, e^40] and every product of two
// in [e^-80, e^80], inside fp32's normal range.  Chunks of stronger decay
// take the per-element form: P_ij exp(Lam_i - Lam_j) in registers, and Q, K
// rescaled in place once QK^T has read them.
constexpr float kSplitMinLogDecay = -80.f;

// P epilogue of a chunk outside the split decay form (total log decay below
// the bound): mask and exp(Lam_i - Lam_j) per element, from TMEM to the
// swizzled bf16 P tile.  Rare, so one compact out-of-line copy: 16 columns
// per step.  Called by all 32 lanes of each warp of the epilogue warpgroup
// (tcgen05.ld is warp-collective).
__device__ __noinline__ void p_tile_strong_decay(uint32_t t_p, int row, const float *lm,
                                                 unsigned char *ps) {
  const float li = row >= 0 ? lm[row] : 0.f;
#pragma unroll 1
  for (int j16 = 0; j16 < 64; j16 += 16) {
    uint32_t r[16];
    __syncwarp();
    tmem_ld16(t_p + j16, r);
    tmem_ld_wait();
    if (row >= 0) {
      uint32_t pk[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const int j0 = j16 + j;
        const float v0 = j0 <= row ? __uint_as_float(r[j]) * __expf(fminf(li - lm[j0], 0.f)) : 0.f;
        const float v1 =
            j0 + 1 <= row ? __uint_as_float(r[j + 1]) * __expf(fminf(li - lm[j0 + 1], 0.f)) : 0.f;
        pk[j >> 1] = pack_bf16(v0, v1);
      }
      st_row16(ps, 8192, row, j16, pk);
    }
  }
}

// Rows of the chunk's Q and K tiles scaled in place for the per-element decay
// form: Qt_i = exp(Lam_i) q_i, Kt_j = exp(A - Lam_j) k_j.  Rare; out of line.
template <int DK>
__device__ __noinline__ void rescale_qk_rows(unsigned char *stage, const float *lm, int t, int n) {
  const float A = lm[63];
  tile_pass<DK, 2, false, true>(
      stage, [lm, A](int kt, int r) { return __expf(kt == 0 ? lm[r] : A - lm[r]); }, t, n);
}

// Two values picked by a 0/1 index known only at run time: a select between
// two registers (an array indexed at run time would sit in local memory,
// and these are read on every chunk).
template <typename T>
struct Pair2 {
  T v0, v1;
  __device__ __forceinline__ T operator[](int i) const { return i ? v1 : v0; }
  __device__ __forceinline__ void set(int i, T x) {
    if (i)
      v1 = x;
    else
      v0 = x;
  }
};

// The virtual-chunk order of a CTA's two segments (d = 64), or of its one
// segment (d = 128: nc[1] = 0).
struct Streams {
  Pair2<int> nc;  // chunks per segment (the second may have none)
  int m;       // chunks both have: virtual 0 .. 2m-1 alternate
  int longer;  // the segment whose chunks follow alone
  __device__ void at(int k, int &sg, int &c) const {
    if (k < 2 * m) {
      sg = k & 1;
      c = k >> 1;
    } else {
      sg = longer;
      c = m + (k - 2 * m);
    }
  }
  __device__ int index(int sg, int c) const { return c < m ? 2 * c + sg : 2 * m + (c - m); }
};

template <int DK, bool PHI, bool DECAY, bool NORM = false>
__global__ void __launch_bounds__((kThreadsOut<DK, DECAY, NORM>), 1)
chunk_output_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmO, TcParams p) {
  using SM = OutSmem<DK, NORM>;
  constexpr int NST = SM::NST;
  constexpr bool PAIRS = SM::PAIRS;
  constexpr int NCHAIN = SM::NCHAIN, CW = SM::CW, CWT = SM::CWT, ZW = SM::ZW;
  constexpr int D = DK;  // d_k = d_v: the state row length
  extern __shared__ __align__(1024) unsigned char smem[];
  float *lam = reinterpret_cast<float *>(smem + SM::OFF_LAM);
  float *vfac = reinterpret_cast<float *>(smem + SM::OFF_VF);
  float *ofac = reinterpret_cast<float *>(smem + SM::OFF_OF);
  uint32_t *split = reinterpret_cast<uint32_t *>(smem + SM::OFF_SPLIT);
  float *scr = reinterpret_cast<float *>(smem + SM::OFF_SCR);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::OFF_BAR);
  uint64_t *empty = full + NST;
  uint64_t *xdone = empty + NST;       // [NST] phi applied, Lam, V rows and factors ready
  uint64_t *qk_ready = xdone + NST;    // [NST] Q, K, V rows hold what MMA2-4 need
  uint64_t *p_full = qk_ready + NST;   // [2] MMA1 done
  uint64_t *p_ready = p_full + 2;      // [2] P in smem
  uint64_t *o_full = p_ready + 2;      // [2] MMA2 done: O complete in TMEM, P smem free
  uint64_t *o_free = o_full + 2;       // [2] O TMEM buffer read
  uint64_t *s_ready = o_free + 2;      // [chain] S_c in smem, scaled S_c in TMEM
  uint64_t *s_done = s_ready + 2;      // [chain] the chain's MMA4 and MMA3 of a chunk done
  uint64_t *drain = s_done + 2;        // abort path: all issued MMAs done
  Ctl *ctl = reinterpret_cast<Ctl *>(smem + SM::OFF_CTL);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) LA_CTA_STAMP(2, 0);
  // Grid (B*H, segment pairs or segments): blocks launch segment by segment,
  // so the shorter last segments of every sequence come last.
  const int bh = blockIdx.x, h = bh % p.H;
  const size_t bhL = (size_t)bh * p.L;
  // Segments of this CTA (one for d = 128).
  Streams st;
  Pair2<int> tok0, seg;
  Pair2<const float *> S_seg;
  Pair2<int> S_ld;  // floats per row of S_seg (a workspace slot row holds z after S when NORM)
#pragma unroll
  for (int sg = 0; sg < 2; ++sg) {
    const int sgi = PAIRS ? 2 * (int)blockIdx.y + sg : (sg == 0 ? (int)blockIdx.y : p.n_seg);
    seg.set(sg, sgi);
    const int c0 = sgi * p.seg_chunks;
    st.nc.set(sg, sgi < p.n_seg ? min(p.seg_chunks, p.n_chunks - c0) : 0);
    tok0.set(sg, c0 * CH);
    const float *src = nullptr;
    if (p.n_seg > 1) {
      S_ld.set(sg, p.srow);
      if (sgi > 0 || p.S0 || (NORM && p.z0))
        src = p.ws_state + ((size_t)bh * p.n_seg + sgi) * D * p.srow;
    } else {
      S_ld.set(sg, D);
      src = p.S0 ? p.S0 + (size_t)bh * D * D : nullptr;
    }
    S_seg.set(sg, src);
  }
  st.m = min(st.nc[0], st.nc[1]);
  st.longer = st.nc[0] >= st.nc[1] ? 0 : 1;
  const int nk = st.nc[0] + st.nc[1];
  // Chain ch: its segment, its first state column, and its chunk index in
  // virtual chunk k.
  auto ch_seg = [&](int ch) { return PAIRS ? ch : 0; };
  auto ch_col = [](int ch) { return PAIRS ? 0 : CW * ch; };
  auto ch_chunk = [&](int ch, int k) {
    int sg, c;
    st.at(k, sg, c);
    return PAIRS ? c : k;
  };
  if (tid == 0) {
    (void)LA_CHK(bh < p.BH && seg[0] < p.n_seg && st.nc[0] >= 1, KID_PREFILL_TC_OUT, 5);
    (void)LA_CHK(!p.S_final || bh < p.BH, KID_PREFILL_TC_OUT, 6);
  }

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&xdone[s], 1);
      mbar_init(&qk_ready[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_ready[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 1);
      mbar_init(&s_ready[i], 1);
      mbar_init(&s_done[i], 1);
    }
    mbar_init(drain, 1);
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
  const bool trace_on = blockIdx.x == 0 && blockIdx.y == 0;
  const long long t0 = clock64();
  (void)trace_on;
  (void)t0;

  float *ofr = reinterpret_cast<float *>(smem + SM::OFF_OFR);  // [2][64] (TRANS)
  // The O epilogue of virtual chunk k, run by one warpgroup (t = 0..127 within
  // it, its lane quarter, its named barrier): WG2, or WG4 where there is one.
  auto o_epilogue_by = [&](int k, int t, int quarter, uint32_t bar) -> bool {
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int b = k & 1;
    if (!wait_wg(&o_full[b], (k >> 1) & 1, ctl, p.err, KID_PREFILL_TC_OUT, 11, bar))
      return false;
    tc_fence_after();
    if (t == 0) tma_store_wait_read<SM::NOB - 1>();  // the store that used this buffer is done
    __syncwarp();
    named_bar_sync(bar, 128);
    unsigned char *o_sm = smem + SM::OFF_O + (b % SM::NOB) * SM::TILE;
    if constexpr (SM::TRANS) {
      // O^T: TMEM lanes are value columns, columns the chunk's 64 tokens.
      // Per 16 lanes (16x256b loads), each 8x8 block (8 value columns x 8
      // tokens) is scaled by its tokens' factors, packed to bf16 and stored
      // transposed (stmatrix .trans): one 16-byte chunk of a token's row of
      // the swizzled staging tile per stored row.
      const int tq = lane & 3;
      float2 fq[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        fq[q] = DECAY ? *reinterpret_cast<const float2 *>(ofr + b * 64 + 8 * q + 2 * tq)
                      : make_float2(1.f, 1.f);
      const uint32_t o_base = smem_u32(o_sm);
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {
        __syncwarp();
        uint32_t r[32];
        tmem_ld_16x256b_x8(tmem + ((uint32_t)(quarter * 32 + 16 * g) << 16) + SM::T_O +
                               SM::T_OW * b,
                           r);
        tmem_ld_wait();
        uint32_t pa[8], pb[8];  // value rows 0-7 and 8-15 of the 16, per token chunk
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          pa[q] = pack_bf16(__uint_as_float(r[4 * q]) * fq[q].x,
                            __uint_as_float(r[4 * q + 1]) * fq[q].y);
          pb[q] = pack_bf16(__uint_as_float(r[4 * q + 2]) * fq[q].x,
                            __uint_as_float(r[4 * q + 3]) * fq[q].y);
        }
#pragma unroll
        for (int qq = 0; qq < 8; qq += 2) {
          // matrices (qq, rows 0-7), (qq, 8-15), (qq+1, 0-7), (qq+1, 8-15)
          const int mi = lane >> 3, tok = 8 * (qq + (mi >> 1)) + (lane & 7);
          const int dv0 = quarter * 32 + 16 * g + 8 * (mi & 1);
          const uint32_t addr = o_base + (dv0 >> 6) * BOX_BYTES + tok * 128 +
                                ((((dv0 & 63) >> 3) ^ (tok & 7)) << 4);
          stmatrix_x4_trans(addr, pa[qq], pb[qq], pa[qq + 1], pb[qq + 1]);
        }
      }
    } else {
      // O has M = 64 as P: 16x256b loads, the rows' output factors, stmatrix.
      const int ra = 16 * quarter + (lane >> 2);
      float fa = DECAY ? ofr[b * 64 + ra] : 1.f, fb = DECAY ? ofr[b * 64 + ra + 8] : 1.f;
      if constexpr (NORM) {
        // The denominator rides in O's column DK (the ones column), with the
        // same output row factor as the numerator: the factor cancels.
        uint32_t dr[4];
        __syncwarp();
        tmem_ld_16x256b_x1(tmem + lane_off + SM::T_O + SM::T_OW * b + DK, dr);
        tmem_ld_wait();
        fa = 1.f / __shfl_sync(0xffffffffu, __uint_as_float(dr[0]), lane & ~3);
        fb = 1.f / __shfl_sync(0xffffffffu, __uint_as_float(dr[2]), lane & ~3);
      }
      const int mi = lane >> 3, srow = 16 * quarter + 8 * (mi & 1) + (lane & 7);
#pragma unroll 1
      for (int col = 0; col < DK; col += 64) {
        __syncwarp();
        uint32_t r[32];
        tmem_ld_16x256b_x8(tmem + lane_off + SM::T_O + SM::T_OW * b + col, r);
        tmem_ld_wait();
        uint32_t pa[8], pb[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          pa[q] = pack_bf16(__uint_as_float(r[4 * q]) * fa, __uint_as_float(r[4 * q + 1]) * fa);
          pb[q] = pack_bf16(__uint_as_float(r[4 * q + 2]) * fb, __uint_as_float(r[4 * q + 3]) * fb);
        }
        const uint32_t rbase = smem_u32(o_sm) + (col / 64) * BOX_BYTES + srow * 128;
#pragma unroll
        for (int qq = 0; qq < 8; qq += 2) {
          const int q = qq + (mi >> 1);
          stmatrix_x4(rbase + ((q ^ (srow & 7)) << 4), pa[qq], pb[qq], pa[qq + 1], pb[qq + 1]);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar_sync(bar, 128);
    if (t == 0) {
      mbar_arrive(&o_free[b]);
      int sg, c;
      st.at(k, sg, c);
      const int tok = tok0[sg] + c * CH;
      for (int bb = 0; bb < DK / BOX; ++bb)
        if (LA_CHK(bb * BOX + BOX <= DK && tok < p.L && bh < p.BH, KID_PREFILL_TC_OUT, 3))
          tma_store_3d(&tmO, o_sm + bb * BOX_BYTES, bb * BOX, tok, bh);
      tma_store_commit();
      LA_TRACE_EVENT(trace_on, t0, 12, k);
    }
    return true;
  };
  if (warp == W_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
      int issued = 0;
      for (int k = 0; k < nk; ++k) {
        const int s = k % NST;
        if (k >= NST &&
            !wait1(&empty[s], ((k / NST) - 1) & 1, ctl, p.err, KID_PREFILL_TC_OUT, 1))
          break;
        int sg, c;
        st.at(k, sg, c);
        unsigned char *stg = smem + s * SM::STAGE;
        mbar_arrive_expect_tx(&full[s], 3 * SM::TILE);  // Q, K, V (not the ones block)
        const int tok = tok0[sg] + c * CH;
        for (int b = 0; b < DK / BOX; ++b) {
          if (!LA_CHK(b * BOX + BOX <= DK && tok < p.L && bh < p.BH, KID_PREFILL_TC_OUT, 2))
            continue;
          tma_load_3d(stg + b * BOX_BYTES, &tmQ, &full[s], b * BOX, tok, bh);
          tma_load_3d(stg + SM::TILE + b * BOX_BYTES, &tmK, &full[s], b * BOX, tok, bh);
          tma_load_3d(stg + 2 * SM::TILE + b * BOX_BYTES, &tmV, &full[s], b * BOX, tok, bh);
        }
        LA_TRACE_EVENT(trace_on, t0, 0, k);
        issued = k + 1;
      }
      if (*(volatile uint32_t *)&ctl->abort)  // loads still landing must land first
        for (int k = max(0, issued - NST); k < issued; ++k) drain_wait(&full[k % NST], (k / NST) & 1);
      // Producer tail: the releases of the last stages come from tcgen05.commit
      // and land asynchronously; wait for them so that no mbarrier arrival
      // reaches this CTA's shared memory after it has exited.
      for (int k = max(0, nk - NST); k < nk; ++k) drain_wait(&empty[k % NST], (k / NST) & 1);
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the scheduler, with every readiness test made
    // warp-uniform by a vote, and one elected lane issues each group of MMAs
    // and its commits.  Operands go in as 32-bit descriptor low words (the
    // high word is one constant): the per-MMA operand arithmetic then stays a
    // 32-bit add, which roughly halves the issue cost of a small MMA against
    // one thread adding 64-bit descriptors.
    if (nk > 0) {
      constexpr uint32_t FULL = 0xffffffffu;
      constexpr uint32_t id_qk = idesc_bf16_f32(64, 64, false, false);
      // NORM: N includes the ones block (V) / z block (S), read as the second
      // 64-column MN block of the operand (V's next tile / the S copy's z block).
      constexpr uint32_t id_pv = idesc_bf16_f32(64, DK + ZW, false, true);
      constexpr uint32_t id_qs = idesc_bf16_f32(64, CW + ZW, false, true);
      constexpr uint32_t id_kv = idesc_bf16_f32(DK, CW + ZW, true, true);
      // Transposed forms (TRANS): S^T += V^T K, O^T = S^T Q^T (A in TMEM),
      // O^T += V^T P^T.  M = 128 value columns in every one.
      constexpr uint32_t id_kvT = idesc_bf16_f32(DK, DK, true, true);
      constexpr uint32_t id_qsT = idesc_bf16_f32(DK, 64, false, false);
      constexpr uint32_t id_pvT = idesc_bf16_f32(DK, 64, true, false);
      // Descriptor low words of each layout at the start of shared memory;
      // an operand at byte offset off adds off >> 4 (shared memory ends below
      // 256 KB, so the 14-bit address field never carries).
      constexpr uint32_t HI = smem_desc_sw128_hi(1024);
      const uint32_t sbase = smem_u32(smem);
      const uint32_t dKM = smem_desc_sw128_lo(sbase, 16);          // K-major rows
      const uint32_t dMN = smem_desc_sw128_lo(sbase, BOX_BYTES);   // MN-major, 8 KB blocks
      const uint32_t dMS = smem_desc_sw128_lo(sbase, SM::S_BLOCK); // MN-major state blocks
      auto at = [](uint32_t d, uint32_t off) { return d + (off >> 4); };
      auto ready = [&](uint64_t *bar, uint32_t par) { return __all_sync(FULL, mbar_test(bar, par)); };
      // Three streams of MMA work, issued as each becomes ready (non-blocking
      // tests), so that a late input of one never holds up another:
      //   chain step kc: per chain, S += K^T V and O = Q S_c (needs the
      //     chain's state, Q/K/V rows in final form, O buffer kc & 1 free);
      //   P V of chunk km (needs P in smem; after its chain step);
      //   QK^T of chunk kq (needs its tiles; the shared-memory P tile it
      //     leads to is free once P V of chunk kq - NPB is issued:
      //     kq <= km + NPB - 1; MMAs complete in issue order).
      // In each stream the chunks go in order, and every test is of a phase
      // that cannot yet be overtaken by the next one on the same barrier.
      int kq = 0, kc = 0, cc = 0, km = 0;  // cc: next chain within step kc
      bool ok = true;
      uint64_t idle_since = 0;
      uint32_t idle_polls = 0;
      while (ok && km < nk) {
        bool did = false;
        if (kc < nk) {  // ---- chain step
          int sg, c;
          st.at(kc, sg, c);
          const int s = kc % NST, b = kc & 1;
          const int ch = PAIRS ? sg : cc;
          // Q, K, V of the chunk in their final form: phi applied (xdone) and,
          // with decay, the rows scaled (qk_ready, which follows xdone).
          const bool inputs =
              (cc > 0) || ((kc < 2 || ready(&o_free[b], ((kc >> 1) - 1) & 1)) &&
                           ready(DECAY ? &qk_ready[s] : &xdone[s], (kc / NST) & 1));
          if (inputs && ready(&s_ready[ch], ch_chunk(ch, kc) & 1)) {
            tc_fence_after();
            LA_TRACE_EVENT(trace_on && lane == 0 && cc == 0, t0, 8, kc);
            const uint32_t qo = s * SM::STAGE, ko = qo + SM::TILE, vo = qo + 2 * SM::TILE;
            const uint32_t o_t = tmem + SM::T_O + SM::T_OW * b;
            const bool inter = NORM || S_seg[sg] != nullptr || c > 0;
            if constexpr (SM::TRANS) {
              // The chain is S^T += V^T K alone; O^T = S^T Q^T follows it off the
              // chain (its bf16 S^T copy is double-buffered in TMEM).
              const uint32_t sb = tmem + SM::T_SB + 64 * (c & 1);
              if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < CH / 16; ++kk)
                  mma_bf16_w(tmem + SM::T_S, at(dMN, vo + 2048 * kk), at(dMN, ko + 2048 * kk), HI,
                             id_kvT, (inter || kk > 0) ? 1u : 0u);
                mma_commit(&s_done[0]);
                if (inter) {
#pragma unroll
                  for (int kk = 0; kk < DK / 16; ++kk)
                    mma_bf16_ta_w(o_t, sb + 8 * kk,
                                  at(dKM, qo + (kk / 4) * BOX_BYTES + 32 * (kk % 4)), HI, id_qsT,
                                  kk > 0);
                }
              }
              __syncwarp();
              ++kc;
            } else {
              const uint32_t vb = vo + (PAIRS ? 0u : (uint32_t)(ch * (CW / 64)) * BOX_BYTES);
              const uint32_t so = SM::OFF_S + ch * SM::S_BYTES;
              if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < CH / 16; ++kk)  // chain state: S (TMEM) += K^T V
                  mma_bf16_w(tmem + SM::T_S + CWT * ch, at(dMN, ko + 2048 * kk),
                             at(dMN, vb + 2048 * kk), HI, id_kv, (inter || kk > 0) ? 1u : 0u);
                if (inter) {
#pragma unroll
                  for (int kk = 0; kk < DK / 16; ++kk)  // O[:, chain] = Q S_c[:, chain]
                    mma_bf16_w(o_t + ch_col(ch), at(dKM, qo + (kk / 4) * BOX_BYTES + 32 * (kk % 4)),
                               at(dMS, so + 2048 * kk), HI, id_qs, kk > 0);
                }
                mma_commit(&s_done[ch]);
              }
              __syncwarp();
              if (PAIRS || ++cc == NCHAIN) {
                cc = 0;
                ++kc;
              }
            }
            if (cc == 0) LA_TRACE_EVENT(trace_on && lane == 0, t0, 9, kc - 1);
            did = true;
          }
        }
        if (km < kc) {  // ---- P V
          int sg, c;
          st.at(km, sg, c);
          const int s = km % NST, b = km & 1;
          if (ready(&p_ready[b], (km >> 1) & 1)) {
            tc_fence_after();
            LA_TRACE_EVENT(trace_on && lane == 0, t0, 5, km);
            const uint32_t vo = s * SM::STAGE + 2 * SM::TILE, po = SM::OFF_P + 8192 * (b % SM::NPB);
            const bool inter = NORM || S_seg[sg] != nullptr || c > 0;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < CH / 16; ++kk) {  // O += P V   (TRANS: O^T += V^T P^T)
                if constexpr (SM::TRANS)
                  mma_bf16_w(tmem + SM::T_O + SM::T_OW * b, at(dMN, vo + 2048 * kk),
                             at(dKM, po + 32 * kk), HI, id_pvT, (inter || kk > 0) ? 1u : 0u);
                else
                  mma_bf16_w(tmem + SM::T_O + SM::T_OW * b, at(dKM, po + 32 * kk),
                             at(dMN, vo + 2048 * kk), HI, id_pv, (inter || kk > 0) ? 1u : 0u);
              }
              mma_commit(&o_full[b]);
              mma_commit(&empty[s]);
            }
            __syncwarp();
            LA_TRACE_EVENT(trace_on && lane == 0, t0, 6, km);
            ++km;
            did = true;
          }
        }
        if (kq < nk && kq <= km + SM::NPB - 1) {  // ---- QK^T
          const int s = kq % NST;
          if (ready(&xdone[s], (kq / NST) & 1)) {
            tc_fence_after();
            const uint32_t so = s * SM::STAGE;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < DK / 16; ++kk) {
                const uint32_t off = so + (kk / 4) * BOX_BYTES + 32 * (kk % 4);
                mma_bf16_w(tmem + SM::T_P + 64 * (kq & 1), at(dKM, off), at(dKM, off + SM::TILE), HI,
                           id_qk, kk > 0);
              }
              mma_commit(&p_full[kq & 1]);
            }
            __syncwarp();
            LA_TRACE_EVENT(trace_on && lane == 0, t0, 7, kq);
            ++kq;
            did = true;
          }
        }
        if (did) {
          idle_polls = 0;
          idle_since = 0;
        } else if (++idle_polls == 256) {  // spin (a sleep delays the reaction to a barrier
                                        // by far more than asked); bounded: give up after the limit
          idle_polls = 0;
          const uint64_t now = __shfl_sync(FULL, global_timer_ns(), 0);
          if (idle_since == 0) {
            idle_since = now;
          } else if (now - idle_since > kWaitNs ||
                     __any_sync(FULL, *(volatile uint32_t *)&ctl->abort != 0)) {
            if (lane == 0 && !*(volatile uint32_t *)&ctl->abort) {
              atomicExch(&ctl->abort, 1u);
              record_device_error(p.err, KID_PREFILL_TC_OUT, 20);
            }
            ok = false;
          }
        }
      }
      if (!ok) {  // let every issued MMA finish before TMEM is released
        if (elect_one()) {  // the lane that issued them
          mma_commit(drain);
          drain_wait(drain, 0);
        }
        __syncwarp();
      }
    }
  } else if (warp >= W_PREP && warp < WG2) {
    // ------------------------------------------------------------ PREP: Lam, phi, decay factors
    const int t = tid - W_PREP * 32;  // 0..191
    auto gwait = [&](uint64_t *bar, uint32_t par, uint32_t site) {
      return wait_grp<kPrepThreads>(bar, par, ctl, p.err, KID_PREFILL_TC_OUT, site, BAR_PREP, t);
    };
    // Threads t < 64 fetch their token's decay input three chunks ahead, as an
    // asynchronous copy into a ring of four chunk slots: a DRAM round trip under
    // full load can take longer than a chunk, and no register waits on it.
    // Each fetch is one copy group of the thread (empty past the last chunk),
    // so at prep(k) the groups of chunks k, k + 1, k + 2 are the pending ones.
    float *rawbuf = reinterpret_cast<float *>(smem + SM::OFF_RAW);
    auto fetch = [&](int k) {
      if (k < nk) {
        int sg, c;
        st.at(k, sg, c);
        const int tok = tok0[sg] + c * CH + t;
        float *dst = rawbuf + (k & 3) * 64 + t;
        if (tok < p.L)
          cp_async_4(dst, p.decay_kind == LA_DECAY_HEAD ? p.decay + h : p.decay + bhL + tok);
        else
          *dst = token_decay_raw(p.decay_kind, p.decay, h, bhL, tok, p.L);
      }
      cp_async_commit();
    };
    if (DECAY && t < 64) {
      fetch(0);
      fetch(1);
      fetch(2);
    }
    auto prep = [&](int k) -> bool {
      const int s = k % NST;
      if (!gwait(&full[s], (k / NST) & 1, 7)) return false;
      LA_TRACE_EVENT(trace_on && t == 0, t0, 1, k);
      unsigned char *qt = smem + s * SM::STAGE;
      bool sp = false;  // uniform over the group
      if constexpr (DECAY) {
        if (t < 64) {  // inclusive prefix of the chunk's log decays (warps 2, 3)
          cp_async_wait<2>();  // chunk k's group is complete
          float x = token_log_decay(p.decay_kind, rawbuf[(k & 3) * 64 + t]);
          fetch(k + 3);  // into chunk k - 1's slot, read by this thread at prep(k - 1)
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
          }
          if (t == 31) scr[0] = x;
          lam[s * 64 + t] = x;
        }
        named_bar_sync(BAR_PREP, kPrepThreads);
        if (t >= 32 && t < 64) lam[s * 64 + t] += scr[0];
        named_bar_sync(BAR_PREP, kPrepThreads);
        const float A = lam[s * 64 + 63];
        sp = A >= kSplitMinLogDecay;
        if (t < 64 && sp) {
          const float li = lam[s * 64 + t];
          vfac[s * 64 + t] = __expf(0.5f * A - li);
          ofac[s * 64 + t] = __expf(li - 0.5f * A);
        }
        if (t == 0) split[s] = sp ? 1u : 0u;
        if (sp) named_bar_sync(BAR_PREP, kPrepThreads);  // factors visible to the V pass
      }
      if constexpr (NORM) {  // the ones block after V: column 0 = V's row factor, the rest 0
        if (t < 64) {
          // Rows past the sequence end hold zero-filled keys that phi may map
          // to non-zero values (elu + 1 gives 1): their ones must be zero, as
          // their zero-filled values are, or they would be added to z.
          int sg, c;
          st.at(k, sg, c);
          const bool live = tok0[sg] + c * CH + t < p.L;
          const float f = !live ? 0.f : (DECAY && sp) ? vfac[s * 64 + t] : 1.f;
          unsigned char *ob = qt + 3 * SM::TILE + t * 128;
          *reinterpret_cast<uint4 *>(ob + ((0 ^ (t & 7)) << 4)) = make_uint4(pack_bf16(f, 0.f), 0u, 0u, 0u);
          *reinterpret_cast<uint4 *>(ob + ((1 ^ (t & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      if constexpr (PHI) {  // Q and K tiles are adjacent in the stage: one pass
        tile_pass<DK, 2, true, false>(qt, [](int, int) { return 1.f; }, t, kPrepThreads);
        fence_proxy_async_smem();
      }
      named_bar_sync(BAR_PREP, kPrepThreads);
      if (t == 0) mbar_arrive(&xdone[s]);  // QK^T may start; V is scaled meanwhile
      LA_TRACE_EVENT(trace_on && t == 0, t0, 2, k);
      if (DECAY && sp) {  // the MMAs that read V wait for qk_ready
        const float *vf = vfac + s * 64;
        tile_pass<DK, 1, false, true>(qt + 2 * SM::TILE, [vf](int, int r) { return vf[r]; }, t,
                                      kPrepThreads);
        fence_proxy_async_smem();
        named_bar_sync(BAR_PREP, kPrepThreads);
        if (t == 0) mbar_arrive(&qk_ready[s]);
        LA_TRACE_EVENT(trace_on && t == 0, t0, 15, k);
      }
      return true;
    };
    // Per-element decay form: once QK^T of the chunk has consumed the
    // unscaled tiles, scale the rows in place: Qt_i = exp(Lam_i) q_i,
    // Kt_j = exp(A - Lam_j) k_j (both factors <= 1).
    auto rescale = [&](int k) -> bool {
      const int s = k % NST, b = k & 1;
      if (!gwait(&p_full[b], (k >> 1) & 1, 8)) return false;
      LA_TRACE_EVENT(trace_on && t == 0, t0, 13, k);
      rescale_qk_rows<DK>(smem + s * SM::STAGE, lam + s * 64, t, kPrepThreads);
      fence_proxy_async_smem();
      named_bar_sync(BAR_PREP, kPrepThreads);
      if (t == 0) mbar_arrive(&qk_ready[s]);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 14, k);
      return true;
    };
    // prep(0), then prep(k + 1) before rescale(k): each lambda has one call
    // site, so it is inlined and its captures (the decay ring) stay in registers.
    bool ok = true;
    for (int k = 0; ok && k <= nk; ++k) {
      if (k < nk && !(ok = prep(k))) break;
      if constexpr (DECAY) {
        if (k > 0 && !split[(k - 1) % NST] && !(ok = rescale(k - 1))) break;
      }
    }
  } else if (warp >= WG2 && warp < WG3) {
    // ------------------------------------------------------------ WG2: P and O epilogues
    const int t = tid - WG2 * 32;
    const int quarter = warp & 3;
    const int row = acc_row<64>(quarter, lane);   // row within the chunk
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    auto p_epilogue = [&](int k) -> bool {
      const int s = k % NST, b = k & 1;
      if (DECAY && !wait_wg(&xdone[s], (k / NST) & 1, ctl, p.err, KID_PREFILL_TC_OUT, 15, BAR_WG2))
        return false;
      if (!wait_wg(&p_full[b], (k >> 1) & 1, ctl, p.err, KID_PREFILL_TC_OUT, 9, BAR_WG2))
        return false;
      tc_fence_after();
      LA_TRACE_EVENT(trace_on && t == 0, t0, 3, k);
      unsigned char *ps = smem + SM::OFF_P + 8192 * (b % SM::NPB);
      // Causal mask.  Split-form chunks need nothing more here (their row
      // factor is applied by the O epilogue); others take their decay per
      // element, out of line.
      const bool sp = !DECAY || split[s];
      if (DECAY && t < 64)  // the chunk's output row factors, for its O epilogue
        ofr[b * 64 + t] = sp ? ofac[s * 64 + t] : 1.f;
      if (!sp) {
        p_tile_strong_decay(tmem + lane_off + SM::T_P + 64 * b, row, lam + s * 64, ps);
      } else {
        // P has M = 64: rows 16 quarter + 0..15 sit in the quarter's first 16
        // lanes.  A 16x256b load spreads them over all 32 threads in the 8x8
        // fragment layout (rows ra and ra + 8, columns 8 q + c2, +1), which
        // stmatrix stores into the swizzled tile, 16 bytes per matrix row.
        __syncwarp();
        uint32_t r[32];
        tmem_ld_16x256b_x8(tmem + lane_off + SM::T_P + 64 * b, r);
        tmem_ld_wait();
        const int ra = 16 * quarter + (lane >> 2), c2 = 2 * (lane & 3);
        uint32_t pa[8], pb[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int j = 8 * q + c2;  // causal mask: keep key j <= query row
          pa[q] = pack_bf16(j <= ra ? __uint_as_float(r[4 * q]) : 0.f,
                            j + 1 <= ra ? __uint_as_float(r[4 * q + 1]) : 0.f);
          pb[q] = pack_bf16(j <= ra + 8 ? __uint_as_float(r[4 * q + 2]) : 0.f,
                            j + 1 <= ra + 8 ? __uint_as_float(r[4 * q + 3]) : 0.f);
        }
        const int mi = lane >> 3, srow = 16 * quarter + 8 * (mi & 1) + (lane & 7);
        const uint32_t rbase = smem_u32(ps) + srow * 128;
#pragma unroll
        for (int qq = 0; qq < 8; qq += 2) {
          const int q = qq + (mi >> 1);
          stmatrix_x4(rbase + ((q ^ (srow & 7)) << 4), pa[qq], pb[qq], pa[qq + 1], pb[qq + 1]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_WG2, 128);
      if (t == 0) mbar_arrive(&p_ready[b]);
      LA_TRACE_EVENT(trace_on && t == 0, t0, 4, k);
      return true;
    };
    auto o_epilogue = [&](int k) { return o_epilogue_by(k, t, quarter, BAR_WG2); };
    bool ok = true;
    constexpr bool own_o = !kOutWG4<DK, DECAY, NORM>;
    for (int k = 0; ok && k < nk; ++k) {
      ok = p_epilogue(k);
      if (own_o && ok && k >= 1) ok = o_epilogue(k - 1);
    }
    if (own_o && ok && nk > 0) o_epilogue(nk - 1);
    if (own_o && t == 0) tma_store_wait_all();
  } else if (kOutWG4<DK, DECAY, NORM> && warp >= WG4) {
    // ------------------------------------------------------------ WG4: O epilogues
    const int t = tid - WG4 * 32;
    bool ok = true;
    for (int k = 0; ok && k < nk; ++k) ok = o_epilogue_by(k, t, warp & 3, BAR_WG4);
    if (t == 0) tma_store_wait_all();
  } else if (warp >= WG3) {
    // ------------------------------------------------------------ WG3: the state chains
    const int t = tid - WG3 * 32;
    const int quarter = warp & 3;
    const int srow = acc_row<DK>(quarter, lane);    // state row (d_k index)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // 32 columns of state row srow: r * sm_scale as bf16 into a chain's S
    // buffer, and optionally r * tm_scale back into the chain's TMEM state.
    auto put32 = [&](int ch, int col, uint32_t (&r)[32], float sm_scale, float tm_scale,
                     bool to_tmem) {
      if (srow >= 0) {
#pragma unroll
        for (int q16 = 0; q16 < 2; ++q16) {
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            pk[j] = pack_bf16(__uint_as_float(r[q16 * 16 + 2 * j]) * sm_scale,
                              __uint_as_float(r[q16 * 16 + 2 * j + 1]) * sm_scale);
          st_row16(smem + SM::OFF_S + ch * SM::S_BYTES, SM::S_BLOCK, srow, col + q16 * 16, pk);
        }
      }
      if (to_tmem) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * tm_scale);
        __syncwarp();
        tmem_st32(tmem + lane_off + SM::T_S + CWT * ch + col, r);
      }
    };
    // NORM: the chain's z column (state column DK; the next 15 stay zero):
    // z * sm_scale into the bf16 copy's z block, z * tm_scale back into TMEM.
    auto putz = [&](int ch, float z, float sm_scale, float tm_scale, bool to_tmem) {
      if (srow >= 0) {
        const uint32_t pk[8] = {pack_bf16(z * sm_scale, 0.f), 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        st_row16(smem + SM::OFF_S + ch * SM::S_BYTES, SM::S_BLOCK, srow, CW, pk);
      }
      if (to_tmem) {
        uint32_t r16[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) r16[j] = 0u;
        r16[0] = __float_as_uint(z * tm_scale);
        __syncwarp();
        tmem_st16(tmem + lane_off + SM::T_S + CWT * ch + CW, r16);
      }
    };
    auto getz = [&](int ch) -> float {  // the chain's z from TMEM (warp-collective)
      uint32_t r16[16];
      __syncwarp();
      tmem_ld16(tmem + lane_off + SM::T_S + CWT * ch + CW, r16);
      tmem_ld_wait();
      return __uint_as_float(r16[0]);
    };
    // TRANS: this thread's TMEM lane is value column dv = t of S^T.  32 state
    // rows (d_k = 32 cb ..) of that column: r * sm packed to bf16 pairs into
    // A-operand copy `buf` (column = pair of d_k), and r * tm back into the
    // fp32 S^T when to_fp32.
    auto put_trans = [&](int cb, int buf, uint32_t (&r)[32], float sm, float tm, bool to_fp32) {
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = pack_bf16(__uint_as_float(r[2 * j]) * sm, __uint_as_float(r[2 * j + 1]) * sm);
      __syncwarp();
      tmem_st16(tmem + lane_off + SM::T_SB + 64 * buf + 16 * cb, pk);
      if (to_fp32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * tm);
        __syncwarp();
        tmem_st32(tmem + lane_off + SM::T_S + 32 * cb, r);
      }
    };
    // Scales of a chain's state at one of its chunks (decay kernels), as
    // natural logarithms:
    //   smem copy  S_c * e^{m}   (m = r = A/2 in the split form, else 0),
    //   TMEM       S_c * e^{t}   (t = r in the split form, else A),
    // and after the chunk's MMA4 the TMEM holds S_c+1 * e^{-g} (g = A - r =
    // A/2 in the split form, else 0).  k is the chunk's virtual index.
    auto log_scales = [&](int k, float &m, float &tt, float &g) {
      const int s = k % NST;
      const float A = lam[s * 64 + 63];
      if (split[s]) {
        m = tt = g = 0.5f * A;
      } else {
        m = g = 0.f;
        tt = A;
      }
    };
    Pair2<float> g_prev{0.f, 0.f};  // per chain: g of its chunk whose MMA4 is next awaited
    bool ok = true;
    // The incoming segment states come from the scan, which this kernel may
    // have been launched alongside (programmatic dependent launch): only this
    // warpgroup reads them, so only it waits for the scan grid to finish.
    if (p.n_seg > 1) pdl_wait_previous();
    if (t == 0) LA_CTA_STAMP(2, 1);
    // Initial states, chain by chain (a chain's first chunk is virtual 0 or 1).
    for (int ch = 0; ok && ch < NCHAIN; ++ch) {
      const int sg = ch_seg(ch);
      if (st.nc[sg] == 0) continue;
      const int k = PAIRS ? st.index(sg, 0) : 0;
      float m0 = 0.f, t0s = 0.f;
      if constexpr (DECAY) {
        ok = wait_wg(&xdone[k % NST], (k / NST) & 1, ctl, p.err, KID_PREFILL_TC_OUT, 12, BAR_WG3);
        if (!ok) break;
        float g0;
        log_scales(k, m0, t0s, g0);
        g_prev.set(ch, g0);
      }
      if (SM::TRANS && S_seg[sg] != nullptr) {
        const float sm0 = __expf(m0), tm0 = __expf(t0s);
#pragma unroll 1
        for (int cb = 0; cb < DK / 32; ++cb) {
          uint32_t r[32];
          const float *src = S_seg[sg] + (size_t)(32 * cb) * D + t;  // column t, rows 32 cb ..
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(src[(size_t)j * D]);
          put_trans(cb, 0, r, sm0, tm0, true);
        }
        tmem_st_wait();
      } else if (NORM || S_seg[sg] != nullptr) {
        const float sm0 = __expf(m0), tm0 = __expf(t0s);
        if constexpr (NORM) {  // z: column D of a slot row, or z0 at the sequence start
          float z = 0.f;
          if (srow >= 0) {
            if (p.n_seg > 1 && S_seg[sg] != nullptr) z = S_seg[sg][(size_t)srow * S_ld[sg] + D];
            else if (p.n_seg == 1 && p.z0) z = p.z0[(size_t)bh * D + srow];
          }
          putz(ch, z, sm0, tm0, true);
        }
#pragma unroll 1
        for (int col = 0; col < CW; col += 32) {
          uint32_t r[32];
          if (srow >= 0 && S_seg[sg] != nullptr) {
            const float4 *src = reinterpret_cast<const float4 *>(S_seg[sg] + (size_t)srow * S_ld[sg] +
                                                                 ch_col(ch) + col);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float4 f = src[j];
              r[4 * j] = __float_as_uint(f.x);
              r[4 * j + 1] = __float_as_uint(f.y);
              r[4 * j + 2] = __float_as_uint(f.z);
              r[4 * j + 3] = __float_as_uint(f.w);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
          put32(ch, col, r, sm0, tm0, true);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(BAR_WG3, 128);
      if (t == 0) mbar_arrive(&s_ready[ch]);
    }
    for (int k = 0; ok && k < nk; ++k) {
      int sg, c;
      st.at(k, sg, c);
      const bool more = c + 1 < st.nc[sg];
      const int kn = PAIRS ? (more ? st.index(sg, c + 1) : 0) : k + 1;
      float lm1 = 0.f, lt1 = 0.f, lg1 = 0.f;  // log scales of the chain's next chunk
      if (DECAY && more) {
        if (!(ok = wait_wg(&xdone[kn % NST], (kn / NST) & 1, ctl, p.err, KID_PREFILL_TC_OUT, 14,
                           BAR_WG3)))
          break;
        log_scales(kn, lm1, lt1, lg1);
      }
      for (int ch = PAIRS ? sg : 0; ok && ch <= (PAIRS ? sg : NCHAIN - 1); ++ch) {
        if (!(ok = wait_wg(&s_done[ch], c & 1, ctl, p.err, KID_PREFILL_TC_OUT, 13, BAR_WG3)))
          break;
        tc_fence_after();
        LA_TRACE_EVENT(trace_on && t == 0, t0, 10, k);
        if (more) {
          // TMEM holds S_c+1 * e^{-g_c}.  Copy S_c+1 * e^{m_c+1} to bf16 for
          // the next chunk's Q S, and leave S_c+1 * e^{t_c+1} in TMEM for its
          // state update.  Each scale is one exponential of a sum >= -80.
          float sm = 1.f, tm = 1.f;
          if constexpr (DECAY) {
            sm = __expf(g_prev[ch] + lm1);
            tm = __expf(g_prev[ch] + lt1);
            g_prev.set(ch, lg1);
          }
          if constexpr (SM::TRANS) {
            // TMEM to TMEM: the copy for chunk c+1 goes to buffer (c+1) & 1;
            // the Q S of chunk c-1 that read it finished before this chunk's
            // state MMA (s_done tracks every earlier MMA).
#pragma unroll 1
            for (int cb = 0; cb < DK / 32; ++cb) {
              __syncwarp();
              uint32_t r[32];
              tmem_ld32(tmem + lane_off + SM::T_S + 32 * cb, r);
              tmem_ld_wait();
              put_trans(cb, (c + 1) & 1, r, sm, tm, DECAY);
            }
            tmem_st_wait();
          } else {
#pragma unroll 1
          for (int col = 0; col < CW; col += 64) {
            __syncwarp();
            uint32_t r[2][32];
            tmem_ld32(tmem + lane_off + SM::T_S + CWT * ch + col, r[0]);
            tmem_ld32(tmem + lane_off + SM::T_S + CWT * ch + col + 32, r[1]);
            tmem_ld_wait();
            put32(ch, col, r[0], sm, tm, DECAY);
            put32(ch, col + 32, r[1], sm, tm, DECAY);
          }
          if constexpr (NORM) putz(ch, getz(ch), sm, tm, DECAY);
          if (DECAY) tmem_st_wait();
          }
          fence_proxy_async_smem();
          tc_fence_before();
          named_bar_sync(BAR_WG3, 128);
          if (t == 0) mbar_arrive(&s_ready[ch]);
          LA_TRACE_EVENT(trace_on && t == 0, t0, 11, k);
        } else if (SM::TRANS && seg[sg] == p.n_seg - 1 && p.S_final) {
          const float fin = DECAY ? __expf(g_prev[ch]) : 1.f;
#pragma unroll 1
          for (int cb = 0; cb < DK / 32; ++cb) {
            __syncwarp();
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + SM::T_S + 32 * cb, r);
            tmem_ld_wait();
            float *dst = p.S_final + ((size_t)bh * D + 32 * cb) * D + t;  // column t
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[(size_t)j * D] = __uint_as_float(r[j]) * fin;
          }
        } else if (seg[sg] == p.n_seg - 1 && (p.S_final || (NORM && p.z_final))) {
          const float fin = DECAY ? __expf(g_prev[ch]) : 1.f;
          if constexpr (NORM) {
            const float z = getz(ch);
            if (srow >= 0 && p.z_final) p.z_final[(size_t)bh * D + srow] = z * fin;
          }
#pragma unroll 1
          for (int col = 0; col < CW && p.S_final; col += 32) {
            __syncwarp();
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + SM::T_S + CWT * ch + col, r);
            tmem_ld_wait();
            if (srow >= 0) {
              float4 *dst = reinterpret_cast<float4 *>(p.S_final + ((size_t)bh * D + srow) * D +
                                                       ch_col(ch) + col);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(__uint_as_float(r[4 * j]) * fin,
                                     __uint_as_float(r[4 * j + 1]) * fin,
                                     __uint_as_float(r[4 * j + 2]) * fin,
                                     __uint_as_float(r[4 * j + 3]) * fin);
            }
          }
        }
      }
    }
  }
  __syncwarp();  // lanes that skipped a lane-0 role loop wait for lane 0
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) {
    __syncwarp();
    tmem_dealloc(tmem, SM::T_COLS);
  }
  LA_TRACE_FLUSH(trace_on, &g_trace[0][0]);
  if (tid == 0) LA_CTA_STAMP(2, 2);
}

// ---------------------------------------------------------------- planning
struct Plan {
  int n_chunks, seg_chunks, n_seg;
};

// Segment count.  The output kernel runs ceil(NS/2) x BH CTAs of two
// segments each (d = 64) or NS x BH CTAs of one (d = 128); the segment-state
// kernel (NS > 1) runs (NS-1) x BH CTAs, two per SM, and reads K and V of all
// but the last segment once more; the scan moves the segment states.  The estimate of each
// kernel is the larger of its wave time -- waves x (fixed CTA cost + chunk
// steps x step time) -- and its bytes over the HBM bandwidth; step times and
// fixed costs are measured ones for these kernels on GB300 (microseconds; the
// d = 128 output step is the ~1.45 us per chunk of the traced steady state).
// G <= 32 bounds the segment-state kernel's suffix table.
Plan make_plan(int B, int H, int L, int D) {
  const int nc = (L + CH - 1) / CH;
  const bool halves = D == 128;  // one segment per output CTA
  const double bh = (double)B * H, sms = sm_count();
  const double t_out = 1.5, t_state = halves ? 0.7 : 0.4;
  const double fill_out = 3.0, fill_state = 2.0, t_launch = 3.0, bw = 6.5e3;  // bytes per us / 1e3
  const double tile = 64.0 * D * 2, state = (double)D * D * 4;
  Plan best{nc, nc, 1};
  double best_t = 1e300;
  for (int ns = 1; ns <= std::min(nc, 256); ++ns) {
    const int g = (nc + ns - 1) / ns;
    const int n_seg = (nc + g - 1) / g;
    if (g > kMaxSegChunks || n_seg != ns) continue;
    const double ctas = (halves ? (double)n_seg : std::ceil(n_seg / 2.0)) * bh;
    const double steps = (halves || n_seg == 1) ? (double)g : 2.0 * g;
    const double out_bytes = bh * (nc * 4.0 * tile + (n_seg > 1 ? n_seg * state : 0.0));
    double t = std::max(std::ceil(ctas / sms) * (fill_out + steps * t_out), out_bytes / bw * 1e-3);
    if (n_seg > 1) {
      const double sctas = (n_seg - 1) * bh;
      const double st_bytes = bh * ((n_seg - 1) * (g * 2.0 * tile + state));
      // (a last partial wave at two CTAs per SM runs its CTAs faster: fractional)
      t += std::max(sctas / (2 * sms) * (fill_state + g * t_state), st_bytes / bw * 1e-3);
      t += 2 * t_launch + bh * n_seg * 2.0 * state / bw * 1e-3;
    }
    if (t < best_t) {
      best_t = t;
      best = Plan{nc, g, n_seg};
    }
  }
  return best;
}

// srow: floats per state row in a slot (D, or D + 16 for the normalised form).
size_t ws_bytes_for(int B, int H, int L, int D, int srow) {
  Plan pl = make_plan(B, H, L, D);
  if (pl.n_seg <= 1) return 0;
  const size_t bh = (size_t)B * H;
  const size_t st = bh * pl.n_seg * (size_t)D * srow * sizeof(float);
  return st + ((bh * pl.n_seg * sizeof(float) + 255) & ~(size_t)255);
}

// The segment-state pass over grid = (segments, sequences).  At d = 128, when
// K is transformed (phi or decay weights) and the grid fits in one wave of two
// blocks per SM, the deep three-stage form, whose two groups share each
// chunk's transform; else the two-stage form, of which three blocks fit on an
// SM.  (Measured on B1 H16 L32768: 3.4 us less per call with decay, none
// without a transform.)
template <int D, bool PHI, bool DECAY, bool NORM>
cudaError_t launch_state(dim3 grid, const CUtensorMap &tk, const CUtensorMap &tv,
                         const TcParams &p, cudaStream_t stream) {
  cudaError_t e;
  if constexpr (D == 128 && !NORM && (PHI || DECAY)) {
    if ((long)grid.x * grid.y <= 2L * sm_count()) {
      using SS = StateSmem<D, NORM, true>;
      auto ks = segment_state_kernel<D, PHI, DECAY, NORM, true>;
      static int smem_set_deep[64];
      if ((e = set_smem_once(ks, SS::BYTES, smem_set_deep)) != cudaSuccess) return e;
      ks<<<grid, kThreadsState, SS::BYTES, stream>>>(tk, tv, p);
      return cudaGetLastError();
    }
  }
  using SS = StateSmem<D, NORM>;
  auto ks = segment_state_kernel<D, PHI, DECAY, NORM>;
  static int smem_set_state[64];
  if ((e = set_smem_once(ks, SS::BYTES, smem_set_state)) != cudaSuccess) return e;
  ks<<<grid, kThreadsState, SS::BYTES, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int D, bool PHI, bool DECAY, bool NORM = false>
cudaError_t launch_d(const PrefillArgs &a, const char **why, const float *z0 = nullptr,
                     float *z_final = nullptr) {
  const Plan pl = make_plan(a.B, a.H, a.L, D);
  const int BH = a.B * a.H;
  TcParams p{};
  p.H = a.H;
  p.L = a.L;
  p.BH = BH;
  p.n_chunks = pl.n_chunks;
  p.seg_chunks = pl.seg_chunks;
  p.n_seg = pl.n_seg;
  p.phi = a.phi;
  p.decay_kind = a.decay_kind;
  p.decay = a.decay;
  p.S0 = a.S0;
  p.S_final = a.S_final;
  p.err = device_error_word();
  p.srow = NORM ? D + 16 : D;
  p.z0 = z0;
  p.z_final = z_final;
  if (pl.n_seg > 1) {
    p.ws_state = static_cast<float *>(a.workspace);
    p.ws_logdec = p.ws_state + (size_t)BH * pl.n_seg * D * p.srow;
  }
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_bf16_3d(&tq, a.q, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&tk, a.k, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&tv, a.v, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&to, a.O, D, a.L, BH, BOX, BOX)) {
    if (why) *why = "la_chunk_fwd: TMA tensor map creation failed";
    return cudaErrorInvalidValue;
  }
  cudaError_t e;
  if (pl.n_seg > 1) {
    if ((e = launch_state<D, PHI, DECAY, NORM>(dim3(pl.n_seg - 1, BH), tk, tv, p, a.stream)) !=
        cudaSuccess) {
      if (why) *why = "la_chunk_fwd: segment-state kernel launch";
      return e;
    }
#ifdef LA_CHECKED
    if ((e = cudaStreamSynchronize(a.stream)) != cudaSuccess) {
      if (why) *why = "la_chunk_fwd [checked]: segment-state kernel failed";
      return e;
    }
#endif
    const int n4 = D * p.srow / 4;
    e = launch_pdl(state_scan_kernel, dim3((n4 + 255) / 256, BH), 256, 0, a.stream, D, p.srow,
                   pl.n_seg, a.S0, z0, p.ws_state, (const float *)p.ws_logdec);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) {
      if (why) *why = "la_chunk_fwd: state-scan kernel launch";
      return e;
    }
#ifdef LA_CHECKED
    if ((e = cudaStreamSynchronize(a.stream)) != cudaSuccess) {
      if (why) *why = "la_chunk_fwd [checked]: state-scan kernel failed";
      return e;
    }
#endif
  }
  using OS = OutSmem<D, NORM>;
  auto ko = chunk_output_kernel<D, PHI, DECAY, NORM>;
  static int smem_set_out[64];
  e = set_smem_once(ko, OS::BYTES, smem_set_out);
  if (e != cudaSuccess) return e;
  const int out_x = OS::PAIRS ? (pl.n_seg + 1) / 2 : pl.n_seg;
  // With segments, the output kernel is a programmatic dependent of the scan
  // (its inputs were complete before the segment-state kernel started).  A
  // single segment has no predecessor of its own: ordinary stream order.
  if (pl.n_seg > 1)
    e = launch_pdl(ko, dim3(BH, out_x), kThreadsOut<D, DECAY, NORM>, OS::BYTES, a.stream, tq, tk, tv, to, p);
  else
    ko<<<dim3(BH, out_x), kThreadsOut<D, DECAY, NORM>, OS::BYTES, a.stream>>>(tq, tk, tv, to, p);
  if ((e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) && why)
    *why = "la_chunk_fwd: chunk-output kernel launch";
#ifdef LA_CHECKED
  if (e == cudaSuccess && (e = cudaStreamSynchronize(a.stream)) != cudaSuccess && why)
    *why = "la_chunk_fwd [checked]: chunk-output kernel failed";
#endif
  return e;
}


// ================================================================ non-causal form
// O = phi(Q) S for every token of a (b,h) sequence, with S = phi(K)^T V over
// the whole sequence ("adv13 - Linear Attention / SSM" section 4.3,
// linear_attention_matrix; "CS336 lecture 4, code 1", demo_associativity).
// S comes from the segment-state kernel run over every chunk and summed by
// the scan into the sequence's last workspace slot.  This kernel reads S once
// per sequence as the bf16 B operand of O_c = phi(Q_c) S and streams Q to O.
// The grid is a fixed number of blocks per SM; block j takes the j-th equal
// run of the (b,h)-major list of all chunks, so every SM gets the same share
// (a run may cross into the next sequence, which reloads S).  One warpgroup:
// thread 0 issues the TMA loads, the MMAs and the stores; all 128 threads
// apply phi and run the epilogue.
template <int D>
struct NcSmem {
  static constexpr int NQ = D == 64 ? 2 : 3;      // Q stages (d = 64: five blocks per SM)
  static constexpr uint32_t TILE = 64 * D * 2;    // [64][D] bf16 in D/64 boxes
  static constexpr uint32_t S_BLOCK = D * 128;    // [D][64] bf16 block of S, MN-major
  static constexpr uint32_t OFF_S = NQ * TILE;
  static constexpr uint32_t OFF_O = OFF_S + (D / 64) * S_BLOCK;  // 2 x O staging
  static constexpr uint32_t OFF_BAR = OFF_O + 2 * TILE;          // full[NQ], mma_done
  static constexpr uint32_t OFF_CTL = OFF_BAR + 8 * (NQ + 1);
  static constexpr uint32_t BYTES = OFF_CTL + 64;
  static_assert(TILE % 1024 == 0 && OFF_S % 1024 == 0 && OFF_O % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
};
constexpr int kNcThreads = 128;
constexpr uint32_t BAR_NC = 1;

template <int D, bool PHI>
__global__ void __launch_bounds__(kNcThreads)
noncausal_output_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmO, TcParams p,
                        int chunks_per_cta) {
  using SM = NcSmem<D>;
  constexpr int NQ = SM::NQ;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + SM::OFF_BAR);
  uint64_t *mma_done = full + NQ;
  Ctl *ctl = reinterpret_cast<Ctl *>(smem + SM::OFF_CTL);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long total = (long)p.BH * p.n_chunks;
  const long g0 = (long)blockIdx.x * chunks_per_cta;
  const int n = (int)max(0L, min((long)chunks_per_cta, total - g0));
  auto item_bh = [&](int i) { return (int)((g0 + i) / p.n_chunks); };
  auto item_c = [&](int i) { return (int)((g0 + i) % p.n_chunks); };
  if (tid == 0) {
    for (int s = 0; s < NQ; ++s) mbar_init(&full[s], 1);
    mbar_init(mma_done, 1);
    ctl->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem_base, D);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  int issued = 0;  // thread 0: Q tiles requested
  auto load_q = [&](int i) {
    const int s = i % NQ, bh = item_bh(i), tok = item_c(i) * CH;
    mbar_arrive_expect_tx(&full[s], SM::TILE);
    for (int b = 0; b < D / BOX; ++b)
      if (LA_CHK(tok < p.L && bh < p.BH, KID_NONCAUSAL, 3))
        tma_load_3d(smem + s * SM::TILE + b * BOX_BYTES, &tmQ, &full[s], b * BOX, tok, bh);
    issued = i + 1;
  };
  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmO);
    for (int i = 0; i < min(n, NQ); ++i) load_q(i);  // Q does not depend on S
  }
  // The segments' own states (slots 1 .. n_seg - 1 of a sequence) or, at
  // d = 128, their sum (the scan's last slot) are written by the kernel
  // before this one (a programmatic dependent launch): wait for them once.
  // load_s forms sequence bh's S and converts it to the bf16 B operand,
  // MN-major with the 128-byte swizzle; every thread calls it, after every
  // MMA that read the previous S has completed.  At d = 64 the block that
  // holds the sequence's first chunk also writes S, fp32, to S_final.
  pdl_wait_previous();
  constexpr bool FOLD = D == 64;
  auto load_s = [&](int bh, bool write_final) {
    const float *slots = p.ws_state + (size_t)bh * p.n_seg * D * D;
    float *fin = FOLD && write_final && p.S_final ? p.S_final + (size_t)bh * D * D : nullptr;
    unsigned char *sb = smem + SM::OFF_S;
    for (int idx = tid; idx < D * D / 8; idx += kNcThreads) {
      const int i = idx / (D / 8), j0 = (idx % (D / 8)) * 8;
      float4 x, y;
      if constexpr (FOLD) {
        x = make_float4(0.f, 0.f, 0.f, 0.f);
        y = x;
        for (int sg = 1; sg < p.n_seg; ++sg) {
          const float *S = slots + (size_t)sg * D * D + (size_t)i * D + j0;
          const float4 a = *reinterpret_cast<const float4 *>(S);
          const float4 b = *reinterpret_cast<const float4 *>(S + 4);
          x = make_float4(x.x + a.x, x.y + a.y, x.z + a.z, x.w + a.w);
          y = make_float4(y.x + b.x, y.y + b.y, y.z + b.z, y.w + b.w);
        }
      } else {
        const float *S = slots + (size_t)(p.n_seg - 1) * D * D + (size_t)i * D + j0;
        x = *reinterpret_cast<const float4 *>(S);
        y = *reinterpret_cast<const float4 *>(S + 4);
      }
      if (fin) {
        *reinterpret_cast<float4 *>(fin + (size_t)i * D + j0) = x;
        *reinterpret_cast<float4 *>(fin + (size_t)i * D + j0 + 4) = y;
      }
      *reinterpret_cast<uint4 *>(sb + (j0 / 64) * SM::S_BLOCK + i * 128 +
                                 ((((j0 % 64) >> 3) ^ (i & 7)) << 4)) =
          make_uint4(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w), pack_bf16(y.x, y.y),
                     pack_bf16(y.z, y.w));
    }
    fence_proxy_async_smem();
    __syncthreads();
  };
  int s_bh = -1;  // the sequence whose S is in shared memory
  constexpr uint32_t HI = smem_desc_sw128_hi(1024);
  constexpr uint32_t idesc = idesc_bf16_f32(64, D, false, true);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t dKM = smem_desc_sw128_lo(sbase, 16);          // Q: K-major rows
  const uint32_t dMS = smem_desc_sw128_lo(sbase, SM::S_BLOCK); // S: MN-major blocks
  // The accumulator has M = 64: rows 16 w + 0..15 in the first 16 lanes of
  // warp w's quarter.  A 16x256b load gives each thread rows ra and ra + 8 in
  // the 8x8 fragment layout, which stmatrix writes to the swizzled tile.
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const int mi = lane >> 3, srow = 16 * warp + 8 * (mi & 1) + (lane & 7);
  bool ok = true;
  int consumed = 0, mma_pending = -1;
  for (int i = 0; ok && i < n; ++i) {
    const int s = i % NQ, b = i & 1;
    if (!wait_grp<kNcThreads>(&full[s], (i / NQ) & 1, ctl, p.err, KID_NONCAUSAL, 1, BAR_NC, tid)) {
      ok = false;
      break;
    }
    consumed = i + 1;
    if (item_bh(i) != s_bh) {
      s_bh = item_bh(i);
      load_s(s_bh, item_c(i) == 0);
    }
    if constexpr (PHI) {
      tile_pass<D, 1, true, false>(smem + s * SM::TILE, [](int, int) { return 1.f; }, tid,
                                   kNcThreads);
      fence_proxy_async_smem();
      named_bar_sync(BAR_NC, kNcThreads);
    }
    if (tid == 0) {
      tc_fence_after();
      const uint32_t qo = s * SM::TILE;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16_w(tmem, dKM + ((qo + (kk / 4) * BOX_BYTES + 32 * (kk % 4)) >> 4),
                   dMS + ((SM::OFF_S + 2048 * kk) >> 4), HI, idesc, kk > 0 ? 1u : 0u);
      mma_commit(mma_done);
    }
    mma_pending = i;
    if (!wait_grp<kNcThreads>(mma_done, i & 1, ctl, p.err, KID_NONCAUSAL, 2, BAR_NC, tid)) {
      ok = false;
      break;
    }
    mma_pending = -1;
    tc_fence_after();
    if (tid == 0) {
      if (i + NQ < n) load_q(i + NQ);  // the MMA has read this stage
      tma_store_wait_read<1>();        // the store that used staging tile b has read it
    }
    __syncwarp();
    named_bar_sync(BAR_NC, kNcThreads);
    unsigned char *o_sm = smem + SM::OFF_O + b * SM::TILE;
#pragma unroll 1
    for (int col = 0; col < D; col += 64) {
      __syncwarp();
      uint32_t r[32];
      tmem_ld_16x256b_x8(tmem + lane_off + col, r);
      tmem_ld_wait();
      uint32_t pa[8], pb[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        pa[q] = pack_bf16(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]));
        pb[q] = pack_bf16(__uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
      }
      const uint32_t rbase = smem_u32(o_sm) + (col / 64) * BOX_BYTES + srow * 128;
#pragma unroll
      for (int qq = 0; qq < 8; qq += 2) {
        const int q = qq + (mi >> 1);
        stmatrix_x4(rbase + ((q ^ (srow & 7)) << 4), pa[qq], pb[qq], pa[qq + 1], pb[qq + 1]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar_sync(BAR_NC, kNcThreads);
    if (tid == 0) {
      const int tok = item_c(i) * CH, bh = item_bh(i);
      for (int bb = 0; bb < D / BOX; ++bb)
        if (LA_CHK(tok < p.L && bh < p.BH, KID_NONCAUSAL, 4))
          tma_store_3d(&tmO, o_sm + bb * BOX_BYTES, bb * BOX, tok, bh);
      tma_store_commit();
    }
  }
  if (tid == 0) {
    tma_store_wait_all();
    if (!ok) {  // asynchronous work still in flight lands before the CTA exits
      for (int c = consumed; c < issued; ++c) drain_wait(&full[c % NQ], (c / NQ) & 1);
      if (mma_pending >= 0) drain_wait(mma_done, mma_pending & 1);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, D);
  }
}

// Segments of the non-causal state pass: G <= 32 chunks, and about two
// segment-state blocks per SM.  Slot s + 1 takes segment s's state; at
// d = 128 the scan turns the slots into prefix sums (slot 0 = 0), the last
// one the sum of all.
Plan make_noncausal_plan(int B, int H, int L) {
  const int nc = (L + CH - 1) / CH;
  const int bh = std::max(1, B * H);
  int ns = std::max((nc + kMaxSegChunks - 1) / kMaxSegChunks,
                    std::min(nc, std::max(1, 2 * sm_count() / bh)));  // one wave at 2 per SM
  const int g = (nc + ns - 1) / ns;
  ns = (nc + g - 1) / g;
  return Plan{nc, g, ns};
}

size_t noncausal_ws_bytes_for(int B, int H, int L, int D) {
  const Plan pl = make_noncausal_plan(B, H, L);
  const size_t bh = (size_t)B * H, slots = (size_t)pl.n_seg + 1;
  return bh * slots * D * D * sizeof(float) + ((bh * slots * sizeof(float) + 255) & ~(size_t)255);
}

template <int D, bool PHI>
cudaError_t launch_noncausal_d(const NoncausalArgs &a, const char **why) {
  const Plan pl = make_noncausal_plan(a.B, a.H, a.L);
  const int BH = a.B * a.H, slots = pl.n_seg + 1;
  TcParams p{};
  p.H = a.H;
  p.L = a.L;
  p.BH = BH;
  p.n_chunks = pl.n_chunks;
  p.seg_chunks = pl.seg_chunks;
  p.n_seg = slots;  // segments 0..NS-1 cover every chunk; segment s writes slot s + 1
  p.S_final = a.S;  // d = 64: the sum, written by the output kernel
  p.phi = a.phi;
  p.decay_kind = LA_DECAY_NONE;
  p.err = device_error_word();
  p.srow = D;
  p.ws_state = static_cast<float *>(a.workspace);
  p.ws_logdec = p.ws_state + (size_t)BH * slots * D * D;
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_bf16_3d(&tq, a.q, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&tk, a.k, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&tv, a.v, D, a.L, BH, BOX, BOX) ||
      !make_tmap_bf16_3d(&to, a.O, D, a.L, BH, BOX, BOX)) {
    if (why) *why = "la_noncausal_fwd: TMA tensor map creation failed";
    return cudaErrorInvalidValue;
  }
  cudaError_t e;
  if ((e = launch_state<D, PHI, false, false>(dim3(pl.n_seg, BH), tk, tv, p, a.stream)) !=
      cudaSuccess) {
    if (why) *why = "la_noncausal_fwd: segment-state kernel launch";
    return e;
  }
  if constexpr (D != 64) {  // the scan sums the segments into the last slot
    const int n4 = D * D / 4;
    e = launch_pdl(state_scan_kernel, dim3((n4 + 255) / 256, BH), 256, 0, a.stream, D, D, slots,
                   (const float *)nullptr, (const float *)nullptr, p.ws_state,
                   (const float *)p.ws_logdec);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) {
      if (why) *why = "la_noncausal_fwd: state-scan kernel launch";
      return e;
    }
  }
  using NS_ = NcSmem<D>;
  auto kn = noncausal_output_kernel<D, PHI>;
  static int smem_set_nc[64];
  if ((e = set_smem_once(kn, NS_::BYTES, smem_set_nc)) != cudaSuccess) return e;
  const int per_sm = D == 64 ? 5 : 2;  // blocks per SM that fit in shared memory
  const long total = (long)pl.n_chunks * BH, slots_all = (long)per_sm * sm_count();
  const int cpc = (int)std::max(1L, (total + slots_all - 1) / slots_all);
  const int nx = (int)((total + cpc - 1) / cpc);
  e = launch_pdl(kn, dim3(nx), kNcThreads, NS_::BYTES, a.stream, tq, to, p, cpc);
  if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) {
    if (why) *why = "la_noncausal_fwd: output kernel launch";
    return e;
  }
  if (D != 64 && a.S) {  // the sum slot of every sequence
    e = cudaMemcpy2DAsync(a.S, (size_t)D * D * sizeof(float),
                          p.ws_state + (size_t)pl.n_seg * D * D,
                          (size_t)slots * D * D * sizeof(float), (size_t)D * D * sizeof(float),
                          BH, cudaMemcpyDeviceToDevice, a.stream);
    if (e != cudaSuccess && why) *why = "la_noncausal_fwd: state copy";
  }
  return e;
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs &a) {
  return a.dtype == LA_BF16 && a.chunk == CH && a.dk == a.dv && (a.dk == 64 || a.dk == 128);
}

size_t prefill_tc_workspace_bytes(int B, int H, int L, int d) {
  if (B <= 0 || H <= 0 || L <= 0) return 0;
  return ws_bytes_for(B, H, L, d, d);
}

bool prefill_tc_norm_supported(const PrefillArgs &a) {
  return prefill_tc_supported(a) && a.dk == 64;
}

size_t prefill_tc_norm_workspace_bytes(int B, int H, int L) {
  if (B <= 0 || H <= 0 || L <= 0) return 0;
  return ws_bytes_for(B, H, L, 64, 64 + 16);
}

cudaError_t launch_prefill_tc_norm(const PrefillArgs &a, const float *z0, float *z_final,
                                   const char **why) {
  const bool phi = a.phi != LA_PHI_IDENTITY, decay = a.decay_kind != LA_DECAY_NONE;
  if (phi && decay) return launch_d<64, true, true, true>(a, why, z0, z_final);
  if (phi) return launch_d<64, true, false, true>(a, why, z0, z_final);
  if (decay) return launch_d<64, false, true, true>(a, why, z0, z_final);
  return launch_d<64, false, false, true>(a, why, z0, z_final);
}

int prefill_tc_kernel_count(int B, int H, int L, int d) {
  return make_plan(B, H, L, d).n_seg > 1 ? 3 : 1;
}

template <int D>
cudaError_t launch_variant(const PrefillArgs &a, const char **why) {
  const bool phi = a.phi != LA_PHI_IDENTITY, decay = a.decay_kind != LA_DECAY_NONE;
  if (phi && decay) return launch_d<D, true, true>(a, why);
  if (phi) return launch_d<D, true, false>(a, why);
  if (decay) return launch_d<D, false, true>(a, why);
  return launch_d<D, false, false>(a, why);
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, const char **why) {
  if (a.dk == 128) return launch_variant<128>(a, why);
  return launch_variant<64>(a, why);
}

size_t noncausal_workspace_bytes(int B, int H, int L, int d) {
  if (B <= 0 || H <= 0 || L <= 0) return 0;
  return noncausal_ws_bytes_for(B, H, L, d);
}

cudaError_t launch_noncausal(const NoncausalArgs &a, const char **why) {
  const bool phi = a.phi != LA_PHI_IDENTITY;
  if (a.d == 128) return phi ? launch_noncausal_d<128, true>(a, why) : launch_noncausal_d<128, false>(a, why);
  return phi ? launch_noncausal_d<64, true>(a, why) : launch_noncausal_d<64, false>(a, why);
}

}  // namespace la
