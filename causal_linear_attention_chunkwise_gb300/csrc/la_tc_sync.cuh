// la_tc_sync.cuh -- pieces shared by the tcgen05 kernels: tile constants,
// bounded mbarrier waits (single thread and group-wide), the abort control
// word, bf16 packing, elu + 1, swizzled row stores, and the host-side launch
// helpers (shared-memory opt-in, programmatic dependent launch, SM count).
// Every wait gives up after a time or poll limit, records the site in the
// device error word and sets the CTA abort flag, so no kernel spins forever.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "la_common.cuh"
#include "la_ptx.cuh"

namespace la {
namespace tc {

constexpr int CH = 64;                  // tokens per chunk
constexpr int BOX = 64;                 // TMA box: 64 rows x 64 bf16 (128 bytes)
constexpr uint32_t BOX_BYTES = 8192;
constexpr uint64_t kWaitNs = 2000000000ull;  // a wait gives up after 2 s
constexpr uint32_t kSpinCap = 1u << 26;       // and after this many polls regardless
constexpr uint32_t kSleepNs = 1000;           // suspend-time hint of one poll

struct Ctl {
  uint32_t abort;
  uint32_t tmem_base;
};

// ---------------------------------------------------------------- waits
// Single-thread bounded wait; on timeout records the error and sets abort.
// The first test is inline; the polling loop is one shared out-of-line copy.
static __device__ __noinline__ bool wait1_slow(uint64_t *bar, uint32_t parity, Ctl *ctl,
                                        unsigned int *err, uint32_t kid, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < kSpinCap; ++i) {
    // Suspend (up to kSleepNs) rather than spin: the other warps of this
    // sub-partition keep its issue slots.
    if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
    if ((i & 63u) == 0) {
      if (*(volatile uint32_t *)&ctl->abort) return false;
      if (global_timer_ns() - t0 > kWaitNs) break;
    }
  }
  atomicExch(&ctl->abort, 1u);
  record_device_error(err, kid, site);
  return false;
}

__device__ __forceinline__ bool wait1(uint64_t *bar, uint32_t parity, Ctl *ctl,
                                      unsigned int *err, uint32_t kid, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait1_slow(bar, parity, ctl, err, kid, site);
}

// After an abort: wait (bounded, ignoring the abort flag) for a phase that
// in-flight asynchronous work will still complete, so that no TMA write or
// MMA outlives the CTA's shared memory and TMEM.
static __device__ __noinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0; i < kSpinCap; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 63u) == 63u && global_timer_ns() - t0 > kWaitNs) return;
  }
}

// Group-wide bounded wait for NT threads (t = index within the group, whole
// warps): the group's first thread polls while the others sleep in a reducing
// named barrier (the .aligned form, entered converged after a __syncwarp) that
// also hands them the outcome, so all leave together.  The barrier orders the
// group's later accesses after the leader's acquire of the mbarrier phase.
template <int NT>
__device__ __forceinline__ bool wait_grp(uint64_t *bar, uint32_t parity, Ctl *ctl,
                                         unsigned int *err, uint32_t kid, uint32_t site,
                                         uint32_t bar_id, int t) {
  bool ok = true;
  if (t == 0) ok = wait1(bar, parity, ctl, err, kid, site);
  __syncwarp();
  uint32_t any_fail;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.eq.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(any_fail)
      : "r"(ok ? 1u : 0u), "r"(bar_id), "n"(NT)
      : "memory");
  if (any_fail) return false;
  __syncwarp();
  return true;
}

// The same for a warpgroup (four consecutive warps starting at a multiple of 4).
// Barrier bar_id over n threads that ORs a predicate across them.
__device__ __forceinline__ bool bar_red_or(uint32_t bar_id, uint32_t n, bool pred) {
  uint32_t any;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(any)
      : "r"(pred ? 1u : 0u), "r"(bar_id), "r"(n)
      : "memory");
  return any != 0;
}

__device__ __forceinline__ bool wait_wg(uint64_t *bar, uint32_t parity, Ctl *ctl,
                                        unsigned int *err, uint32_t kid, uint32_t site,
                                        uint32_t bar_id) {
  return wait_grp<128>(bar, parity, ctl, err, kid, site, bar_id, threadIdx.x & 127);
}

// Debug builds (-DLA_CHECKED) bounds-check every runtime-computed TMA
// coordinate and global index, record the first violation in the device
// error word (wait site 200 + n) and skip the access.
#ifdef LA_CHECKED
#define LA_CHK(cond, kid, site) ((cond) ? true : (record_device_error(p.err, (kid), 200u + (site)), false))
#else
#define LA_CHK(cond, kid, site) true
#endif

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Rows of an M=64 accumulator: row 16*i + t lives in TMEM lane 32*i + t
// (t < 16) of lane quarter i; lanes 16..31 of each quarter are unused.
// M=128: row = lane.
template <int M>
__device__ __forceinline__ int acc_row(int quarter, int lane) {
  if (M == 128) return quarter * 32 + lane;
  return lane < 16 ? quarter * 16 + lane : -1;
}

// ================================================================ shared pieces
// elu(x) + 1 without a branch: for x > 0 it is x + 1 > 1 = 2^0, and for x <= 0
// exp(x) >= x + 1 (convexity), so max(x + 1, 2^(min(x, 0) log2 e)) takes the
// right side in both cases.  The NaN-propagating max keeps a NaN input NaN.
__device__ __forceinline__ float elu1_fast(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fminf(x, 0.f) * 1.4426950408889634f));
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(x + 1.f), "f"(e));
  return r;
}

// The same on a pair of bf16 values, in packed bf16 arithmetic.  For x > 0,
// x + 1 is computed exactly and rounded once, as from fp32.  For x <= 0 the
// argument t = x log2 e takes log2 e as the bf16 pair hi + lo
// (hi = 0x3FB9 = 1.4453125, lo = 0xBB2C ~ -2.6245e-3; hi + lo matches log2 e
// to 5e-6 relative), so that t carries one bf16 rounding and no bias; 2^t
// then adds the rounding of its bf16 result.
__device__ __forceinline__ uint32_t elu1_bf16x2(uint32_t x) {
  uint32_t m, tl, tt, e, p1, r;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(x), "r"(0u));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(tl) : "r"(m), "r"(0xBB2CBB2Cu));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(tt) : "r"(m), "r"(0x3FB93FB9u), "r"(tl));
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(tt));
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(p1) : "r"(x), "r"(0x3F803F80u));
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(p1), "r"(e));
  return r;
}

// Store 16 consecutive bf16 values (8 packed words) of `row` at column `col`
// (a multiple of 16) into a swizzled tile whose 64-column blocks are `blk`
// bytes apart.
__device__ __forceinline__ void st_row16(unsigned char *base, uint32_t blk, int row, int col,
                                         const uint32_t *pk) {
  unsigned char *p = base + (col / 64) * blk + row * 128;
  const int ch0 = (col % 64) >> 3;
  *reinterpret_cast<uint4 *>(p + ((ch0 ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  *reinterpret_cast<uint4 *>(p + (((ch0 + 1) ^ (row & 7)) << 4)) =
      make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

// Elementwise pass over NT consecutive bf16 tiles of ROWS rows x D columns
// (D/64 swizzled boxes of ROWS x 128 bytes per tile, 8 sixteen-byte chunks per
// row): x <- phi(x) * fac(k, row) in tile k.  Threads t = 0..n-1 take chunks
// t, t + n, ...; four loads are issued before any use.
template <int D, int NT, bool PHI, bool SCALE, typename Fac, int ROWS = 64>
__device__ __forceinline__ void tile_pass(unsigned char *tile, Fac fac, int t, int n) {
  constexpr int kTileChunks = ROWS * D * 2 / 16;
  constexpr int kBoxChunks = ROWS * 8;
  constexpr int kChunks = NT * kTileChunks;
#pragma unroll 1
  for (int base = 0; base < kChunks; base += 4 * n) {
    uint4 u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int x = base + j * n + t;
      if (x < kChunks) u[j] = *reinterpret_cast<const uint4 *>(tile + (size_t)x * 16);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int x = base + j * n + t;
      if (x >= kChunks) continue;
      float sc = 1.f;
      if (SCALE) sc = fac(NT == 1 || x < kTileChunks ? 0 : 1, (x % kBoxChunks) >> 3);
      uint32_t w[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (PHI && !SCALE) {  // phi alone: packed bf16 arithmetic
          w[e] = elu1_bf16x2(w[e]);
          continue;
        }
        float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
        if (PHI) {
          lo = elu1_fast(lo);
          hi = elu1_fast(hi);
        }
        w[e] = pack_bf16(lo * sc, hi * sc);
      }
      u[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int x = base + j * n + t;
      if (x < kChunks) *reinterpret_cast<uint4 *>(tile + (size_t)x * 16) = u[j];
    }
  }
}

// ---------------------------------------------------------------- host helpers
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  return n;
}

// Opt the kernels into their dynamic shared memory once per device.
template <typename K>
cudaError_t set_smem_once(K kern, size_t bytes, int *done_for_device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && done_for_device[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev < 64) done_for_device[dev] = 1;
  return e;
}

// Launch `kern` as a programmatic dependent of the previous kernel on the
// stream: it may start before that kernel finishes, and waits for it
// (griddepcontrol.wait) before it reads what that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, int threads, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace tc
}  // namespace la
