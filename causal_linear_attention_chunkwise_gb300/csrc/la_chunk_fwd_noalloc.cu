// la_chunk_fwd_noalloc.cu -- la_chunk_fwd for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they run prefill: code
// inside a custom allocator or a memory-pool callback, runtimes that forbid
// allocation after start-up (fixed-footprint serving processes), or code
// running while another component holds the allocator lock.  For them the
// segment-state workspace that la_chunk_fwd takes from the caller lives here
// instead, in one fixed-size array in device memory.
//
// When the bytes are reserved.  The CUDA runtime loads a module lazily by
// default (CUDA_MODULE_LOADING=LAZY): the array is placed in device memory
// when this file's module is first used on a device, which is the
// cudaGetSymbolAddress below.  la_chunk_fwd_noalloc_prepare() does that
// lookup for the current device, so a caller that cannot allocate later calls
// it once per device at start-up; la_chunk_fwd_noalloc does it itself on its
// first call on a device that was not prepared.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/la_gb300.h"
#include "la_internal.h"

namespace {

// The scratch.  The workspace of la_chunk_fwd is B*H*NS*d_k*d_v*4 bytes of
// segment states plus B*H*NS log decays (NS = segments per sequence, chosen
// by the launcher), so 32 MiB holds, for instance, about 250 sequences of
// 128 x 128 state at 2 segments each.  Every GPU on which the module is loaded
// holds these bytes until the process exits.
constexpr size_t kScratchBytes = LA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];  // device address of g_scratch, per device

// Look up (again, when `refresh`) the array's device address for the current
// device, with that device current, and cache it.  In host code `g_scratch`
// names a host-side stand-in, not device memory, so it is never passed to a
// kernel: only the address returned here is.
cudaError_t scratch_for_current_device(void **out, bool refresh) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (refresh || !g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

la_status lookup_failed(cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof msg, "la_chunk_fwd_noalloc: scratch address lookup: %s",
           cudaGetErrorString(e));
  la::set_last_error(msg);
  return LA_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t la_chunk_fwd_noalloc_scratch_bytes(void) { return kScratchBytes; }

la_status la_chunk_fwd_noalloc_prepare(void) {
  void *p = nullptr;
  const cudaError_t e = scratch_for_current_device(&p, true);
  return e == cudaSuccess ? LA_OK : lookup_failed(e);
}

la_status la_chunk_fwd_noalloc(const void *q, const void *k, const void *v, int dtype, int B,
                               int H, int L, int d_k, int d_v, int chunk, int decay_kind,
                               const float *decay, const float *S0, void *O, float *S_final,
                               void *cuda_stream) {
  const size_t need = la_chunk_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk, dtype);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "la_chunk_fwd_noalloc: this problem needs %zu bytes of scratch; the static "
             "scratch holds %zu (use la_chunk_fwd with a caller workspace)",
             need, kScratchBytes);
    la::set_last_error(msg);
    return LA_ERR_UNSUPPORTED;
  }
  void *scratch = nullptr;
  if (need > 0) {
    const cudaError_t e = scratch_for_current_device(&scratch, false);
    if (e != cudaSuccess) return lookup_failed(e);
  }
  return la_chunk_fwd(q, k, v, dtype, B, H, L, d_k, d_v, chunk, decay_kind, decay, S0, O,
                      S_final, scratch, need > 0 ? kScratchBytes : 0, cuda_stream);
}

}  // extern "C"
