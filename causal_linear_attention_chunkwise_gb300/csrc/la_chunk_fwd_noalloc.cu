// la_chunk_fwd_noalloc.cu -- la_chunk_fwd for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they run prefill: code
// inside a custom allocator or a memory-pool callback, runtimes that forbid
// allocation after start-up (fixed-footprint serving processes), or code
// running while another component holds the allocator lock.  For them the
// segment-state workspace that la_chunk_fwd takes from the caller lives here
// instead, in one fixed-size array in device memory that the CUDA module
// reserves when the library is loaded.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/la_gb300.h"
#include "la_internal.h"

namespace {

// The scratch: enough for the segment states of about 300 sequences of 128x128
// state at 2 segments each (every workload this library is tuned for needs at
// most 21 MB).  Every GPU that loads the library holds these bytes until the
// process exits.
constexpr size_t kScratchBytes = LA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];  // device address of g_scratch, per device

// The array's device address for the current device, looked up once per device
// with that device current.  (In host code `g_scratch` names a host-side
// stand-in, not device memory, so it must never be passed to a kernel.)
cudaError_t scratch_for_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t la_chunk_fwd_noalloc_scratch_bytes(void) { return kScratchBytes; }

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
    cudaError_t e = scratch_for_current_device(&scratch);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof msg, "la_chunk_fwd_noalloc: scratch address lookup: %s",
               cudaGetErrorString(e));
      la::set_last_error(msg);
      return LA_ERR_CUDA;
    }
  }
  return la_chunk_fwd(q, k, v, dtype, B, H, L, d_k, d_v, chunk, decay_kind, decay, S0, O,
                      S_final, scratch, need > 0 ? kScratchBytes : 0, cuda_stream);
}

}  // extern "C"
