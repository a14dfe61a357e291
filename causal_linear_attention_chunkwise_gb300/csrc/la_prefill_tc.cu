// la_prefill_tc.cu -- tensor-core (tcgen05) chunkwise prefill.  Not yet enabled:
// every bf16 request currently runs the SIMT kernel.
#include "la_internal.h"

namespace la {

bool prefill_tc_supported(const PrefillArgs &) { return false; }

size_t prefill_tc_workspace_bytes(int, int, int, int) { return 0; }

int prefill_tc_kernel_count(int, int, int, int) { return 0; }

cudaError_t launch_prefill_tc(const PrefillArgs &, const char **why) {
  if (why) *why = "tcgen05 prefill not available";
  return cudaErrorNotSupported;
}

}  // namespace la
