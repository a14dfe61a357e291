// la_abi.cu -- the extern "C" boundary: argument validation, dispatch to the
// kernel launchers, the process-wide feature map, error reporting.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "../../include/la_gb300.h"
#include "la_common.cuh"
#include "la_internal.h"

namespace la {

__device__ unsigned int g_device_error;

namespace {
std::atomic<int> g_phi{LA_PHI_IDENTITY};
thread_local char g_msg[512] = "";

la_status fail(la_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return s;
}

la_status ok() {
  g_msg[0] = '\0';
  return LA_OK;
}

la_status cuda_fail(cudaError_t e, const char *where) {
  return fail(LA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

bool supported_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// Copy `src` to `dst` (or zero `dst` when src is null): the state after no tokens.
cudaError_t pass_through_state(float *dst, const float *src, size_t bytes, cudaStream_t st) {
  if (!dst) return cudaSuccess;
  if (!src) return cudaMemsetAsync(dst, 0, bytes, st);
  if (src == dst) return cudaSuccess;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
}

// Checks shared by la_normalised_fwd, la_channel_gate_fwd and la_delta_fwd.
// Returns LA_OK with *done = false when the kernel is to run; otherwise the
// call ends with the returned status (LA_OK with *done = true: an empty batch,
// or L = 0 with the states passed through).
la_status check_variant(const char *fn, const void *q, const void *k, const void *v, int dtype,
                        int B, int H, int L, int d_k, int d_v, int chunk, bool uses_chunk,
                        const float *S0, const float *z0, void *O, float *S_final,
                        float *z_final, cudaStream_t st, bool *done) {
  *done = true;
  if (dtype != LA_F32 && dtype != LA_BF16)
    return fail(LA_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, dtype);
  if (B < 0 || H < 0 || L < 0 || d_k <= 0 || d_v <= 0 || (uses_chunk && chunk <= 0))
    return fail(LA_ERR_INVALID_ARG, "%s: bad sizes B=%d H=%d L=%d d_k=%d d_v=%d chunk=%d", fn,
                B, H, L, d_k, d_v, chunk);
  if (!supported_d(d_k) || !supported_d(d_v))
    return fail(LA_ERR_UNSUPPORTED, "%s: d_k=%d d_v=%d not in {16,32,64,128}", fn, d_k, d_v);
  if (uses_chunk && chunk > 64)
    return fail(LA_ERR_UNSUPPORTED, "%s: chunk %d > 64 is not supported", fn, chunk);
  if ((size_t)B * H == 0) return ok();
  if ((S0 && !aligned16(S0)) || (S_final && !aligned16(S_final)) || (z0 && !aligned16(z0)) ||
      (z_final && !aligned16(z_final)))
    return fail(LA_ERR_INVALID_ARG, "%s: state pointers must be 16-byte aligned", fn);
  if (L == 0) {
    const size_t sb = (size_t)B * H * d_k * d_v * sizeof(float);
    const size_t zb = (size_t)B * H * d_k * sizeof(float);
    cudaError_t e = pass_through_state(S_final, S0, sb, st);
    if (e == cudaSuccess) e = pass_through_state(z_final, z0, zb, st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return ok();
  }
  if (!q || !k || !v || !O)
    return fail(LA_ERR_INVALID_ARG, "%s: q, k, v and O must be non-null", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(O))
    return fail(LA_ERR_INVALID_ARG, "%s: tensors must start on a 16-byte boundary", fn);
  *done = false;
  return ok();
}

la_status run_variant(const char *fn, const VariantArgs &a) {
  cudaError_t e = launch_variant(a);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

const char *kernel_name(unsigned int id) {
  switch (id) {
    case KID_PREFILL_TC_STATE: return "prefill segment-state kernel";
    case KID_PREFILL_TC_OUT: return "prefill chunk-output kernel";
    case KID_SELFTEST: return "wait-timeout self-test kernel";
    case KID_NONCAUSAL: return "non-causal output kernel";
    case KID_CHANNEL_GATE_TC: return "per-channel gate tensor-core kernel";
    case KID_DELTA_TC: return "delta-rule tensor-core kernel";
    default: return "unknown kernel";
  }
}
}  // namespace

void set_last_error(const char *msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

unsigned int *device_error_word() {
  // The symbol's device address, looked up for the current device on each
  // call (cheap; avoids caching an address across devices).
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<unsigned int *>(p);
}

}  // namespace la

using namespace la;

extern "C" {

la_status la_set_feature_map(int phi) {
  if (phi != LA_PHI_IDENTITY && phi != LA_PHI_ELU1)
    return fail(LA_ERR_INVALID_ARG, "la_set_feature_map: unknown feature map %d", phi);
  g_phi.store(phi);
  return ok();
}

int la_get_feature_map(void) { return g_phi.load(); }

size_t la_chunk_fwd_workspace_bytes(int B, int H, int L, int d_k, int d_v, int chunk, int dtype) {
  PrefillArgs a{};
  a.dtype = dtype; a.B = B; a.H = H; a.L = L; a.dk = d_k; a.dv = d_v; a.chunk = chunk;
  if (B <= 0 || H <= 0 || L <= 0) return 0;
  if (prefill_tc_supported(a)) return prefill_tc_workspace_bytes(B, H, L, d_k);
  return 0;
}

int la_chunk_fwd_kernel_count(int B, int H, int L, int d_k, int d_v, int chunk, int dtype) {
  if (B <= 0 || H <= 0 || L <= 0) return 0;
  if ((dtype != LA_F32 && dtype != LA_BF16) || !supported_d(d_k) || !supported_d(d_v) ||
      chunk < 1 || chunk > 64)
    return 0;
  PrefillArgs a{};
  a.dtype = dtype; a.B = B; a.H = H; a.L = L; a.dk = d_k; a.dv = d_v; a.chunk = chunk;
  if (prefill_tc_supported(a)) return prefill_tc_kernel_count(B, H, L, d_k);
  return 1;
}

la_status la_chunk_fwd(const void *q, const void *k, const void *v, int dtype, int B, int H,
                       int L, int d_k, int d_v, int chunk, int decay_kind, const float *decay,
                       const float *S0, void *O, float *S_final, void *workspace,
                       size_t ws_bytes, void *cuda_stream) {
  if (dtype != LA_F32 && dtype != LA_BF16)
    return fail(LA_ERR_INVALID_ARG, "la_chunk_fwd: unknown dtype %d", dtype);
  if (B < 0 || H < 0 || L < 0 || d_k <= 0 || d_v <= 0 || chunk <= 0)
    return fail(LA_ERR_INVALID_ARG,
                "la_chunk_fwd: bad sizes B=%d H=%d L=%d d_k=%d d_v=%d chunk=%d", B, H, L, d_k,
                d_v, chunk);
  if (decay_kind < LA_DECAY_NONE || decay_kind > LA_DECAY_GATE_LOGIT)
    return fail(LA_ERR_INVALID_ARG, "la_chunk_fwd: unknown decay kind %d", decay_kind);
  if (!supported_d(d_k) || !supported_d(d_v))
    return fail(LA_ERR_UNSUPPORTED, "la_chunk_fwd: d_k=%d d_v=%d not in {16,32,64,128}", d_k,
                d_v);
  if (chunk > 64)
    return fail(LA_ERR_UNSUPPORTED, "la_chunk_fwd: chunk %d > 64 is not supported", chunk);
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const size_t state_bytes = (size_t)B * H * d_k * d_v * sizeof(float);
  if ((size_t)B * H == 0) return ok();
  if (L == 0) {  // nothing to attend to: the final state is the initial one
    if (!S_final) return ok();
    if (!aligned16(S_final) || (S0 && !aligned16(S0)))
      return fail(LA_ERR_INVALID_ARG, "la_chunk_fwd: state pointers must be 16-byte aligned");
    cudaError_t e = S0 ? (S0 == S_final ? cudaSuccess
                                        : cudaMemcpyAsync(S_final, S0, state_bytes,
                                                          cudaMemcpyDeviceToDevice, st))
                       : cudaMemsetAsync(S_final, 0, state_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "la_chunk_fwd (L=0)");
    return ok();
  }
  if (!q || !k || !v || !O)
    return fail(LA_ERR_INVALID_ARG, "la_chunk_fwd: q, k, v and O must be non-null");
  if (decay_kind != LA_DECAY_NONE && !decay)
    return fail(LA_ERR_INVALID_ARG, "la_chunk_fwd: decay kind %d needs a decay pointer",
                decay_kind);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(O) ||
      (S0 && !aligned16(S0)) || (S_final && !aligned16(S_final)))
    return fail(LA_ERR_INVALID_ARG, "la_chunk_fwd: tensors must start on a 16-byte boundary");

  PrefillArgs a{q, k, v, dtype, B, H, L, d_k, d_v, chunk, g_phi.load(), decay_kind,
                decay_kind == LA_DECAY_NONE ? nullptr : decay, S0, O, S_final,
                workspace, ws_bytes, st};
  if (prefill_tc_supported(a)) {
    size_t need = prefill_tc_workspace_bytes(B, H, L, d_k);
    if (need > 0 && (!workspace || ws_bytes < need))
      return fail(LA_ERR_INVALID_ARG,
                  "la_chunk_fwd: workspace of %zu bytes needed, %zu given", need,
                  workspace ? ws_bytes : (size_t)0);
    if (need > 0 && !aligned16(workspace))
      return fail(LA_ERR_INVALID_ARG, "la_chunk_fwd: workspace must be 16-byte aligned");
    const char *why = nullptr;
    cudaError_t e = launch_prefill_tc(a, &why);
    if (e != cudaSuccess) return cuda_fail(e, why ? why : "la_chunk_fwd (tcgen05 path)");
    return ok();
  }
  cudaError_t e = launch_prefill_simt(a);
  if (e != cudaSuccess) return cuda_fail(e, "la_chunk_fwd (SIMT path)");
  return ok();
}

size_t la_noncausal_fwd_workspace_bytes(int B, int H, int L, int d_k, int d_v) {
  if (d_k != d_v || (d_k != 64 && d_k != 128)) return 0;
  return noncausal_workspace_bytes(B, H, L, d_k);
}

la_status la_noncausal_fwd(const void *q, const void *k, const void *v, int dtype, int B, int H,
                           int L, int d_k, int d_v, void *O, float *S, void *workspace,
                           size_t ws_bytes, void *cuda_stream) {
  if (dtype != LA_F32 && dtype != LA_BF16)
    return fail(LA_ERR_INVALID_ARG, "la_noncausal_fwd: unknown dtype %d", dtype);
  if (B < 0 || H < 0 || L < 0 || d_k <= 0 || d_v <= 0)
    return fail(LA_ERR_INVALID_ARG, "la_noncausal_fwd: bad sizes B=%d H=%d L=%d d_k=%d d_v=%d",
                B, H, L, d_k, d_v);
  if (dtype != LA_BF16 || d_k != d_v || (d_k != 64 && d_k != 128))
    return fail(LA_ERR_UNSUPPORTED,
                "la_noncausal_fwd: needs bf16 with d_k = d_v in {64, 128} (dtype %d, %d x %d)",
                dtype, d_k, d_v);
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if ((size_t)B * H == 0) return ok();
  if (S && !aligned16(S))
    return fail(LA_ERR_INVALID_ARG, "la_noncausal_fwd: S must start on a 16-byte boundary");
  if (L == 0) {  // no tokens: the state is zero and there is no output
    if (S) {
      cudaError_t e = cudaMemsetAsync(S, 0, (size_t)B * H * d_k * d_v * sizeof(float), st);
      if (e != cudaSuccess) return cuda_fail(e, "la_noncausal_fwd (L=0)");
    }
    return ok();
  }
  if (!q || !k || !v || !O)
    return fail(LA_ERR_INVALID_ARG, "la_noncausal_fwd: q, k, v and O must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(O))
    return fail(LA_ERR_INVALID_ARG, "la_noncausal_fwd: tensors must start on a 16-byte boundary");
  const size_t need = noncausal_workspace_bytes(B, H, L, d_k);
  if (!workspace || ws_bytes < need)
    return fail(LA_ERR_INVALID_ARG, "la_noncausal_fwd: workspace of %zu bytes needed, %zu given",
                need, workspace ? ws_bytes : (size_t)0);
  if (!aligned16(workspace))
    return fail(LA_ERR_INVALID_ARG, "la_noncausal_fwd: workspace must be 16-byte aligned");
  NoncausalArgs a{q, k, v, B, H, L, d_k, g_phi.load(), O, S, workspace, ws_bytes, st};
  const char *why = nullptr;
  cudaError_t e = launch_noncausal(a, &why);
  if (e != cudaSuccess) return cuda_fail(e, why ? why : "la_noncausal_fwd");
  return ok();
}

la_status la_decode_step(const void *q, const void *k, const void *v, int dtype, int B, int H,
                         int d_k, int d_v, const float *log_alpha, float *S, void *o,
                         void *cuda_stream) {
  if (dtype != LA_F32 && dtype != LA_BF16)
    return fail(LA_ERR_INVALID_ARG, "la_decode_step: unknown dtype %d", dtype);
  if (B < 0 || H < 0 || d_k <= 0 || d_v <= 0)
    return fail(LA_ERR_INVALID_ARG, "la_decode_step: bad sizes B=%d H=%d d_k=%d d_v=%d", B, H,
                d_k, d_v);
  if (!decode_supported(d_k, d_v))
    return fail(LA_ERR_UNSUPPORTED,
                "la_decode_step: d_k=%d d_v=%d unsupported (need d_k = d_v in {16,32,64,128})",
                d_k, d_v);
  if ((size_t)B * H == 0) return ok();
  if (!q || !k || !v || !S || !o)
    return fail(LA_ERR_INVALID_ARG, "la_decode_step: q, k, v, S and o must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(S) || !aligned16(o))
    return fail(LA_ERR_INVALID_ARG, "la_decode_step: tensors must start on a 16-byte boundary");
  DecodeArgs a{q, k, v, dtype, B, H, d_k, d_v, g_phi.load(), log_alpha, S, o,
               static_cast<cudaStream_t>(cuda_stream)};
  cudaError_t e = launch_decode(a);
  if (e != cudaSuccess) return cuda_fail(e, "la_decode_step");
  return ok();
}

size_t la_normalised_fwd_workspace_bytes(int B, int H, int L, int d_k, int d_v, int chunk,
                                         int dtype) {
  if (B <= 0 || H <= 0 || L <= 0 || !supported_d(d_k) || !supported_d(d_v)) return 0;
  PrefillArgs probe{};
  probe.dtype = dtype;
  probe.B = B;
  probe.H = H;
  probe.L = L;
  probe.dk = d_k;
  probe.dv = d_v;
  probe.chunk = chunk;
  if (prefill_tc_norm_supported(probe)) return prefill_tc_norm_workspace_bytes(B, H, L);
  return align256(la_chunk_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk, dtype)) +
         normaliser_workspace_bytes(B, H, L, d_k);
}

la_status la_normalised_fwd(const void *q, const void *k, const void *v, int dtype, int B,
                            int H, int L, int d_k, int d_v, int chunk, int decay_kind,
                            const float *decay, const float *S0, const float *z0, void *O,
                            float *S_final, float *z_final, void *workspace, size_t ws_bytes,
                            void *cuda_stream) {
  const char *fn = "la_normalised_fwd";
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (decay_kind < LA_DECAY_NONE || decay_kind > LA_DECAY_GATE_LOGIT)
    return fail(LA_ERR_INVALID_ARG, "%s: unknown decay kind %d", fn, decay_kind);
  if (decay_kind != LA_DECAY_NONE && !decay)
    return fail(LA_ERR_INVALID_ARG, "%s: decay kind %d needs a decay pointer", fn, decay_kind);
  bool done = false;
  la_status s = check_variant(fn, q, k, v, dtype, B, H, L, d_k, d_v, chunk, true, S0, z0, O,
                              S_final, z_final, st, &done);
  if (s != LA_OK || done) return s;
  const int phi = g_phi.load();
  const float *dec = decay_kind == LA_DECAY_NONE ? nullptr : decay;
  {
    // One pass on the d = 64 tensor-core kernels: the denominator and z ride
    // with the numerator and the state as one more value column.
    PrefillArgs a{q, k, v, dtype, B, H, L, d_k, d_v, chunk, phi, decay_kind, dec, S0, O,
                  S_final, workspace, ws_bytes, st};
    if (prefill_tc_norm_supported(a)) {
      const size_t need = prefill_tc_norm_workspace_bytes(B, H, L);
      if (need > 0 && (!workspace || ws_bytes < need))
        return fail(LA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                    workspace ? ws_bytes : (size_t)0);
      if (need > 0 && !aligned16(workspace))
        return fail(LA_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", fn);
      const char *why = nullptr;
      const cudaError_t e = launch_prefill_tc_norm(a, z0, z_final, &why);
      if (e != cudaSuccess) return cuda_fail(e, why ? why : fn);
      return ok();
    }
  }
  const size_t num_ws = la_chunk_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk, dtype);
  const size_t need = align256(num_ws) + normaliser_workspace_bytes(B, H, L, d_k);
  if (!workspace || ws_bytes < need)
    return fail(LA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                workspace ? ws_bytes : (size_t)0);
  if (!aligned16(workspace))
    return fail(LA_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", fn);
  // The numerator phi(q_t)^T S_t goes to O (and S_final) through the prefill
  // kernels; the normaliser then forms z and divides O in place.
  PrefillArgs a{q, k, v, dtype, B, H, L, d_k, d_v, chunk, phi, decay_kind, dec, S0, O,
                S_final, num_ws ? workspace : nullptr, num_ws, st};
  cudaError_t e;
  const char *why = nullptr;
  if (prefill_tc_supported(a)) {
    e = launch_prefill_tc(a, &why);
  } else {
    e = launch_prefill_simt(a);
  }
  if (e != cudaSuccess) return cuda_fail(e, why ? why : fn);
  NormaliserArgs n{q, k, dtype, B, H, L, d_k, d_v, phi, decay_kind, dec, z0, O, z_final,
                   static_cast<char *>(workspace) + align256(num_ws), st};
  e = launch_normaliser(n);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

size_t la_channel_gate_fwd_workspace_bytes(int B, int H, int L, int d_k, int d_v, int chunk,
                                           int dtype) {
  if (dtype != LA_BF16 || chunk != 64 || d_k != d_v) return 0;
  return channel_gate_tc_workspace_bytes(B, H, L, d_k);
}

la_status la_channel_gate_fwd(const void *q, const void *k, const void *v, int dtype, int B,
                              int H, int L, int d_k, int d_v, int chunk, const float *log_alpha,
                              const float *S0, void *O, float *S_final, void *workspace,
                              size_t ws_bytes, void *cuda_stream) {
  const char *fn = "la_channel_gate_fwd";
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  bool done = false;
  la_status s = check_variant(fn, q, k, v, dtype, B, H, L, d_k, d_v, chunk, true, S0, nullptr,
                              O, S_final, nullptr, st, &done);
  if (s != LA_OK || done) return s;
  if (!log_alpha) return fail(LA_ERR_INVALID_ARG, "%s: log_alpha must be non-null", fn);
  if (!aligned16(log_alpha))
    return fail(LA_ERR_INVALID_ARG, "%s: log_alpha must start on a 16-byte boundary", fn);
  if (workspace) {
    const size_t need = la_channel_gate_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk, dtype);
    if (ws_bytes < need)
      return fail(LA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                  ws_bytes);
    if (!aligned16(workspace))
      return fail(LA_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", fn);
  }
  VariantArgs a{VARIANT_CHANNEL_GATE, q, k, v, dtype, B, H, L, d_k, d_v, chunk, g_phi.load(),
                log_alpha, nullptr, S0, O, S_final, st};
  a.workspace = workspace;
  a.ws_bytes = workspace ? ws_bytes : 0;
  return run_variant(fn, a);
}

la_status la_delta_fwd(const void *q, const void *k, const void *v, int dtype, int B, int H,
                       int L, int d_k, int d_v, const float *beta, const float *log_alpha,
                       const float *S0, void *O, float *S_final, void *cuda_stream) {
  const char *fn = "la_delta_fwd";
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  bool done = false;
  la_status s = check_variant(fn, q, k, v, dtype, B, H, L, d_k, d_v, 0, false, S0, nullptr, O,
                              S_final, nullptr, st, &done);
  if (s != LA_OK || done) return s;
  if (!beta) return fail(LA_ERR_INVALID_ARG, "%s: beta must be non-null", fn);
  VariantArgs a{VARIANT_DELTA, q, k, v, dtype, B, H, L, d_k, d_v, 0, g_phi.load(), log_alpha,
                beta, S0, O, S_final, st};
  return run_variant(fn, a);
}

la_status la_device_status(void *cuda_stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "la_device_status: stream synchronize");
  unsigned int word = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&word, g_device_error, sizeof word);
  if (e != cudaSuccess) return cuda_fail(e, "la_device_status: read error word");
  if (word == 0) return ok();
  e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(e, "la_device_status: clear error word");
  return fail(LA_ERR_DEVICE_TIMEOUT, "bounded wait timed out in %s (wait site %u)",
              kernel_name(word & 0xffu), (word >> 8) & 0xffu);
}

la_status la_selftest_wait_timeout(unsigned int spin_limit, void *cuda_stream) {
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = launch_wait_timeout_selftest(spin_limit, st);
  if (e != cudaSuccess) return cuda_fail(e, "la_selftest_wait_timeout: launch");
  return la_device_status(cuda_stream);
}

const char *la_last_error(void) { return g_msg; }

}  // extern "C"
