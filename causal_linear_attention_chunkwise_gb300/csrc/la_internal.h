// la_internal.h -- launchers shared between the ABI translation unit and the
// kernel translation units.  Host-only declarations; no device code.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

namespace la {

// Device error word set by kernels whose bounded waits run out.  Codes:
// bits 0..7 kernel id, bits 8..15 wait site (see la_common.cuh).
unsigned int *device_error_word();  // device address for the current device

struct PrefillArgs {
  const void *q, *k, *v;
  int dtype;  // LA_F32 / LA_BF16
  int B, H, L, dk, dv, chunk;
  int phi;
  int decay_kind;
  const float *decay;
  const float *S0;
  void *O;
  float *S_final;
  void *workspace;
  size_t ws_bytes;
  cudaStream_t stream;
};

struct DecodeArgs {
  const void *q, *k, *v;
  int dtype;
  int B, H, dk, dv;
  int phi;
  const float *log_alpha;
  float *S;
  void *o;
  cudaStream_t stream;
};

// General SIMT prefill (fp32 or bf16, 1 <= chunk <= 64, d <= 128).
cudaError_t launch_prefill_simt(const PrefillArgs &a);

// Tensor-core (tcgen05) prefill: bf16, chunk 64, dk == dv in {64, 128}.
bool prefill_tc_supported(const PrefillArgs &a);
size_t prefill_tc_workspace_bytes(int B, int H, int L, int d);
int prefill_tc_kernel_count(int B, int H, int L, int d);
cudaError_t launch_prefill_tc(const PrefillArgs &a, const char **why);

// The normalised form in one pass on the d = 64 tensor-core kernels: a ones
// column rides with V, so O carries the denominator (divided out before the
// store) and the state carries z.  Supported when prefill_tc_supported and
// d_k = d_v = 64; the workspace holds segment states of 64 + 16 columns.
bool prefill_tc_norm_supported(const PrefillArgs &a);
size_t prefill_tc_norm_workspace_bytes(int B, int H, int L);
cudaError_t launch_prefill_tc_norm(const PrefillArgs &a, const float *z0, float *z_final,
                                   const char **why);

// Non-causal form O = phi(Q) (phi(K)^T V): bf16, d_k == d_v in {64, 128}.
struct NoncausalArgs {
  const void *q, *k, *v;
  int B, H, L, d;
  int phi;
  void *O;
  float *S;  // [B,H,d,d] fp32 or null
  void *workspace;
  size_t ws_bytes;
  cudaStream_t stream;
};
size_t noncausal_workspace_bytes(int B, int H, int L, int d);
cudaError_t launch_noncausal(const NoncausalArgs &a, const char **why);

// Per-channel gate and delta rule (CUDA cores, fp32 or bf16 inputs,
// d_k, d_v <= 128).
enum VariantForm { VARIANT_CHANNEL_GATE = 1, VARIANT_DELTA = 2 };
struct VariantArgs {
  int form;  // VariantForm
  const void *q, *k, *v;
  int dtype;
  int B, H, L, dk, dv, chunk;  // chunk: 1..64 (unused by the delta rule)
  int phi;
  const float *decay;  // channel gate: log alpha [B,H,L,dk]; delta rule: log alpha [B,H,L] or null
  const float *beta;   // delta rule: [B,H,L]
  const float *S0;
  void *O;
  float *S_final;
  cudaStream_t stream;
  void *workspace = nullptr;  // channel gate: segment states (optional)
  size_t ws_bytes = 0;
};
cudaError_t launch_variant(const VariantArgs &a);

// The per-channel gate on the tensor cores: bf16, chunk 64, d_k == d_v in
// {64, 128}; launch_variant takes this path when it applies.
bool channel_gate_tc_supported(const VariantArgs &a);
cudaError_t launch_channel_gate_tc(const VariantArgs &a);
// Workspace for running each sequence as several segments (0: one per sequence).
size_t channel_gate_tc_workspace_bytes(int B, int H, int L, int d);

// The delta rule a chunk of 64 tokens at a time on the tensor cores (the WY
// form): bf16, d_k == d_v in {64, 128}; launch_variant takes this path when it
// applies.
bool delta_tc_supported(const VariantArgs &a);
cudaError_t launch_delta_tc(const VariantArgs &a);

// Denominator of the normalised form and the division of O by it, after the
// numerator has been written to O (d_k <= 128).
struct NormaliserArgs {
  const void *q, *k;
  int dtype;
  int B, H, L, dk, dv;
  int phi;
  int decay_kind;
  const float *decay;
  const float *z0;
  void *O;
  float *z_final;
  void *workspace;  // normaliser_workspace_bytes(...) bytes, float-aligned
  cudaStream_t stream;
};
size_t normaliser_workspace_bytes(int B, int H, int L, int dk);
cudaError_t launch_normaliser(const NormaliserArgs &a);

// Decode step.
bool decode_supported(int dk, int dv);
cudaError_t launch_decode(const DecodeArgs &a);

// Set the message la_last_error() returns on the calling thread.
void set_last_error(const char *msg);

// Self-test of the bounded-wait timeout path.
cudaError_t launch_wait_timeout_selftest(unsigned int spin_limit, cudaStream_t s);

}  // namespace la
