/*
 * la_gb300.h -- C ABI of the GB300 (sm_103a) causal linear attention library.
 *
 * What the library computes.  For every (batch b, head h) sequence of L tokens
 * with queries q_t, keys k_t (width d_k) and values v_t (width d_v), a matrix
 * state S in R^{d_k x d_v} evolves as
 *
 *     S_t = a_t S_{t-1} + phi(k_t) v_t^T,        o_t = phi(q_t)^T S_t
 *
 * (update before read; S_{-1} = S0 or zero).  Sources:
 *   - "Linear / Sparse Attention - minimal runnable implementation",
 *     linear_attn_recurrent (the self-inclusive recurrence, S in R^{d_k x d_v})
 *     and linear_attn_chunkwise (the chunk form the prefill kernels evaluate:
 *     inter-chunk read Q_c S, intra-chunk ((Q_c K_c^T) .* tril) V_c with the
 *     diagonal included, then S += K_c^T V_c; a ragged last chunk);
 *   - "CS336 lecture 4, code 1: linear attention",
 *     gated_linear_attention_recurrent (S_t = gamma_t S_{t-1} + k_t v_t^T;
 *     constant gamma is RetNet, input-dependent gamma_t the Mamba-2 gate) and
 *     gated_linear_attention_parallel (decay factors taken in log space);
 *   - "Linear / sparse attention tutorial" section 6.2 (the two-part chunk
 *     computation; gates multiply the state and the in-chunk mask by the
 *     cumulative decay) and section 8.1 (decode keeps only the fixed-size
 *     state);
 *   - "adv13 - Linear Attention / SSM" section 3.2 / 4.2 (phi applied to q
 *     and k, never to v) and Q1 (phi = elu + 1).
 *
 * Conventions for every entry point:
 *   - Pointers to tensors are DEVICE pointers owned by the caller; the library
 *     never frees them and never allocates device memory.  Tensors are dense,
 *     row-major, contiguous, and must start on a 16-byte boundary.
 *   - Calls are asynchronous on the CUDA stream passed as `cuda_stream`
 *     (a cudaStream_t; NULL = the legacy default stream).  The return status
 *     covers argument validation and kernel launch; a device-side timeout of a
 *     bounded wait is reported by la_device_status().
 *   - No call aborts, throws or prints.  On any non-zero status the reason is
 *     available from la_last_error() on the calling thread.
 */
#ifndef LA_GB300_H
#define LA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int la_status;

#define LA_OK                 0  /* success */
#define LA_ERR_INVALID_ARG    1  /* bad pointer, size, alignment or enum value */
#define LA_ERR_UNSUPPORTED    2  /* valid request the library has no kernel for */
#define LA_ERR_CUDA           3  /* a CUDA runtime call or launch failed */
#define LA_ERR_DEVICE_TIMEOUT 4  /* a kernel's bounded wait ran out (la_device_status) */

/* Feature map phi applied to q and k. */
#define LA_PHI_IDENTITY 0        /* phi(x) = x ("tutorial" 2.1: RetNet / GLA use phi = id) */
#define LA_PHI_ELU1     1        /* phi(x) = elu(x) + 1 = x + 1 (x > 0), exp(x) (x <= 0) */

/* Element type of q, k, v and of the outputs O / o.  The state is always fp32. */
#define LA_F32  0
#define LA_BF16 1

/* How the per-token decay a_t is given (always in log space, fp32). */
#define LA_DECAY_NONE       0   /* a_t = 1; decay pointer ignored (may be NULL)    */
#define LA_DECAY_HEAD       1   /* decay[h] = log gamma_h, shape [H] (RetNet)      */
#define LA_DECAY_TOKEN      2   /* decay[b,h,t] = log alpha_t, shape [B,H,L]       */
#define LA_DECAY_GATE_LOGIT 3   /* decay[b,h,t] = g_t, alpha_t = exp(-softplus(g_t)),
                                   shape [B,H,L] (Mamba-2-style input gate)       */

/* Select phi for all later calls in this process (atomic; default identity).
 * Returns LA_ERR_INVALID_ARG for an unknown value. */
la_status la_set_feature_map(int phi);

/* The feature map currently selected. */
int la_get_feature_map(void);

/* Bytes of device workspace la_chunk_fwd needs for this problem (0 if none).
 * The workspace holds per-segment partial states when the sequence is split
 * across CTAs; its contents need no initialisation and are not kept. */
size_t la_chunk_fwd_workspace_bytes(int B, int H, int L, int d_k, int d_v, int chunk,
                                    int dtype);

/* Number of kernel launches one la_chunk_fwd call makes for this problem
 * (host-only query; 0 for an empty problem or an unsupported one). */
int la_chunk_fwd_kernel_count(int B, int H, int L, int d_k, int d_v, int chunk, int dtype);

/*
 * Chunkwise-parallel causal linear attention over whole sequences (prefill).
 *
 *   q, k      [B,H,L,d_k]  dtype            (read)
 *   v         [B,H,L,d_v]  dtype            (read)
 *   dtype     LA_F32 or LA_BF16
 *   chunk     chunk size C (tokens per chunk); the result does not depend on
 *             it up to rounding.  The tensor-core path takes C = 64; the
 *             fp32 / general path takes 1 <= C <= 64.
 *   decay_kind / decay   see LA_DECAY_*; decay is fp32 device memory.
 *   S0        [B,H,d_k,d_v] fp32 initial state, or NULL for zero   (read)
 *   O         [B,H,L,d_v]   dtype, every row written                (write)
 *   S_final   [B,H,d_k,d_v] fp32 state after the last token, or NULL
 *             (write; may be the same buffer as S0)
 *   workspace device scratch of at least la_chunk_fwd_workspace_bytes(...)
 *             bytes (may be NULL when that is 0); ws_bytes = its size.
 *
 * Supported: d_k, d_v in {16, 32, 64, 128}; fp32 inputs run the fp32 SIMT
 * kernel, bf16 inputs with d_k = d_v in {64, 128} and C = 64 run the tcgen05
 * tensor-core kernels, other bf16 shapes the SIMT kernel.  L = 0 writes
 * S_final = S0 (or zero).  Errors: LA_ERR_INVALID_ARG (null or misaligned
 * pointer, negative size, unknown enum, workspace too small),
 * LA_ERR_UNSUPPORTED (a d or C outside the list), LA_ERR_CUDA.
 */
la_status la_chunk_fwd(const void *q, const void *k, const void *v, int dtype,
                       int B, int H, int L, int d_k, int d_v, int chunk,
                       int decay_kind, const float *decay,
                       const float *S0, void *O, float *S_final,
                       void *workspace, size_t ws_bytes, void *cuda_stream);

/*
 * One recurrent decode step for B*H sequences, state updated in place:
 *
 *     S <- alpha S + phi(k) v^T ;   o = phi(q)^T S      (update, then read)
 *
 *   q, k       [B,H,d_k] dtype   (read)
 *   v          [B,H,d_v] dtype   (read)
 *   log_alpha  [B,H] fp32 log of the decay, or NULL for alpha = 1  (read)
 *   S          [B,H,d_k,d_v] fp32, read and overwritten             (in/out)
 *   o          [B,H,d_v] dtype                                      (write)
 *
 * Supported: d_k = d_v in {16, 32, 64, 128}.  Errors as for la_chunk_fwd.
 */
la_status la_decode_step(const void *q, const void *k, const void *v, int dtype,
                         int B, int H, int d_k, int d_v,
                         const float *log_alpha, float *S, void *o, void *cuda_stream);

/*
 * The non-causal matrix form, for B*H independent sequences of L tokens:
 *
 *     S = phi(K)^T V  (summed over all L tokens) ;   O = phi(Q) S
 *
 * (page "adv13 - Linear Attention / SSM", section 4.3, linear_attention_matrix;
 * page "CS336 lecture 4, code 1: linear attention", demo_associativity: the
 * order (Q K^T) V = Q (K^T V)).  Every token reads the same state: there is no
 * causal mask, no decay and no initial state.  The feature map is the one set
 * by la_set_feature_map.
 *
 *   q, k       [B,H,L,d] bf16                          (read)
 *   v          [B,H,L,d] bf16                          (read)
 *   O          [B,H,L,d] bf16                          (write)
 *   S          [B,H,d,d] fp32, the state phi(K)^T V, or NULL (write)
 *   workspace  device scratch of la_noncausal_fwd_workspace_bytes(...) bytes
 *
 * All pointers are device pointers owned by the caller, row-major and
 * 16-byte aligned; the call is asynchronous on `cuda_stream`.
 * Supported: bf16 with d_k = d_v = d in {64, 128}.  L = 0 writes S = 0.
 * Errors: LA_ERR_INVALID_ARG (null or misaligned pointer, negative size,
 * workspace too small), LA_ERR_UNSUPPORTED (another dtype or d), LA_ERR_CUDA.
 */
la_status la_noncausal_fwd(const void *q, const void *k, const void *v, int dtype,
                           int B, int H, int L, int d_k, int d_v,
                           void *O, float *S, void *workspace, size_t ws_bytes,
                           void *cuda_stream);
size_t la_noncausal_fwd_workspace_bytes(int B, int H, int L, int d_k, int d_v);

/*
 * Three further forms of the recurrence (q, k, v and O in dtype = LA_F32 or
 * LA_BF16; states fp32).  Each runs over whole sequences like la_chunk_fwd,
 * and each is also its own decode step:
 * with L = 1 and the output state aliasing the input state, one call advances
 * every sequence by one token.  phi is the one set by la_set_feature_map.
 * Supported: d_k, d_v in {16, 32, 64, 128}; chunk 1..64 where one is taken
 * (the result does not depend on it up to rounding).  L = 0 passes the
 * initial states through (or zeroes the outputs when none is given).  Errors:
 * LA_ERR_INVALID_ARG (null or misaligned pointer, negative size, unknown
 * enum), LA_ERR_UNSUPPORTED (a d or chunk outside the list), LA_ERR_CUDA.
 * Pointers are device pointers owned by the caller, row-major, 16-byte
 * aligned; the calls are asynchronous on `cuda_stream` and allocate nothing.
 * The per-channel gate and the delta rule run on the CUDA cores in fp32.
 */

/*
 * Normalised linear attention ("Linear / sparse attention tutorial" Q11 and
 * section 2.2): the state carries a key sum z next to S, which decays with S,
 *
 *     S_t = a_t S_{t-1} + phi(k_t) v_t^T,   z_t = a_t z_{t-1} + phi(k_t),
 *     o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t).
 *
 * For bf16 with d_k = d_v = 64 and chunk 64 it is one pass of the tensor-core
 * prefill kernels: a column of ones rides with v, so z travels as one more
 * state column and each row's denominator comes out of the same products as
 * its numerator, and the epilogue divides before it stores O.  Otherwise the
 * numerator runs on the la_chunk_fwd kernels (the tensor-core ones for bf16,
 * d_k = d_v = 128, chunk 64), then a scan of z forms the denominators and
 * divides O in place.  There is no epsilon in the denominator: choose a
 * positive feature map (LA_PHI_ELU1), as the tutorial does, or the quotient
 * may be undefined.
 *
 *   q, k   [B,H,L,d_k] dtype;  v, O [B,H,L,d_v] dtype
 *   decay_kind / decay   as for la_chunk_fwd
 *   S0     [B,H,d_k,d_v] fp32 or NULL (zero);  z0 [B,H,d_k] fp32 or NULL (zero)
 *   S_final, z_final   the states after the last token, or NULL; each may be
 *          the same buffer as S0 / z0.
 *   workspace  device scratch of la_normalised_fwd_workspace_bytes(...) bytes,
 *          or NULL when that is 0 (the one-pass form on a sequence short
 *          enough for one CTA); ws_bytes = its size.  Its contents need no
 *          initialisation and are not kept.
 */
la_status la_normalised_fwd(const void *q, const void *k, const void *v, int dtype,
                            int B, int H, int L, int d_k, int d_v, int chunk,
                            int decay_kind, const float *decay,
                            const float *S0, const float *z0, void *O,
                            float *S_final, float *z_final,
                            void *workspace, size_t ws_bytes, void *cuda_stream);
size_t la_normalised_fwd_workspace_bytes(int B, int H, int L, int d_k, int d_v, int chunk,
                                         int dtype);

/*
 * Per-channel (diagonal) gate, as in GLA ("Linear / sparse attention
 * tutorial" Q21):
 *
 *     S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T,   o_t = phi(q_t)^T S_t,
 *
 * one decay per key channel and token.
 *
 *   log_alpha  [B,H,L,d_k] fp32, log alpha_t[i] (expected <= 0), 16-byte
 *              aligned like the other tensors                      (read)
 *   S0         [B,H,d_k,d_v] fp32 or NULL;  S_final may alias S0.
 *   workspace  device scratch of la_channel_gate_fwd_workspace_bytes(...)
 *              bytes (16-byte aligned), or NULL; ws_bytes = its size.  With it
 *              (bf16, d_k = d_v in {64, 128}, chunk 64, when the query is not
 *              0) each sequence is cut into segments that run side by side: a
 *              state pass over every segment but the last, then the segments'
 *              outputs, each folding in the states of the segments before it.
 *              With NULL each sequence runs in one piece.
 *              A non-NULL workspace smaller than the query or misaligned is
 *              LA_ERR_INVALID_ARG.  Its contents need no initialisation and are
 *              not kept.
 */
la_status la_channel_gate_fwd(const void *q, const void *k, const void *v, int dtype,
                              int B, int H, int L, int d_k, int d_v, int chunk,
                              const float *log_alpha, const float *S0, void *O,
                              float *S_final, void *workspace, size_t ws_bytes,
                              void *cuda_stream);
size_t la_channel_gate_fwd_workspace_bytes(int B, int H, int L, int d_k, int d_v, int chunk,
                                           int dtype);

/*
 * The (gated) delta rule ("Linear / Sparse Attention - minimal runnable
 * implementation", delta_rule_recurrent; "Linear / sparse attention tutorial"
 * Q21 for the gate), with the state as [d_k, d_v] like the others:
 *
 *     S_t = alpha_t (S_{t-1} - beta_t k (k^T S_{t-1})) + beta_t k v_t^T,
 *     o_t = phi(q_t)^T S_t,      k = phi(k_t).
 *
 * Keys are used as given (after phi): the rule assumes unit-norm keys, and
 * normalising them is the caller's step.  Runs token by token.
 *
 *   beta       [B,H,L] fp32 write strengths                        (read)
 *   log_alpha  [B,H,L] fp32 log of the gate, or NULL for alpha = 1  (read)
 *   S0         [B,H,d_k,d_v] fp32 or NULL;  S_final may alias S0.
 */
la_status la_delta_fwd(const void *q, const void *k, const void *v, int dtype,
                       int B, int H, int L, int d_k, int d_v,
                       const float *beta, const float *log_alpha,
                       const float *S0, void *O, float *S_final, void *cuda_stream);

/*
 * la_chunk_fwd for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this is a deployment variant of la_chunk_fwd.)
 *
 * Some callers cannot call cudaMalloc where they run prefill -- code inside
 * an allocator or memory-pool callback, processes whose device footprint is
 * fixed after start-up, or code that runs while another component holds the
 * allocator.  This entry point takes the same arguments as la_chunk_fwd
 * without the workspace: the segment states live in one static device array
 * of LA_NOALLOC_SCRATCH_BYTES, held on each GPU until the process exits.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   - When the bytes are reserved: the CUDA runtime loads modules lazily by
 *     default, so the array is placed on a device when it is first looked
 *     up there.  Call la_chunk_fwd_noalloc_prepare() once per device, with
 *     that device current, at start-up (before any stream capture and before
 *     the point where allocation is forbidden).  A device not prepared is
 *     prepared by its first la_chunk_fwd_noalloc call, which may then
 *     reserve the bytes itself.
 *   - The looked-up address is cached per device.  It does not survive
 *     cudaDeviceReset: call la_chunk_fwd_noalloc_prepare() again after one.
 *   - Problems whose workspace (la_chunk_fwd_workspace_bytes) exceeds
 *     LA_NOALLOC_SCRATCH_BYTES are rejected with LA_ERR_UNSUPPORTED before
 *     any device work; la_last_error() names both sizes.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  Nothing in it has to start at zero (each call writes every
 *     part it reads before reading it), but calls whose kernels overlap on
 *     the GPU (different streams, or different host threads without
 *     ordering) race on it and give wrong results: order them.
 * Errors: as la_chunk_fwd, plus LA_ERR_UNSUPPORTED for a too-large problem.
 */
#define LA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
la_status la_chunk_fwd_noalloc(const void *q, const void *k, const void *v, int dtype,
                               int B, int H, int L, int d_k, int d_v, int chunk,
                               int decay_kind, const float *decay,
                               const float *S0, void *O, float *S_final, void *cuda_stream);

/* Look up (again) the static scratch on the current device and cache its
 * address; under lazy module loading this is where the scratch is reserved.
 * LA_OK, or LA_ERR_CUDA with the runtime's message. */
la_status la_chunk_fwd_noalloc_prepare(void);

/* Size in bytes of the static scratch la_chunk_fwd_noalloc uses. */
size_t la_chunk_fwd_noalloc_scratch_bytes(void);

/* Synchronise `cuda_stream`, then report and clear the device error word that
 * kernels set when a bounded wait runs out: LA_OK, LA_ERR_DEVICE_TIMEOUT (the
 * message names the kernel and the wait) or LA_ERR_CUDA. */
la_status la_device_status(void *cuda_stream);

/* Self-test of the timeout path: launches one CTA that waits on an mbarrier
 * nothing ever arrives at, with a spin limit of `spin_limit` polls; the
 * kernel records the timeout, releases what it holds and exits.  Returns the
 * status la_device_status() then reports (LA_ERR_DEVICE_TIMEOUT expected). */
la_status la_selftest_wait_timeout(unsigned int spin_limit, void *cuda_stream);

/* Message for the last non-zero status on this thread ("" if none). */
const char *la_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* LA_GB300_H */
