"""Python binding of the C ABI, with the same names.  Argument marshalling only:
tensors become device pointers, torch supplies output memory and the current
CUDA stream, and every step of the computation runs in the library's kernels.

Host (CPU) tensors are accepted too: they are copied to the current device,
the same kernels run, and the outputs are copied back (this is the
end-to-end path the benchmark times with host buffers).
"""
from __future__ import annotations

import torch

from . import _native

PHI = {"identity": 0, "elu1": 1}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
DECAY = {"none": 0, "head": 1, "token": 2, "logit": 3}

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_DEVICE_TIMEOUT = range(5)


class LAError(RuntimeError):
    """A non-zero la_status, with the library's message."""

    def __init__(self, status: int, message: str):
        super().__init__(f"la_status {status}: {message}")
        self.status = status


def _check(status: int):
    if status != LA_OK:
        raise LAError(status, _native.load().la_last_error().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("expected CUDA tensors")
        if t is not None and not t.is_contiguous():
            raise ValueError("expected contiguous tensors")


def la_set_feature_map(phi) -> None:
    """Select phi ("identity" | "elu1" or 0 | 1) for all later calls."""
    _check(_native.load().la_set_feature_map(PHI.get(phi, phi)))


def la_get_feature_map() -> int:
    return _native.load().la_get_feature_map()


def la_chunk_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk=64, dtype=torch.bfloat16) -> int:
    return int(_native.load().la_chunk_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk,
                                                           DTYPE[dtype]))


def la_chunk_fwd_kernel_count(B, H, L, d_k, d_v, chunk=64, dtype=torch.bfloat16) -> int:
    return int(_native.load().la_chunk_fwd_kernel_count(B, H, L, d_k, d_v, chunk, DTYPE[dtype]))


_ws_cache: dict = {}


def _workspace(nbytes, device, stream=None):
    """A cached scratch buffer per (device, stream): calls ordered on one
    stream may share it, calls on different streams never do."""
    if nbytes == 0:
        return None
    s = torch.cuda.current_stream(device) if stream is None else stream
    key = (device.index, s.cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        if stream is not None:
            buf.record_stream(s)  # the allocator must not hand it out while s may use it
        _ws_cache[key] = buf
    return buf


def la_chunk_fwd(q, k, v, chunk=64, decay_kind="none", decay=None, S0=None, O=None,
                 S_final=None, want_final_state=True, workspace=None, stream=None):
    """Chunkwise causal linear attention over [B,H,L,d] sequences.

    Returns ``(O, S_final)`` (``S_final`` is None when ``want_final_state`` is
    false and no buffer is given).  ``decay_kind``: "none" | "head" (decay =
    fp32 [H] log gamma) | "token" (fp32 [B,H,L] log alpha) | "logit" (fp32
    [B,H,L] gate logits g).  ``S0``: fp32 [B,H,d_k,d_v] or None.
    """
    if not q.is_cuda:
        return _chunk_fwd_host(q, k, v, chunk, decay_kind, decay, S0, want_final_state)
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or v.dtype != q.dtype or k.dtype != q.dtype:
        raise ValueError("q, k, v must agree in [B,H,L] and dtype")
    if O is None:
        O = torch.empty(B, H, L, dv, dtype=q.dtype, device=q.device)
    if S_final is None and want_final_state:
        S_final = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    _need_cuda(q, k, v, decay, S0, O, S_final)
    lib = _native.load()
    ws_need = la_chunk_fwd_workspace_bytes(B, H, L, dk, dv, chunk, q.dtype)
    if workspace is None:
        workspace = _workspace(ws_need, q.device, stream)
    _check(lib.la_chunk_fwd(
        _ptr(q), _ptr(k), _ptr(v), DTYPE[q.dtype], B, H, L, dk, dv, chunk,
        DECAY[decay_kind], _ptr(decay), _ptr(S0), _ptr(O), _ptr(S_final),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return O, S_final


def la_noncausal_fwd_workspace_bytes(B, H, L, d_k, d_v) -> int:
    return int(_native.load().la_noncausal_fwd_workspace_bytes(B, H, L, d_k, d_v))


def la_noncausal_fwd(q, k, v, O=None, S=None, want_state=True, workspace=None, stream=None):
    """Non-causal linear attention O = phi(Q) (phi(K)^T V) over [B,H,L,d] bf16
    sequences on the GPU.  Returns ``(O, S)`` with S = phi(K)^T V, fp32
    [B,H,d,d] (None when ``want_state`` is false and no buffer is given)."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or v.dtype != q.dtype or k.dtype != q.dtype:
        raise ValueError("q, k, v must agree in [B,H,L] and dtype")
    if O is None:
        O = torch.empty(B, H, L, dv, dtype=q.dtype, device=q.device)
    if S is None and want_state:
        S = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    _need_cuda(q, k, v, O, S)
    lib = _native.load()
    if workspace is None:
        workspace = _workspace(la_noncausal_fwd_workspace_bytes(B, H, L, dk, dv), q.device,
                               stream)
    _check(lib.la_noncausal_fwd(
        _ptr(q), _ptr(k), _ptr(v), DTYPE[q.dtype], B, H, L, dk, dv, _ptr(O), _ptr(S),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return O, S


def la_chunk_fwd_noalloc(q, k, v, chunk=64, decay_kind="none", decay=None, S0=None, O=None,
                         S_final=None, want_final_state=True, stream=None):
    """la_chunk_fwd without a caller workspace, for callers that cannot
    allocate device memory at call time: the library's fixed static scratch
    (la_chunk_fwd_noalloc_scratch_bytes() bytes per GPU) holds the segment
    states.  Calls on one device share that scratch, so calls that may run
    concurrently on the GPU must be ordered by the caller.  Output buffers
    are allocated here only when not given; pass O and S_final to allocate
    nothing at all."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if O is None:
        O = torch.empty(B, H, L, dv, dtype=q.dtype, device=q.device)
    if S_final is None and want_final_state:
        S_final = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    _need_cuda(q, k, v, decay, S0, O, S_final)
    _check(_native.load().la_chunk_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), DTYPE[q.dtype], B, H, L, dk, dv, chunk, DECAY[decay_kind],
        _ptr(decay), _ptr(S0), _ptr(O), _ptr(S_final), _stream(stream)))
    return O, S_final


def la_chunk_fwd_noalloc_prepare():
    """Look up the static scratch on the current device (which is where lazy
    module loading reserves it).  Call once per device at start-up, before
    the point where the caller may no longer allocate."""
    _check(_native.load().la_chunk_fwd_noalloc_prepare())


def la_chunk_fwd_noalloc_scratch_bytes() -> int:
    return int(_native.load().la_chunk_fwd_noalloc_scratch_bytes())


def _chunk_fwd_host(q, k, v, chunk, decay_kind, decay, S0, want_final_state):
    dev = torch.device("cuda", torch.cuda.current_device())
    to = lambda t: None if t is None else t.to(dev, non_blocking=True)  # noqa: E731
    O, Sf = la_chunk_fwd(to(q), to(k), to(v), chunk, decay_kind, to(decay), to(S0),
                         want_final_state=want_final_state)
    O_h = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
    O_h.copy_(O, non_blocking=True)
    Sf_h = None
    if Sf is not None:
        Sf_h = torch.empty(Sf.shape, dtype=Sf.dtype, pin_memory=True)
        Sf_h.copy_(Sf, non_blocking=True)
    torch.cuda.current_stream().synchronize()
    return O_h, Sf_h


def la_decode_step(q, k, v, S, log_alpha=None, o=None, stream=None):
    """One decode step: S <- alpha S + phi(k) v^T in place, returns o = phi(q)^T S.
    q, k [B,H,d_k], v [B,H,d_v], S fp32 [B,H,d_k,d_v], log_alpha fp32 [B,H]."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, S, log_alpha, o)
    if S.dtype != torch.float32:
        raise ValueError("the state S must be fp32")
    _check(_native.load().la_decode_step(
        _ptr(q), _ptr(k), _ptr(v), DTYPE[q.dtype], B, H, dk, dv, _ptr(log_alpha), _ptr(S),
        _ptr(o), _stream(stream)))
    return o


def _state_bufs(q, v, want, S_final, extra=False, z_final=None):
    B, H, _, dk = q.shape
    dv = v.shape[-1]
    if S_final is None and want:
        S_final = torch.empty(B, H, dk, dv, dtype=torch.float32, device=q.device)
    if extra and z_final is None and want:
        z_final = torch.empty(B, H, dk, dtype=torch.float32, device=q.device)
    return S_final, z_final


def _qkv(q, k, v, O):
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or v.dtype != q.dtype or k.dtype != q.dtype:
        raise ValueError("q, k, v must agree in [B,H,L] and dtype")
    B, H, L, _ = q.shape
    if O is None:
        O = torch.empty(B, H, L, v.shape[-1], dtype=q.dtype, device=q.device)
    return O


def la_normalised_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk=64, dtype=torch.bfloat16) -> int:
    return int(_native.load().la_normalised_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk,
                                                                DTYPE[dtype]))


def la_normalised_fwd(q, k, v, chunk=64, decay_kind="none", decay=None, S0=None, z0=None,
                      O=None, S_final=None, z_final=None, want_final_state=True,
                      workspace=None, stream=None):
    """Normalised form o_t = phi(q_t)^T S_t / phi(q_t)^T z_t over [B,H,L,d]
    sequences, z the decayed key sum.  Returns ``(O, S_final, z_final)``.
    ``S0`` fp32 [B,H,d_k,d_v], ``z0`` fp32 [B,H,d_k]; the outputs may be the
    same tensors as the inputs (with L = 1 that is one decode step)."""
    O = _qkv(q, k, v, O)
    S_final, z_final = _state_bufs(q, v, want_final_state, S_final, True, z_final)
    _need_cuda(q, k, v, decay, S0, z0, O, S_final, z_final)
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if workspace is None:
        workspace = _workspace(la_normalised_fwd_workspace_bytes(B, H, L, dk, dv, chunk, q.dtype),
                               q.device, stream)
    _check(_native.load().la_normalised_fwd(
        _ptr(q), _ptr(k), _ptr(v), DTYPE[q.dtype], B, H, L, dk, dv, chunk,
        DECAY[decay_kind], _ptr(decay), _ptr(S0), _ptr(z0), _ptr(O), _ptr(S_final),
        _ptr(z_final), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return O, S_final, z_final


def la_channel_gate_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk=64, dtype=torch.bfloat16) -> int:
    return int(_native.load().la_channel_gate_fwd_workspace_bytes(B, H, L, d_k, d_v, chunk,
                                                                  DTYPE[dtype]))


def la_channel_gate_fwd(q, k, v, log_alpha, chunk=64, S0=None, O=None, S_final=None,
                        want_final_state=True, workspace=None, segments=True, stream=None):
    """Per-channel gate S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T with
    ``log_alpha`` fp32 [B,H,L,d_k].  Returns ``(O, S_final)``.  With
    ``segments`` (the default) a cached workspace lets the library run each
    sequence as several segments side by side; ``segments=False`` runs each
    sequence in one piece."""
    O = _qkv(q, k, v, O)
    S_final, _ = _state_bufs(q, v, want_final_state, S_final)
    _need_cuda(q, k, v, log_alpha, S0, O, S_final)
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if log_alpha.shape != (B, H, L, dk) or log_alpha.dtype != torch.float32:
        raise ValueError("log_alpha must be fp32 [B,H,L,d_k]")
    if workspace is None and segments:
        workspace = _workspace(la_channel_gate_fwd_workspace_bytes(B, H, L, dk, dv, chunk, q.dtype),
                               q.device, stream)
    _check(_native.load().la_channel_gate_fwd(
        _ptr(q), _ptr(k), _ptr(v), DTYPE[q.dtype], B, H, L, dk, dv, chunk,
        _ptr(log_alpha), _ptr(S0), _ptr(O), _ptr(S_final), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return O, S_final


def la_delta_fwd(q, k, v, beta, log_alpha=None, S0=None, O=None, S_final=None,
                 want_final_state=True, stream=None):
    """(Gated) delta rule S <- alpha (S - beta k (k^T S)) + beta k v^T,
    o = phi(q)^T S, token by token; ``beta`` and ``log_alpha`` fp32 [B,H,L]
    (``log_alpha`` None: alpha = 1).  Returns ``(O, S_final)``."""
    O = _qkv(q, k, v, O)
    S_final, _ = _state_bufs(q, v, want_final_state, S_final)
    _need_cuda(q, k, v, beta, log_alpha, S0, O, S_final)
    B, H, L, dk = q.shape
    for t in (beta, log_alpha):
        if t is not None and (t.shape != (B, H, L) or t.dtype != torch.float32):
            raise ValueError("beta and log_alpha must be fp32 [B,H,L]")
    _check(_native.load().la_delta_fwd(
        _ptr(q), _ptr(k), _ptr(v), DTYPE[q.dtype], B, H, L, dk, v.shape[-1], _ptr(beta),
        _ptr(log_alpha), _ptr(S0), _ptr(O), _ptr(S_final), _stream(stream)))
    return O, S_final


def la_device_status(stream=None) -> None:
    """Synchronise and raise LAError if a kernel's bounded wait timed out."""
    _check(_native.load().la_device_status(_stream(stream)))


def la_selftest_wait_timeout(spin_limit: int = 1000, stream=None) -> int:
    """Run the timeout self-test kernel; returns the status it reports."""
    lib = _native.load()
    return lib.la_selftest_wait_timeout(spin_limit, _stream(stream))


def la_last_error() -> str:
    return _native.load().la_last_error().decode()
