"""fp64 CPU oracle for causal linear attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library in
``causal_linear_attention_chunkwise_gb300`` never imports it, and it imports
nothing from the library: the two share no code.

The arithmetic lives in ``la_oracle.c`` (plain C, fp64, OpenMP over the
independent (b, h) sequences).  This module only compiles it with gcc, loads it
with ctypes and converts arrays to contiguous float64.

Functions (each cites the definition it follows in ``la_oracle.c``):

* :func:`recurrent`  -- token-by-token recurrence, the definition
  ("Linear / Sparse Attention - minimal runnable implementation",
  ``linear_attn_recurrent``; "CS336 lecture 4, code 1: linear attention",
  ``gated_linear_attention_recurrent``).
* :func:`parallel`   -- O(L^2) masked / decay-matrix form ("CS336 lecture 4,
  code 1", ``causal_linear_attention_parallel`` and
  ``gated_linear_attention_parallel``).
* :func:`chunkwise`  -- the chunkwise form for any chunk size C >= 1
  ("Linear / Sparse Attention - minimal runnable implementation",
  ``linear_attn_chunkwise``; "Linear / sparse attention tutorial" section 6.2).
* :func:`decode`     -- consecutive single-token decode steps; the recurrence
  run along the step axis ("adv13 - Linear Attention / SSM" section 3.2).

Decay kinds: ``"none"``, ``"head"`` (log gamma per head, shape [H]),
``"token"`` (log alpha per token, [B,H,L]) and ``"logit"`` (gate logits g,
[B,H,L], alpha = exp(-softplus(g))).  Feature maps: ``"identity"``, ``"elu1"``.

Parity: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (hand-worked golden values, closed forms,
special cases, cross-form equalities) and ``tests/test_oracle_mutants.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")

PHI = {"identity": 0, "elu1": 1}
DECAY = {"none": 0, "head": 1, "token": 2, "logit": 3}

_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = _SO, extra_flags=()) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc (OpenMP on).

    Plain portable flags only (the same source builds on x86-64 and aarch64).
    Returns the path of the library.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build(force: bool = False) -> str:
    """Build ``liboracle.so`` if missing or older than its source."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        compile_library()
    return _SO


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    sig = [i, i, i, i, i, dp, dp, dp, i, i, dp, dp, dp, dp]
    lib.oracle_recurrent.argtypes = sig
    lib.oracle_parallel.argtypes = sig
    lib.oracle_noncausal.argtypes = sig
    lib.oracle_normalised.argtypes = [i, i, i, i, i, dp, dp, dp, i, i, dp, dp, dp, dp, dp, dp]
    lib.oracle_channel_gate.argtypes = [i, i, i, i, i, dp, dp, dp, i, dp, dp, dp, dp]
    lib.oracle_delta.argtypes = [i, i, i, i, i, dp, dp, dp, i, dp, dp, dp, dp, dp]
    lib.oracle_chunkwise.argtypes = [i, i, i, i, i, i, dp, dp, dp, i, i, dp, dp, dp, dp]
    lib.oracle_delta_chunkwise.argtypes = [i, i, i, i, i, i, dp, dp, dp, i, dp, dp, dp, dp, dp]
    for f in (lib.oracle_recurrent, lib.oracle_parallel, lib.oracle_chunkwise, lib.oracle_noncausal,
              lib.oracle_normalised, lib.oracle_channel_gate, lib.oracle_delta,
              lib.oracle_delta_chunkwise):
        f.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle library.  ``path`` loads a
    different build of the same source, e.g. a test's planted-mistake copy."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def num_threads(lib=None) -> int:
    return (lib or load_library()).oracle_num_threads()


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact upcast of bf16 / fp32 values
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _prepare(q, k, v, phi, decay_kind, decay, S0):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim == 2:  # a single [L, d] sequence, as on the pages
        q, k, v = q[None, None], k[None, None], v[None, None]
        if decay is not None and decay_kind in ("token", "logit"):
            decay = _f64(decay).reshape(1, 1, -1)
        if S0 is not None:
            S0 = _f64(S0)[None, None]
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if k.shape != (B, H, L, dk) or v.shape != (B, H, L, dv):
        raise ValueError("q, k, v shapes disagree")
    decay = _f64(decay)
    if decay_kind != "none" and decay is None:
        raise ValueError("decay values required")
    if decay_kind == "head":
        decay = decay.reshape(H)
    elif decay_kind in ("token", "logit"):
        decay = decay.reshape(B, H, L)
    elif decay_kind != "none":
        raise ValueError(f"unknown decay kind {decay_kind!r}")
    S0 = _f64(S0)
    if S0 is not None and S0.shape != (B, H, dk, dv):
        raise ValueError("S0 must be [B,H,dk,dv]")
    return q, k, v, PHI[phi], DECAY[decay_kind], decay, S0, (B, H, L, dk, dv)


def _run(fn_name, q, k, v, phi, decay_kind, decay, S0, chunk=None, lib=None):
    squeeze = np.ndim(q) == 2 if not hasattr(q, "dim") else q.dim() == 2
    q, k, v, p, dkind, decay, S0, (B, H, L, dk, dv) = _prepare(q, k, v, phi, decay_kind, decay, S0)
    O = np.zeros((B, H, L, dv))
    Sf = np.zeros((B, H, dk, dv))
    lib = lib or load_library()
    fn = getattr(lib, fn_name)
    args = [B, H, L, dk, dv]
    if chunk is not None:
        args.append(int(chunk))
    rc = fn(*args, _ptr(q), _ptr(k), _ptr(v), p, dkind, _ptr(decay), _ptr(S0), _ptr(O), _ptr(Sf))
    if rc != 0:
        raise RuntimeError(f"{fn_name} failed with code {rc}")
    if squeeze:
        return O[0, 0], Sf[0, 0]
    return O, Sf


def recurrent(q, k, v, phi="identity", decay_kind="none", decay=None, S0=None, lib=None):
    """Token-by-token recurrence; returns (O, S_final) as float64 arrays."""
    return _run("oracle_recurrent", q, k, v, phi, decay_kind, decay, S0, lib=lib)


def parallel(q, k, v, phi="identity", decay_kind="none", decay=None, S0=None, lib=None):
    """O(L^2) masked / decay-matrix form; returns (O, S_final)."""
    return _run("oracle_parallel", q, k, v, phi, decay_kind, decay, S0, lib=lib)


def chunkwise(q, k, v, chunk, phi="identity", decay_kind="none", decay=None, S0=None, lib=None):
    """Chunkwise form with chunk size ``chunk``; returns (O, S_final)."""
    return _run("oracle_chunkwise", q, k, v, phi, decay_kind, decay, S0, chunk=chunk, lib=lib)


def noncausal(q, k, v, phi="identity", lib=None):
    """Non-causal matrix form O = phi(Q) (phi(K)^T V); returns (O, S) with S
    = phi(K)^T V, the state every token reads."""
    return _run("oracle_noncausal", q, k, v, phi, "none", None, None, lib=lib)


def normalised(q, k, v, phi="elu1", decay_kind="none", decay=None, S0=None, z0=None, lib=None):
    """Normalised form o_t = phi(q_t)^T S_t / phi(q_t)^T z_t, with z the state of
    a value column of ones; returns (O, S_final, z_final)."""
    q, k, v, p, dkind, decay, S0, (B, H, L, dk, dv) = _prepare(q, k, v, phi, decay_kind, decay, S0)
    z0 = _f64(z0)
    if z0 is not None and z0.shape != (B, H, dk):
        raise ValueError("z0 must be [B,H,dk]")
    O, Sf, zf = np.zeros((B, H, L, dv)), np.zeros((B, H, dk, dv)), np.zeros((B, H, dk))
    rc = (lib or load_library()).oracle_normalised(
        B, H, L, dk, dv, _ptr(q), _ptr(k), _ptr(v), p, dkind, _ptr(decay), _ptr(S0), _ptr(z0),
        _ptr(O), _ptr(Sf), _ptr(zf))
    if rc != 0:
        raise RuntimeError(f"oracle_normalised failed with code {rc}")
    return O, Sf, zf


def channel_gate(q, k, v, log_alpha, phi="identity", S0=None, lib=None):
    """Per-channel gate S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T, with
    log_alpha [B,H,L,dk]; returns (O, S_final)."""
    q, k, v, p, _, _, S0, (B, H, L, dk, dv) = _prepare(q, k, v, phi, "none", None, S0)
    la = _f64(log_alpha)
    if la.shape != (B, H, L, dk):
        raise ValueError("log_alpha must be [B,H,L,dk]")
    O, Sf = np.zeros((B, H, L, dv)), np.zeros((B, H, dk, dv))
    rc = (lib or load_library()).oracle_channel_gate(
        B, H, L, dk, dv, _ptr(q), _ptr(k), _ptr(v), p, _ptr(la), _ptr(S0), _ptr(O), _ptr(Sf))
    if rc != 0:
        raise RuntimeError(f"oracle_channel_gate failed with code {rc}")
    return O, Sf


def delta(q, k, v, beta, log_alpha=None, phi="identity", S0=None, lib=None):
    """(Gated) delta rule with the state as [d_k, d_v]: S <- alpha (S - beta k
    (k^T S)) + beta k v^T, o = q^T S.  beta [B,H,L]; log_alpha [B,H,L] or None.
    Returns (O, S_final)."""
    q, k, v, p, _, _, S0, (B, H, L, dk, dv) = _prepare(q, k, v, phi, "none", None, S0)
    be = _f64(beta)
    la = _f64(log_alpha)
    if be.shape != (B, H, L) or (la is not None and la.shape != (B, H, L)):
        raise ValueError("beta and log_alpha must be [B,H,L]")
    O, Sf = np.zeros((B, H, L, dv)), np.zeros((B, H, dk, dv))
    rc = (lib or load_library()).oracle_delta(
        B, H, L, dk, dv, _ptr(q), _ptr(k), _ptr(v), p, _ptr(be), _ptr(la), _ptr(S0), _ptr(O),
        _ptr(Sf))
    if rc != 0:
        raise RuntimeError(f"oracle_delta failed with code {rc}")
    return O, Sf


def delta_chunkwise(q, k, v, beta, chunk, log_alpha=None, phi="identity", S0=None, lib=None):
    """The delta rule of ``delta`` evaluated a chunk of ``chunk`` tokens at a
    time (the WY form: per chunk, a unit lower-triangular solve for the
    written values u_t, then dense products).  Returns (O, S_final)."""
    q, k, v, p, _, _, S0, (B, H, L, dk, dv) = _prepare(q, k, v, phi, "none", None, S0)
    be = _f64(beta)
    la = _f64(log_alpha)
    if be.shape != (B, H, L) or (la is not None and la.shape != (B, H, L)):
        raise ValueError("beta and log_alpha must be [B,H,L]")
    O, Sf = np.zeros((B, H, L, dv)), np.zeros((B, H, dk, dv))
    rc = (lib or load_library()).oracle_delta_chunkwise(
        B, H, L, dk, dv, int(chunk), _ptr(q), _ptr(k), _ptr(v), p, _ptr(be), _ptr(la), _ptr(S0),
        _ptr(O), _ptr(Sf))
    if rc != 0:
        raise RuntimeError(f"oracle_delta_chunkwise failed with code {rc}")
    return O, Sf


def decode(q, k, v, S0, log_alpha=None, phi="elu1", lib=None):
    """``steps`` consecutive decode steps from state ``S0``.

    q, k [steps,B,H,dk]; v [steps,B,H,dv]; log_alpha [steps,B,H] or None;
    S0 [B,H,dk,dv].  Each step is S <- alpha S + phi(k) v^T, o = phi(q)^T S,
    i.e. the recurrence with the step axis as the token axis.  Returns
    (o [steps,B,H,dv], S_final [B,H,dk,dv]).
    """
    q, k, v = (np.moveaxis(_f64(x), 0, 2) for x in (q, k, v))
    kind, dec = "none", None
    if log_alpha is not None:
        kind, dec = "token", np.moveaxis(_f64(log_alpha), 0, 2)
    O, Sf = recurrent(q, k, v, phi=phi, decay_kind=kind, decay=dec, S0=S0, lib=lib)
    return np.moveaxis(O, 2, 0), Sf
