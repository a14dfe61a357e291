"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` takes a loaded oracle library (the real one, or a copy with a
planted mistake) and raises AssertionError when the oracle disagrees with:

* values worked by hand from the recurrence (``golden/hand_worked.json``);
* closed forms (final state phi(K)^T V; the geometric sum for a constant gamma;
  the L = 1 case; one-hot queries and keys; orthonormal keys);
* library routines for the pieces (torch ELU for phi, numpy logaddexp for
  softplus, numpy QR for orthonormal keys);
* equalities the pages check themselves: chunkwise == recurrent for
  C in {1, 4, 7, L} at L = 13, d = 6 ("Linear / Sparse Attention - minimal
  runnable implementation", checks [a], [b], [c]); parallel == recurrent ==
  chunked at n = 300, d = 16, chunk 64, and gated parallel == gated recurrent
  at n = 200, d = 16, gamma = sigmoid(k.w + 3) ("CS336 lecture 4, code 1:
  linear attention", demo_two_forms and demo_gating);
* the resume invariant: running [0, m) then [m, L) from the carried state
  equals one run over [0, L);
* for the non-causal form: the causal final state and last row, the n x n
  association order, one-hot values and L = 0 (``pin_noncausal``);
* for the normalised form and the per-channel gate (rows the library does not
  build yet): the ratio of two plain recurrences, constant values, one token;
  equal-channel and zero gates, and an O(L^2) form written with numpy
  (``pin_normalised``, ``pin_channel_gate``);
* for the delta rule: the page's checks [d]/[e] (orthonormal keys give the
  additive rule, random keys do not), exact retrieval of the value just
  written, beta = 0, one token (``pin_delta``);
* for the delta rule's chunkwise (WY) form: equality with the token-by-token
  rule for chunk sizes 1, 4, 7 and L (``pin_delta_chunkwise``).

``tests/test_oracle_mutants.py`` plants plausible mistakes in a copy of the
oracle's C source and checks that at least one pin fails for each.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_worked.json")
FORMS = ("recurrent", "parallel", "chunk1", "chunk2", "chunk7")


def _run(form, lib, *args, **kw):
    if form == "recurrent":
        return oracle.recurrent(*args, lib=lib, **kw)
    if form == "parallel":
        return oracle.parallel(*args, lib=lib, **kw)
    return oracle.chunkwise(*args, chunk=int(form[5:]), lib=lib, **kw)


def _close(a, b, tol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(1.0, np.max(np.abs(b)) if b.size else 1.0)
    assert err <= tol * scale, f"{what}: max |diff| {err:.3e} > {tol:.1e} x {scale:.3g}"


def _rng(seed):
    return np.random.default_rng(seed)


def _elu1(x):
    """phi via torch's ELU (alpha = 1), a library routine independent of the oracle."""
    return (torch.nn.functional.elu(torch.as_tensor(x, dtype=torch.float64)) + 1.0).numpy()


# --------------------------------------------------------------------------
def pin_golden(lib):
    """Hand-worked values (golden/hand_worked.json) for every form."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    decays = {
        "plain_additive": None,
        "constant_decay_half": [math.log(0.5)],
        "token_gate_elu1_with_S0": [math.log(0.5), math.log(0.25)],
        "gate_logits_softplus": [0.0, math.log(3.0)],
    }
    for c in cases:
        q, k, v = (np.array(c[x], dtype=np.float64) for x in ("q", "k", "v"))
        S0 = None if c["S0"] is None else np.array(c["S0"], dtype=np.float64)
        dec = decays[c["name"]]
        for form in FORMS:
            O, S = _run(form, lib, q, k, v, phi=c["phi"], decay_kind=c["decay_kind"],
                        decay=None if dec is None else np.array(dec), S0=S0)
            _close(O, c["O"], 1e-12, f"{c['name']}/{form} O")
            _close(S, c["S_final"], 1e-12, f"{c['name']}/{form} S_final")


def pin_closed_form_additive(lib):
    """No decay, S0 = 0: S_final = phi(K)^T V, and the last output row is
    phi(q_{L-1})^T S_final -- the associativity (QK^T)V = Q(K^T V) on the
    whole sequence."""
    r = _rng(1)
    B, H, L, dk, dv = 2, 3, 37, 5, 4
    q, k, v = r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dv))
    for phi in ("identity", "elu1"):
        kf = k if phi == "identity" else _elu1(k)
        qf = q if phi == "identity" else _elu1(q)
        S_ref = np.einsum("bhti,bhtj->bhij", kf, v)
        for form in ("recurrent", "parallel", "chunk7"):
            O, S = _run(form, lib, q, k, v, phi=phi)
            _close(S, S_ref, 1e-12, f"additive S_final {phi}/{form}")
            _close(O[:, :, -1], np.einsum("bhi,bhij->bhj", qf[:, :, -1], S_ref), 1e-12,
                   f"additive last row {phi}/{form}")


def pin_closed_form_constant_decay(lib):
    """Constant per-head gamma_h (distinct per head):
    S_final = gamma^L S0 + sum_t gamma^(L-1-t) k_t v_t^T."""
    r = _rng(2)
    B, H, L, dk, dv = 2, 4, 29, 3, 5
    q, k, v = r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dv))
    S0 = r.normal(size=(B, H, dk, dv))
    gam = np.array([0.5, 0.9, 0.97, 0.75])
    w = gam[None, :, None] ** (L - 1 - np.arange(L))[None, None, :]      # [1,H,L]
    S_ref = (gam ** L)[None, :, None, None] * S0 + np.einsum("ht,bhti,bhtj->bhij", w[0], k, v)
    for form in ("recurrent", "parallel", "chunk7"):
        _, S = _run(form, lib, q, k, v, decay_kind="head", decay=np.log(gam), S0=S0)
        _close(S, S_ref, 1e-12, f"constant-decay S_final/{form}")


def pin_single_token(lib):
    """L = 1: o = alpha phi(q)^T S0 + (phi(q).phi(k)) v, S = alpha S0 + phi(k) v^T."""
    r = _rng(3)
    dk, dv = 4, 3
    q, k, v = r.normal(size=(1, dk)), r.normal(size=(1, dk)), r.normal(size=(1, dv))
    S0 = r.normal(size=(dk, dv))
    la = np.array([math.log(0.8)])
    qf, kf = _elu1(q[0]), _elu1(k[0])
    o_ref = 0.8 * (qf @ S0) + (qf @ kf) * v[0]
    S_ref = 0.8 * S0 + np.outer(kf, v[0])
    for form in FORMS:
        O, S = _run(form, lib, q, k, v, phi="elu1", decay_kind="token", decay=la, S0=S0)
        _close(O[0], o_ref, 1e-12, f"L=1 o/{form}")
        _close(S, S_ref, 1e-12, f"L=1 S/{form}")


def pin_one_hot(lib):
    """One-hot q_t = e_{j_t}, k_t = e_{i_t} (identity phi, per-token decay):
    o_t = sum over s <= t with i_s == j_t of exp(c_t - c_s) v_s, plus
    exp(c_t) S0[j_t, :], where c is the running sum of log alpha.  Computed
    by index selection alone, no dot products."""
    r = _rng(4)
    L, d, dv = 23, 4, 3
    jq, ik = r.integers(0, d, size=L), r.integers(0, d, size=L)
    q, k = np.eye(d)[jq], np.eye(d)[ik]
    v = r.normal(size=(L, dv))
    la = np.log(r.uniform(0.5, 1.0, size=L))
    S0 = r.normal(size=(d, dv))
    c = np.cumsum(la)
    O_ref = np.zeros((L, dv))
    for t in range(L):
        O_ref[t] = math.exp(c[t]) * S0[jq[t]]
        for s in range(t + 1):
            if ik[s] == jq[t]:
                O_ref[t] += math.exp(c[t] - c[s]) * v[s]
    for form in FORMS:
        O, _ = _run(form, lib, q, k, v, decay_kind="token", decay=la, S0=S0)
        _close(O, O_ref, 1e-12, f"one-hot/{form}")


def pin_orthonormal_keys(lib):
    """Identity phi, no decay, L = d orthonormal keys (numpy QR): the state
    maps each key to its value, k_i^T S = v_i^T."""
    r = _rng(5)
    d, dv = 6, 4
    Qm, _ = np.linalg.qr(r.normal(size=(d, d)))
    K = Qm.T
    V = r.normal(size=(d, dv))
    Q = r.normal(size=(d, d))
    for form in FORMS:
        _, S = _run(form, lib, Q, K, V)
        _close(K @ S, V, 1e-12, f"orthonormal keys/{form}")


def pin_chunk_invariance(lib):
    """chunkwise == recurrent for C in {1, 4, 7, L} at L = 13, d = 6, for every
    phi / decay / S0 combination, plus C = 64 at L = 300 with a ragged tail."""
    r = _rng(6)
    B, H, L, d = 1, 2, 13, 6
    q, k, v = r.normal(size=(B, H, L, d)), r.normal(size=(B, H, L, d)), r.normal(size=(B, H, L, d))
    S0 = r.normal(size=(B, H, d, d))
    variants = [("identity", "none", None, None), ("elu1", "none", None, S0),
                ("identity", "head", np.log([0.9, 0.6]), S0),
                ("elu1", "token", np.log(r.uniform(0.3, 1.0, size=(B, H, L))), S0),
                ("identity", "logit", r.normal(size=(B, H, L)) * 3.0, S0)]
    for phi, kind, dec, s0 in variants:
        O_ref, S_ref = oracle.recurrent(q, k, v, phi=phi, decay_kind=kind, decay=dec, S0=s0, lib=lib)
        for C in (1, 4, 7, L):
            O, S = oracle.chunkwise(q, k, v, C, phi=phi, decay_kind=kind, decay=dec, S0=s0, lib=lib)
            _close(O, O_ref, 1e-11, f"chunk C={C} {phi}/{kind} O")
            _close(S, S_ref, 1e-11, f"chunk C={C} {phi}/{kind} S")
    q, k, v = r.normal(size=(300, 16)), r.normal(size=(300, 16)), r.normal(size=(300, 16))
    O_ref, S_ref = oracle.recurrent(q, k, v, lib=lib)
    O, S = oracle.chunkwise(q, k, v, 64, lib=lib)
    _close(O, O_ref, 1e-11, "chunk 64 ragged O")
    _close(S, S_ref, 1e-11, "chunk 64 ragged S")


def pin_parallel_equals_recurrent(lib):
    """The page's two demos: parallel == recurrent == chunked (n = 300, d = 16,
    chunk 64) and gated parallel == gated recurrent (n = 200, d = 16,
    gamma_t = sigmoid(k_t . w + 3), given here as log gamma_t)."""
    g = torch.Generator().manual_seed(0)
    n, d = 300, 16
    q, k, v = (torch.randn(n, d, generator=g, dtype=torch.float64) for _ in range(3))
    Op, _ = oracle.parallel(q, k, v, lib=lib)
    Or, _ = oracle.recurrent(q, k, v, lib=lib)
    Oc, _ = oracle.chunkwise(q, k, v, 64, lib=lib)
    _close(Op, Or, 1e-11, "parallel vs recurrent")
    _close(Oc, Or, 1e-11, "chunked vs recurrent")
    n = 200
    q, k, v = (torch.randn(n, d, generator=g, dtype=torch.float64) for _ in range(3))
    w = torch.randn(d, generator=g, dtype=torch.float64)
    log_gamma = torch.nn.functional.logsigmoid(k @ w + 3.0)
    Op, Sp = oracle.parallel(q, k, v, decay_kind="token", decay=log_gamma, lib=lib)
    Or, Sr = oracle.recurrent(q, k, v, decay_kind="token", decay=log_gamma, lib=lib)
    _close(Op, Or, 1e-11, "gated parallel vs recurrent O")
    _close(Sp, Sr, 1e-11, "gated parallel vs recurrent S")


def pin_split_invariance(lib):
    """Resume: run [0, m), then [m, L) from the carried state == one run."""
    r = _rng(7)
    B, H, L, dk, dv = 2, 2, 50, 4, 5
    q, k, v = r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dv))
    g = r.normal(size=(B, H, L))
    S0 = r.normal(size=(B, H, dk, dv))
    for form in ("recurrent", "parallel", "chunk7"):
        O, S = _run(form, lib, q, k, v, phi="elu1", decay_kind="logit", decay=g, S0=S0)
        for m in (1, 17, 49):
            O1, S1 = _run(form, lib, q[:, :, :m], k[:, :, :m], v[:, :, :m], phi="elu1",
                          decay_kind="logit", decay=g[:, :, :m], S0=S0)
            O2, S2 = _run(form, lib, q[:, :, m:], k[:, :, m:], v[:, :, m:], phi="elu1",
                          decay_kind="logit", decay=g[:, :, m:], S0=S1)
            _close(np.concatenate([O1, O2], axis=2), O, 1e-11, f"split m={m}/{form} O")
            _close(S2, S, 1e-11, f"split m={m}/{form} S")


def pin_library_pieces(lib):
    """phi = elu + 1 equals torch's ELU + 1 applied beforehand with phi = id;
    gate logits equal per-token log alpha = -logaddexp(0, g) (numpy); a
    gamma of exactly 1 equals no decay; L = 0 returns S0 unchanged."""
    r = _rng(8)
    B, H, L, dk, dv = 1, 2, 31, 5, 3
    q, k, v = r.normal(size=(B, H, L, dk)) * 2, r.normal(size=(B, H, L, dk)) * 2, r.normal(size=(B, H, L, dv))
    g = r.normal(size=(B, H, L)) * 4
    S0 = r.normal(size=(B, H, dk, dv))
    for form in ("recurrent", "parallel", "chunk7"):
        O1, S1 = _run(form, lib, q, k, v, phi="elu1")
        O2, S2 = _run(form, lib, _elu1(q), _elu1(k), v, phi="identity")
        _close(O1, O2, 1e-12, f"elu1 vs torch ELU/{form}")
        _close(S1, S2, 1e-12, f"elu1 vs torch ELU S/{form}")
        O1, S1 = _run(form, lib, q, k, v, decay_kind="logit", decay=g, S0=S0)
        O2, S2 = _run(form, lib, q, k, v, decay_kind="token", decay=-np.logaddexp(0.0, g), S0=S0)
        _close(O1, O2, 1e-12, f"logit vs token/{form}")
        _close(S1, S2, 1e-12, f"logit vs token S/{form}")
        O1, S1 = _run(form, lib, q, k, v, decay_kind="head", decay=np.zeros(H), S0=S0)
        O2, S2 = _run(form, lib, q, k, v, S0=S0)
        _close(O1, O2, 0.0, f"gamma=1/{form}")
        _close(S1, S2, 0.0, f"gamma=1 S/{form}")
        O, S = _run(form, lib, q[:, :, :0], k[:, :, :0], v[:, :, :0], S0=S0)
        assert O.shape == (B, H, 0, dv)
        _close(S, S0, 0.0, f"L=0 state/{form}")


def pin_state_shape(lib):
    """The state is [d_k, d_v] whatever L is (page 1, check [c])."""
    r = _rng(9)
    for L in (1, 13, 300):
        q, k, v = r.normal(size=(L, 6)), r.normal(size=(L, 6)), r.normal(size=(L, 4))
        _, S = oracle.recurrent(q, k, v, lib=lib)
        assert S.shape == (6, 4), S.shape


def pin_noncausal(lib):
    """The non-causal form ("adv13 - Linear Attention / SSM" section 4.3):
    - its state is the causal recurrence's final state with no decay and S0 = 0;
    - its last output row is the recurrence's last row (both read that state);
    - (phi(Q) phi(K)^T) V, the n x n order of "CS336 lecture 4, code 1"
      demo_associativity, computed by numpy with torch's ELU for phi, equals it;
    - one-hot queries and keys: o_t = sum_s [q_t = k_s] v_s by hand;
    - L = 0 gives an empty output and a zero state."""
    r = _rng(12)
    B, H, L, dk, dv = 2, 2, 23, 5, 4
    q, k, v = r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dv))
    for phi in ("identity", "elu1"):
        O, S = oracle.noncausal(q, k, v, phi=phi, lib=lib)
        Oc, Sc = oracle.recurrent(q, k, v, phi=phi, lib=lib)
        _close(S, Sc, 1e-12, f"noncausal state = causal final state/{phi}")
        _close(O[:, :, -1], Oc[:, :, -1], 1e-12, f"noncausal last row = causal last row/{phi}")
        fq, fk = (q, k) if phi == "identity" else (_elu1(q), _elu1(k))
        scores = np.matmul(fq, np.swapaxes(fk, -1, -2))  # [B,H,L,L], no mask
        _close(O, np.matmul(scores, v), 1e-12, f"(QK^T)V = Q(K^TV)/{phi}")
    # one-hot: token t has q_t = e_{t mod dk}, k_s = e_{s mod dk}
    Lh, d = 7, 3
    eye = np.eye(d)
    qh = np.stack([eye[t % d] for t in range(Lh)])
    kh = np.stack([eye[(2 * s) % d] for s in range(Lh)])
    vh = np.arange(Lh * 2, dtype=np.float64).reshape(Lh, 2)
    O, S = oracle.noncausal(qh, kh, vh, lib=lib)
    want = np.stack([sum(vh[s] for s in range(Lh) if (2 * s) % d == t % d) for t in range(Lh)])
    _close(O, want, 0.0, "noncausal one-hot")
    O, S = oracle.noncausal(q[:, :, :0], k[:, :, :0], v[:, :, :0], lib=lib)
    assert O.shape == (B, H, 0, dv)
    _close(S, np.zeros((B, H, dk, dv)), 0.0, "noncausal L=0 state")


def pin_normalised(lib):
    """The normalised form ("Linear / sparse attention tutorial" Q11, section 2.2):
    - it is the ratio of two runs of the plain recurrence, one with v and one with a
      value column of ones (z0 as that column's initial state), decay and S0 included;
    - with phi = elu + 1 and the same value vector c at every token (S0 = z0 c^T), every
      output is c: a convex combination of equal vectors;
    - one token from zero state gives o = v;
    - z_final is the ones column's final state."""
    r = _rng(13)
    B, H, L, dk, dv = 2, 2, 29, 5, 3
    q, k, v = r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dv))
    g = r.normal(size=(B, H, L))
    z0 = r.uniform(0.1, 1.0, size=(B, H, dk))
    S0 = r.normal(size=(B, H, dk, dv)) * 0.1
    for phi in ("identity", "elu1"):
        O, S, z = oracle.normalised(q, k, v, phi=phi, decay_kind="logit", decay=g, S0=S0, z0=z0,
                                    lib=lib)
        num, Sn = oracle.recurrent(q, k, v, phi=phi, decay_kind="logit", decay=g, S0=S0, lib=lib)
        den, Sd = oracle.recurrent(q, k, np.ones((B, H, L, 1)), phi=phi, decay_kind="logit",
                                   decay=g, S0=z0[..., None], lib=lib)
        _close(O, num / den, 1e-9, f"normalised = num / den/{phi}")
        _close(S, Sn, 1e-12, f"normalised S/{phi}")
        _close(z, Sd[..., 0], 1e-12, f"normalised z/{phi}")
    c = r.normal(size=dv)
    vc = np.broadcast_to(c, (B, H, L, dv)).copy()
    O, _, _ = oracle.normalised(q, k, vc, phi="elu1", decay_kind="logit", decay=g,
                                S0=z0[..., None] * c, z0=z0, lib=lib)
    _close(O, vc, 1e-12, "normalised constant v")
    O, _, _ = oracle.normalised(q[:, :, :1], k[:, :, :1], v[:, :, :1], phi="elu1", lib=lib)
    _close(O, v[:, :, :1], 1e-12, "normalised one token")


def pin_channel_gate(lib):
    """The per-channel gate ("Linear / sparse attention tutorial" Q21, GLA):
    - equal gates on every channel give the scalar per-token gate of the recurrence;
    - gates of zero log give the plain additive recurrence;
    - it equals the O(L^2) form written with numpy: o_t = sum_{s<=t} sum_i phi(q)_ti
      phi(k)_si exp(cum_ti - cum_si) v_s + sum_i phi(q)_ti exp(cum_ti) S0[i,:], and
      S_L[i,:] = exp(cum_Li) S0[i,:] + sum_s exp(cum_Li - cum_si) phi(k)_si v_s."""
    r = _rng(14)
    B, H, L, dk, dv = 2, 2, 23, 5, 4
    q, k, v = r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dk)), r.normal(size=(B, H, L, dv))
    S0 = r.normal(size=(B, H, dk, dv))
    lam = -np.logaddexp(0.0, r.normal(size=(B, H, L)))
    O, S = oracle.channel_gate(q, k, v, np.repeat(lam[..., None], dk, axis=-1), S0=S0, lib=lib)
    Oc, Sc = oracle.recurrent(q, k, v, decay_kind="token", decay=lam, S0=S0, lib=lib)
    _close(O, Oc, 1e-12, "channel gate, equal channels")
    _close(S, Sc, 1e-12, "channel gate S, equal channels")
    O, S = oracle.channel_gate(q, k, v, np.zeros((B, H, L, dk)), S0=S0, lib=lib)
    Oc, Sc = oracle.recurrent(q, k, v, S0=S0, lib=lib)
    _close(O, Oc, 1e-12, "channel gate, no decay")
    la = -np.logaddexp(0.0, r.normal(size=(B, H, L, dk)) * 2)
    for phi in ("identity", "elu1"):
        O, S = oracle.channel_gate(q, k, v, la, phi=phi, S0=S0, lib=lib)
        fq, fk = (q, k) if phi == "identity" else (_elu1(q), _elu1(k))
        cum = np.cumsum(la, axis=2)                                         # [B,H,L,dk]
        w = np.exp(cum[:, :, :, None, :] - cum[:, :, None, :, :])          # [B,H,t,s,dk]
        mask = np.tril(np.ones((L, L)))[None, None, :, :, None]
        scores = np.einsum("bhti,bhtsi,bhsi->bhts", fq, w * mask, fk)
        ref = np.einsum("bhts,bhse->bhte", scores, v)
        ref += np.einsum("bhti,bhie->bhte", fq * np.exp(cum), S0)
        _close(O, ref, 1e-10, f"channel gate O(L^2) form/{phi}")
        SL = np.exp(cum[:, :, -1, :])[..., None] * S0 + np.einsum(
            "bhsi,bhse->bhie", fk * np.exp(cum[:, :, -1:, :] - cum), v)
        _close(S, SL, 1e-10, f"channel gate final state/{phi}")


def pin_delta(lib):
    """The (gated) delta rule ("Linear / Sparse Attention - minimal runnable
    implementation", delta_rule_recurrent and its checks [d], [e]):
    - orthonormal keys with beta = 1 give the additive recurrence (check [e]), and
      random unit keys do not;
    - reading with the key just written (unit norm, beta = 1) returns exactly its
      value whatever the history and alpha: k^T S_t = v_t^T (the erase-then-write);
    - beta = 0 only decays the initial state: o_t = exp(cum_t) q_t^T S0;
    - one token from zero state: o = beta (q . k) v."""
    r = _rng(15)
    B, H, d, dv = 2, 2, 6, 4
    Q, _ = np.linalg.qr(r.normal(size=(B, H, d, d)))        # columns orthonormal
    Ko = np.swapaxes(Q, -1, -2)                               # rows orthonormal: L = d keys
    v = r.normal(size=(B, H, d, dv))
    q = r.normal(size=(B, H, d, d))
    ones = np.ones((B, H, d))
    O, S = oracle.delta(q, Ko, v, ones, lib=lib)
    Oa, Sa = oracle.recurrent(q, Ko, v, lib=lib)
    _close(O, Oa, 1e-12, "delta = additive for orthonormal keys")
    _close(S, Sa, 1e-12, "delta state = additive for orthonormal keys")
    L = 17
    kr = r.normal(size=(B, H, L, d))
    kr /= np.linalg.norm(kr, axis=-1, keepdims=True)
    vr = r.normal(size=(B, H, L, dv))
    S0 = r.normal(size=(B, H, d, dv))
    la = -np.logaddexp(0.0, r.normal(size=(B, H, L)))
    _, Sd = oracle.delta(kr, kr, vr, np.ones((B, H, L)), lib=lib)
    _, Sadd = oracle.recurrent(kr, kr, vr, lib=lib)
    assert np.linalg.norm(Sd - Sadd) > 1e-3, "delta must differ from additive for random keys"
    O, _ = oracle.delta(kr, kr, vr, np.ones((B, H, L)), log_alpha=la, S0=S0, lib=lib)
    _close(O, vr, 1e-12, "delta: reading the key just written returns its value")
    qz = r.normal(size=(B, H, L, d))
    O, S = oracle.delta(qz, kr, vr, np.zeros((B, H, L)), log_alpha=la, S0=S0, lib=lib)
    cum = np.cumsum(la, axis=2)
    _close(O, np.exp(cum)[..., None] * np.einsum("bhti,bhie->bhte", qz, S0), 1e-12,
           "delta with beta = 0")
    be = r.uniform(0.1, 1.0, size=(B, H, 1))
    O, _ = oracle.delta(qz[:, :, :1], kr[:, :, :1], vr[:, :, :1], be, lib=lib)
    want = be[..., None] * np.einsum("bhti,bhti->bht", qz[:, :, :1], kr[:, :, :1])[..., None] * vr[:, :, :1]
    _close(O, want, 1e-12, "delta one token")


def pin_delta_chunkwise(lib):
    """The chunkwise (WY) form of the delta rule equals the token-by-token rule
    for every chunk size: C = 1 is the recurrence itself, C = L one chunk, and
    C in {4, 7} ragged chunks (the check [a]/[b] of "Linear / Sparse Attention -
    minimal runnable implementation", chunkwise == recurrent, carried over to
    the delta rule), with and without the gate, from S0, for both phi."""
    r = _rng(16)
    B, H, L, d, dv = 2, 2, 23, 5, 3
    k = r.normal(size=(B, H, L, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.normal(size=(B, H, L, dv))
    q = r.normal(size=(B, H, L, d))
    S0 = r.normal(size=(B, H, d, dv))
    la = -np.logaddexp(0.0, r.normal(size=(B, H, L)))
    for phi, bmax in (("identity", 1.0), ("elu1", 1.0 / d)):
        be = r.uniform(0.0, bmax, size=(B, H, L))
        for gate in (None, la):
            Or, Sr = oracle.delta(q, k, v, be, log_alpha=gate, phi=phi, S0=S0, lib=lib)
            for C in (1, 4, 7, L):
                O, S = oracle.delta_chunkwise(q, k, v, be, C, log_alpha=gate, phi=phi, S0=S0,
                                              lib=lib)
                what = f"delta chunkwise C={C}/{phi}/{'gated' if gate is not None else 'plain'}"
                _close(O, Or, 1e-11, what)
                _close(S, Sr, 1e-11, what + " state")


PINS = [pin_golden, pin_closed_form_additive, pin_closed_form_constant_decay, pin_single_token,
        pin_one_hot, pin_orthonormal_keys, pin_chunk_invariance, pin_parallel_equals_recurrent,
        pin_split_invariance, pin_library_pieces, pin_state_shape, pin_noncausal, pin_normalised,
        pin_channel_gate, pin_delta, pin_delta_chunkwise]
