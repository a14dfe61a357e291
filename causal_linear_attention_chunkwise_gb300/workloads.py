"""Seeded synthetic inputs for the prefill and decode workloads.

This module only draws random numbers and encodes the decay parameters the
workloads specify; it holds none of the attention arithmetic, and both the CUDA
path's tests and the oracle's tests take their inputs from here.

Every tensor comes from one CPU ``torch.Generator`` seeded per workload (seed 0
by default, as the pages seed their demos), in a fixed order: Q, K, V (fp32
``randn`` times ``scale``, then cast to the workload dtype), then the decay
input (gate logits g or decode alpha), then the initial state S0.  Layout is
``[B, H, L, d]`` for prefill and ``[steps, B, H, d]`` for decode.

Decay parameters are handed to the library in log space:
* per-head constant decay (RetNet): gamma_h = 1 - 2^(-5 - 3h/31) for
  h = 0..H-1, encoded as log(gamma_h) = log1p(-2^(-5 - 3h/31)) computed in
  double and rounded to fp32;
* per-token gate: the logits g ~ N(0, 1) fp32 themselves (the kernel forms
  alpha = exp(-softplus(g)));
* decode gate: alpha ~ U(0.9, 1.0) drawn in fp32, encoded as fp32(log alpha).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class PrefillWorkload:
    """One chunkwise-prefill problem.  ``decay`` is "none", "head" (constant
    per-head gamma) or "logit" (per-token gate logits g)."""
    name: str
    B: int
    H: int
    L: int
    dk: int
    dv: int
    dtype: str = "bf16"
    phi: str = "identity"
    decay: str = "none"
    chunk: int = 64
    scale: float = 1.0
    s0_std: float | None = None  # None: zero initial state

    @property
    def tokens(self) -> int:
        return self.B * self.L


@dataclass(frozen=True)
class DecodeWorkload:
    """Consecutive single-token decode steps on an fp32 state held in place."""
    name: str
    B: int
    H: int
    dk: int
    dv: int
    steps: int = 64
    dtype: str = "bf16"
    phi: str = "elu1"
    scale: float = 1.0
    alpha_range: tuple = field(default=(0.9, 1.0))
    s0_std: float = 0.1


_INV_SQRT_128 = 1.0 / math.sqrt(128.0)

# The four prefill problems (N(0, 0.01) for S0 is read as variance 0.01,
# i.e. standard deviation 0.1).
PREFILL = {
    w.name: w for w in (
        PrefillWorkload("L300_d16_f32", 1, 1, 300, 16, 16, "f32", "identity", "none", 64),
        PrefillWorkload("B4_H16_L4096_d64_elu1", 4, 16, 4096, 64, 64, "bf16", "elu1", "none", 64),
        PrefillWorkload("B2_H32_L8192_d128_retnet", 2, 32, 8192, 128, 128, "bf16", "identity",
                        "head", 64, _INV_SQRT_128),
        PrefillWorkload("B1_H16_L32768_d128_gate", 1, 16, 32768, 128, 128, "bf16", "identity",
                        "logit", 64, _INV_SQRT_128, 0.1),
    )
}

DECODE = {
    w.name: w for w in (
        DecodeWorkload("B512_H32_d128_decode", 512, 32, 128, 128, 64, "bf16", "elu1",
                       _INV_SQRT_128, (0.9, 1.0), 0.1),
    )
}


def retnet_log_gamma(H: int) -> torch.Tensor:
    """fp32 log(gamma_h), gamma_h = 1 - 2^(-5 - 3h/31), evaluated in double."""
    return torch.tensor([math.log1p(-2.0 ** (-5.0 - 3.0 * h / 31.0)) for h in range(H)],
                        dtype=torch.float32)


def make_prefill_inputs(w: PrefillWorkload, seed: int = 0) -> dict:
    """Draw one workload's inputs on the CPU.

    Returns a dict with q, k [B,H,L,dk] and v [B,H,L,dv] in the workload dtype,
    ``decay_kind`` ("none" | "head" | "logit"), ``decay`` (fp32 [H] log gamma,
    fp32 [B,H,L] logits, or None) and ``S0`` (fp32 [B,H,dk,dv] or None).
    """
    gen = torch.Generator().manual_seed(seed)
    dt = DTYPES[w.dtype]

    def draw(*shape):
        return (torch.randn(*shape, generator=gen, dtype=torch.float32) * w.scale).to(dt)

    q = draw(w.B, w.H, w.L, w.dk)
    k = draw(w.B, w.H, w.L, w.dk)
    v = draw(w.B, w.H, w.L, w.dv)
    decay = None
    if w.decay == "head":
        decay = retnet_log_gamma(w.H)
    elif w.decay == "logit":
        decay = torch.randn(w.B, w.H, w.L, generator=gen, dtype=torch.float32)
    elif w.decay != "none":
        raise ValueError(f"unknown decay {w.decay!r}")
    S0 = None
    if w.s0_std is not None:
        S0 = torch.randn(w.B, w.H, w.dk, w.dv, generator=gen, dtype=torch.float32) * w.s0_std
    return {"q": q, "k": k, "v": v, "decay_kind": w.decay, "decay": decay, "S0": S0}


def make_decode_inputs(w: DecodeWorkload, seed: int = 0, steps: int | None = None) -> dict:
    """Draw the decode workload: S0 fp32 [B,H,dk,dv], then per step q, k
    [steps,B,H,dk] and v [steps,B,H,dv] in the workload dtype and
    log_alpha fp32 [steps,B,H]."""
    steps = w.steps if steps is None else steps
    gen = torch.Generator().manual_seed(seed)
    dt = DTYPES[w.dtype]
    S0 = torch.randn(w.B, w.H, w.dk, w.dv, generator=gen, dtype=torch.float32) * w.s0_std
    q = (torch.randn(steps, w.B, w.H, w.dk, generator=gen) * w.scale).to(dt)
    k = (torch.randn(steps, w.B, w.H, w.dk, generator=gen) * w.scale).to(dt)
    v = (torch.randn(steps, w.B, w.H, w.dv, generator=gen) * w.scale).to(dt)
    lo, hi = w.alpha_range
    alpha = torch.rand(steps, w.B, w.H, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    log_alpha = torch.log(alpha.double()).float()
    return {"S0": S0, "q": q, "k": k, "v": v, "log_alpha": log_alpha, "phi": w.phi}


def small_prefill(B=1, H=2, L=200, dk=32, dv=32, dtype="bf16", phi="identity", decay="none",
                  chunk=64, scale=None, s0_std=None, name="small") -> PrefillWorkload:
    """A custom-size workload for tests (scale defaults to 1/sqrt(dk) for bf16)."""
    if scale is None:
        scale = 1.0 if dtype == "f32" else 1.0 / math.sqrt(dk)
    return PrefillWorkload(name, B, H, L, dk, dv, dtype, phi, decay, chunk, scale, s0_std)


def make_variant_inputs(form: str, B: int, H: int, L: int, dk: int, dv: int, dtype: str = "bf16",
                        seed: int = 0, with_state: bool = False, gated: bool = True,
                        beta_max: float = 1.0) -> dict:
    """Inputs of the three further forms (``form`` "normalised" |
    "channel_gate" | "delta"), drawn in this order from one generator:

    * q, k, v: ``randn`` (fp32) scaled by 1/sqrt(dk) for q and k, 1 for v, cast
      to the dtype; for "delta" each key row is rescaled to unit L2 norm
      before the cast (the rule assumes unit-norm keys);
    * "channel_gate": log_alpha fp32 [B,H,L,dk] = -U(0.005, 0.7), i.e. alpha
      per channel in (0.50, 0.995);
    * "delta": beta fp32 [B,H,L] ~ U(0, beta_max), then (``gated``)
      log_alpha fp32 [B,H,L] = -U(0.005, 0.3);
    * "normalised": gate logits g ~ N(0, 1) fp32 [B,H,L] when ``gated``;
    * with ``with_state``: S0 ~ 0.5 randn fp32 [B,H,dk,dv] and, for
      "normalised", z0 ~ U(0.5, 2.5) fp32 [B,H,dk] (a positive key sum).
    """
    gen = torch.Generator().manual_seed(seed)
    dt = DTYPES[dtype]
    s = 1.0 / math.sqrt(dk)
    q = torch.randn(B, H, L, dk, generator=gen) * s
    k = torch.randn(B, H, L, dk, generator=gen) * s
    v = torch.randn(B, H, L, dv, generator=gen)
    if form == "delta":
        k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    out = {"q": q.to(dt), "k": k.to(dt), "v": v.to(dt), "log_alpha": None, "beta": None,
           "decay_kind": "none", "decay": None, "S0": None, "z0": None}
    if form == "channel_gate":
        out["log_alpha"] = -(torch.rand(B, H, L, dk, generator=gen) * 0.695 + 0.005)
    elif form == "delta":
        out["beta"] = torch.rand(B, H, L, generator=gen) * beta_max
        if gated:
            out["log_alpha"] = -(torch.rand(B, H, L, generator=gen) * 0.295 + 0.005)
    elif form == "normalised":
        if gated:
            out["decay_kind"] = "logit"
            out["decay"] = torch.randn(B, H, L, generator=gen)
    else:
        raise ValueError(f"unknown form {form!r}")
    if with_state:
        out["S0"] = torch.randn(B, H, dk, dv, generator=gen) * 0.5
        if form == "normalised":
            out["z0"] = torch.rand(B, H, dk, generator=gen) * 2.0 + 0.5
    return out
