"""The seeded input generators (CPU only): same seed, same tensors; the
distributions and structure the design states for each workload."""
import math

import pytest
import torch

from causal_linear_attention_chunkwise_gb300 import workloads as W


def _same(a, b):
    for key in a:
        x, y = a[key], b[key]
        if isinstance(x, torch.Tensor):
            assert torch.equal(x, y), key
        else:
            assert x == y, key


@pytest.mark.parametrize("form", ["normalised", "channel_gate", "delta"])
def test_variant_inputs_are_seeded(form):
    a = W.make_variant_inputs(form, 2, 3, 70, 32, 16, "bf16", seed=5, with_state=True)
    b = W.make_variant_inputs(form, 2, 3, 70, 32, 16, "bf16", seed=5, with_state=True)
    c = W.make_variant_inputs(form, 2, 3, 70, 32, 16, "bf16", seed=6, with_state=True)
    _same(a, b)
    assert not torch.equal(a["q"], c["q"])
    assert a["q"].shape == (2, 3, 70, 32) and a["v"].shape == (2, 3, 70, 16)
    assert a["q"].dtype == torch.bfloat16 and a["S0"].dtype == torch.float32


def test_variant_input_ranges():
    B, H, L, d = 2, 2, 500, 64
    g = W.make_variant_inputs("channel_gate", B, H, L, d, d, "f32", seed=1)
    la = g["log_alpha"]
    assert la.shape == (B, H, L, d) and la.dtype == torch.float32
    assert float(la.max()) <= -0.005 + 1e-7 and float(la.min()) >= -0.7 - 1e-7
    dl = W.make_variant_inputs("delta", B, H, L, d, d, "f32", seed=1, beta_max=0.25)
    norms = dl["k"].double().norm(dim=-1)
    assert torch.allclose(norms, torch.ones_like(norms), atol=1e-6)  # unit keys
    assert float(dl["beta"].min()) >= 0 and float(dl["beta"].max()) <= 0.25
    assert float(dl["log_alpha"].max()) <= -0.005 + 1e-7
    assert float(dl["log_alpha"].min()) >= -0.3 - 1e-7
    un = W.make_variant_inputs("delta", B, H, L, d, d, "f32", seed=1, gated=False)
    assert un["log_alpha"] is None
    nm = W.make_variant_inputs("normalised", B, H, L, d, d, "f32", seed=1, with_state=True)
    assert nm["decay_kind"] == "logit" and nm["decay"].shape == (B, H, L)
    assert float(nm["z0"].min()) >= 0.5 and float(nm["z0"].max()) <= 2.5  # a positive key sum
    q = nm["q"].double()
    assert abs(float(q.std()) - 1 / math.sqrt(d)) < 0.05 / math.sqrt(d)
    with pytest.raises(ValueError):
        W.make_variant_inputs("unknown", 1, 1, 4, 16, 16)


def test_prefill_workloads_are_seeded_and_shaped():
    for name, w in W.PREFILL.items():
        if w.B * w.H * w.L > 1 << 20:
            continue  # the full-size workloads are drawn by the GPU tests
        a = W.make_prefill_inputs(w, seed=3)
        b = W.make_prefill_inputs(w, seed=3)
        _same(a, b)
        assert a["q"].shape == (w.B, w.H, w.L, w.dk) and a["v"].shape == (w.B, w.H, w.L, w.dv)


def test_retnet_gamma_closed_form():
    lg = W.retnet_log_gamma(32).double()
    for h in (0, 7, 31):
        gamma = 1 - 2.0 ** (-5 - 3 * h / 31)
        assert abs(float(lg[h]) - math.log(gamma)) < 1e-6
    assert bool((lg < 0).all()) and bool((lg[1:] > lg[:-1]).all())  # decays weaken with h
