"""GPU parity of la_decode_step against the oracle, and decode == prefill over
the same tokens.  Needs a GB300."""
import numpy as np
import pytest
import torch

import oracle
from causal_linear_attention_chunkwise_gb300 import api
from causal_linear_attention_chunkwise_gb300 import workloads as W
from tests import parity
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


def run_decode(inp, steps, phi):
    api.la_set_feature_map(phi)
    S = to_dev(inp["S0"]).clone()
    q, k, v = to_dev(inp["q"]), to_dev(inp["k"]), to_dev(inp["v"])
    la = None if inp["log_alpha"] is None else to_dev(inp["log_alpha"])
    outs = []
    for t in range(steps):
        outs.append(api.la_decode_step(q[t], k[t], v[t], S, None if la is None else la[t]))
    api.la_device_status()
    return torch.stack(outs).cpu(), S.cpu()


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("phi,gated", [("elu1", True), ("identity", False)])
def test_small_decode_matches_oracle(d, dtype, phi, gated):
    w = W.DecodeWorkload("small", 3, 2, d, d, 6, dtype, phi, 1.0 / np.sqrt(d))
    inp = W.make_decode_inputs(w, seed=1)
    if not gated:
        inp["log_alpha"] = None
    o, S = run_decode(inp, w.steps, phi)
    o_ref, S_ref = oracle.decode(inp["q"], inp["k"], inp["v"], inp["S0"], inp["log_alpha"], phi=phi)
    parity.check(o, o_ref, dtype, "o")
    parity.check(S, S_ref, dtype, "S")


def test_full_decode_workload_on_sampled_states():
    """B=512, H=32, d=128, 64 consecutive steps on the 1 GiB fp32 state, as
    the benchmark runs it; the oracle recomputes a sample of (b, h) states
    through all 64 steps."""
    w = W.DECODE["B512_H32_d128_decode"]
    inp = W.make_decode_inputs(w)
    o, S = run_decode(inp, w.steps, w.phi)
    pairs = [(0, 0), (511, 31), (137, 5), (256, 16), (400, 30)]
    sel = lambda x, b, h: x[:, b, h]  # noqa: E731
    for b, h in pairs:
        o_ref, S_ref = oracle.decode(sel(inp["q"], b, h)[:, None, None], sel(inp["k"], b, h)[:, None, None],
                                     sel(inp["v"], b, h)[:, None, None], inp["S0"][b:b + 1, h:h + 1],
                                     sel(inp["log_alpha"], b, h)[:, None, None], phi=w.phi)
        parity.check(o[:, b, h], o_ref[:, 0, 0], "bf16", f"o ({b},{h})")
        parity.check(S[b, h], S_ref[0, 0], "bf16", f"S ({b},{h})")
    assert torch.isfinite(S).all()


def test_decode_equals_prefill_over_same_tokens():
    """64 decode steps from S0 == la_chunk_fwd over the same 64 tokens with a
    per-token gate and the same S0 (both checked against the oracle)."""
    steps, B, H, d = 64, 2, 4, 128
    w = W.DecodeWorkload("x", B, H, d, d, steps, "bf16", "identity", 1.0 / np.sqrt(d))
    inp = W.make_decode_inputs(w, seed=3)
    o_dec, S_dec = run_decode(inp, steps, "identity")
    api.la_set_feature_map("identity")
    q, k, v = (to_dev(inp[x].permute(1, 2, 0, 3).contiguous()) for x in ("q", "k", "v"))
    la = to_dev(inp["log_alpha"].permute(1, 2, 0).contiguous())
    O_pre, S_pre = api.la_chunk_fwd(q, k, v, 64, "token", la, to_dev(inp["S0"]))
    api.la_device_status()
    O_pre = O_pre.cpu().permute(2, 0, 1, 3)
    o_ref, S_ref = oracle.decode(inp["q"], inp["k"], inp["v"], inp["S0"], inp["log_alpha"],
                                 phi="identity")
    parity.check(o_dec, o_ref, "bf16", "decode o")
    parity.check(O_pre, o_ref, "bf16", "prefill O")
    parity.check(S_dec, S_ref, "bf16", "decode S")
    parity.check(S_pre.cpu(), S_ref, "bf16", "prefill S")
    parity.check(o_dec, O_pre, "bf16", "decode vs prefill")


def test_decode_rejects_non_fp32_state():
    q = torch.zeros(1, 1, 64, dtype=torch.bfloat16, device="cuda")
    S = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        api.la_decode_step(q, q, q, S)
