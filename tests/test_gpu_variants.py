"""GPU parity of the three further forms of the recurrence against the fp64
oracle on the same seeded inputs: the normalised form (la_normalised_fwd,
"Linear / sparse attention tutorial" Q11 and section 2.2), the per-channel
gate (la_channel_gate_fwd, the tutorial's Q21, GLA) and the (gated) delta rule
(la_delta_fwd, "Linear / Sparse Attention - minimal runnable implementation",
delta_rule_recurrent).  Needs a GB300."""
import numpy as np
import pytest
import torch

import oracle
from causal_linear_attention_chunkwise_gb300 import api
from causal_linear_attention_chunkwise_gb300 import workloads as W
from tests import parity
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

# (B, H, L, dk, dv, dtype, chunk, phi, gated, with_state): one token, one chunk,
# several chunks with a ragged tail, d_k != d_v, an odd chunk size.
CASES = [
    (1, 1, 1, 16, 16, "f32", 64, "elu1", False, False),
    (2, 2, 200, 32, 32, "f32", 64, "elu1", True, True),
    (1, 2, 130, 64, 64, "bf16", 64, "elu1", True, False),
    (2, 2, 300, 128, 128, "bf16", 64, "elu1", True, True),
    (1, 2, 150, 64, 128, "f32", 7, "identity", True, True),
    (1, 1, 100, 128, 16, "bf16", 33, "identity", False, False),
]
IDS = [f"{c[0]}x{c[1]}x{c[2]}_dk{c[3]}_dv{c[4]}_{c[5]}_C{c[6]}_{c[7]}_{'g' if c[8] else 'ng'}"
       f"{'_S0' if c[9] else ''}" for c in CASES]


def _d(x):
    return to_dev(x)


# The quotient needs a positive feature map: the normalised form runs under elu + 1 only.
NORM_CASES = [c[:7] + ("elu1",) + c[8:] for c in CASES]
NORM_IDS = [i.replace("identity", "elu1") for i in IDS]


@pytest.mark.parametrize("case", NORM_CASES, ids=NORM_IDS)
def test_normalised_matches_oracle(case):
    B, H, L, dk, dv, dtype, chunk, phi, gated, with_state = case
    inp = W.make_variant_inputs("normalised", B, H, L, dk, dv, dtype, seed=1,
                                with_state=with_state, gated=gated)
    api.la_set_feature_map(phi)
    O, S, z = api.la_normalised_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), chunk,
                                    inp["decay_kind"], _d(inp["decay"]), _d(inp["S0"]),
                                    _d(inp["z0"]))
    api.la_device_status()
    O_ref, S_ref, z_ref = oracle.normalised(inp["q"], inp["k"], inp["v"], phi=phi,
                                            decay_kind=inp["decay_kind"], decay=inp["decay"],
                                            S0=inp["S0"], z0=inp["z0"])
    parity.check(O.cpu(), O_ref, dtype, "O")
    parity.check(S.cpu(), S_ref, dtype, "S")
    parity.check(z.cpu()[..., None], z_ref[..., None], dtype, "z")


def _normalised_check(inp, phi, dtype, tag=""):
    api.la_set_feature_map(phi)
    O, S, z = api.la_normalised_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), 64,
                                    inp["decay_kind"], _d(inp["decay"]), _d(inp["S0"]),
                                    _d(inp["z0"]))
    api.la_device_status()
    O_ref, S_ref, z_ref = oracle.normalised(inp["q"], inp["k"], inp["v"], phi=phi,
                                            decay_kind=inp["decay_kind"], decay=inp["decay"],
                                            S0=inp["S0"], z0=inp["z0"])
    parity.check(O.cpu(), O_ref, dtype, f"O{tag}")
    parity.check(S.cpu(), S_ref, dtype, f"S{tag}")
    parity.check(z.cpu()[..., None], z_ref[..., None], dtype, f"z{tag}")


@pytest.mark.parametrize("decay", ["none", "head", "logit"])
@pytest.mark.parametrize("with_state", [False, True])
@pytest.mark.parametrize("L", [1, 64, 65, 1000, 5000])
def test_normalised_one_pass_path(decay, with_state, L):
    """bf16, d_k = d_v = 64, chunk 64: z rides with the numerator through the
    tensor-core prefill kernels as a 65th value column.  One token, one chunk,
    a ragged tail, and sequences long enough to be split into segments whose z
    partials go through the scan; no decay, a per-head decay and gate logits
    (whose chunks often pass the split form's range); with and without S0, z0."""
    inp = W.make_variant_inputs("normalised", 2, 3, L, 64, 64, "bf16", seed=40 + L,
                                with_state=with_state, gated=decay == "logit")
    if decay == "head":
        inp["decay_kind"] = "head"
        inp["decay"] = torch.log(1 - 2.0 ** (-5 - torch.arange(3, dtype=torch.float32)))
    _normalised_check(inp, "elu1", "bf16")


def test_normalised_full_workload_shape_on_sampled_sequences():
    """The benchmarked shape (B4 H16 L4096 d64, bf16, elu + 1, gate logits, S0
    and z0) in one call, three sequences recomputed by the oracle."""
    B, H, L, d = 4, 16, 4096, 64
    inp = W.make_variant_inputs("normalised", B, H, L, d, d, "bf16", seed=0, with_state=True)
    api.la_set_feature_map("elu1")
    O, S, z = api.la_normalised_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), 64,
                                    inp["decay_kind"], _d(inp["decay"]), _d(inp["S0"]),
                                    _d(inp["z0"]))
    api.la_device_status()
    for b, h in [(0, 0), (1, 7), (3, 15)]:
        sl = lambda x: x[b:b + 1, h:h + 1]  # noqa: E731
        O_ref, S_ref, z_ref = oracle.normalised(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]),
                                                phi="elu1", decay_kind="logit",
                                                decay=sl(inp["decay"]), S0=sl(inp["S0"]),
                                                z0=sl(inp["z0"]))
        parity.check(sl(O).cpu(), O_ref, "bf16", f"O[{b},{h}]")
        parity.check(sl(S).cpu(), S_ref, "bf16", f"S[{b},{h}]")
        parity.check(sl(z).cpu()[..., None], z_ref[..., None], "bf16", f"z[{b},{h}]")


def test_normalised_one_pass_outputs_may_alias_the_initial_states():
    """S_final and z_final may be the S0 and z0 buffers (one-pass path, split
    into segments so the scan reads S0 and z0 while the outputs are written)."""
    inp = W.make_variant_inputs("normalised", 2, 2, 3000, 64, 64, "bf16", seed=47, with_state=True)
    api.la_set_feature_map("elu1")
    S, z = _d(inp["S0"]).clone(), _d(inp["z0"]).clone()
    O, S_out, z_out = api.la_normalised_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), 64, "logit",
                                            _d(inp["decay"]), S, z, S_final=S, z_final=z)
    api.la_device_status()
    assert S_out.data_ptr() == S.data_ptr() and z_out.data_ptr() == z.data_ptr()
    O_ref, S_ref, z_ref = oracle.normalised(inp["q"], inp["k"], inp["v"], phi="elu1",
                                            decay_kind="logit", decay=inp["decay"], S0=inp["S0"],
                                            z0=inp["z0"])
    parity.check(O.cpu(), O_ref, "bf16", "O")
    parity.check(S.cpu(), S_ref, "bf16", "S")
    parity.check(z.cpu()[..., None], z_ref[..., None], "bf16", "z")


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_channel_gate_matches_oracle(case):
    B, H, L, dk, dv, dtype, chunk, phi, _, with_state = case
    inp = W.make_variant_inputs("channel_gate", B, H, L, dk, dv, dtype, seed=2,
                                with_state=with_state)
    api.la_set_feature_map(phi)
    O, S = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]),
                                   _d(inp["log_alpha"]), chunk, _d(inp["S0"]))
    api.la_device_status()
    O_ref, S_ref = oracle.channel_gate(inp["q"], inp["k"], inp["v"], inp["log_alpha"], phi=phi,
                                       S0=inp["S0"])
    parity.check(O.cpu(), O_ref, dtype, "O")
    parity.check(S.cpu(), S_ref, dtype, "S")


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_delta_matches_oracle(case):
    B, H, L, dk, dv, dtype, _, phi, gated, with_state = case
    # unit-norm keys; under elu + 1 the keys grow to norm ~ sqrt(dk), so the
    # write strength shrinks to keep I - beta k k^T a contraction
    beta_max = 1.0 if phi == "identity" else 1.0 / dk
    inp = W.make_variant_inputs("delta", B, H, L, dk, dv, dtype, seed=3, with_state=with_state,
                                gated=gated, beta_max=beta_max)
    api.la_set_feature_map(phi)
    O, S = api.la_delta_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(inp["beta"]),
                            _d(inp["log_alpha"]), _d(inp["S0"]))
    api.la_device_status()
    O_ref, S_ref = oracle.delta(inp["q"], inp["k"], inp["v"], inp["beta"], inp["log_alpha"],
                                phi=phi, S0=inp["S0"])
    parity.check(O.cpu(), O_ref, dtype, "O")
    parity.check(S.cpu(), S_ref, dtype, "S")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("phi", ["identity", "elu1"])
@pytest.mark.parametrize("gated", [True, False])
@pytest.mark.parametrize("L", [65, 300, 1000])
def test_delta_tensor_core_path(d, phi, gated, L):
    """bf16, d_k = d_v in {64, 128}: with identity phi, the chunkwise (WY)
    tcgen05 kernel; with elu + 1 (long keys, beta shrunk to keep the erase a
    contraction) the fp32 CUDA-core kernel.  One chunk and a token, ragged
    tails and a longer run, from a non-zero S0, with and without the gate."""
    beta_max = 1.0 if phi == "identity" else 1.0 / d
    inp = W.make_variant_inputs("delta", 2, 2, L, d, d, "bf16", seed=30 + L, with_state=True,
                                gated=gated, beta_max=beta_max)
    api.la_set_feature_map(phi)
    O, S = api.la_delta_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(inp["beta"]),
                            _d(inp["log_alpha"]), _d(inp["S0"]))
    api.la_device_status()
    O_ref, S_ref = oracle.delta(inp["q"], inp["k"], inp["v"], inp["beta"], inp["log_alpha"],
                                phi=phi, S0=inp["S0"])
    parity.check(O.cpu(), O_ref, "bf16", "O")
    parity.check(S.cpu(), S_ref, "bf16", "S")


@pytest.mark.parametrize("d", [64, 128])
def test_delta_tensor_core_recalls_the_key_just_written(d):
    """beta = 1, unit keys, no gate, on the tensor-core path: every read with
    the key just written returns its value (up to bf16), however much of the
    chunk's solve cancels."""
    B, H, L = 2, 2, 200
    inp = W.make_variant_inputs("delta", B, H, L, d, d, "bf16", seed=41, with_state=True,
                                gated=False)
    beta = torch.ones(B, H, L)
    api.la_set_feature_map("identity")
    O, _ = api.la_delta_fwd(_d(inp["k"]), _d(inp["k"]), _d(inp["v"]), _d(beta), None,
                            _d(inp["S0"]))
    api.la_device_status()
    parity.check(O.cpu(), inp["v"].double(), "bf16", "recall")


def test_delta_full_workload_shape_on_sampled_sequences():
    """The benchmarked shape (B4 H16 L4096 d64, bf16, identity, gated, S0,
    beta ~ U(0, 1)) in one call; three sequences recomputed by the oracle."""
    B, H, L, d = 4, 16, 4096, 64
    inp = W.make_variant_inputs("delta", B, H, L, d, d, "bf16", seed=0, with_state=True)
    api.la_set_feature_map("identity")
    O, S = api.la_delta_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(inp["beta"]),
                            _d(inp["log_alpha"]), _d(inp["S0"]))
    api.la_device_status()
    for b, h in [(0, 0), (2, 9), (3, 15)]:
        sl = lambda x: x[b:b + 1, h:h + 1]  # noqa: E731
        O_ref, S_ref = oracle.delta(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["beta"]),
                                    sl(inp["log_alpha"]), phi="identity", S0=sl(inp["S0"]))
        parity.check(sl(O).cpu(), O_ref, "bf16", f"O[{b},{h}]")
        parity.check(sl(S).cpu(), S_ref, "bf16", f"S[{b},{h}]")


@pytest.mark.parametrize("L,d,dtype", [(2, 16, "f32"), (31, 128, "bf16"), (32, 64, "f32"),
                                       (33, 32, "f32"), (64, 128, "f32"), (65, 64, "bf16")])
def test_delta_short_sequences(L, d, dtype):
    """Short sequences with gate and initial state around the kernel's staging
    of 32 tokens at a time: inside one pass, exactly one, one and a token, two,
    two and a token."""
    inp = W.make_variant_inputs("delta", 2, 3, L, d, d, dtype, seed=12, with_state=True)
    api.la_set_feature_map("identity")
    O, S = api.la_delta_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(inp["beta"]),
                            _d(inp["log_alpha"]), _d(inp["S0"]))
    api.la_device_status()
    O_ref, S_ref = oracle.delta(inp["q"], inp["k"], inp["v"], inp["beta"], inp["log_alpha"],
                                phi="identity", S0=inp["S0"])
    parity.check(O.cpu(), O_ref, dtype, "O")
    parity.check(S.cpu(), S_ref, dtype, "S")


def test_delta_recalls_the_key_just_written():
    """beta = 1 with unit keys and no gate: reading with the key just written
    returns its value exactly (the write replaces the old association)."""
    B, H, L, d = 2, 3, 64, 64
    inp = W.make_variant_inputs("delta", B, H, L, d, d, "f32", seed=4, with_state=True,
                                gated=False)
    beta = torch.ones(B, H, L)
    api.la_set_feature_map("identity")
    O, _ = api.la_delta_fwd(_d(inp["k"]), _d(inp["k"]), _d(inp["v"]), _d(beta), None,
                            _d(inp["S0"]))
    api.la_device_status()
    parity.check(O.cpu(), inp["v"], "f32", "recall")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_steps_equal_one_call(dtype):
    """L calls with one token each, every call writing its states over its input
    states (the decode step of each form), give the oracle's outputs over the L
    tokens."""
    B, H, L, d = 3, 2, 6, 64
    api.la_set_feature_map("elu1")
    # normalised
    inp = W.make_variant_inputs("normalised", B, H, L, d, d, dtype, seed=5, with_state=True)
    q, k, v, g = _d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(inp["decay"])
    S, z = _d(inp["S0"]).clone(), _d(inp["z0"]).clone()
    outs = []
    for t in range(L):
        sl = lambda x: x[:, :, t:t + 1].contiguous()  # noqa: E731
        o, _, _ = api.la_normalised_fwd(sl(q), sl(k), sl(v), 64, "logit", sl(g), S, z,
                                        S_final=S, z_final=z)
        outs.append(o)
    O_ref, S_ref, z_ref = oracle.normalised(inp["q"], inp["k"], inp["v"], phi="elu1",
                                            decay_kind="logit", decay=inp["decay"],
                                            S0=inp["S0"], z0=inp["z0"])
    api.la_device_status()
    parity.check(torch.cat(outs, 2).cpu(), O_ref, dtype, "normalised steps")
    parity.check(S.cpu(), S_ref, dtype, "normalised S")
    parity.check(z.cpu()[..., None], z_ref[..., None], dtype, "normalised z")
    # channel gate
    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, dtype, seed=6, with_state=True)
    q, k, v, la = _d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(inp["log_alpha"])
    S = _d(inp["S0"]).clone()
    outs = []
    for t in range(L):
        sl = lambda x: x[:, :, t:t + 1].contiguous()  # noqa: E731
        o, _ = api.la_channel_gate_fwd(sl(q), sl(k), sl(v), sl(la), 64, S, S_final=S)
        outs.append(o)
    O_ref, S_ref = oracle.channel_gate(inp["q"], inp["k"], inp["v"], inp["log_alpha"],
                                       phi="elu1", S0=inp["S0"])
    api.la_device_status()
    parity.check(torch.cat(outs, 2).cpu(), O_ref, dtype, "channel gate steps")
    parity.check(S.cpu(), S_ref, dtype, "channel gate S")
    # delta rule
    inp = W.make_variant_inputs("delta", B, H, L, d, d, dtype, seed=7, with_state=True,
                                beta_max=1.0 / d)
    q, k, v = _d(inp["q"]), _d(inp["k"]), _d(inp["v"])
    be, la = _d(inp["beta"]), _d(inp["log_alpha"])
    S = _d(inp["S0"]).clone()
    outs = []
    for t in range(L):
        sl = lambda x: x[:, :, t:t + 1].contiguous()  # noqa: E731
        o, _ = api.la_delta_fwd(sl(q), sl(k), sl(v), sl(be), sl(la), S, S_final=S)
        outs.append(o)
    O_ref, S_ref = oracle.delta(inp["q"], inp["k"], inp["v"], inp["beta"], inp["log_alpha"],
                                phi="elu1", S0=inp["S0"])
    api.la_device_status()
    parity.check(torch.cat(outs, 2).cpu(), O_ref, dtype, "delta steps")
    parity.check(S.cpu(), S_ref, dtype, "delta S")


def test_channel_gate_with_equal_channels_is_the_token_gate():
    """Equal per-channel decays reduce the channel gate to la_chunk_fwd with
    a per-token decay: two different kernels, one answer."""
    B, H, L, d = 2, 2, 333, 64
    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, "f32", seed=8, with_state=True)
    la_tok = inp["log_alpha"][..., 0].contiguous()
    la_ch = la_tok[..., None].expand(B, H, L, d).contiguous()
    api.la_set_feature_map("elu1")
    O1, S1 = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(la_ch), 64,
                                     _d(inp["S0"]))
    O2, S2 = api.la_chunk_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), 64, "token",
                              _d(la_tok), _d(inp["S0"]))
    api.la_device_status()
    parity.check(O1.cpu(), O2.cpu(), "f32", "O")
    parity.check(S1.cpu(), S2.cpu(), "f32", "S")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("phi", ["identity", "elu1"])
@pytest.mark.parametrize("L", [64, 65, 200, 1000])
def test_channel_gate_tensor_core_path(d, phi, L):
    """bf16, chunk 64, d_k = d_v in {64, 128}: the tcgen05 kernel.  One chunk,
    one chunk and a token, ragged tails and a longer run, from a non-zero S0;
    identity phi leaves q . k free to cancel, elu + 1 keeps it positive."""
    B, H = 2, 2
    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, "bf16", seed=21 + L,
                                with_state=True)
    api.la_set_feature_map(phi)
    O, S = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]),
                                   _d(inp["log_alpha"]), 64, _d(inp["S0"]))
    api.la_device_status()
    O_ref, S_ref = oracle.channel_gate(inp["q"], inp["k"], inp["v"], inp["log_alpha"], phi=phi,
                                       S0=inp["S0"])
    parity.check(O.cpu(), O_ref, "bf16", "O")
    parity.check(S.cpu(), S_ref, "bf16", "S")


def test_channel_gate_full_workload_shape_on_sampled_sequences():
    """The benchmarked shape (B4 H16 L4096 d64, bf16, elu + 1, S0) in one call,
    three sequences recomputed by the oracle."""
    B, H, L, d = 4, 16, 4096, 64
    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, "bf16", seed=0, with_state=True)
    api.la_set_feature_map("elu1")
    O, S = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]),
                                   _d(inp["log_alpha"]), 64, _d(inp["S0"]))
    api.la_device_status()
    for b, h in [(0, 0), (1, 7), (3, 15)]:
        sl = lambda x: x[b:b + 1, h:h + 1]  # noqa: E731
        O_ref, S_ref = oracle.channel_gate(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]),
                                           sl(inp["log_alpha"]), phi="elu1", S0=sl(inp["S0"]))
        parity.check(sl(O).cpu(), O_ref, "bf16", f"O[{b},{h}]")
        parity.check(sl(S).cpu(), S_ref, "bf16", f"S[{b},{h}]")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("phi,strong", [("identity", False), ("elu1", False), ("elu1", True),
                                        ("identity", True)])
def test_channel_gate_segments(d, phi, strong):
    """A sequence long enough to be cut into several segments (B1 H2 L3000: 47
    chunks, five segments): per-segment state passes with per-channel weights,
    the scan with a per-row decay, and the segments' outputs from their
    incoming states, from a non-zero S0.  With ``strong``, one chunk per
    segment decays ten times harder, so segment totals underflow in places.
    Every case must match the same call run in one piece.  Identity phi with
    strong decay leaves some output rows at ~1% of the typical row norm (a
    token's own score q.k nearly cancelling where everything before it has
    decayed away); the bf16 rounding of the rescaled operands then shows as up
    to ~0.4 relative error in those rows, identically in one piece, so there
    the oracle checks the final state and the outputs are held to the one-piece
    run.  Identity phi without strong decay has such rows too (one at 0.17 of
    the median row norm here, 2.7e-2 off): its outputs are held to the oracle
    with each row's norm floored at half the RMS row norm, the scale of the
    terms whose rounding the row carries."""
    B, H, L = 1, 2, 3000
    assert api.la_channel_gate_fwd_workspace_bytes(B, H, L, d, d) > 0
    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, "bf16", seed=50 + d, with_state=True)
    la = inp["log_alpha"].clone()
    if strong:
        for c in range(3, 47, 10):
            la[:, :, 64 * c:64 * c + 64] *= 10.0
    api.la_set_feature_map(phi)
    O, S = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(la), 64,
                                   _d(inp["S0"]))
    api.la_device_status()
    O1, S1 = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(la), 64,
                                     _d(inp["S0"]), segments=False)
    api.la_device_status()
    parity.check(O.cpu(), O1.cpu(), "bf16", "O segmented vs one piece")
    parity.check(S.cpu(), S1.cpu(), "bf16", "S segmented vs one piece")
    O_ref, S_ref = oracle.channel_gate(inp["q"], inp["k"], inp["v"], la, phi=phi, S0=inp["S0"])
    parity.check(S.cpu(), S_ref, "bf16", "S")
    if not (strong and phi == "identity"):
        parity.check(O.cpu(), O_ref, "bf16", "O", row_floor=0.5 if phi == "identity" else 1e-6)


@pytest.mark.parametrize("d", [64, 128])
def test_channel_gate_segments_final_state_may_alias_initial_state(d):
    """S_final given as the S0 buffer while the sequence runs as five segments:
    the first segment and the scan read S0 before the last segment writes it."""
    B, H, L = 1, 2, 3000
    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, "bf16", seed=60 + d, with_state=True)
    api.la_set_feature_map("elu1")
    S = _d(inp["S0"]).clone()
    O, S_out = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]),
                                       _d(inp["log_alpha"]), 64, S, S_final=S)
    api.la_device_status()
    assert S_out.data_ptr() == S.data_ptr()
    O_ref, S_ref = oracle.channel_gate(inp["q"], inp["k"], inp["v"], inp["log_alpha"], phi="elu1",
                                       S0=inp["S0"])
    parity.check(O.cpu(), O_ref, "bf16", "O")
    parity.check(S.cpu(), S_ref, "bf16", "S")


@pytest.mark.parametrize("d", [64, 128])
def test_channel_gate_chunk_forms_alternate(d):
    """The tensor-core kernel picks a form per chunk: one reference point per
    key channel when every part of the chunk (8 or 16 tokens) falls by at
    most its share of 80 and none rises, 16-token blocks otherwise.  Here
    chunk 1 falls evenly by 69 (one reference, factors up to e^35), chunk 2
    by ~140 (blocks), chunk 3 has log decays above zero in a few channels
    (blocks), chunks 0 and 4 are plain; each hands its state to the next."""
    B, H, L = 1, 2, 320
    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, "bf16", seed=70 + d, with_state=True)
    la = inp["log_alpha"].clone()
    la[:, :, 64:128] = -1.1
    la[:, :, 128:192] *= 5.0
    la[:, :, 200:204, : d // 8] = 0.05
    assert float((-la[:, :, 65:128].sum(2)).max()) < 80 < float((-la[:, :, 129:192].sum(2)).max())
    api.la_set_feature_map("elu1")
    O, S = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(la), 64,
                                   _d(inp["S0"]))
    api.la_device_status()
    O_ref, S_ref = oracle.channel_gate(inp["q"], inp["k"], inp["v"], la, phi="elu1",
                                       S0=inp["S0"])
    parity.check(O.cpu(), O_ref, "bf16", "O")
    parity.check(S.cpu(), S_ref, "bf16", "S")


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 64), ("bf16", 128), ("f32", 16)])
def test_channel_gate_strong_decay_chunks(dtype, d):
    """Chunks whose cumulative log decay leaves [-80, 80] take the exact
    per-element form, the others the split form: the second and fourth chunks
    here decay ten times harder (down to e^-448 over a chunk), so the two forms
    alternate and hand the state to each other.  On the tensor-core path (bf16)
    those chunks have 16-token blocks whose decay span passes 80, whose
    diagonal scores are then recomputed exactly."""
    B, H, L = 2, 2, 300
    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, dtype, seed=13, with_state=True)
    la = inp["log_alpha"].clone()
    la[:, :, 64:128] *= 10.0
    la[:, :, 192:256] *= 10.0
    api.la_set_feature_map("elu1")
    O, S = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(la), 64,
                                   _d(inp["S0"]))
    api.la_device_status()
    O_ref, S_ref = oracle.channel_gate(inp["q"], inp["k"], inp["v"], la, phi="elu1",
                                       S0=inp["S0"])
    parity.check(O.cpu(), O_ref, dtype, "O")
    parity.check(S.cpu(), S_ref, dtype, "S")


def test_empty_sequences_pass_the_state_through_and_bad_shapes_are_refused():
    B, H, d = 2, 2, 32
    x = torch.zeros(B, H, 0, d, device="cuda")
    S0 = torch.randn(B, H, d, d, device="cuda")
    z0 = torch.rand(B, H, d, device="cuda")
    _, S, z = api.la_normalised_fwd(x, x, x, 64, "none", None, S0, z0)
    _, S2 = api.la_channel_gate_fwd(x, x, x, torch.zeros(B, H, 0, d, device="cuda"), 64, None)
    _, S3 = api.la_delta_fwd(x, x, x, torch.zeros(B, H, 0, device="cuda"), None, S0)
    api.la_device_status()
    assert torch.equal(S, S0) and torch.equal(z, z0) and torch.equal(S3, S0)
    assert torch.count_nonzero(S2) == 0
    y = torch.zeros(1, 1, 8, 48, device="cuda")
    for call in (lambda: api.la_normalised_fwd(y, y, y),
                 lambda: api.la_channel_gate_fwd(y, y, y, torch.zeros(1, 1, 8, 48, device="cuda")),
                 lambda: api.la_delta_fwd(y, y, y, torch.zeros(1, 1, 8, device="cuda"))):
        with pytest.raises(api.LAError) as e:
            call()
        assert e.value.status == api.LA_ERR_UNSUPPORTED


def test_larger_shapes_on_sampled_sequences():
    """A longer run of each form at d = 128 (B2 H4 L2048, bf16), checked on
    two sequences the oracle recomputes alone."""
    B, H, L, d = 2, 4, 2048, 128
    api.la_set_feature_map("elu1")
    pairs = [(0, 0), (1, 3)]

    def sl(x, b, h):
        return None if x is None else x[b:b + 1, h:h + 1]

    inp = W.make_variant_inputs("normalised", B, H, L, d, d, "bf16", seed=9, with_state=True)
    O, S, z = api.la_normalised_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), 64, "logit",
                                    _d(inp["decay"]), _d(inp["S0"]), _d(inp["z0"]))
    api.la_device_status()
    for b, h in pairs:
        O_ref, S_ref, _ = oracle.normalised(sl(inp["q"], b, h), sl(inp["k"], b, h),
                                            sl(inp["v"], b, h), phi="elu1", decay_kind="logit",
                                            decay=sl(inp["decay"], b, h), S0=sl(inp["S0"], b, h),
                                            z0=sl(inp["z0"], b, h))
        parity.check(sl(O, b, h).cpu(), O_ref, "bf16", f"normalised O[{b},{h}]")
        parity.check(sl(S, b, h).cpu(), S_ref, "bf16", f"normalised S[{b},{h}]")

    inp = W.make_variant_inputs("channel_gate", B, H, L, d, d, "bf16", seed=10, with_state=True)
    O, S = api.la_channel_gate_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]),
                                   _d(inp["log_alpha"]), 64, _d(inp["S0"]))
    api.la_device_status()
    for b, h in pairs:
        O_ref, S_ref = oracle.channel_gate(sl(inp["q"], b, h), sl(inp["k"], b, h),
                                           sl(inp["v"], b, h), sl(inp["log_alpha"], b, h),
                                           phi="elu1", S0=sl(inp["S0"], b, h))
        parity.check(sl(O, b, h).cpu(), O_ref, "bf16", f"channel gate O[{b},{h}]")
        parity.check(sl(S, b, h).cpu(), S_ref, "bf16", f"channel gate S[{b},{h}]")

    inp = W.make_variant_inputs("delta", B, H, L, d, d, "bf16", seed=11, with_state=True,
                                beta_max=1.0 / d)
    O, S = api.la_delta_fwd(_d(inp["q"]), _d(inp["k"]), _d(inp["v"]), _d(inp["beta"]),
                            _d(inp["log_alpha"]), _d(inp["S0"]))
    api.la_device_status()
    for b, h in pairs:
        O_ref, S_ref = oracle.delta(sl(inp["q"], b, h), sl(inp["k"], b, h), sl(inp["v"], b, h),
                                    sl(inp["beta"], b, h), sl(inp["log_alpha"], b, h),
                                    phi="elu1", S0=sl(inp["S0"], b, h))
        parity.check(sl(O, b, h).cpu(), O_ref, "bf16", f"delta O[{b},{h}]")
        parity.check(sl(S, b, h).cpu(), S_ref, "bf16", f"delta S[{b},{h}]")
    assert np.isfinite(S.cpu().numpy()).all()
