"""GPU parity of la_chunk_fwd against the fp64 oracle (element by element on
the same seeded inputs), plus its edge cases.  Needs a GB300."""
import numpy as np
import pytest
import torch

import oracle
from causal_linear_attention_chunkwise_gb300 import api
from causal_linear_attention_chunkwise_gb300 import workloads as W
from tests import parity
from tests.gpu_helpers import gpu_prefill, oracle_prefill, select_pairs, to_dev

pytestmark = pytest.mark.gpu

# Small cases: several chunks and a ragged tail, every phi / decay / dtype /
# head size, chosen so the oracle finishes in well under a second each.
SMALL = [
    # (B, H, L, dk, dv, dtype, phi, decay, chunk, s0)
    (1, 1, 300, 16, 16, "f32", "identity", "none", 64, None),
    (2, 3, 200, 32, 32, "f32", "elu1", "head", 64, 0.1),
    (1, 2, 130, 64, 64, "f32", "identity", "logit", 64, 0.1),
    (1, 2, 77, 128, 128, "f32", "elu1", "token", 64, None),
    (1, 1, 45, 16, 32, "f32", "identity", "none", 7, 0.5),
    (2, 2, 257, 64, 64, "bf16", "elu1", "none", 64, None),
    (1, 3, 321, 64, 64, "bf16", "identity", "head", 64, 0.1),
    (1, 2, 200, 64, 64, "bf16", "identity", "logit", 64, 0.1),
    (2, 2, 257, 128, 128, "bf16", "identity", "none", 64, None),
    (1, 2, 321, 128, 128, "bf16", "elu1", "head", 64, None),
    (1, 2, 190, 128, 128, "bf16", "identity", "logit", 64, 0.1),
    (1, 2, 129, 128, 128, "bf16", "identity", "token", 64, 0.1),
    (1, 1, 64, 128, 128, "bf16", "identity", "none", 64, None),
    (1, 1, 1, 64, 64, "bf16", "elu1", "logit", 64, 0.1),
    (1, 2, 63, 32, 16, "bf16", "identity", "head", 64, None),
    (3, 1, 100, 16, 16, "bf16", "elu1", "none", 4, None),
]


def _make(B, H, L, dk, dv, dtype, phi, decay, chunk, s0, seed=0):
    w = W.small_prefill(B, H, L, dk, dv, dtype, phi, "logit" if decay == "token" else decay,
                        chunk, s0_std=s0)
    inp = W.make_prefill_inputs(w, seed=seed)
    if decay == "token":  # per-token log alpha given directly: log alpha = -softplus(g)
        inp["decay_kind"] = "token"
        inp["decay"] = -torch.nn.functional.softplus(inp["decay"].double()).float()
    return w, inp


@pytest.mark.parametrize("case", SMALL, ids=[f"{c[0]}x{c[1]}x{c[2]}_d{c[3]}x{c[4]}_{c[5]}_{c[6]}_{c[7]}_C{c[8]}"
                                             for c in SMALL])
def test_small_cases_match_oracle(case):
    w, inp = _make(*case)
    O, S = gpu_prefill(inp, w.phi, case[8])
    O_ref, S_ref = oracle_prefill(inp, w.phi)
    parity.check(O, O_ref, w.dtype, "O")
    parity.check(S, S_ref, w.dtype, "S_final")


@pytest.mark.parametrize("chunk", [1, 4, 7, 33, 64])
def test_chunk_size_invariance_fp32(chunk):
    """The output does not depend on C (page 1 checks [a], [b]) -- here on the
    GPU against the oracle at fp32 tolerance, L = 300, d = 16."""
    w = W.PREFILL["L300_d16_f32"]
    inp = W.make_prefill_inputs(w)
    O, S = gpu_prefill(inp, w.phi, chunk)
    O_ref, S_ref = oracle_prefill(inp, w.phi)
    parity.check(O, O_ref, "f32", f"O C={chunk}")
    parity.check(S, S_ref, "f32", f"S C={chunk}")


def test_headline_fp32_workload():
    """B=1, H=1, L=300, d=16, fp32, chunk 64 (ragged 44-token tail): the whole
    output at relative Frobenius error <= 1e-5."""
    w = W.PREFILL["L300_d16_f32"]
    inp = W.make_prefill_inputs(w)
    O, S = gpu_prefill(inp, w.phi, w.chunk)
    O_ref, S_ref = oracle_prefill(inp, w.phi)
    parity.check(O, O_ref, "f32", "O")
    parity.check(S, S_ref, "f32", "S_final")


# Many (b, h) sequences of ten chunks each: the launcher keeps each sequence
# in one segment, so every output CTA runs one long state chain through the
# stage ring and the lookahead (d = 128 over two value-column slices).
MULTI = [
    # (B, H, L, d, phi, decay, s0)
    (2, 76, 640, 64, "identity", "none", None),
    (2, 76, 640, 64, "elu1", "head", None),
    (2, 76, 640, 64, "identity", "logit", 0.1),
    (2, 76, 640, 128, "identity", "none", None),
    (2, 76, 640, 128, "identity", "head", None),
    (2, 76, 600, 128, "elu1", "logit", 0.1),
    (4, 76, 640, 128, "identity", "head", 0.1),
    (4, 76, 630, 64, "elu1", "token", None),
]


@pytest.mark.parametrize("case", MULTI, ids=[f"{c[0]}x{c[1]}x{c[2]}_d{c[3]}_{c[4]}_{c[5]}" for c in MULTI])
def test_multi_chunk_segments_match_oracle(case):
    B, H, L, d, phi, decay, s0 = case
    w, inp = _make(B, H, L, d, d, "bf16", phi, decay, 64, s0)
    O, S = gpu_prefill(inp, w.phi, 64)
    pairs = [(0, 0), (B - 1, H - 1), (B // 2, H // 3), (1, 5)]
    O_ref, S_ref = oracle_prefill(inp, w.phi, pairs)
    parity.check(select_pairs(O, pairs), O_ref, "bf16", "O")
    parity.check(select_pairs(S, pairs), S_ref, "bf16", "S_final")


# Sequences the launcher cuts into segments: a segment-state pass and a scan
# give each segment its incoming state, and each output CTA interleaves two
# segments (d = 64).  The shapes cover one-chunk segments, odd segment counts
# (the last d = 64 CTA has one segment), a short last segment, both head
# sizes, and both forms of the d = 128 state pass with decay.
SEGMENTED = [
    # (B, H, L, d, phi, decay, s0, sampled pairs or None for all)
    (1, 2, 1000, 64, "elu1", "none", None, None),
    (1, 2, 2100, 128, "identity", "head", 0.1, None),
    (2, 4, 3000, 64, "identity", "logit", 0.1, None),
    (1, 2, 6000, 64, "elu1", "head", None, None),
    (2, 4, 3100, 64, "elu1", "head", None, None),
    (2, 4, 2800, 64, "identity", "logit", 0.1, None),
    (2, 4, 1500, 128, "elu1", "none", 0.1, None),
    (2, 4, 6000, 128, "identity", "logit", 0.1, [(0, 0), (1, 3), (0, 2)]),
    # 4 segments of 32 chunks x 128 sequences: 384 segment-state blocks, more
    # than one wave of two per SM, so the d = 128 pass with decay runs in its
    # two-stage form (three blocks per SM)
    (4, 32, 8192, 128, "identity", "head", None, [(0, 0), (3, 31), (2, 17)]),
]


@pytest.mark.parametrize("case", SEGMENTED,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}_d{c[3]}_{c[4]}_{c[5]}" for c in SEGMENTED])
def test_segmented_sequences_match_oracle(case):
    B, H, L, d, phi, decay, s0, pairs = case
    assert api.la_chunk_fwd_workspace_bytes(B, H, L, d, d, 64) > 0  # segments in use
    w, inp = _make(B, H, L, d, d, "bf16", phi, decay, 64, s0)
    O, S = gpu_prefill(inp, w.phi, 64)
    if pairs is None:
        O_ref, S_ref = oracle_prefill(inp, w.phi)
        parity.check(O, O_ref, "bf16", "O")
        parity.check(S, S_ref, "bf16", "S_final")
    else:
        O_ref, S_ref = oracle_prefill(inp, w.phi, pairs)
        parity.check(select_pairs(O, pairs), O_ref, "bf16", "O")
        parity.check(select_pairs(S, pairs), S_ref, "bf16", "S_final")


# elu + 1 over a wide input range: q and k scaled by a power of two (exact in
# bf16) to a standard deviation of about 4, so that many entries lie deep in
# the exponential branch, where the packed-bf16 form
# of phi rounds the exponent argument.  Covers the output kernel (phi alone on
# Q and K), the segment-state kernel without decay (phi alone on K) and with
# decay (phi and K's weight in one fp32 pass).
WIDE = [
    # (B, H, L, d, decay)
    (2, 4, 1000, 64, "none"),
    (1, 2, 2100, 128, "none"),
    (1, 3, 1500, 64, "head"),
    (1, 2, 1300, 128, "logit"),
]


@pytest.mark.parametrize("case", WIDE, ids=[f"{c[0]}x{c[1]}x{c[2]}_d{c[3]}_{c[4]}" for c in WIDE])
def test_elu1_on_wide_range_inputs(case):
    B, H, L, d, decay = case
    w, inp = _make(B, H, L, d, d, "bf16", "elu1", decay, 64, None)
    scale = 32 if d == 64 else 64  # inputs are N(0, 1/d)
    inp["q"] = inp["q"] * scale
    inp["k"] = inp["k"] * scale
    assert float((inp["k"].float() < -4).float().mean()) > 0.1  # deep in exp(x)
    O, S = gpu_prefill(inp, w.phi, 64)
    O_ref, S_ref = oracle_prefill(inp, w.phi)
    parity.check(O, O_ref, "bf16", "O")
    parity.check(S, S_ref, "bf16", "S_final")


# Per-token decays whose strength alternates by chunk: odd chunks decay hard
# (log a ~ -2.4 per token, chunk total ~ -155), even chunks gently (~ -15).
# The tensor-core kernel treats the two kinds of chunk differently (the decay
# folded into V rows and output rows, or applied per element), so this checks
# both and the hand-over of the state between them.
MIXED = [
    # (B, H, L, d, phi)
    (1, 2, 300, 64, "identity"),
    (1, 2, 300, 128, "elu1"),
    (2, 76, 640, 128, "identity"),
    (2, 76, 600, 64, "elu1"),
    (2, 4, 3000, 128, "identity"),
    (2, 4, 3000, 64, "elu1"),
]


@pytest.mark.parametrize("case", MIXED, ids=[f"{c[0]}x{c[1]}x{c[2]}_d{c[3]}_{c[4]}" for c in MIXED])
def test_mixed_strong_and_weak_decay_chunks(case):
    B, H, L, d, phi = case
    w, inp = _make(B, H, L, d, d, "bf16", phi, "token", 64, 0.1)
    g = torch.randn(B, H, L, generator=torch.Generator().manual_seed(7), dtype=torch.float64)
    strength = torch.where((torch.arange(L) // 64) % 2 == 1, 3.0, 0.3).double()
    inp["decay"] = (-strength * torch.nn.functional.softplus(g)).float()
    O, S = gpu_prefill(inp, w.phi, 64)
    pairs = [(0, 0), (B - 1, H - 1), (B // 2, H // 3)]
    O_ref, S_ref = oracle_prefill(inp, w.phi, pairs)
    parity.check(select_pairs(O, pairs), O_ref, "bf16", "O")
    parity.check(select_pairs(S, pairs), S_ref, "bf16", "S_final")


FULL = {
    "B4_H16_L4096_d64_elu1": [(0, 0), (1, 7), (2, 13), (3, 15)],
    "B2_H32_L8192_d128_retnet": [(0, 0), (0, 31), (1, 16), (1, 5)],
    "B1_H16_L32768_d128_gate": [(0, 0), (0, 9), (0, 15)],
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_workloads_on_sampled_sequences(name):
    """The bf16 workloads at full size, launched as the benchmark launches
    them; the oracle recomputes a sample of whole (b, h) sequences."""
    w = W.PREFILL[name]
    inp = W.make_prefill_inputs(w)
    O, S = gpu_prefill(inp, w.phi, w.chunk)
    assert torch.isfinite(O.float()).all() and torch.isfinite(S).all()
    pairs = FULL[name]
    O_ref, S_ref = oracle_prefill(inp, w.phi, pairs)
    parity.check(select_pairs(O, pairs), O_ref, w.dtype, f"{name} O")
    parity.check(select_pairs(S, pairs), S_ref, w.dtype, f"{name} S_final")


def test_empty_sequence_returns_initial_state():
    S0 = torch.randn(2, 3, 64, 64, device="cuda")
    q = torch.empty(2, 3, 0, 64, dtype=torch.bfloat16, device="cuda")
    O, S = api.la_chunk_fwd(q, q, q, 64, S0=S0)
    api.la_device_status()
    assert O.shape == (2, 3, 0, 64)
    assert torch.equal(S, S0)
    O, S = api.la_chunk_fwd(q, q, q, 64)
    assert torch.count_nonzero(S) == 0


def test_empty_batch_is_a_no_op():
    q = torch.empty(0, 4, 16, 64, dtype=torch.bfloat16, device="cuda")
    O, S = api.la_chunk_fwd(q, q, q, 64)
    api.la_device_status()
    assert O.numel() == 0 and S.numel() == 0


@pytest.mark.parametrize("dtype,d", [("f32", 16), ("bf16", 64), ("bf16", 128)])
def test_final_state_may_alias_initial_state(dtype, d):
    w, inp = _make(1, 2, 150, d, d, dtype, "identity", "logit", 64, 0.1)
    O_ref, S_ref = gpu_prefill(inp, "identity")
    S = to_dev(inp["S0"])
    api.la_set_feature_map("identity")
    O, S_out = api.la_chunk_fwd(to_dev(inp["q"]), to_dev(inp["k"]), to_dev(inp["v"]), 64, "logit",
                                to_dev(inp["decay"]), S, S_final=S)
    api.la_device_status()
    assert S_out.data_ptr() == S.data_ptr()
    assert torch.equal(O.cpu(), O_ref) and torch.equal(S.cpu(), S_ref)


@pytest.mark.parametrize("dtype,d", [("f32", 32), ("bf16", 128)])
def test_resume_from_carried_state(dtype, d):
    """Running [0, m) and then [m, L) from the returned state equals one run."""
    w, inp = _make(1, 2, 300, d, d, dtype, "identity", "logit", 64, 0.1)
    O_ref, S_ref = oracle_prefill(inp, "identity")
    m = 131
    first = {k_: (v_[:, :, :m].contiguous() if k_ in "qkv" else v_) for k_, v_ in inp.items()}
    first["decay"] = inp["decay"][:, :, :m].contiguous()
    O1, S1 = gpu_prefill(first, "identity")
    second = {k_: (v_[:, :, m:].contiguous() if k_ in "qkv" else v_) for k_, v_ in inp.items()}
    second["decay"] = inp["decay"][:, :, m:].contiguous()
    second["S0"] = S1
    O2, S2 = gpu_prefill(second, "identity")
    parity.check(torch.cat([O1, O2], dim=2), O_ref, dtype, "resumed O")
    parity.check(S2, S_ref, dtype, "resumed S")


def test_unsupported_and_invalid_requests_raise():
    q = torch.zeros(1, 1, 8, 48, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.LAError) as e:
        api.la_chunk_fwd(q, q, q, 64)
    assert e.value.status == api.LA_ERR_UNSUPPORTED
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.LAError) as e:
        api.la_chunk_fwd(q, q, q, 64, "head", None)
    assert e.value.status == api.LA_ERR_INVALID_ARG
    buf = torch.zeros(1 * 1 * 8 * 64 + 1, dtype=torch.bfloat16, device="cuda")
    mis = buf[1:].view(1, 1, 8, 64)  # 2-byte offset: not 16-byte aligned
    with pytest.raises(api.LAError) as e:
        api.la_chunk_fwd(mis, q, q, 64)
    assert e.value.status == api.LA_ERR_INVALID_ARG


def test_host_buffers_roundtrip():
    """CPU tensors in, CPU tensors out: same kernels, copies around them."""
    w, inp = _make(1, 2, 130, 64, 64, "bf16", "elu1", "none", 64, None)
    O_dev, S_dev = gpu_prefill(inp, "elu1")
    api.la_set_feature_map("elu1")
    O_h, S_h = api.la_chunk_fwd(inp["q"].pin_memory(), inp["k"].pin_memory(),
                                inp["v"].pin_memory(), 64)
    assert not O_h.is_cuda
    assert torch.equal(O_h, O_dev) and torch.equal(S_h, S_dev)


def test_timeout_selftest_reports_and_context_survives():
    assert api.la_selftest_wait_timeout(200) == api.LA_ERR_DEVICE_TIMEOUT
    assert "timed out" in api.la_last_error()
    w, inp = _make(1, 1, 70, 64, 64, "bf16", "identity", "none", 64, None)
    O, S = gpu_prefill(inp, "identity")
    O_ref, S_ref = oracle_prefill(inp, "identity")
    parity.check(O, O_ref, "bf16", "O after self-test")
