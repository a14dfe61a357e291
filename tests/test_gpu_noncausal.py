"""GPU parity of la_noncausal_fwd, the non-causal matrix form O = phi(Q)
(phi(K)^T V) ("adv13 - Linear Attention / SSM" section 4.3), against the fp64
oracle on the same seeded inputs.  Needs a GB300."""
import pytest
import torch

import oracle
from causal_linear_attention_chunkwise_gb300 import api
from causal_linear_attention_chunkwise_gb300 import workloads as W
from tests import parity
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, L, d, phi): one token, one chunk, a ragged tail, several segments
    (1, 1, 1, 64, "identity"),
    (2, 2, 64, 64, "identity"),
    (2, 3, 300, 64, "elu1"),
    (1, 2, 200, 128, "identity"),
    (2, 4, 1000, 128, "elu1"),
    (1, 2, 5000, 64, "elu1"),
    (1, 1, 2300, 128, "identity"),
]


def _inputs(B, H, L, d, seed=0):
    w = W.small_prefill(B, H, L, d, d, "bf16", "identity", "none", 64)
    return W.make_prefill_inputs(w, seed=seed)


def _gpu(inp, phi):
    api.la_set_feature_map(phi)
    O, S = api.la_noncausal_fwd(to_dev(inp["q"]), to_dev(inp["k"]), to_dev(inp["v"]))
    api.la_device_status()
    return O.cpu(), S.cpu()


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}_d{c[3]}_{c[4]}" for c in CASES])
def test_noncausal_matches_oracle(case):
    B, H, L, d, phi = case
    inp = _inputs(B, H, L, d)
    O, S = _gpu(inp, phi)
    O_ref, S_ref = oracle.noncausal(inp["q"], inp["k"], inp["v"], phi=phi)
    parity.check(O, O_ref, "bf16", "O")
    parity.check(S, S_ref, "bf16", "S")


def test_noncausal_full_size_on_sampled_sequences():
    """The d = 64 prefill workload's shape, checked on three sequences."""
    B, H, L, d = 4, 16, 4096, 64
    inp = _inputs(B, H, L, d, seed=3)
    O, S = _gpu(inp, "elu1")
    for b, h in [(0, 0), (3, 15), (2, 7)]:
        sl = lambda x: x[b:b + 1, h:h + 1]
        O_ref, S_ref = oracle.noncausal(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), phi="elu1")
        parity.check(sl(O), O_ref, "bf16", f"O[{b},{h}]")
        parity.check(sl(S), S_ref, "bf16", f"S[{b},{h}]")


def test_noncausal_last_row_equals_causal_last_row():
    """Both forms read phi(K)^T V at the last token; the states agree too."""
    B, H, L, d = 2, 2, 700, 128
    inp = _inputs(B, H, L, d, seed=5)
    O, S = _gpu(inp, "elu1")
    api.la_set_feature_map("elu1")
    Oc, Sc = api.la_chunk_fwd(to_dev(inp["q"]), to_dev(inp["k"]), to_dev(inp["v"]), 64)
    api.la_device_status()
    parity.check(O[:, :, -1:], Oc.cpu()[:, :, -1:], "bf16", "last row")
    parity.check(S, Sc.cpu(), "bf16", "state")


def test_noncausal_empty_and_unsupported():
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    S = torch.full((1, 2, 64, 64), 7.0, device="cuda")
    api.la_noncausal_fwd(q, q, q, S=S)
    api.la_device_status()
    assert torch.count_nonzero(S) == 0  # no tokens: the state is zero
    x = torch.zeros(1, 1, 64, 32, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.LAError) as e:
        api.la_noncausal_fwd(x, x, x)
    assert e.value.status == api.LA_ERR_UNSUPPORTED
    x = torch.zeros(1, 1, 64, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(api.LAError) as e:
        api.la_noncausal_fwd(x, x, x)
    assert e.value.status == api.LA_ERR_UNSUPPORTED
