"""The allocation-free prefill entry point, la_chunk_fwd_noalloc.

It serves callers that cannot allocate device memory when they run prefill
(allocator or memory-pool callbacks, fixed-footprint serving processes): the
segment states live in the library's static device scratch instead of a caller
workspace.  These tests call it through the C ABI and compare it with
la_chunk_fwd, the entry point that takes a caller workspace, on two calls in a
row (the scratch keeps the first call's contents when the second starts).
The file is named to be collected last."""
import pytest
import torch

from causal_linear_attention_chunkwise_gb300 import api
from causal_linear_attention_chunkwise_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


def _inputs(B, H, L, d, phi, decay, s0, seed):
    w = W.small_prefill(B, H, L, d, d, "bf16", phi, decay, 64, s0_std=s0)
    inp = W.make_prefill_inputs(w, seed=seed)
    return w, {k: (t.cuda() if torch.is_tensor(t) else t) for k, t in inp.items()}


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_matches_workspace_entry_point_on_two_calls(d):
    cases = [  # both split each sequence into segments, so the scratch is used
        (2, 4, 3000, d, "identity", "head", None, 0),
        (2, 4, 1500, d, "identity", "logit", 0.1, 1),
    ]
    api.la_set_feature_map("identity")
    runs = []
    for B, H, L, dd, phi, decay, s0, seed in cases:
        w, inp = _inputs(B, H, L, dd, phi, decay, s0, seed)
        need = api.la_chunk_fwd_workspace_bytes(B, H, L, dd, dd, 64)
        assert 0 < need <= api.la_chunk_fwd_noalloc_scratch_bytes()
        ref = api.la_chunk_fwd(inp["q"], inp["k"], inp["v"], 64, inp["decay_kind"], inp["decay"],
                               inp["S0"])
        runs.append((inp, ref, torch.empty_like(ref[0]), torch.empty_like(ref[1])))
    api.la_device_status()
    for inp, _, O_na, S_na in runs:  # two calls in a row on the shared scratch
        api.la_chunk_fwd_noalloc(inp["q"], inp["k"], inp["v"], 64, inp["decay_kind"], inp["decay"],
                                 inp["S0"], O=O_na, S_final=S_na)
    api.la_device_status()
    for i, (_, (O_ref, S_ref), O_na, S_na) in enumerate(runs):
        parity.check(O_na.cpu(), O_ref.cpu(), "bf16", f"call {i}: O")
        parity.check(S_na.cpu(), S_ref.cpu(), "bf16", f"call {i}: S_final")


def test_noalloc_rejects_problems_larger_than_its_scratch():
    B, H, L, d = 8, 32, 32768, 128  # needs far more segment-state scratch than it has
    assert api.la_chunk_fwd_workspace_bytes(B, H, L, d, d, 64) > api.la_chunk_fwd_noalloc_scratch_bytes()
    q = torch.empty(1, dtype=torch.bfloat16, device="cuda")  # never touched: rejected first
    lib = api._native.load()
    st = lib.la_chunk_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), 1, B, H, L, d, d, 64,
                                  0, None, None, q.data_ptr(), None, None)
    assert st == api.LA_ERR_UNSUPPORTED
    assert "static scratch holds" in api.la_last_error()
