"""The allocation-free prefill entry point, la_chunk_fwd_noalloc.

It serves callers that cannot allocate device memory when they run prefill
(allocator or memory-pool callbacks, fixed-footprint serving processes): the
segment states live in the library's static device scratch instead of a caller
workspace.  These tests call it through the C ABI and compare it with
la_chunk_fwd, the entry point that takes a caller workspace, on two calls in a
row (the scratch keeps the first call's contents when the second starts), after
a call that leaves NaN states behind in the scratch, and check that a call
after the first grows neither the device's nor torch's memory use.
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


def _noalloc(inp, O, S):
    api.la_chunk_fwd_noalloc(inp["q"], inp["k"], inp["v"], 64, inp["decay_kind"], inp["decay"],
                             inp["S0"], O=O, S_final=S)


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_matches_workspace_entry_point_on_two_calls(d):
    api.la_chunk_fwd_noalloc_prepare()
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
        _noalloc(inp, O_na, S_na)
    api.la_device_status()
    for i, (_, (O_ref, S_ref), O_na, S_na) in enumerate(runs):
        parity.check(O_na.cpu(), O_ref.cpu(), "bf16", f"call {i}: O")
        parity.check(S_na.cpu(), S_ref.cpu(), "bf16", f"call {i}: S_final")


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_ignores_nan_states_left_in_the_scratch(d):
    """A call whose values are NaN fills the scratch's segment states with NaN;
    the next call of the same shape must not read any of them."""
    api.la_chunk_fwd_noalloc_prepare()
    api.la_set_feature_map("identity")
    _, inp = _inputs(2, 4, 3000, d, "identity", "logit", 0.1, 2)
    poison = dict(inp, v=torch.full_like(inp["v"], float("nan")))
    O_p, S_p = torch.empty_like(inp["v"]), torch.empty_like(inp["S0"])
    _noalloc(poison, O_p, S_p)
    api.la_device_status()
    assert torch.isnan(S_p).all()  # the poisoned states did pass through the scratch
    O_ref, S_ref = api.la_chunk_fwd(inp["q"], inp["k"], inp["v"], 64, inp["decay_kind"],
                                    inp["decay"], inp["S0"])
    O_na, S_na = torch.empty_like(O_ref), torch.empty_like(S_ref)
    _noalloc(inp, O_na, S_na)
    api.la_device_status()
    parity.check(O_na.cpu(), O_ref.cpu(), "bf16", "O after NaN leftovers")
    parity.check(S_na.cpu(), S_ref.cpu(), "bf16", "S_final after NaN leftovers")


def test_noalloc_call_after_the_first_grows_no_memory():
    api.la_chunk_fwd_noalloc_prepare()
    api.la_set_feature_map("identity")
    _, inp = _inputs(1, 16, 8192, 128, "identity", "logit", 0.1, 3)
    assert api.la_chunk_fwd_workspace_bytes(1, 16, 8192, 128, 128, 64) > 0
    O, S = torch.empty_like(inp["v"]), torch.empty_like(inp["S0"])
    _noalloc(inp, O, S)  # the first call may load the prefill kernels' module
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    _noalloc(inp, O, S)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0
    api.la_device_status()


def test_noalloc_rejects_problems_larger_than_its_scratch():
    B, H, L, d = 8, 32, 32768, 128  # needs far more segment-state scratch than it has
    assert api.la_chunk_fwd_workspace_bytes(B, H, L, d, d, 64) > api.la_chunk_fwd_noalloc_scratch_bytes()
    q = torch.empty(1, dtype=torch.bfloat16, device="cuda")  # never touched: rejected first
    lib = api._native.load()
    st = lib.la_chunk_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), 1, B, H, L, d, d, 64,
                                  0, None, None, q.data_ptr(), None, None)
    assert st == api.LA_ERR_UNSUPPORTED
    assert "static scratch holds" in api.la_last_error()
