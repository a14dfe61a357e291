"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU.  CPU only
(the library must have been built; the build runs here without a GPU)."""
import ctypes
import os
import re

import pytest

from causal_linear_attention_chunkwise_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_symbols():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(la_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_native.LIB_PATH):
        build.build()
    return _native.load()


def test_header_declares_the_three_core_calls():
    names = declared_symbols()
    assert {"la_chunk_fwd", "la_decode_step", "la_set_feature_map"} <= names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in sorted(declared_symbols()) if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert set(_native.SIGNATURES) == declared_symbols()


def test_feature_map_roundtrip(lib):
    assert lib.la_set_feature_map(7) == 1
    assert b"unknown feature map" in lib.la_last_error()
    assert lib.la_set_feature_map(1) == 0 and lib.la_get_feature_map() == 1
    assert lib.la_set_feature_map(0) == 0 and lib.la_get_feature_map() == 0


def test_validation_before_any_device_work(lib):
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    # unknown dtype
    assert lib.la_chunk_fwd(p, p, p, 9, 1, 1, 8, 16, 16, 64, 0, None, None, p, None, None, 0,
                            None) == 1
    # negative size
    assert lib.la_chunk_fwd(p, p, p, 1, 1, 1, -1, 16, 16, 64, 0, None, None, p, None, None, 0,
                            None) == 1
    # unsupported head size and chunk
    assert lib.la_chunk_fwd(p, p, p, 1, 1, 1, 8, 48, 48, 64, 0, None, None, p, None, None, 0,
                            None) == 2
    assert lib.la_chunk_fwd(p, p, p, 1, 1, 1, 8, 64, 64, 128, 0, None, None, p, None, None, 0,
                            None) == 2
    # null tensors, decay without values, misaligned pointer
    assert lib.la_chunk_fwd(None, p, p, 1, 1, 1, 8, 16, 16, 64, 0, None, None, p, None, None, 0,
                            None) == 1
    assert lib.la_chunk_fwd(p, p, p, 1, 1, 1, 8, 16, 16, 64, 2, None, None, p, None, None, 0,
                            None) == 1
    assert b"decay pointer" in lib.la_last_error()
    q = ctypes.c_void_p(0x1002)
    assert lib.la_chunk_fwd(q, p, p, 1, 1, 1, 8, 16, 16, 64, 0, None, None, p, None, None, 0,
                            None) == 1
    assert b"16-byte" in lib.la_last_error()
    # empty batch and empty sequence without a final state are no-ops
    assert lib.la_chunk_fwd(p, p, p, 1, 0, 4, 8, 16, 16, 64, 0, None, None, p, None, None, 0,
                            None) == 0
    assert lib.la_chunk_fwd(None, None, None, 1, 2, 2, 0, 16, 16, 64, 0, None, None, None, None,
                            None, 0, None) == 0
    # decode: unsupported shapes and null state
    assert lib.la_decode_step(p, p, p, 1, 1, 1, 128, 64, None, p, p, None) == 2
    assert lib.la_decode_step(p, p, p, 1, 1, 1, 128, 128, None, None, p, None) == 1


def test_workspace_query_is_host_only(lib):
    for args in [(4, 16, 4096, 64, 64, 64, 1), (1, 16, 32768, 128, 128, 64, 1),
                 (1, 1, 300, 16, 16, 64, 0), (0, 1, 10, 64, 64, 64, 1)]:
        n = lib.la_chunk_fwd_workspace_bytes(*args)
        assert n >= 0


def test_noalloc_scratch_holds_every_prefill_workload(lib):
    """The static scratch of la_chunk_fwd_noalloc is sized so that every prefill workload's
    segment states fit (on the 152-SM plan the query assumes without a GPU)."""
    from causal_linear_attention_chunkwise_gb300 import workloads as W
    cap = lib.la_chunk_fwd_noalloc_scratch_bytes()
    for w in W.PREFILL.values():
        need = lib.la_chunk_fwd_workspace_bytes(w.B, w.H, w.L, w.dk, w.dv, w.chunk,
                                                1 if w.dtype == "bf16" else 0)
        assert need <= cap, (w.name, need, cap)


def test_noncausal_validation_and_workspace(lib):
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    # fp32, mismatched or unsupported head sizes: unsupported
    assert lib.la_noncausal_fwd(p, p, p, 0, 1, 1, 64, 64, 64, p, None, p, 1 << 20, None) == 2
    assert lib.la_noncausal_fwd(p, p, p, 1, 1, 1, 64, 64, 128, p, None, p, 1 << 20, None) == 2
    assert lib.la_noncausal_fwd(p, p, p, 1, 1, 1, 64, 32, 32, p, None, p, 1 << 20, None) == 2
    assert b"bf16" in lib.la_last_error()
    # unknown dtype, negative size, null tensors, misaligned pointer
    assert lib.la_noncausal_fwd(p, p, p, 5, 1, 1, 64, 64, 64, p, None, p, 1 << 20, None) == 1
    assert lib.la_noncausal_fwd(p, p, p, 1, 1, 1, -3, 64, 64, p, None, p, 1 << 20, None) == 1
    assert lib.la_noncausal_fwd(None, p, p, 1, 1, 1, 64, 64, 64, p, None, p, 1 << 20, None) == 1
    assert lib.la_noncausal_fwd(ctypes.c_void_p(0x1004), p, p, 1, 1, 1, 64, 64, 64, p, None, p,
                                1 << 20, None) == 1
    # workspace too small or missing
    need = lib.la_noncausal_fwd_workspace_bytes(2, 3, 1000, 64, 64)
    assert need > 0
    assert lib.la_noncausal_fwd(p, p, p, 1, 2, 3, 1000, 64, 64, p, None, p, need - 1, None) == 1
    assert b"workspace" in lib.la_last_error()
    assert lib.la_noncausal_fwd(p, p, p, 1, 2, 3, 1000, 64, 64, p, None, None, 0, None) == 1
    # the workspace holds one fp32 d x d state per segment and sequence plus the
    # sum slot, then one log decay per slot (256-byte aligned); segments are at
    # most 32 chunks
    for B, H, L, d in [(1, 1, 1, 64), (4, 16, 4096, 64), (2, 32, 8192, 128), (1, 16, 32768, 128)]:
        ws = lib.la_noncausal_fwd_workspace_bytes(B, H, L, d, d)
        bh, nc = B * H, (L + 63) // 64
        slots = [n for n in range(2, nc + 2)
                 if bh * n * d * d * 4 + (bh * n * 4 + 255) // 256 * 256 == ws]
        assert len(slots) == 1, (B, H, L, d, ws)
        assert -(-nc // (slots[0] - 1)) <= 32
    assert lib.la_noncausal_fwd_workspace_bytes(1, 1, 64, 64, 128) == 0
    # empty batch is a no-op
    assert lib.la_noncausal_fwd(p, p, p, 1, 0, 4, 64, 64, 64, p, None, None, 0, None) == 0


def test_prefill_plan_invariants(lib):
    """The tensor-core launcher's segment plan, seen through the workspace query: segments of at
    most 32 chunks, at most one per chunk, and three kernels exactly when a workspace is used."""
    for B, H, L in [(1, 1, 64), (1, 1, 100), (4, 16, 4096), (2, 32, 8192), (1, 16, 32768),
                    (8, 32, 32768), (1, 2, 6000), (2, 4, 3000), (64, 64, 512), (1, 1, 1 << 17)]:
        for d in (64, 128):
            ws = lib.la_chunk_fwd_workspace_bytes(B, H, L, d, d, 64, 1)
            kernels = lib.la_chunk_fwd_kernel_count(B, H, L, d, d, 64, 1)
            bh, nc = B * H, (L + 63) // 64
            if ws == 0:
                assert kernels == 1 and nc <= 32, (B, H, L, d)
                continue
            assert kernels == 3
            ns = [n for n in range(2, nc + 1)
                  if bh * n * d * d * 4 + (bh * n * 4 + 255) // 256 * 256 == ws]
            assert len(ns) == 1, (B, H, L, d, ws)
            g = -(-nc // ns[0])
            assert g <= 32 and -(-nc // g) == ns[0], (B, H, L, d, ns[0])
    # fp32 and other shapes take the SIMT path: no workspace
    assert lib.la_chunk_fwd_workspace_bytes(4, 16, 4096, 64, 64, 64, 0) == 0
    assert lib.la_chunk_fwd_workspace_bytes(4, 16, 4096, 32, 32, 64, 1) == 0


def _prefill_segments(lib, B, H, L, d):
    ws = lib.la_chunk_fwd_workspace_bytes(B, H, L, d, d, 64, 1)
    if ws == 0:
        return 1
    bh, nc = B * H, (L + 63) // 64
    ns = [n for n in range(2, nc + 1) if bh * n * d * d * 4 + (bh * n * 4 + 255) // 256 * 256 == ws]
    assert len(ns) == 1, (B, H, L, d, ws)
    return ns[0]


def test_prefill_plan_picks_the_measured_segment_counts(lib):
    """The cost model's picks on 152 SMs, at the segment counts that measured fastest on a
    GB300 when every count within the 32-chunk bound was timed: 19 for B1 H16 L32768 d128
    (160.6 us against 166.4 at 18 and 191.3 at 20), 4 for B2 H32 L8192 d128 (171.3 us
    against 175.4 at 7), 4 for B4 H32 L8192 d128, 2 for B8 H32 L4096 d128 and 4 for B1 H64
    L8192 d128; the d64 workload B4 H16 L4096 keeps 4."""
    try:
        import torch
        if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 152:
            pytest.skip("the plan depends on the SM count; these picks are for 152 SMs")
    except ImportError:
        pass
    for (B, H, L, d), ns in [((1, 16, 32768, 128), 19), ((2, 32, 8192, 128), 4),
                             ((4, 32, 8192, 128), 4), ((8, 32, 4096, 128), 2),
                             ((1, 64, 8192, 128), 4), ((4, 16, 4096, 64), 4)]:
        assert _prefill_segments(lib, B, H, L, d) == ns, (B, H, L, d)


def test_channel_gate_plan_invariants(lib):
    """The per-channel gate's segment plan, seen through its workspace query: with segments,
    one fp32 state and one log-decay row per slot, and the slots are the state pass's pieces
    plus a copy of S0 -- at d = 64 each segment but the last in two pieces (2 (NS - 1) + 1
    slots; the chunks / 8 cap on NS leaves every segment two chunks or more), at d = 128 in
    one (NS slots) -- for 2 <= NS <= chunks / 8."""
    for B, H, L in [(4, 16, 4096), (2, 32, 8192), (1, 16, 32768), (2, 16, 4096), (1, 2, 3000),
                    (8, 16, 2048), (1, 1, 1 << 16), (64, 64, 512)]:
        for d in (64, 128):
            ws = lib.la_channel_gate_fwd_workspace_bytes(B, H, L, d, d, 64, 1)
            if ws == 0:
                continue
            bh, nc = B * H, (L + 63) // 64
            per_slot = bh * (d * d + d) * 4
            assert ws % per_slot == 0, (B, H, L, d, ws)
            slots = ws // per_slot
            if d == 64:
                assert slots % 2 == 1, (B, H, L, d, slots)
                n_seg = (slots - 1) // 2 + 1
            else:
                n_seg = slots
            assert 2 <= n_seg <= nc // 8, (B, H, L, d, n_seg)
    # the tensor-core gate takes bf16, chunk 64, d in {64, 128}: no workspace otherwise
    assert lib.la_channel_gate_fwd_workspace_bytes(4, 16, 4096, 64, 64, 64, 0) == 0
    assert lib.la_channel_gate_fwd_workspace_bytes(4, 16, 4096, 32, 32, 64, 1) == 0


def test_variant_validation_before_any_device_work(lib):
    """la_normalised_fwd, la_channel_gate_fwd and la_delta_fwd reject bad
    arguments before any device work."""
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    odd = ctypes.c_void_p(0x1008)
    W = 1 << 20
    nf = lambda *a: lib.la_normalised_fwd(*a, p, W, None)  # noqa: E731
    # (q, k, v, dtype, B, H, L, d_k, d_v, chunk, decay_kind, decay, S0, z0, O, S_final, z_final)
    # + (workspace, ws_bytes, stream)
    assert nf(p, p, p, 7, 1, 1, 8, 16, 16, 64, 0, None, None, None, p, None, None) == 1
    assert nf(p, p, p, 1, 1, 1, 8, 48, 16, 64, 0, None, None, None, p, None, None) == 2
    assert nf(p, p, p, 1, 1, 1, 8, 16, 16, 65, 0, None, None, None, p, None, None) == 2
    assert nf(p, p, p, 1, 1, 1, 8, 16, 16, 0, 0, None, None, None, p, None, None) == 1
    assert nf(p, p, p, 1, 1, 1, 8, 16, 16, 64, 5, None, None, None, p, None, None) == 1
    assert nf(p, p, p, 1, 1, 1, 8, 16, 16, 64, 3, None, None, None, p, None, None) == 1
    assert b"decay pointer" in lib.la_last_error()
    assert nf(p, p, p, 1, 1, 1, 8, 16, 16, 64, 0, None, None, None, None, None, None) == 1
    assert nf(p, p, p, 1, 1, 1, 8, 16, 16, 64, 0, None, None, odd, p, None, None) == 1
    assert b"16-byte" in lib.la_last_error()
    assert nf(p, p, p, 1, 0, 3, 8, 16, 16, 64, 0, None, None, None, p, None, None) == 0
    # the workspace, checked before any launch
    need = lib.la_normalised_fwd_workspace_bytes(4, 16, 4096, 64, 64, 64, 1)
    assert need > lib.la_chunk_fwd_workspace_bytes(4, 16, 4096, 64, 64, 64, 1) > 0
    assert lib.la_normalised_fwd_workspace_bytes(1, 1, 300, 16, 16, 64, 0) > 0
    assert lib.la_normalised_fwd_workspace_bytes(1, 1, 0, 16, 16, 64, 0) == 0
    assert lib.la_normalised_fwd(p, p, p, 1, 4, 16, 4096, 64, 64, 64, 0, None, None, None, p,
                                 None, None, p, need - 1, None) == 1
    assert b"workspace" in lib.la_last_error()
    assert lib.la_normalised_fwd(p, p, p, 1, 4, 16, 4096, 64, 64, 64, 0, None, None, None, p,
                                 None, None, None, 0, None) == 1
    cg = lambda *a: lib.la_channel_gate_fwd(*a, None, 0, None)  # noqa: E731
    # (q, k, v, dtype, B, H, L, d_k, d_v, chunk, log_alpha, S0, O, S_final[, workspace,
    #  ws_bytes, stream])
    assert cg(p, p, p, 1, 1, 1, 8, 16, 16, 64, None, None, p, None) == 1
    assert b"log_alpha" in lib.la_last_error()
    assert cg(p, p, p, 1, 1, 1, 8, 16, 16, 64, odd, None, p, None) == 1
    assert b"log_alpha" in lib.la_last_error()
    assert cg(p, p, p, 1, 1, 1, 8, 16, 256, 64, p, None, p, None) == 2
    assert cg(p, p, p, 1, 1, -1, 8, 16, 16, 64, p, None, p, None) == 1
    assert cg(p, odd, p, 1, 1, 1, 8, 16, 16, 64, p, None, p, None) == 1
    # the segment workspace: none needed for a short or an unsupported problem; a
    # given one that is too small or misaligned is refused before any launch
    need = lib.la_channel_gate_fwd_workspace_bytes(4, 16, 4096, 64, 64, 64, 1)
    assert need > 0
    assert lib.la_channel_gate_fwd_workspace_bytes(1, 1, 300, 64, 64, 64, 1) == 0
    assert lib.la_channel_gate_fwd_workspace_bytes(4, 16, 4096, 64, 64, 64, 0) == 0
    assert lib.la_channel_gate_fwd_workspace_bytes(4, 16, 4096, 64, 64, 32, 1) == 0
    full = lambda *a: lib.la_channel_gate_fwd(*a)  # noqa: E731
    assert full(p, p, p, 1, 4, 16, 4096, 64, 64, 64, p, None, p, None, p, need - 1, None) == 1
    assert b"workspace" in lib.la_last_error()
    assert full(p, p, p, 1, 4, 16, 4096, 64, 64, 64, p, None, p, None, odd, need, None) == 1
    assert b"16-byte" in lib.la_last_error()
    dl = lambda *a: lib.la_delta_fwd(*a)  # noqa: E731
    # (q, k, v, dtype, B, H, L, d_k, d_v, beta, log_alpha, S0, O, S_final, stream)
    assert dl(p, p, p, 1, 1, 1, 8, 16, 16, None, None, None, p, None, None) == 1
    assert b"beta" in lib.la_last_error()
    assert dl(p, p, p, 0, 1, 1, 8, 16, 24, p, None, None, p, None, None) == 2
    assert dl(p, p, p, 1, 1, 1, 8, 16, 16, p, None, None, p, odd, None) == 1
    assert dl(p, p, p, 2, 1, 1, 8, 16, 16, p, None, None, p, None, None) == 1


def _segments(num, bh, d):
    """Segments per sequence of a prefill workspace of num bytes: per segment a
    d x d fp32 state, then a 256-byte-rounded fp32 log decay per segment."""
    for n in range(1, 4096):
        if bh * n * d * d * 4 + (bh * n * 4 + 255) // 256 * 256 == num:
            return n
    raise AssertionError(f"no segment count gives {num} bytes")


def test_normalised_workspace_layout(lib):
    """la_normalised_fwd's workspace.  The two-pass form (every case but bf16,
    d_k = d_v = 64, chunk 64) is the prefill's workspace (rounded up to 256
    bytes) followed by the z scan's: per sequence and 256-token block a d_k
    total and a log decay, and one incoming z0 per sequence, all fp32.  The
    one-pass d = 64 form keeps the same segments, with each segment state 16
    columns wider (z in the first of them), and has no scan of its own."""
    for B, H, L, dk, dv, chunk, dtype in [(4, 16, 4096, 64, 64, 64, 1), (1, 16, 32768, 128, 128, 64, 1),
                                          (2, 3, 300, 32, 16, 7, 0), (1, 1, 1, 16, 16, 64, 0),
                                          (2, 32, 8192, 128, 128, 64, 1), (4, 16, 4096, 64, 64, 64, 0),
                                          (1, 2, 300, 64, 64, 64, 1), (8, 16, 16384, 64, 64, 64, 1)]:
        num = lib.la_chunk_fwd_workspace_bytes(B, H, L, dk, dv, chunk, dtype)
        bh, nblk = B * H, -(-L // 256)
        if (dk, dv, chunk, dtype) == (64, 64, 64, 1):
            n = _segments(num, bh, 64) if num else 0
            want = bh * n * 64 * 80 * 4 + (bh * n * 4 + 255) // 256 * 256
        else:
            scan = 4 * (bh * nblk * dk + bh * nblk + bh * dk)
            want = (num + 255) // 256 * 256 + scan
        assert lib.la_normalised_fwd_workspace_bytes(B, H, L, dk, dv, chunk, dtype) == want
    assert lib.la_normalised_fwd_workspace_bytes(1, 1, 64, 48, 48, 64, 1) == 0  # unsupported d
