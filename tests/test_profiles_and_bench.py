"""Host checks of the measurement side: the committed ncu summaries and DRAM
traffic figures were taken on the kernel sources as they stand, and the
bench's algorithmic byte counts and roofline arithmetic.  CPU only."""
import glob
import hashlib
import json
import os
import re

import pytest

import bench
from causal_linear_attention_chunkwise_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sha16(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def test_traffic_figures_match_the_current_sources():
    """Every DRAM traffic figure the bench line may quote was captured on the
    kernel source as it stands (else the bench reports no traffic)."""
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        entries = json.load(f)
    assert entries
    for key in entries:
        assert bench.traffic_from_profiles(key) is not None, key


def test_ncu_summaries_name_the_current_sources():
    """Each summary under profiles/ that records its sources records their
    current contents: a kernel changed after its capture fails here."""
    pat = re.compile(r"`([^`]+\.cu)` sha256 ([0-9a-f]{16})")
    seen = 0
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            text = f.read()
        for rel, sha in pat.findall(text):
            assert _sha16(rel) == sha, (os.path.basename(path), rel)
            seen += 1
    assert seen > 0


def test_algorithmic_bytes_of_the_measured_workloads():
    """The per-call byte counts the roofline fractions divide by, written out
    term by term."""
    w = W.PREFILL["B1_H16_L32768_d128_gate"]
    n = 1 * 16 * 32768                      # head-tokens
    qkv_o = n * (128 + 128 + 128 + 128) * 2  # q, k, v read and O written, bf16
    gate = n * 4                            # one fp32 gate logit per head-token
    states = 2 * 16 * 128 * 128 * 4         # S0 read, S_final written, fp32
    assert bench.prefill_bytes(w) == qkv_o + gate + states == 541065216

    w = W.PREFILL["B2_H32_L8192_d128_retnet"]  # per-head decay: 32 floats, no S0
    assert bench.prefill_bytes(w) == 2 * 32 * 8192 * 512 * 2 + 32 * 4 + 64 * 128 * 128 * 4

    dw = W.DECODE["B512_H32_d128_decode"]
    bh = 512 * 32
    state_rmw = 2 * bh * 128 * 128 * 4      # the fp32 state read and written back
    qkv = bh * (128 + 128 + 128) * 2        # this step's q, k, v
    assert bench.decode_bytes(dw) == state_rmw + qkv + bh * 4 + bh * 128 * 2 == 2164326400


def test_roofline_arithmetic():
    peaks = {"hbm_gbs": 6683.8, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    w = W.PREFILL["B1_H16_L32768_d128_gate"]
    r = bench.roofline(bench.prefill_bytes(w), bench.prefill_flops(w), 0.1646e-3, peaks,
                       "measured", False)
    # 541 MB against 51.5 GFLOP: the copy bandwidth bounds it, not the tensor cores
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(541065216 / 0.1646e-3 / 1e9, abs=0.1)
    assert r["frac"] == pytest.approx(r["achieved"] / 6683.8, abs=1e-4)
    # a pure contraction with few bytes is tensor-bound, against the bf16 peak
    t = bench.roofline(1e6, 1e12, 1e-3, peaks, "measured", True)
    assert t["bound"] == "tensor" and t["peak"] == 1700.0
    assert t["frac"] == pytest.approx(1000.0 / 1700.0, abs=1e-4)
