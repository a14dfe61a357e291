#!/usr/bin/env python3
"""Benchmark: chunkwise causal linear attention prefill (and the decode step)
on one GB300 per process.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--no-cpu-baseline] [--legs main|all]

One "step" is one la_chunk_fwd call over the whole workload batch (every
prefill row of the path: feature map, gate prep, intra/inter products, state
update, output and final-state stores).  The headline workload is the largest
single-GPU prefill problem: B=1, H=16, L=32768, d=128, bf16, per-token gate
logits, a non-zero fp32 initial state, chunk 64.  ``value`` is prefill
tokens/s (B*L tokens per step, all heads of a token counted once) with inputs
resident in HBM.  The same line carries, each with its own time and roofline:
the other prefill workloads (``legs``), the decode step (B=512, H=32, d=128,
fp32 state in place) as ``decode``, the non-causal form (``noncausal``) and
the normalised, per-channel-gate and delta-rule forms (``variants``).

Timing: W untimed warm-up steps (at least ~1 s of them for the headline, so
the clock sampler sees the GPU under load), then a barrier and a synchronize,
K steps bracketed by CUDA events on the launching stream, a synchronize and a
barrier; the max over ranks.  Inputs rotate over enough copies that each
step's working set is out of L2 (129 MB).  Under torchrun (N > 1) every rank
runs its own replica of the workload (no data-path collective; weak scaling).

``--impl reference`` times the fp64 CPU oracle on the same workload (bounded
samples per step) on the host cores; only rank 0 works under torchrun.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from causal_linear_attention_chunkwise_gb300 import workloads as W  # noqa: E402

METRIC = "tokens/s per GB300 (chunkwise prefill, decode step); % of roofline"
DEFAULT_WORKLOAD = "B1_H16_L32768_d128_gate"
# Further prefill workloads timed beside the headline (the fp32 L = 300 one is a
# correctness / latency case: it fits in L2 and is launch-bound).
SUB_LEGS = ("B2_H32_L8192_d128_retnet", "B4_H16_L4096_d64_elu1", "L300_d16_f32")
NONCAUSAL_LEGS = ("B4_H16_L4096_d64_elu1", "B2_H32_L8192_d128_retnet")
VARIANT_SHAPE = "B4_H16_L4096_d64_elu1"
DECODE_WORKLOAD = "B512_H32_d128_decode"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
ELT = {"f32": 4, "bf16": 2}


# ---------------------------------------------------------------- ranks
def world():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, ws, local


def init_dist(backend=None):
    rank, ws, _ = world()
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        torch.distributed.init_process_group(backend, rank=rank, world_size=ws)
    return rank, ws


def barrier():
    if torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over all ranks (identity on one rank)."""
    if not torch.distributed.is_initialized():
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank_step: int, steps: int, elapsed_ms_max: float, n_ranks: int):
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    return tokens_per_rank_step * n_ranks * steps / (elapsed_ms_max / 1e3)


# ---------------------------------------------------------------- peaks and clocks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            flat = {}

            def walk(x, prefix=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, k if not prefix else f"{prefix}.{k}")
                elif isinstance(x, (int, float)):
                    flat[prefix.split(".")[-1]] = float(x)
            walk(d)
            if "hbm_gbs" in flat:
                return flat, "measured"
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the GPU works."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- algorithmic work
def prefill_bytes(w) -> int:
    """Bytes the path must move: q, k, v read and O written once, gate input,
    S0 read and S_final written."""
    e = ELT[w.dtype]
    n = w.B * w.H * w.L
    b = n * (2 * w.dk + w.dv) * e + n * w.dv * e
    if w.decay == "logit":
        b += n * 4
    elif w.decay == "head":
        b += w.H * 4
    st = w.B * w.H * w.dk * w.dv * 4
    b += st  # S_final
    if w.s0_std is not None:
        b += st
    return b


def prefill_flops(w) -> int:
    """Dense chunk products per head-token: 2C d_k + 2C d_v + 4 d_k d_v."""
    return w.B * w.H * w.L * (2 * w.chunk * w.dk + 2 * w.chunk * w.dv + 4 * w.dk * w.dv)


def decode_bytes(w) -> int:
    e = ELT[w.dtype]
    bh = w.B * w.H
    return 2 * bh * w.dk * w.dv * 4 + bh * (2 * w.dk + w.dv) * e + bh * 4 + bh * w.dv * e


def roofline(bytes_, flops, seconds, peaks, peak_kind, sustained):
    gbs = bytes_ / seconds / 1e9
    tfs = flops / seconds / 1e12
    t_mem = bytes_ / (peaks["hbm_gbs"] * 1e9)
    bf16 = peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops",
                     peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    t_fl = flops / (bf16 * 1e12)
    if t_mem >= t_fl:
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                "peak_source": peak_kind, "algorithmic_bytes": bytes_,
                "tflops_achieved": round(tfs, 2)}
    return {"bound": "tensor", "achieved": round(tfs, 2), "peak": bf16, "unit": "TFLOP/s",
            "frac": round(tfs / bf16, 4), "peak_source": peak_kind, "algorithmic_flops": flops}


def traffic_from_profiles(kernel_key: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel_key)
    if not ent:
        return None
    import hashlib
    src = os.path.join(ROOT, ent.get("source", ""))
    try:
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    if digest != ent.get("source_sha256_16"):
        return None
    return ent.get("bytes_per_launch")


# ---------------------------------------------------------------- GPU arm
def _dev_inputs(inp, dev):
    return {k: (v.to(dev).contiguous() if torch.is_tensor(v) else v) for k, v in inp.items()}


def rotation(w):
    """(input sets, bytes per set) of the L2 rotation of prefill workload w."""
    set_bytes = prefill_bytes(w)
    return min(16, max(2, math.ceil(3 * L2_BYTES / set_bytes))), set_bytes


def workload_config(w, n_ranks):
    """The ``config`` object of a line on prefill workload w (the same for
    both arms)."""
    n_sets, set_bytes = rotation(w)
    l2 = (f"inputs rotate over {n_sets} sets of {set_bytes / 2**20:.0f} MiB (> L2)"
          if n_sets * set_bytes > L2_BYTES else
          f"inputs rotate over {n_sets} sets of {set_bytes / 2**10:.0f} KiB (fit in L2)")
    return {"workload": w.name, "global_batch": w.B * n_ranks, "seq_len": w.L, "heads": w.H,
            "d_k": w.dk, "d_v": w.dv, "chunk": w.chunk, "phi": w.phi, "decay": w.decay,
            "initial_state": w.s0_std is not None,
            "parallelism": f"replicas{n_ranks}" if n_ranks > 1 else "single", "l2": l2}


def bench_prefill(w, steps, warmup, dev, peaks, peak_kind, min_warmup_s=1.0):
    from causal_linear_attention_chunkwise_gb300 import api
    api.la_set_feature_map(w.phi)
    host = W.make_prefill_inputs(w, seed=0)
    n_sets, set_bytes = rotation(w)
    sets = []
    for i in range(n_sets):
        d = _dev_inputs(host if i == 0 else W.make_prefill_inputs(w, seed=i), dev)
        d["O"] = torch.empty(w.B, w.H, w.L, w.dv, dtype=d["q"].dtype, device=dev)
        d["S"] = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)
        sets.append(d)
    ws_bytes = api.la_chunk_fwd_workspace_bytes(w.B, w.H, w.L, w.dk, w.dv, w.chunk, sets[0]["q"].dtype)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        s = sets[i % n_sets]
        api.la_chunk_fwd(s["q"], s["k"], s["v"], w.chunk, s["decay_kind"], s["decay"], s["S0"],
                         O=s["O"], S_final=s["S"], workspace=ws, stream=stream)

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    t0 = time.time()
    i = 0
    while i < warmup or time.time() - t0 < min_warmup_s:
        step(i)
        i += 1
        if i % 50 == 0:
            torch.cuda.synchronize(dev)
    api.la_device_status()
    barrier()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for j in range(steps):
        starts[j].record(stream)
        step(i + j)
        ends[j].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    api.la_device_status()
    elapsed_ms = starts[0].elapsed_time(ends[-1])
    per_call_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    kernels = api.la_chunk_fwd_kernel_count(w.B, w.H, w.L, w.dk, w.dv, w.chunk, sets[0]["q"].dtype)
    rl = roofline(prefill_bytes(w), prefill_flops(w), per_call_ms / 1e3, peaks, peak_kind, False)
    rl["kernel"] = "la_chunk_fwd call (all its kernels)"
    rl["traffic"] = traffic_from_profiles(f"prefill:{w.name}")
    return {"elapsed_ms": elapsed_ms, "per_call_ms": per_call_ms, "clocks": clocks,
            "roofline": rl, "gpu_launches": kernels * steps, "n_sets": n_sets,
            "set_bytes": set_bytes}


def noncausal_bytes(w) -> int:
    """Bytes the non-causal form must move: q, k, v read and O written once,
    and the state phi(K)^T V written."""
    e = ELT[w.dtype]
    n = w.B * w.H * w.L
    return n * (2 * w.dk + 2 * w.dv) * e + w.B * w.H * w.dk * w.dv * 4


def bench_noncausal(w, steps, warmup, dev, peaks, peak_kind):
    """la_noncausal_fwd on the shape (and phi) of prefill workload ``w``, its
    decay and initial state dropped: the form has neither."""
    from causal_linear_attention_chunkwise_gb300 import api
    api.la_set_feature_map(w.phi)
    set_bytes = noncausal_bytes(w)
    n_sets = min(16, max(2, math.ceil(3 * L2_BYTES / set_bytes)))
    sets = []
    for i in range(n_sets):
        d = _dev_inputs(W.make_prefill_inputs(w, seed=i), dev)
        d["O"] = torch.empty(w.B, w.H, w.L, w.dv, dtype=d["q"].dtype, device=dev)
        d["S"] = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)
        sets.append(d)
    ws = torch.empty(max(api.la_noncausal_fwd_workspace_bytes(w.B, w.H, w.L, w.dk, w.dv), 16),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        s = sets[i % n_sets]
        api.la_noncausal_fwd(s["q"], s["k"], s["v"], O=s["O"], S=s["S"], workspace=ws,
                             stream=stream)

    for i in range(warmup):
        step(i)
    api.la_device_status()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for j in range(steps):
        starts[j].record(stream)
        step(warmup + j)
        ends[j].record(stream)
    torch.cuda.synchronize(dev)
    api.la_device_status()
    per_call_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    flops = 4 * w.B * w.H * w.L * w.dk * w.dv  # phi(K)^T V and phi(Q) S
    rl = roofline(set_bytes, flops, per_call_ms / 1e3, peaks, peak_kind, False)
    rl["kernel"] = "la_noncausal_fwd call (all its kernels)"
    rl["traffic"] = traffic_from_profiles(f"noncausal:{w.name}")
    return per_call_ms, rl


def variant_bytes(form, w) -> int:
    """Bytes a further form must move at least: q, k, v read and O written once,
    its per-token gate inputs read, and the final state written."""
    e = ELT["bf16"]
    n = w.B * w.H * w.L
    per_token = {"normalised": 4, "channel_gate": 4 * w.dk, "delta": 8}[form]
    state = w.B * w.H * (w.dk * w.dv + (w.dk if form == "normalised" else 0)) * 4
    return n * ((2 * w.dk + 2 * w.dv) * e + per_token) + state


def bench_variants(w, steps, warmup, dev, peaks, peak_kind):
    """The normalised form, the per-channel gate and the delta rule, each on
    the shape of prefill workload ``w`` in bf16 (elu + 1 for the first two;
    identity with unit-norm keys for the delta rule).  One input set per form:
    these CUDA-core kernels are bound by arithmetic, not by HBM."""
    from causal_linear_attention_chunkwise_gb300 import api
    stream = torch.cuda.current_stream(dev)
    out = {}
    for form in ("normalised", "channel_gate", "delta"):
        inp = W.make_variant_inputs(form, w.B, w.H, w.L, w.dk, w.dv, "bf16", seed=0,
                                    with_state=True)
        d = {k: (v.to(dev) if hasattr(v, "to") else v) for k, v in inp.items()}
        if form == "normalised":
            api.la_set_feature_map("elu1")
            call = lambda: api.la_normalised_fwd(  # noqa: E731
                d["q"], d["k"], d["v"], 64, d["decay_kind"], d["decay"], d["S0"], d["z0"],
                stream=stream)
        elif form == "channel_gate":
            api.la_set_feature_map("elu1")
            call = lambda: api.la_channel_gate_fwd(  # noqa: E731
                d["q"], d["k"], d["v"], d["log_alpha"], 64, d["S0"], stream=stream)
        else:
            api.la_set_feature_map("identity")
            call = lambda: api.la_delta_fwd(  # noqa: E731
                d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["S0"], stream=stream)
        for _ in range(warmup):
            call()
        api.la_device_status()
        torch.cuda.synchronize(dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for j in range(steps):
            starts[j].record(stream)
            call()
            ends[j].record(stream)
        torch.cuda.synchronize(dev)
        api.la_device_status()
        ms = statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends))
        rl = roofline(variant_bytes(form, w), 0, ms / 1e3, peaks, peak_kind, False)
        out[form] = {"per_call_ms": round(ms, 4),
                     "tokens_per_s": w.B * w.L / (ms / 1e3), "roofline": rl}
    return out


def bench_prefill_e2e(w, steps, dev):
    """Same metric with host buffers: pinned Q/K/V (+gate, S0) copied in and
    O and S_final copied out inside the timed region, every step.  The
    copies are pipelined the way a streaming caller would run them: two sets
    of device buffers, inputs copied in on one stream while the previous
    step computes, results copied out on a third while the next step's
    inputs copy in.  The timed region runs from the first copy in to the
    last copy out."""
    from causal_linear_attention_chunkwise_gb300 import api
    api.la_set_feature_map(w.phi)
    host = W.make_prefill_inputs(w, seed=0)
    h_in = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in host.items()}
    names = [k for k in ("q", "k", "v", "decay", "S0") if torch.is_tensor(h_in.get(k))]
    comp = torch.cuda.current_stream(dev)
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = []
    for _ in range(2):
        d = _dev_inputs(host, dev)
        d["O"] = torch.empty(w.B, w.H, w.L, w.dv, dtype=d["q"].dtype, device=dev)
        d["S"] = torch.empty(w.B, w.H, w.dk, w.dv, dtype=torch.float32, device=dev)
        d["in_done"], d["comp_done"], d["out_done"] = (torch.cuda.Event() for _ in range(3))
        sets.append(d)
    O_h = torch.empty(sets[0]["O"].shape, dtype=sets[0]["O"].dtype, pin_memory=True)
    S_h = torch.empty(sets[0]["S"].shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(h_in[k].numel() * h_in[k].element_size() for k in names)
    d2h = O_h.numel() * O_h.element_size() + S_h.numel() * S_h.element_size()

    def step(i):
        d = sets[i % 2]
        cin.wait_event(d["comp_done"])  # step i - 2 has read this set's inputs
        with torch.cuda.stream(cin):
            for k in names:
                d[k].copy_(h_in[k], non_blocking=True)
        d["in_done"].record(cin)
        comp.wait_event(d["in_done"])
        comp.wait_event(d["out_done"])  # step i - 2's results have been copied out
        api.la_chunk_fwd(d["q"], d["k"], d["v"], w.chunk, d["decay_kind"], d["decay"], d["S0"],
                         O=d["O"], S_final=d["S"], stream=comp)
        d["comp_done"].record(comp)
        cout.wait_event(d["comp_done"])
        with torch.cuda.stream(cout):
            O_h.copy_(d["O"], non_blocking=True)
            S_h.copy_(d["S"], non_blocking=True)
        d["out_done"].record(cout)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(dev)
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cin)
    for i in range(steps):
        step(3 + i)
    b.record(cout)
    torch.cuda.synchronize(dev)
    barrier()
    api.la_device_status()
    return a.elapsed_time(b), h2d, d2h


def bench_decode(steps, warmup, dev, peaks, peak_kind):
    from causal_linear_attention_chunkwise_gb300 import api
    w = W.DECODE[DECODE_WORKLOAD]
    api.la_set_feature_map(w.phi)
    n_in = min(w.steps, 16)
    inp = W.make_decode_inputs(w, seed=0, steps=n_in)
    S = inp["S0"].to(dev)
    q, k, v, la = (inp[x].to(dev) for x in ("q", "k", "v", "log_alpha"))
    o = torch.empty(w.B, w.H, w.dv, dtype=q.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        t = i % n_in
        api.la_decode_step(q[t], k[t], v[t], S, la[t], o=o, stream=stream)

    for i in range(max(warmup, 3)):
        step(i)
    torch.cuda.synchronize(dev)
    barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for j in range(steps):
        starts[j].record(stream)
        step(j)
        ends[j].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    api.la_device_status()
    elapsed_ms = starts[0].elapsed_time(ends[-1])
    per_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    rl = roofline(decode_bytes(w), 5 * w.B * w.H * w.dk * w.dv, per_ms / 1e3, peaks, peak_kind,
                  False)
    rl["kernel"] = "decode_kernel"
    rl["traffic"] = traffic_from_profiles(f"decode:{w.name}")
    return w, elapsed_ms, per_ms, rl


# ---------------------------------------------------------------- CPU oracle
def cpu_oracle_prefill_sample(w, inp, budget_s=8.0):
    """Time the oracle on whole (b, h) sequences of the workload until about
    ``budget_s`` seconds; returns (tokens/s, description, threads)."""
    import oracle
    nseq = w.B * w.H
    order = [(b, h) for b in range(w.B) for h in range(w.H)]
    t_start = time.perf_counter()
    done = 0
    batch = max(1, min(nseq, oracle.num_threads()))
    while done < nseq and time.perf_counter() - t_start < budget_s:
        chunk_pairs = order[done:done + batch]
        bs = sorted({b for b, _ in chunk_pairs})
        for b in bs:
            hs = [h for bb, h in chunk_pairs if bb == b]
            h0, h1 = min(hs), max(hs) + 1
            dec = inp["decay"]
            if inp["decay_kind"] == "head":
                dec = dec[h0:h1]
            elif dec is not None:
                dec = dec[b:b + 1, h0:h1]
            s0 = None if inp["S0"] is None else inp["S0"][b:b + 1, h0:h1]
            oracle.recurrent(inp["q"][b:b + 1, h0:h1], inp["k"][b:b + 1, h0:h1],
                             inp["v"][b:b + 1, h0:h1], phi=w.phi, decay_kind=inp["decay_kind"],
                             decay=dec, S0=s0)
        done += len(chunk_pairs)
    el = time.perf_counter() - t_start
    tokens = done * w.L / w.H  # head-sequences -> batch tokens (all heads of a token = 1)
    desc = (f"{done} of {nseq} (b,h) sequences of {w.L} tokens (fp64 recurrence), "
            f"tokens counted as head-tokens / H")
    return tokens / el, desc, oracle.num_threads(), el


def cpu_oracle_decode_sample(w, budget_s=6.0):
    import oracle
    n_states = 1024
    inp = W.make_decode_inputs(W.DecodeWorkload("sample", n_states // w.H, w.H, w.dk, w.dv, 4,
                                                w.dtype, w.phi, w.scale), seed=0, steps=4)
    t0 = time.perf_counter()
    reps = 0
    while reps == 0 or time.perf_counter() - t0 < budget_s:
        oracle.decode(inp["q"], inp["k"], inp["v"], inp["S0"], inp["log_alpha"], phi=w.phi)
        reps += 1
    el = time.perf_counter() - t0
    tokens = reps * 4 * n_states / w.H
    return tokens / el, f"{n_states} (b,h) states x 4 steps x {reps} repeats", el


# ---------------------------------------------------------------- arms
def prefill_leg(w, steps, warmup, dev, peaks, peak_kind, n_ranks, min_warmup_s):
    """One prefill workload's sub-object: time, throughput, roofline, clocks."""
    r = bench_prefill(w, steps, warmup, dev, peaks, peak_kind, min_warmup_s=min_warmup_s)
    el_max = max_over_ranks(r["elapsed_ms"], dev)
    return r, {"workload": w.name, "dtype": w.dtype,
               "value": round(aggregate(w.tokens, steps, el_max, n_ranks), 1),
               "unit": "tokens/s", "ms_per_step": round(el_max / steps, 5),
               "per_call_ms": round(r["per_call_ms"], 5), "roofline": r["roofline"],
               "gpu_launches": r["gpu_launches"], "clocks": r["clocks"],
               "config": workload_config(w, n_ranks)}


def run_gpu_arm(args):
    rank, ws = init_dist()
    _, _, local = world()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from causal_linear_attention_chunkwise_gb300 import api  # noqa: F401  (loads the library)
    peaks, peak_kind = load_peaks()
    w = W.PREFILL[args.workload]
    res, head = prefill_leg(w, args.steps, args.warmup, dev, peaks, peak_kind, ws, 1.0)
    el_max = max_over_ranks(res["elapsed_ms"], dev)
    value = aggregate(w.tokens, args.steps, el_max, ws)
    e2e_ms, h2d, d2h = bench_prefill_e2e(w, args.steps, dev)
    e2e_max = max_over_ranks(e2e_ms, dev)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, ws),
        "clocks": res["clocks"],
        "e2e": {"value": round(aggregate(w.tokens, args.steps, e2e_max, ws), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": res["gpu_launches"],
        "roofline": res["roofline"],
    }
    if args.legs == "all":
        legs = {}
        for name in SUB_LEGS:
            if name == w.name:
                continue
            _, legs[name] = prefill_leg(W.PREFILL[name], args.steps, args.warmup, dev, peaks,
                                        peak_kind, ws, 0.3)
        line["legs"] = legs
    dw, d_el, d_per, d_rl = bench_decode(args.decode_steps, args.warmup, dev, peaks, peak_kind)
    d_max = max_over_ranks(d_el, dev)
    line["decode"] = {"workload": dw.name,
                      "value": round(aggregate(dw.B, args.decode_steps, d_max, ws), 1),
                      "unit": "tokens/s", "steps": args.decode_steps,
                      "ms_per_step": round(d_max / args.decode_steps, 5), "roofline": d_rl,
                      "gpu_launches": args.decode_steps}
    if args.legs == "all":
        nc = {}
        for name in NONCAUSAL_LEGS:
            nw = W.PREFILL[name]
            per, rl = bench_noncausal(nw, args.steps, args.warmup, dev, peaks, peak_kind)
            nc[name] = {"per_call_ms": round(per, 5), "unit": "tokens/s",
                        "value": round(nw.tokens / (per / 1e3), 1), "roofline": rl}
        line["noncausal"] = nc
        vw = W.PREFILL[VARIANT_SHAPE]
        line["variants"] = {"shape": vw.name, "dtype": "bf16",
                            **bench_variants(vw, args.steps, args.warmup, dev, peaks, peak_kind)}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        inp = W.make_prefill_inputs(w, seed=0)
        tps, desc, cores, _ = cpu_oracle_prefill_sample(w, inp)
        line["cpu_baseline"] = {"value": round(tps, 1), "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "sample": desc,
                                "cpu": _cpu_name()}
        dtps, ddesc, _ = cpu_oracle_decode_sample(dw)
        line["decode"]["cpu_baseline"] = {"value": round(dtps, 1), "unit": "tokens/s",
                                          "cores": cores, "kind": "oracle", "sample": ddesc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


def run_profile(args):
    """One leg only, W warm-up and K timed steps, no minimum warm-up time: the
    command the committed ncu summaries are taken with."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks, peak_kind = load_peaks()
    if args.profile == "prefill":
        w = W.PREFILL[args.workload]
        r = bench_prefill(w, args.steps, args.warmup, dev, peaks, peak_kind, min_warmup_s=0.0)
        print(json.dumps({"profile": "prefill", "workload": w.name,
                          "per_call_ms": round(r["per_call_ms"], 5), "roofline": r["roofline"]}))
    elif args.profile == "noncausal":
        w = W.PREFILL[args.workload]
        per, rl = bench_noncausal(w, args.steps, args.warmup, dev, peaks, peak_kind)
        print(json.dumps({"profile": "noncausal", "workload": w.name, "per_call_ms": round(per, 5),
                          "roofline": rl}))
    elif args.profile == "variants":
        w = W.PREFILL[args.workload]
        r = bench_variants(w, args.steps, args.warmup, dev, peaks, peak_kind)
        print(json.dumps({"profile": "variants", "workload": w.name, "dtype": "bf16", **r}))
    else:
        dw, _, per, rl = bench_decode(args.steps, args.warmup, dev, peaks, peak_kind)
        print(json.dumps({"profile": "decode", "workload": dw.name, "per_step_ms": round(per, 5),
                          "roofline": rl}))


def _cpu_name():
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


def run_reference_arm(args):
    rank, ws, _ = world()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = W.PREFILL[args.workload]
    inp = W.make_prefill_inputs(w, seed=0)
    budget = 2.0
    for _ in range(args.warmup):
        cpu_oracle_prefill_sample(w, inp, budget_s=0.5)
    rates, secs = [], []
    desc, cores = "", 1
    for _ in range(args.steps):
        tps, desc, cores, el = cpu_oracle_prefill_sample(w, inp, budget_s=budget)
        rates.append(tps)
        secs.append(el)
    value = statistics.mean(rates)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(secs), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": workload_config(w, ws),
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": "each step: " + desc, "cpu": _cpu_name()},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--decode-steps", type=int, default=64)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.PREFILL))
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--legs", choices=["main", "all"], default="all",
                   help="main: the headline workload and decode only; all: also the other "
                        "prefill workloads, the non-causal form and the further forms")
    p.add_argument("--profile", choices=["prefill", "decode", "noncausal", "variants"], default=None,
                   help="run one leg only (for ncu captures); prints no benchmark line")
    args = p.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference_arm(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
