"""Shared helpers for the GPU parity tests: run a workload through the C ABI
(via the thin binding) and through the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from causal_linear_attention_chunkwise_gb300 import api


def to_dev(x, dev="cuda"):
    return None if x is None else x.to(dev).contiguous()


def gpu_prefill(inp, phi, chunk=64, **kw):
    api.la_set_feature_map(phi)
    O, Sf = api.la_chunk_fwd(to_dev(inp["q"]), to_dev(inp["k"]), to_dev(inp["v"]), chunk,
                             inp["decay_kind"], to_dev(inp["decay"]), to_dev(inp["S0"]), **kw)
    api.la_device_status()
    return O.cpu(), None if Sf is None else Sf.cpu()


def oracle_prefill(inp, phi, pairs=None):
    """Oracle O and S_final; with ``pairs`` (a list of (b, h)) only those
    sequences, each run on its own, stacked in the order given."""
    q, k, v, dec, S0, kind = inp["q"], inp["k"], inp["v"], inp["decay"], inp["S0"], inp["decay_kind"]
    if pairs is None:
        return oracle.recurrent(q, k, v, phi=phi, decay_kind=kind, decay=dec, S0=S0)
    Os, Ss = [], []
    for b, h in pairs:
        d = None
        if kind == "head":
            d = dec[h:h + 1]
        elif kind in ("token", "logit"):
            d = dec[b:b + 1, h:h + 1]
        s0 = None if S0 is None else S0[b:b + 1, h:h + 1]
        O, S = oracle.recurrent(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                phi=phi, decay_kind=kind, decay=d, S0=s0)
        Os.append(O[0, 0])
        Ss.append(S[0, 0])
    return np.stack(Os), np.stack(Ss)


def select_pairs(x, pairs):
    return np.stack([x[b, h].double().numpy() for b, h in pairs])
