"""The fp64 oracle against its pins (hand-worked values, closed forms, library
routines, the pages' own equalities).  CPU only."""
import pytest

import oracle
from tests.oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.load_library())


def test_decode_is_recurrence_along_steps():
    """Decode steps equal the token recurrence with the step axis as tokens."""
    import numpy as np
    r = np.random.default_rng(11)
    steps, B, H, d = 5, 2, 3, 4
    q, k, v = r.normal(size=(steps, B, H, d)), r.normal(size=(steps, B, H, d)), r.normal(size=(steps, B, H, d))
    la = np.log(r.uniform(0.9, 1.0, size=(steps, B, H)))
    S0 = r.normal(size=(B, H, d, d))
    o, S = oracle.decode(q, k, v, S0, la, phi="elu1")
    # one step at a time, carrying the state
    Sc = S0
    for t in range(steps):
        ot, Sc = oracle.decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], Sc, la[t:t + 1], phi="elu1")
        assert np.allclose(ot[0], o[t], rtol=0, atol=1e-12)
    assert np.allclose(Sc, S, rtol=0, atol=1e-12)


def test_bad_arguments_rejected():
    import numpy as np
    lib = oracle.load_library()
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.recurrent(q, q, q, decay_kind="head", decay=None)
    with pytest.raises(RuntimeError):
        oracle.chunkwise(q, q, q, 0, lib=lib)
