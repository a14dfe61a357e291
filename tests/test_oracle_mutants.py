"""Plant plausible mistakes in a copy of the oracle's C source and check that
the pins catch every one.  Runs on the CPU only; the real oracle source is
never modified."""
import os

import pytest

import oracle
from tests.oracle_pins import PINS

with open(os.path.join(os.path.dirname(oracle.__file__), "la_oracle.c")) as _f:
    SRC = _f.read()

_UPDATE = (
    "            for (int i = 0; i < dk; ++i)\n"
    "                for (int j = 0; j < dv; ++j)\n"
    "                    S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + kf[i] * vt[j];\n")
_READ = (
    "            for (int i = 0; i < dk; ++i) qf[i] = feature(phi, qt[i]);\n"
    "            double *ot = O + ((size_t)bh * L + t) * dv;\n"
    "            for (int j = 0; j < dv; ++j) {\n"
    "                double acc = 0.0;\n"
    "                for (int i = 0; i < dk; ++i) acc += qf[i] * S[(size_t)i * dv + j];\n"
    "                ot[j] = acc;\n"
    "            }\n")

# (name, text in la_oracle.c, replacement): each a mistake someone could make
# while writing the oracle from the pages.
MUTANTS = [
    ("read_before_update", _UPDATE + _READ, _READ + _UPDATE),
    ("decay_scales_new_write",
     "S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + kf[i] * vt[j];",
     "S[(size_t)i * dv + j] = a * (S[(size_t)i * dv + j] + kf[i] * vt[j]);"),
    ("transposed_state_read",
     "for (int i = 0; i < dk; ++i) acc += qf[i] * S[(size_t)i * dv + j];",
     "for (int i = 0; i < dk; ++i) acc += qf[i] * S[(size_t)j * dk + i];"),
    ("elu_branch_plus_one",
     "return x > 0.0 ? x + 1.0 : exp(x);",
     "return x > 0.0 ? x + 1.0 : exp(x) + 1.0;"),
    ("elu_threshold_wrong_side",
     "return x > 0.0 ? x + 1.0 : exp(x);",
     "return x > 0.0 ? exp(x) : x + 1.0;"),
    ("softplus_wrong_branch",
     "return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));",
     "return x > 0.0 ? log1p(exp(-x)) : log1p(exp(x));"),
    ("gate_sign",
     "case 3: return -softplus(decay[((size_t)b * H + h) * L + t]);",
     "case 3: return softplus(-decay[((size_t)b * H + h) * L + t]);"),
    ("head_decay_wrong_index",
     "case 1: return decay[h];",
     "case 1: return decay[b];"),
    ("initial_state_ignored",
     "        if (S0) memcpy(S, S0 + (size_t)bh * dk * dv, sizeof(double) * (size_t)dk * dv);\n"
     "        else memset(S, 0, sizeof(double) * (size_t)dk * dv);\n"
     "        for (int t = 0; t < L; ++t) {",
     "        memset(S, 0, sizeof(double) * (size_t)dk * dv);\n"
     "        for (int t = 0; t < L; ++t) {"),
    ("q_used_as_key",
     "for (int i = 0; i < dk; ++i) kf[i] = feature(phi, kt[i]);",
     "for (int i = 0; i < dk; ++i) kf[i] = feature(phi, qt[i]);"),
    ("parallel_exclusive_cumsum",
     "            run += log_decay(kind, decay, H, L, b, h, t);\n            cum[t] = run;",
     "            cum[t] = run;\n            run += log_decay(kind, decay, H, L, b, h, t);"),
    ("parallel_strict_mask",
     "for (int s = 0; s <= t; ++s) {",
     "for (int s = 0; s < t; ++s) {"),
    ("parallel_initial_state_undecayed",
     "double e = exp(cum[t]);",
     "double e = 1.0;"),
    ("chunk_inter_undecayed",
     "double e = exp(lam[i]);",
     "double e = 1.0;"),
    ("chunk_state_weight_wrong",
     "double w = exp(lam[n - 1] - lam[jj]);",
     "double w = exp(-lam[jj]);"),
    ("chunk_state_not_decayed",
     "for (size_t x = 0; x < (size_t)dk * dv; ++x) S[x] *= eEnd;",
     "for (size_t x = 0; x < (size_t)dk * dv; ++x) S[x] *= 1.0;"),
    ("chunk_intra_excludes_diagonal",
     "for (int jj = 0; jj <= i; ++jj) {",
     "for (int jj = 0; jj < i; ++jj) {"),
    ("noncausal_state_transposed",
     "for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += f[i] * vt[j];",
     "for (int j = 0; j < dv; ++j) S[(size_t)j * dk + i] += f[i] * vt[j];"),
    ("noncausal_phi_not_on_q",
     "for (int i = 0; i < dk; ++i) f[i] = feature(phi, qt[i]);",
     "for (int i = 0; i < dk; ++i) f[i] = qt[i];"),
    ("normaliser_not_decayed",
     "z[i] = a * z[i] + kf[i];",
     "z[i] = z[i] + kf[i];"),
    ("normaliser_uses_key",
     "for (int i = 0; i < dk; ++i) den += qf[i] * z[i];",
     "for (int i = 0; i < dk; ++i) den += kf[i] * z[i];"),
    ("channel_gate_one_channel",
     "const double a = exp(la[i]);",
     "const double a = exp(la[0]);"),
    ("delta_gate_on_write",
     "S[(size_t)i * dv + j] = a * (S[(size_t)i * dv + j] - bt * kf[i] * ks[j]) +\n"
     "                                            bt * kf[i] * vt[j];",
     "S[(size_t)i * dv + j] = a * (S[(size_t)i * dv + j] - bt * kf[i] * ks[j] +\n"
     "                                            bt * kf[i] * vt[j]);"),
    ("delta_no_erase",
     "a * (S[(size_t)i * dv + j] - bt * kf[i] * ks[j])",
     "a * (S[(size_t)i * dv + j])"),
    ("delta_write_without_beta",
     "                                            bt * kf[i] * vt[j];",
     "                                            kf[i] * vt[j];"),
    ("delta_chunk_solve_includes_diagonal",
     "                    for (int i = 0; i < t; ++i) {\n"
     "                        double kk = 0.0;",
     "                    for (int i = 0; i <= t; ++i) {\n"
     "                        double kk = 0.0;"),
    ("delta_chunk_rhs_state_not_decayed",
     "double acc = v[row * dv + j] - et * kS;",
     "double acc = v[row * dv + j] - kS;"),
    ("delta_chunk_output_excludes_own_write",
     "                    for (int i = 0; i <= t; ++i) {\n"
     "                        double qk = 0.0;",
     "                    for (int i = 0; i < t; ++i) {\n"
     "                        double qk = 0.0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    assert SRC.count(old) >= 1, f"mutant {name}: pattern not found in la_oracle.c"
    src = tmp_path / f"{name}.c"
    src.write_text(SRC.replace(old, new, 1))
    so = oracle.compile_library(str(src), str(tmp_path / f"lib{name}.so"))
    lib = oracle.load_library(so)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError as e:
            caught.append(f"{pin.__name__}: {str(e).splitlines()[0][:80]}")
    assert caught, f"no pin caught the planted mistake {name!r}"
