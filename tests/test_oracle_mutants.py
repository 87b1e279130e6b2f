"""Plant plausible mistakes in a copy of the oracle's C source (on the CPU)
and check that every one of them is caught by at least one pin."""
import os

import pytest

import oracle
from pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, original text, replacement) -- each a single plausible slip.
MUTANTS = [
    ("dropped_beta", "const double bk = bt * kt[i];", "const double bk = kt[i];"),
    ("erase_against_undecayed_state",
     "pred += kt[i] * S[(size_t)i * dv + j];", "pred += kt[i] * S[(size_t)i * dv + j] / alpha[i];"),
    ("output_before_write",
     "o += qt[i] * S[(size_t)i * dv + j];", "o += qt[i] * (S[(size_t)i * dv + j] - bt * kt[i] * err[j]);"),
    ("decay_sign", "alpha[i] = exp(lat[i]);", "alpha[i] = exp(-lat[i]);"),
    ("decay_columns_not_rows", "S[(size_t)i * dv + j] *= alpha[i];",
     "S[(size_t)i * dv + j] *= alpha[j < dk ? j : i];"),
    ("no_decay", "S[(size_t)i * dv + j] *= alpha[i];", "S[(size_t)i * dv + j] *= 1.0;"),
    ("write_value_not_error", "S[(size_t)i * dv + j] += bk * err[j];",
     "S[(size_t)i * dv + j] += bk * vt[j];"),
    ("error_sign", "err[j] = vt[j] - pred;", "err[j] = pred - vt[j];"),
    ("initial_state_ignored", "J->s0 ? J->s0[sbase + (size_t)i * dv + j] : 0.0", "0.0"),
    ("read_with_key", "o += qt[i] * S[(size_t)i * dv + j];", "o += kt[i] * S[(size_t)i * dv + j];"),
    ("gate_from_previous_token", "const double *lat = J->la + ((size_t)t * H + h) * dk;",
     "const double *lat = J->la + ((size_t)(t > t0 ? t - 1 : t) * H + h) * dk;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mpath), out=str(tmp_path / f"lib{name}.so"))
    O = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(O)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
