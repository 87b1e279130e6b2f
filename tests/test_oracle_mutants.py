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
    # reverse mode
    ("bwd_dk_misses_erase_path", "B->dk_[((size_t)t * H + h) * dk + i] = bt * a - b;",
     "B->dk_[((size_t)t * H + h) * dk + i] = bt * a;"),
    ("bwd_dSp_sign", "dSp[(size_t)i * dv + j] = dS[(size_t)i * dv + j] - kt[i] * de[j];",
     "dSp[(size_t)i * dv + j] = dS[(size_t)i * dv + j] + kt[i] * de[j];"),
    ("bwd_state_grad_not_decayed", "dS[(size_t)i * dv + j] = alpha[i] * dSp[(size_t)i * dv + j];",
     "dS[(size_t)i * dv + j] = dSp[(size_t)i * dv + j];"),
    ("bwd_dq_from_previous_state", "acc += St[(size_t)i * dv + j] * dot[j];",
     "acc += Sprev[(size_t)i * dv + j] * dot[j];"),
    ("bwd_dlog_alpha_without_alpha", "B->dla[((size_t)t * H + h) * dk + i] = alpha[i] * a;",
     "B->dla[((size_t)t * H + h) * dk + i] = a;"),
    ("bwd_dbeta_uses_value", "db += err[j] * a;", "db += vt[j] * a;"),
    ("bwd_checkpoint_off_by_one", "memcpy(cp + SZ * (size_t)((r + 1) / kCheckpoint), cur, sizeof(double) * SZ);",
     "memcpy(cp + SZ * (size_t)((r + 1) / kCheckpoint), nxt, sizeof(double) * SZ);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    # the forward formulas appear in the prefill and again in the reverse mode's
    # recomputation; a slip is planted everywhere its text appears
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
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
