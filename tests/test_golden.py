"""The oracle against its stored golden fixtures (written by tests/golden/make_golden.py,
which calls only the oracle).  Guards the oracle and the generator against drift."""
import json
import os

import numpy as np
import pytest

import oracle
from synthetic import prefill_inputs
from golden.make_golden import CASES

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name", sorted(CASES))
def test_golden(name):
    with open(os.path.join(HERE, name + ".json")) as f:
        fx = json.load(f)
    w = CASES[name]()
    assert w.name == fx["workload"] and w.seqlens == fx["seqlens"]
    d = prefill_inputs(w)
    out, sf = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                             d["cu_seqlens"], d["initial_state"])
    # Different libm builds may round exp() differently in the last place.
    assert np.isclose(np.linalg.norm(out), fx["out_norm"], rtol=1e-11, atol=0)
    assert np.isclose(np.linalg.norm(sf), fx["state_norm"], rtol=1e-11, atol=0)
    for idx, val in fx["out_samples"]:
        assert np.isclose(out[tuple(idx)], float(val), rtol=1e-9, atol=1e-13), idx
    for idx, val in fx["state_samples"]:
        assert np.isclose(sf[tuple(idx)], float(val), rtol=1e-9, atol=1e-13), idx
