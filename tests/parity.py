"""Shared helpers for the GPU-vs-oracle parity tests.

Tolerances (relative L2 over a whole tensor, outputs and final state
separately; max-abs over outputs): fp32 inputs rel-L2 <= 1e-4; bf16 inputs
with fp32 state rel-L2 <= 1e-2 and max-abs <= 2e-2 on outputs.
"""
import numpy as np
import torch

TOL = {"f32": {"rel": 1e-4, "abs": 2e-2}, "bf16": {"rel": 1e-2, "abs": 2e-2}}


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    return float(num / den) if den > 0 else float(num)


def max_abs(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(x - ref))) if x.size else 0.0


def host(t):
    return t.detach().to("cpu", torch.float64).numpy()


# Margins of the named workloads' comparisons, printed in pytest's terminal
# summary (tests/conftest.py): (name, output rel-L2, output max-abs, state rel-L2).
MARGINS = []


def record_margin(name, out_rel, out_max, state_rel):
    MARGINS.append((name, out_rel, out_max, state_rel))


def check_margins(name, out_rel, out_max, state_rel, dtype):
    """Assert already-reduced errors against the tolerances and record them."""
    tol = TOL[dtype]
    record_margin(name, out_rel, out_max, state_rel)
    if out_rel is not None:
        assert out_rel <= tol["rel"], f"{name}: output rel-L2 {out_rel:.3e} > {tol['rel']}"
        assert out_max <= tol["abs"], f"{name}: output max-abs {out_max:.3e} > {tol['abs']}"
    if state_rel is not None:
        assert state_rel <= tol["rel"], f"{name}: state rel-L2 {state_rel:.3e} > {tol['rel']}"


def assert_parity(name, out, ref_out, state, ref_state, dtype):
    tol = TOL[dtype]
    e_o = m_o = e_s = None
    if ref_out is not None and np.size(ref_out):
        e_o = rel_l2(out, ref_out)
        m_o = max_abs(out, ref_out)
        assert np.all(np.isfinite(out)), f"{name}: non-finite outputs"
    if ref_state is not None:
        e_s = rel_l2(state, ref_state)
        assert np.all(np.isfinite(state)), f"{name}: non-finite state"
    record_margin(name, e_o, m_o, e_s)
    if e_o is not None:
        assert e_o <= tol["rel"], f"{name}: output rel-L2 {e_o:.3e} > {tol['rel']}"
        assert m_o <= tol["abs"], f"{name}: output max-abs {m_o:.3e} > {tol['abs']}"
    if e_s is not None:
        assert e_s <= tol["rel"], f"{name}: state rel-L2 {e_s:.3e} > {tol['rel']}"


def to_device(d, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
