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


def assert_parity(name, out, ref_out, state, ref_state, dtype):
    tol = TOL[dtype]
    if ref_out is not None and np.size(ref_out):
        e = rel_l2(out, ref_out)
        m = max_abs(out, ref_out)
        assert np.all(np.isfinite(out)), f"{name}: non-finite outputs"
        assert e <= tol["rel"], f"{name}: output rel-L2 {e:.3e} > {tol['rel']}"
        assert m <= tol["abs"], f"{name}: output max-abs {m:.3e} > {tol['abs']}"
    if ref_state is not None:
        e = rel_l2(state, ref_state)
        assert np.all(np.isfinite(state)), f"{name}: non-finite state"
        assert e <= tol["rel"], f"{name}: state rel-L2 {e:.3e} > {tol['rel']}"


def to_device(d, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
