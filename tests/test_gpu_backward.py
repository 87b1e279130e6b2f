"""Reverse mode of the prefill (kda_prefill_backward) on the GPU against the
fp64 oracle's reverse mode, which is itself pinned by finite differences."""
import numpy as np
import pytest
import torch

import oracle
from parity import host, rel_l2, to_device
from synthetic import custom, prefill_inputs

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "beta")
TOL = 1e-4      # fp32 arithmetic on the GPU against fp64, on the same (rounded) inputs


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


def _cotangents(d, seed, dtype):
    """Seeded dLoss/dout (in the input dtype) and dLoss/dfinal_state (fp32)."""
    g = torch.Generator().manual_seed(seed)
    T, H, dv = d["v"].shape
    N = d["cu_seqlens"].numel() - 1
    dk = d["k"].shape[2]
    do = torch.randn((T, H, dv), generator=g, dtype=torch.float64).to(d["q"].dtype)
    dfin = torch.randn((N, H, dk, dv), generator=g, dtype=torch.float64).float()
    return do, dfin


def _compare(kda, d, do, dfin, what, with_init=True):
    g = to_device(d)
    got = kda.prefill_backward(*(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], d_out=do.cuda(),
                               d_final_state=None if dfin is None else dfin.cuda(), want_initial_grad=with_init)
    torch.cuda.synchronize()
    ref = oracle.backward(*(d[n] for n in NAMES), d["cu_seqlens"], d["initial_state"], do,
                          None if dfin is None else dfin)
    keys = ["dq", "dk", "dv", "dlog_alpha", "dbeta"] + (["d_initial_state"] if with_init else [])
    for key in keys:
        rk = "dinitial_state" if key == "d_initial_state" else key
        err = rel_l2(host(got[key]), ref[rk])
        assert err <= TOL, f"{what}: {key} rel-L2 {err:.3e}"
    return got


@pytest.mark.parametrize("dtype,dim", [("f32", 64), ("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_backward_ragged_varlen(kda, dtype, dim):
    lens = [0, 1, 9, 8, 17, 70]
    d = prefill_inputs(custom(110 + dim, lens, 2, dim, dtype))
    do, dfin = _cotangents(d, 1, dtype)
    _compare(kda, d, do, dfin, f"varlen {dtype} d{dim}")


def test_backward_without_state_gradients(kda):
    d = prefill_inputs(custom(115, [100, 33], 3, 128, "bf16"))
    do, _ = _cotangents(d, 2, "bf16")
    _compare(kda, d, do, None, "no dfinal, no d_initial_state", with_init=False)


def test_backward_zero_initial_state(kda):
    d = prefill_inputs(custom(116, [130], 2, 64, "f32", state_std=None))
    do, dfin = _cotangents(d, 3, "f32")
    _compare(kda, d, do, dfin, "zero initial state")


def test_backward_scalar_gate(kda):
    d = prefill_inputs(custom(117, [50, 0, 77], 2, 128, "bf16", gate="scalar"))
    do, dfin = _cotangents(d, 4, "bf16")
    got = _compare(kda, d, do, dfin, "scalar gate")
    assert tuple(got["dlog_alpha"].shape) == (127, 2)


def test_backward_long_sequence(kda):
    """1,000 tokens: many kept-state blocks; strong and weak decay."""
    d = prefill_inputs(custom(118, [1000], 2, 128, "bf16", la_lo=0.0001, la_hi=0.3))
    do, dfin = _cotangents(d, 5, "bf16")
    _compare(kda, d, do, dfin, "1000 tokens")


def test_backward_deterministic(kda):
    d = prefill_inputs(custom(119, [300, 45], 4, 128, "bf16"))
    do, dfin = _cotangents(d, 6, "bf16")
    g = to_device(d)
    args = [g[n] for n in NAMES]
    a = kda.prefill_backward(*args, g["cu_seqlens"], g["initial_state"], d_out=do.cuda(), d_final_state=dfin.cuda())
    b = kda.prefill_backward(*args, g["cu_seqlens"], g["initial_state"], d_out=do.cuda(), d_final_state=dfin.cuda())
    torch.cuda.synchronize()
    for key in a:
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("nseq,heads", [(10, 2), (20, 2), (4, 2)])
def test_backward_tile_widths(kda, nseq, heads):
    """Sequence x head counts that select 16-, 32- and 8-column tiles."""
    lens = [(7 * i + 5) % 37 + 1 for i in range(nseq)]
    d = prefill_inputs(custom(120 + nseq, lens, heads, 128, "bf16"))
    do, dfin = _cotangents(d, 7, "bf16")
    _compare(kda, d, do, dfin, f"{nseq} sequences x {heads} heads")
