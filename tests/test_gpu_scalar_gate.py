"""The scalar (Gated DeltaNet) gate on the GPU: log_alpha [T, H], one value per
token and head, through the C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, host, to_device
from synthetic import custom, initial_state, prefill_inputs

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


def _prefill(kda, d, flags=0):
    g = to_device(d)
    assert g["log_alpha"].dim() == 2
    out, sf, _ = kda.prefill(*(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], flags=flags)
    torch.cuda.synchronize()
    return out, sf


def _oracle(d):
    return oracle.prefill(*(d[n] for n in NAMES), d["cu_seqlens"], d["initial_state"])


@pytest.mark.parametrize("dtype,dim,flags", [("bf16", 128, 0), ("bf16", 128, 1), ("bf16", 64, 0),
                                             ("f32", 128, 0), ("f32", 64, 0)])
def test_scalar_gate_ragged_varlen(kda, dtype, dim, flags):
    lens = [0, 1, 63, 64, 65, 130, 0, 257]
    d = prefill_inputs(custom(70 + dim, lens, 3, dim, dtype, gate="scalar"))
    out, sf = _prefill(kda, d, flags)
    ro, rs = _oracle(d)
    assert_parity(f"scalar gate {dtype} d{dim} flags {flags}", host(out), ro, host(sf), rs, dtype)


def test_scalar_gate_equals_broadcast_channel_gate(kda):
    """The scalar gate and the per-channel gate holding the same value in every
    channel run the same arithmetic: bit-identical results."""
    d = prefill_inputs(custom(72, [500, 77], 4, 128, "bf16", gate="scalar"))
    out1, sf1 = _prefill(kda, d)
    g = to_device(d)
    la3 = g["log_alpha"][:, :, None].expand(-1, -1, 128).contiguous()
    out2, sf2, _ = kda.prefill(g["q"], g["k"], g["v"], la3, g["beta"], g["cu_seqlens"], g["initial_state"])
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(sf1, sf2)


def test_scalar_gate_strong_decay(kda):
    """Scalar gates strong enough (log alpha ~ -U(0.5, 5)) that full chunks take
    the tensor-core kernel's CUDA-core Gram path, while the short tail chunks
    (8 and 2 tokens) stay on the fast path."""
    d = prefill_inputs(custom(75, [200, 64, 130], 2, 128, "bf16", la_lo=0.5, la_hi=5.0, gate="scalar"))
    out, sf = _prefill(kda, d)
    ro, rs = _oracle(d)
    assert np.isfinite(host(out)).all() and np.isfinite(host(sf)).all()
    assert_parity("scalar gate, strong decay", host(out), ro, host(sf), rs, "bf16")


def test_scalar_gate_segment_scan(kda):
    """A long sequence (split into segments) with the scalar gate."""
    d = prefill_inputs(custom(73, [16384 + 100], 2, 128, "bf16", la_lo=0.0001, la_hi=0.05, gate="scalar"))
    out, sf = _prefill(kda, d)
    ro, rs = _oracle(d)
    assert_parity("scalar gate, segment scan", host(out), ro, host(sf), rs, "bf16")


@pytest.mark.parametrize("dtype,dim", [("bf16", 128), ("f32", 64)])
def test_scalar_gate_decode(kda, dtype, dim):
    w = custom(74, [1] * 6, 4, dim, dtype, gate="scalar")
    s0 = initial_state(w, 6)
    s_gpu = s0.cuda().contiguous()
    s_ref = s0.double().numpy()
    for step in range(5):
        x = prefill_inputs(custom(80 + step, [1] * 6, 4, dim, dtype, gate="scalar"))
        assert x["log_alpha"].shape == (6, 4)
        o = kda.decode_step(*(x[n].cuda() for n in NAMES), s_gpu)
        ro, s_ref = oracle.decode_step(*(x[n] for n in NAMES), s_ref)
        torch.cuda.synchronize()
        assert_parity(f"scalar-gate decode {dtype} d{dim} step {step}", host(o), ro, host(s_gpu), s_ref, dtype)
