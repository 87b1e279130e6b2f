"""Decode step on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, host, rel_l2
from synthetic import custom, decode_inputs, initial_state, prefill_inputs, workload

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


def test_workload3_decode_64_steps(kda):
    """The full decode workload: 256 sequences x 32 heads, 64 chained steps."""
    w = workload(3)
    s_gpu = initial_state(w, w.decode_seqs, "cpu").cuda()
    s_ref = initial_state(w, w.decode_seqs, "cpu").double().numpy()
    for step in range(w.decode_steps):
        x = decode_inputs(w, step)
        o = kda.decode_step(*(x[n].cuda() for n in NAMES), s_gpu)
        ro, s_ref = oracle.decode_step(*(x[n] for n in NAMES), s_ref)
        if step % 8 == 0 or step == w.decode_steps - 1:
            torch.cuda.synchronize()
            assert_parity(f"decode step {step}", host(o), ro, None, None, "bf16")
    torch.cuda.synchronize()
    assert_parity("workload3 decode 256x32, after 64 steps", host(o), ro, host(s_gpu), s_ref, "bf16")
    assert rel_l2(host(s_gpu), s_ref) < 1e-4     # the fp32 state itself is far tighter


@pytest.mark.parametrize("dtype,dim", [("f32", 64), ("f32", 128), ("bf16", 64)])
def test_decode_small(kda, dtype, dim):
    w = custom(40 + dim, [1] * 5, 3, dim, dtype)
    s0 = initial_state(w, 5)
    s_gpu = s0.cuda().contiguous()
    s_ref = s0.double().numpy()
    for step in range(6):
        x = prefill_inputs(custom(50 + step, [1] * 5, 3, dim, dtype))
        o = kda.decode_step(*(x[n].cuda() for n in NAMES), s_gpu)
        ro, s_ref = oracle.decode_step(*(x[n] for n in NAMES), s_ref)
        torch.cuda.synchronize()
        assert_parity(f"decode {dtype} d{dim} step {step}", host(o), ro, host(s_gpu), s_ref, dtype)


def test_decode_steps_equal_prefill(kda):
    """T decode steps reproduce one T-token prefill (the two modes share one state update)."""
    T = 70
    w = custom(60, [T], 2, 128, "bf16")
    d = prefill_inputs(w)
    g = {n: d[n].cuda() for n in NAMES}
    out, sf, _ = kda.prefill(*(g[n] for n in NAMES), None, d["initial_state"].cuda())
    st = d["initial_state"].cuda().clone()
    outs = []
    for t in range(T):
        outs.append(kda.decode_step(*(g[n][t:t + 1].contiguous() for n in NAMES), st))
    torch.cuda.synchronize()
    assert rel_l2(host(torch.cat(outs)), host(out)) < 5e-3
    assert rel_l2(host(st), host(sf)) < 5e-3


def test_prefill_hands_state_to_decode(kda):
    """Final state of a prefill is the decode step's input state (same layout)."""
    w = custom(61, [190, 64], 2, 128, "bf16")
    d = prefill_inputs(w)
    _, sf, _ = kda.prefill(*(d[n].cuda() for n in NAMES), d["cu_seqlens"].cuda(), d["initial_state"].cuda())
    x = prefill_inputs(custom(62, [1, 1], 2, 128, "bf16"))
    o = kda.decode_step(*(x[n].cuda() for n in NAMES), sf)
    ro, rs = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["initial_state"])
    ro2, rs2 = oracle.decode_step(*(x[n] for n in NAMES), rs)
    torch.cuda.synchronize()
    assert_parity("prefill->decode", host(o), ro2, host(sf), rs2, "bf16")
