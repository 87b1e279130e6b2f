"""State snapshots at interior positions (kda_prefill_snapshots) on the GPU:
the state after the first p tokens of a sequence, taken during one prefill,
against the fp64 oracle's final state over that prefix."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, host, rel_l2, to_device
from synthetic import custom, prefill_inputs

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


def _prefix_state(d, n, p):
    """Oracle: final state of sequence n over its first p tokens."""
    cu = d["cu_seqlens"].tolist()
    a = cu[n]
    s0 = None if d["initial_state"] is None else d["initial_state"][n:n + 1]
    x = {k: d[k][a:a + p] for k in NAMES}
    _, sf = oracle.prefill(*(x[k] for k in NAMES), None, s0)
    return sf[0]


def _check(kda, d, pairs, dtype, flags=0):
    g = to_device(d)
    at = torch.tensor(pairs, dtype=torch.int32, device="cuda").view(-1, 2)
    out, sf, ws, snaps = kda.prefill(*(g[k] for k in NAMES), g["cu_seqlens"], g["initial_state"],
                                     snapshot_at=at, flags=flags)
    torch.cuda.synchronize()
    desc = kda.make_desc(len(d["cu_seqlens"]) - 1, d["q"].shape[1], d["q"].shape[2], d["v"].shape[2],
                         d["q"].shape[0], g["q"].dtype, ws)
    assert kda.kda_get_device_status(desc) == kda.KDA_OK
    tol = TOL[dtype]["rel"]
    for m, (n, p) in enumerate(pairs):
        ref = _prefix_state(d, n, p)
        err = rel_l2(host(snaps[m]), ref)
        assert err <= tol, f"snapshot {m} (seq {n}, p={p}): rel-L2 {err:.3e} > {tol}"
    return out, sf, snaps


@pytest.mark.parametrize("dtype,dim,flags", [("bf16", 128, 0), ("f32", 64, 0), ("bf16", 128, 1)])
def test_snapshots_varlen(kda, dtype, dim, flags):
    lens = [300, 0, 64, 130]
    d = prefill_inputs(custom(90 + dim, lens, 2, dim, dtype))
    pairs = [(0, 64), (0, 256), (0, 300), (0, 0), (1, 0), (2, 64), (3, 128), (3, 130), (2, 0)]
    out, sf, snaps = _check(kda, d, pairs, dtype, flags)
    # a snapshot at the full length is the final state, bit for bit
    assert torch.equal(snaps[2], sf[0]) and torch.equal(snaps[7], sf[3]) and torch.equal(snaps[5], sf[2])
    # p = 0 is the initial state
    assert torch.equal(snaps[3].cpu(), d["initial_state"][0]) and torch.equal(snaps[4].cpu(), d["initial_state"][1])


def test_snapshots_do_not_change_outputs(kda):
    d = prefill_inputs(custom(93, [500, 200], 3, 128, "bf16"))
    g = to_device(d)
    args = [g[k] for k in NAMES]
    out1, sf1, _ = kda.prefill(*args, g["cu_seqlens"], g["initial_state"])
    at = torch.tensor([[0, 128], [1, 64], [0, 448]], dtype=torch.int32, device="cuda")
    out2, sf2, _, _ = kda.prefill(*args, g["cu_seqlens"], g["initial_state"], snapshot_at=at)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(sf1, sf2)


def test_snapshots_across_segments(kda):
    """A long sequence split into segments: snapshots inside several segments."""
    T = 16384 + 300
    d = prefill_inputs(custom(94, [T], 2, 128, "bf16", la_lo=0.0001, la_hi=0.05))
    pairs = [(0, 64), (0, 128 * 64), (0, 128 * 64 + 64), (0, 200 * 64), (0, T)]
    _check(kda, d, pairs, "bf16")


@pytest.mark.parametrize("pairs", [[(0, 65)], [(2, 0)], [(0, 64), (0, 64)], [(1, 65)], [(-1, 0)]])
def test_bad_snapshot_requests_set_status(kda, pairs):
    d = prefill_inputs(custom(95, [200, 64], 2, 128, "bf16"))
    g = to_device(d)
    at = torch.tensor(pairs, dtype=torch.int32, device="cuda").view(-1, 2)
    out, sf, ws, snaps = kda.prefill(*(g[k] for k in NAMES), g["cu_seqlens"], g["initial_state"], snapshot_at=at)
    desc = kda.make_desc(2, 2, 128, 128, 264, torch.bfloat16, ws)
    assert kda.kda_get_device_status(desc) == kda.KDA_ERR_BAD_SNAPSHOT
    # the next call on the same workspace starts clean
    out, sf, ws, snaps = kda.prefill(*(g[k] for k in NAMES), g["cu_seqlens"], g["initial_state"],
                                     snapshot_at=torch.tensor([[0, 64]], dtype=torch.int32, device="cuda"),
                                     workspace=ws)
    assert kda.kda_get_device_status(desc) == kda.KDA_OK
