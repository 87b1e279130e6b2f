"""kda_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Some callers only receive input and output buffers (a framework that owns all
allocations, a plugin) and cannot call cudaMalloc for a workspace.  For them
the library runs the prefill in its own fixed 64 MiB device array.  These
tests call that entry point through the C ABI and compare it with the regular
kda_prefill (which gets a workspace allocated here) on two calls in a row, so
that a second call also shows the first one's leftovers in the shared array
do not leak into its result.  This file sorts last so that a run stopping at
the first failure has run every other test before it.
"""
import pytest
import torch

from parity import TOL, host, max_abs, rel_l2, to_device
from synthetic import custom, prefill_inputs

pytestmark = pytest.mark.gpu
NAMES = ("q", "k", "v", "log_alpha", "beta")


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


def _noalloc(kda, d):
    g = to_device(d)
    T, H, dk = g["q"].shape
    N = g["cu_seqlens"].numel() - 1
    out = torch.empty((T, H, g["v"].shape[2]), dtype=g["q"].dtype, device="cuda")
    sf = torch.empty((N, H, dk, dk), dtype=torch.float32, device="cuda")
    desc = kda.make_desc(N, H, dk, dk, T, g["q"].dtype)
    rc = kda.kda_prefill_noalloc(desc, *(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], out, sf)
    assert rc == kda.KDA_OK, kda.kda_status_string(rc)
    return out, sf, g


def _check(a, b, dtype, what):
    tol = TOL[dtype]
    assert rel_l2(host(a), host(b)) <= tol["rel"], what
    assert max_abs(host(a), host(b)) <= tol["abs"], what


def test_noalloc_matches_prefill_on_two_calls(kda):
    cases = [custom(71, [300, 0, 129, 64], 4, 128, "bf16"),      # tensor-core path
             custom(72, [200, 37], 3, 64, "f32")]                 # CUDA-core path, other sizes
    for w in cases:
        d = prefill_inputs(w)
        out, sf, g = _noalloc(kda, d)
        ref_out, ref_sf, _ = kda.prefill(*(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"])
        torch.cuda.synchronize()
        _check(out, ref_out, w.dtype, f"{w.name} output")
        _check(sf, ref_sf, w.dtype, f"{w.name} final state")


def test_noalloc_rejects_problems_beyond_its_scratch(kda):
    # 1M tokens x 16 heads needs ~21 GB of scratch: refused on the host, nothing launched
    # (null buffers would be refused too, before any GPU work).
    desc = kda.make_desc(1, 16, 128, 128, 1 << 20, torch.bfloat16)
    assert kda.kda_prefill_workspace_bytes(desc) > kda.KDA_PREFILL_NOALLOC_SCRATCH_BYTES
    rc = kda.kda_prefill_noalloc(desc, None, None, None, None, None, None, None, None, None)
    assert rc == kda.KDA_ERR_WORKSPACE
