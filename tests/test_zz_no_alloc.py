"""kda_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Some callers only receive input and output buffers (a framework that owns all
allocations, a plugin) and cannot call cudaMalloc for a workspace.  For them
the library runs the prefill in its own fixed 64 MiB device array.  These
tests call that entry point through the C ABI:

  * on two calls in a row, each checked against the fp64 oracle at the
    operator's tolerances, and bit for bit against the regular kda_prefill
    (the same kernels on the same inputs), so that leftovers of the first
    call in the shared array cannot leak into the second;
  * across a cudaDeviceReset in a child process: the array's device address
    is looked up on every call, so the call after the reset runs in the new
    context and gives the same bits.

This file sorts last so that a run stopping at the first failure has run
every other test before it.
"""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import oracle
from parity import assert_parity, host, to_device
from synthetic import custom, prefill_inputs

pytestmark = pytest.mark.gpu
NAMES = ("q", "k", "v", "log_alpha", "beta")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


def _noalloc(kda, g):
    T, H, dk = g["q"].shape
    N = g["cu_seqlens"].numel() - 1
    out = torch.full((T, H, g["v"].shape[2]), float("nan"), dtype=g["q"].dtype, device="cuda")
    sf = torch.full((N, H, dk, dk), float("nan"), dtype=torch.float32, device="cuda")
    desc = kda.make_desc(N, H, dk, dk, T, g["q"].dtype)
    rc = kda.kda_prefill_noalloc(desc, *(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], out, sf)
    assert rc == kda.KDA_OK, kda.kda_status_string(rc)
    return out, sf


def test_noalloc_matches_oracle_on_two_calls(kda):
    # tensor-core path (bf16, d = 128) with empty and partial sequences, the same
    # path again on other lengths (stale records of the same layout in the shared
    # array), then the CUDA-core path at other sizes.
    cases = [custom(71, [300, 0, 129, 64], 4, 128, "bf16"),
             custom(74, [65, 250, 1], 4, 128, "bf16"),
             custom(72, [200, 37], 3, 64, "f32")]
    for w in cases:
        d = prefill_inputs(w)
        g = to_device(d)
        out, sf = _noalloc(kda, g)
        torch.cuda.synchronize()
        ro, rs = oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                                d["initial_state"])
        assert_parity(f"{w.name} no-alloc", host(out), ro, host(sf), rs, w.dtype)
        ref_out, ref_sf, _ = kda.prefill(*(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"])
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"{w.name}: no-alloc output differs from kda_prefill"
        assert torch.equal(sf, ref_sf), f"{w.name}: no-alloc final state differs from kda_prefill"


def test_noalloc_rejects_problems_beyond_its_scratch(kda):
    # 1M tokens x 16 heads needs ~21 GB of scratch: refused on the host, nothing launched
    # (null buffers would be refused too, before any GPU work).
    desc = kda.make_desc(1, 16, 128, 128, 1 << 20, torch.bfloat16)
    assert kda.kda_prefill_workspace_bytes(desc) > kda.KDA_PREFILL_NOALLOC_SCRATCH_BYTES
    rc = kda.kda_prefill_noalloc(desc, None, None, None, None, None, None, None, None, None)
    assert rc == kda.KDA_ERR_WORKSPACE


_CHILD = textwrap.dedent(r"""
    import ctypes, sys
    sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
    import numpy as np
    import torch
    import kda_gated_delta_chunked_gb300 as kda      # loads libkda.so and its CUDA runtime
    from synthetic import custom, prefill_inputs

    rt = ctypes.CDLL("libcudart.so.13")               # the runtime instance libkda.so uses
    vp = ctypes.c_void_p
    rt.cudaMalloc.argtypes = [ctypes.POINTER(vp), ctypes.c_size_t]
    rt.cudaMemcpy.argtypes = [vp, vp, ctypes.c_size_t, ctypes.c_int]
    rt.cudaFree.argtypes = [vp]

    def ok(e, what):
        if e != 0:
            raise SystemExit(f"{what}: cudaError {e}")

    d = prefill_inputs(custom(73, [200, 64, 1], 2, 128, "bf16"))
    host = {n: d[n].contiguous().view(torch.uint8).numpy() for n in
            ("q", "k", "v", "log_alpha", "beta", "cu_seqlens", "initial_state")}
    T, H, D = d["q"].shape
    N = d["cu_seqlens"].numel() - 1
    out_bytes, sf_bytes = T * H * D * 2, N * H * D * D * 4

    def run():
        dev = {}
        for n, a in host.items():
            p = vp()
            ok(rt.cudaMalloc(ctypes.byref(p), a.nbytes), "cudaMalloc")
            ok(rt.cudaMemcpy(p, a.ctypes.data, a.nbytes, 1), "cudaMemcpy H2D")
            dev[n] = p
        for n, nb in (("out", out_bytes), ("sf", sf_bytes)):
            p = vp()
            ok(rt.cudaMalloc(ctypes.byref(p), nb), "cudaMalloc")
            dev[n] = p
        desc = kda.make_desc(N, H, D, D, T, torch.bfloat16)
        args = [dev[n].value for n in ("q", "k", "v", "log_alpha", "beta", "cu_seqlens", "initial_state",
                                       "out", "sf")]
        rc = kda.lib.kda_prefill_noalloc(ctypes.byref(desc), *args, None)
        if rc != 0:
            raise SystemExit(f"kda_prefill_noalloc: {kda.kda_status_string(rc)}")
        res = []
        for n, nb in (("out", out_bytes), ("sf", sf_bytes)):
            buf = np.empty(nb, dtype=np.uint8)
            ok(rt.cudaMemcpy(buf.ctypes.data, dev[n], nb, 2), "cudaMemcpy D2H")
            res.append(buf)
        for p in dev.values():
            ok(rt.cudaFree(p), "cudaFree")
        return res

    first = run()
    ok(rt.cudaDeviceReset(), "cudaDeviceReset")
    second = run()
    if not all(np.array_equal(a, b) for a, b in zip(first, second)):
        raise SystemExit("results differ across cudaDeviceReset")
    print("noalloc across reset: identical")
""")


def test_noalloc_after_device_reset(kda):
    """The call after a cudaDeviceReset (a new context on the same device) looks
    up the scratch array's new address and reproduces the first call's bits."""
    code = f"ROOT = {ROOT!r}\n" + _CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, f"child failed:\n{r.stdout}\n{r.stderr}"
    assert "identical" in r.stdout
