"""The C ABI library: loads, exports every declared entry point, and rejects bad
arguments on the host before any CUDA work (no GPU needed: every call here
fails validation before a kernel could be launched)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
kda = pytest.importorskip("kda_gated_delta_chunked_gb300",
                          reason="libkda.so not built (run __graft_entry__.build())")


def declared_entry_points():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", src)
    return names


def test_exports_every_declared_symbol():
    names = declared_entry_points()
    assert {"kda_prefill", "kda_decode_step", "kda_prefill_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(kda.lib, n), f"libkda.so does not export {n}"


def test_status_strings_and_version():
    assert kda.kda_status_string(kda.KDA_OK) == "KDA_OK"
    assert kda.kda_status_string(kda.KDA_ERR_BAD_SEQLENS) == "KDA_ERR_BAD_SEQLENS"
    assert kda.kda_status_string(999) == "KDA_ERR_UNKNOWN"
    assert kda.kda_version() >= 10000


def test_workspace_bytes():
    import torch
    d = kda.make_desc(1, 16, 128, 128, 4096, torch.bfloat16)
    n1 = kda.kda_prefill_workspace_bytes(d)
    d2 = kda.make_desc(1, 16, 128, 128, 8192, torch.bfloat16)
    assert 0 < n1 < kda.kda_prefill_workspace_bytes(d2)
    for bad in (kda.make_desc(1, 16, 96, 96, 64, torch.bfloat16),      # unsupported head size
                kda.make_desc(1, 16, 128, 64, 64, torch.bfloat16),     # d_k != d_v
                kda.make_desc(-1, 16, 128, 128, 64, torch.bfloat16),
                kda.make_desc(1, 0, 128, 128, 64, torch.bfloat16)):
        assert kda.kda_prefill_workspace_bytes(bad) == 0
    # The bound does not depend on cu_seqlens contents: ceil(T/64) + N chunks per head.
    d3 = kda.make_desc(3, 2, 64, 64, 100, torch.float32)
    d4 = kda.make_desc(4, 2, 64, 64, 100, torch.float32)
    assert kda.kda_prefill_workspace_bytes(d4) > kda.kda_prefill_workspace_bytes(d3)


class _FakePtr:
    """Stands in for a tensor in the pointer slots; never dereferenced (validation fails first)."""
    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def _ptrs(base=1 << 20, n=10, stride=1 << 24):
    return [_FakePtr(base + i * stride) for i in range(n)]


def test_prefill_host_validation():
    import torch
    q, k, v, la, b, cu, s0, out, sf, ws = _ptrs()
    d = kda.make_desc(2, 4, 128, 128, 256, torch.bfloat16)
    # unsupported head size
    bad = kda.make_desc(2, 4, 96, 96, 256, torch.bfloat16)
    assert kda.kda_prefill(bad, q, k, v, la, b, cu, s0, out, sf, 0) == kda.KDA_ERR_UNSUPPORTED
    # unknown flag bits and unknown dtypes are rejected
    bad = kda.make_desc(2, 4, 128, 128, 256, torch.bfloat16); bad.flags = 4
    assert kda.kda_prefill(bad, q, k, v, la, b, cu, s0, out, sf, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    bad = kda.make_desc(2, 4, 128, 128, 256, 7)
    assert kda.kda_prefill(bad, q, k, v, la, b, cu, s0, out, sf, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    # no cu_seqlens with N != 1
    assert kda.kda_prefill(d, q, k, v, la, b, None, s0, out, sf, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    # null required input / misaligned pointer
    assert kda.kda_prefill(d, q, None, v, la, b, cu, s0, out, sf, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_prefill(d, q, k, _FakePtr(v.addr + 8), la, b, cu, s0, out, sf, 0) == \
        kda.KDA_ERR_INVALID_ARGUMENT
    # out overlapping an input
    assert kda.kda_prefill(d, q, k, v, la, b, cu, s0, _FakePtr(q.addr + 1024), sf, 0) == \
        kda.KDA_ERR_INVALID_ARGUMENT
    # partially overlapping state buffers (exact aliasing is allowed)
    assert kda.kda_prefill(d, q, k, v, la, b, cu, s0, out, _FakePtr(s0.addr + 4096), 0) == \
        kda.KDA_ERR_INVALID_ARGUMENT
    # missing / too small / misaligned workspace
    assert kda.kda_prefill(d, q, k, v, la, b, cu, s0, out, sf, 0) == kda.KDA_ERR_WORKSPACE
    d.workspace = ws.addr
    d.workspace_bytes = kda.kda_prefill_workspace_bytes(d) - 1
    assert kda.kda_prefill(d, q, k, v, la, b, cu, s0, out, sf, 0) == kda.KDA_ERR_WORKSPACE
    d.workspace = ws.addr + 64
    d.workspace_bytes = kda.kda_prefill_workspace_bytes(d)
    assert kda.kda_prefill(d, q, k, v, la, b, cu, s0, out, sf, 0) == kda.KDA_ERR_WORKSPACE


def test_scalar_gate_alignment():
    """A per-channel log_alpha needs 16-byte alignment; a scalar gate
    ([T, H], KDA_FLAG_SCALAR_GATE) only its element size, like beta."""
    import torch
    q, k, v, la, b, cu, s0, out, sf, ws = _ptrs()
    la2 = _FakePtr(la.addr + 2)
    d = kda.make_desc(2, 4, 128, 128, 256, torch.bfloat16)
    assert kda.kda_prefill(d, q, k, v, la2, b, cu, s0, out, sf, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    d.flags = kda.KDA_FLAG_SCALAR_GATE          # passes the pointer checks, stops at the workspace
    assert kda.kda_prefill(d, q, k, v, la2, b, cu, s0, out, sf, 0) == kda.KDA_ERR_WORKSPACE
    assert kda.kda_prefill(d, q, k, v, _FakePtr(la.addr + 1), b, cu, s0, out, sf, 0) == \
        kda.KDA_ERR_INVALID_ARGUMENT
    # the decode step: a scalar gate overlapping the state is caught with its own [N, H] size
    q, k, v, la, b, st, o = _ptrs(n=7)
    dd = kda.make_desc(8, 4, 128, 128, 8, torch.bfloat16, flags=kda.KDA_FLAG_SCALAR_GATE)
    assert kda.kda_decode_step(dd, q, k, v, _FakePtr(st.addr + 62), b, st, o, 0) == \
        kda.KDA_ERR_INVALID_ARGUMENT


def test_snapshot_host_validation():
    import torch
    q, k, v, la, b, cu, s0, out, sf, ws = _ptrs()
    at, snaps = _FakePtr(ws.addr + (1 << 24)), _FakePtr(ws.addr + 2 * (1 << 24))
    d = kda.make_desc(2, 4, 128, 128, 256, torch.bfloat16)
    call = lambda m, a, sn: kda.kda_prefill_snapshots(d, q, k, v, la, b, cu, s0, out, sf, m, a, sn, 0)
    assert call(-1, at, snaps) == kda.KDA_ERR_INVALID_ARGUMENT
    assert call(3, None, snaps) == kda.KDA_ERR_INVALID_ARGUMENT
    assert call(3, at, None) == kda.KDA_ERR_INVALID_ARGUMENT
    assert call(3, _FakePtr(at.addr + 2), snaps) == kda.KDA_ERR_INVALID_ARGUMENT     # 4-byte pairs
    assert call(3, at, _FakePtr(snaps.addr + 8)) == kda.KDA_ERR_INVALID_ARGUMENT     # 16-byte states
    assert call(3, at, _FakePtr(sf.addr + 4096)) == kda.KDA_ERR_INVALID_ARGUMENT     # overlaps final state
    assert call(3, at, snaps) == kda.KDA_ERR_WORKSPACE          # arguments fine, no workspace given
    assert call(0, None, None) == kda.KDA_ERR_WORKSPACE


def test_backward_host_validation():
    import torch
    p = _ptrs(n=16)
    q, k, v, la, b, cu, s0, do, dfin, dq, dk, dv, dla, db, ds0, ws = p
    d = kda.make_desc(2, 4, 128, 128, 256, torch.bfloat16)
    call = lambda **kw: kda.kda_prefill_backward(d, *[kw.get(n, x) for n, x in zip(
        ["q", "k", "v", "la", "b", "cu", "s0", "do", "dfin", "dq", "dk", "dv", "dla", "db", "ds0"], p[:15])], 0)
    assert kda.kda_backward_workspace_bytes(d) > 0
    assert call() == kda.KDA_ERR_WORKSPACE                               # arguments fine, no workspace
    assert call(do=None) == kda.KDA_ERR_INVALID_ARGUMENT
    assert call(dbeta=None, db=None) == kda.KDA_ERR_INVALID_ARGUMENT
    assert call(dq=_FakePtr(dq.addr + 2)) == kda.KDA_ERR_INVALID_ARGUMENT  # 4-byte gradients
    assert call(ds0=_FakePtr(ds0.addr + 4)) == kda.KDA_ERR_INVALID_ARGUMENT
    assert call(dk=_FakePtr(q.addr + 64)) == kda.KDA_ERR_INVALID_ARGUMENT  # output over an input
    assert call(dv=_FakePtr(dk.addr + 64)) == kda.KDA_ERR_INVALID_ARGUMENT  # two outputs overlap
    assert call(ds0=None, dfin=None) == kda.KDA_ERR_WORKSPACE
    bad = kda.make_desc(2, 4, 96, 96, 256, torch.bfloat16)
    assert kda.kda_prefill_backward(bad, *p[:15], 0) == kda.KDA_ERR_UNSUPPORTED


def test_decode_host_validation():
    import torch
    q, k, v, la, b, st, out = _ptrs(n=7)
    d = kda.make_desc(8, 4, 128, 128, 8, torch.bfloat16)
    bad = kda.make_desc(8, 4, 128, 128, 9, torch.bfloat16)          # T != N
    assert kda.kda_decode_step(bad, q, k, v, la, b, st, out, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    bad = kda.make_desc(8, 4, 80, 80, 8, torch.bfloat16)
    assert kda.kda_decode_step(bad, q, k, v, la, b, st, out, 0) == kda.KDA_ERR_UNSUPPORTED
    assert kda.kda_decode_step(d, q, k, v, la, b, None, out, 0) == kda.KDA_ERR_INVALID_ARGUMENT
    assert kda.kda_decode_step(d, q, k, v, la, b, _FakePtr(st.addr + 16), out, 0) == \
        kda.KDA_ERR_INVALID_ARGUMENT                                  # state needs 32-byte alignment
    assert kda.kda_decode_step(d, q, k, v, la, b, st, _FakePtr(st.addr + 4096), 0) == \
        kda.KDA_ERR_INVALID_ARGUMENT                                  # out inside the state


def test_empty_batches_are_no_ops():
    import torch
    d = kda.make_desc(0, 4, 128, 128, 0, torch.bfloat16)
    assert kda.kda_prefill(d, None, None, None, None, None, _FakePtr(1 << 20), None, None, None, 0) == kda.KDA_OK
    assert kda.kda_decode_step(d, None, None, None, None, None, None, None, 0) == kda.KDA_OK
