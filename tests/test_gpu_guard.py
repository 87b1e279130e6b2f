"""Guard regions around every buffer the kernels write.

compute-sanitizer is not available on the test machines, so out-of-bounds
writes are looked for directly: each output buffer (and the workspace) is
carved out of a larger allocation with 4 KiB of sentinel bytes on both sides,
the entry point runs, and every sentinel byte must be unchanged.  The lengths
straddle the 64-token chunk (1, 63, 65, 129) and include a sequence long
enough for the segment scan of the tensor-core prefill, so that partial last
chunks, tensor stores at sequence ends, segment scratch and the backward's
partial sums are all exercised.
"""
import pytest
import torch

from parity import to_device
from synthetic import custom, decode_inputs, prefill_inputs, workload

pytestmark = pytest.mark.gpu
PAD = 4096
SENTINEL = 0xA5
NAMES = ("q", "k", "v", "log_alpha", "beta")
LENS = [1, 63, 65, 129, 16384 + 100]


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


class Guarded:
    """Buffers carved out of padded allocations filled with a sentinel byte."""

    def __init__(self):
        self.raw = {}

    def make(self, name, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((PAD + nbytes + PAD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.raw[name] = (raw, nbytes)
        return raw[PAD:PAD + nbytes].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        for name, (raw, nbytes) in self.raw.items():
            lo, hi = raw[:PAD], raw[PAD + nbytes:]
            bad_lo = int((lo != SENTINEL).sum())
            bad_hi = int((hi != SENTINEL).sum())
            assert bad_lo == 0 and bad_hi == 0, \
                f"{what}: {name} guard bytes changed ({bad_lo} before, {bad_hi} after the buffer)"


CASES = [("bf16", 128, "channel"), ("bf16", 128, "scalar"), ("f32", 128, "channel"), ("bf16", 64, "channel")]


@pytest.mark.parametrize("dtype,dim,gate", CASES)
def test_prefill_writes_stay_in_bounds(kda, dtype, dim, gate):
    w = custom(201, LENS, 2, dim, dtype, la_lo=0.0001, la_hi=0.05, gate=gate)
    g = to_device(prefill_inputs(w))
    T, H, N = w.total_tokens, w.num_heads, len(LENS)
    flags = kda.KDA_FLAG_SCALAR_GATE if gate == "scalar" else 0
    G = Guarded()
    out = G.make("out", (T, H, dim), g["q"].dtype)
    sf = G.make("final_state", (N, H, dim, dim), torch.float32)
    desc = kda.make_desc(N, H, dim, dim, T, g["q"].dtype, flags=flags)
    nws = kda.kda_prefill_workspace_bytes(desc)
    ws = G.make("workspace", (nws,), torch.uint8)
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), nws
    rc = kda.kda_prefill(desc, *(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], out, sf)
    assert rc == kda.KDA_OK, kda.kda_status_string(rc)
    G.check(f"prefill {dtype} d{dim} {gate}")
    assert kda.kda_get_device_status(desc) == kda.KDA_OK
    assert torch.isfinite(out.float()).all() and torch.isfinite(sf).all()

    # the same call with state snapshots at chunk boundaries and sequence ends
    cu = g["cu_seqlens"].tolist()
    at = [[0, 0], [0, 1], [1, 63], [2, 64], [2, 65], [3, 128], [4, 64], [4, 8192], [4, LENS[4]]]
    snap_at = torch.tensor(at, dtype=torch.int32, device="cuda")
    snaps = G.make("snapshots", (len(at), H, dim, dim), torch.float32)
    rc = kda.kda_prefill_snapshots(desc, *(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], out, sf,
                                   len(at), snap_at, snaps)
    assert rc == kda.KDA_OK, kda.kda_status_string(rc)
    G.check(f"prefill with snapshots {dtype} d{dim} {gate}")
    assert kda.kda_get_device_status(desc) == kda.KDA_OK
    assert cu[-1] == T


@pytest.mark.parametrize("dtype,dim,gate", CASES)
def test_backward_writes_stay_in_bounds(kda, dtype, dim, gate):
    lens = LENS[:4] + [3000]
    w = custom(202, lens, 2, dim, dtype, gate=gate)
    g = to_device(prefill_inputs(w))
    T, H, N = w.total_tokens, w.num_heads, len(lens)
    flags = kda.KDA_FLAG_SCALAR_GATE if gate == "scalar" else 0
    gen = torch.Generator(device="cuda").manual_seed(5)
    d_out = torch.randn((T, H, dim), generator=gen, device="cuda").to(g["q"].dtype)
    d_fin = torch.randn((N, H, dim, dim), generator=gen, device="cuda")
    G = Guarded()
    la_shape = (T, H) if gate == "scalar" else (T, H, dim)
    bufs = [G.make("dq", (T, H, dim), torch.float32), G.make("dk", (T, H, dim), torch.float32),
            G.make("dv", (T, H, dim), torch.float32), G.make("dlog_alpha", la_shape, torch.float32),
            G.make("dbeta", (T, H), torch.float32), G.make("d_initial_state", (N, H, dim, dim), torch.float32)]
    desc = kda.make_desc(N, H, dim, dim, T, g["q"].dtype, flags=flags)
    nws = kda.kda_backward_workspace_bytes(desc)
    ws = G.make("workspace", (nws,), torch.uint8)
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), nws
    rc = kda.kda_prefill_backward(desc, *(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], d_out,
                                  d_fin, *bufs)
    assert rc == kda.KDA_OK, kda.kda_status_string(rc)
    G.check(f"backward {dtype} d{dim} {gate}")
    assert all(torch.isfinite(b).all() for b in bufs)


@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_decode_writes_stay_in_bounds(kda, gate):
    w = workload(3)
    x = decode_inputs(w, 0)
    N, H = 37, 3                                  # not a multiple of any tile
    x = {n: t[:N, :H].contiguous().cuda() for n, t in x.items()}
    if gate == "scalar":
        x["log_alpha"] = x["log_alpha"][..., 0].contiguous()
    G = Guarded()
    st = G.make("state", (N, H, 128, 128), torch.float32)
    st.copy_(torch.randn((N, H, 128, 128), device="cuda") * 0.02)
    out = G.make("out", (N, H, 128), torch.bfloat16)
    desc = kda.make_desc(N, H, 128, 128, N, torch.bfloat16,
                         flags=kda.KDA_FLAG_SCALAR_GATE if gate == "scalar" else 0)
    rc = kda.kda_decode_step(desc, *(x[n] for n in NAMES), st, out)
    assert rc == kda.KDA_OK, kda.kda_status_string(rc)
    G.check(f"decode {gate}")


def test_noalloc_writes_stay_in_bounds(kda):
    w = custom(203, LENS[:4] + [600], 2, 128, "bf16")
    g = to_device(prefill_inputs(w))
    T, H, N = w.total_tokens, w.num_heads, 5
    G = Guarded()
    out = G.make("out", (T, H, 128), torch.bfloat16)
    sf = G.make("final_state", (N, H, 128, 128), torch.float32)
    desc = kda.make_desc(N, H, 128, 128, T, torch.bfloat16)
    rc = kda.kda_prefill_noalloc(desc, *(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], out, sf)
    assert rc == kda.KDA_OK, kda.kda_status_string(rc)
    G.check("no-alloc prefill")
