"""The seeded input generator: exact 64-bit hashing, slicing, distributions."""
import math

import torch

from synthetic import generator as g


def test_splitmix64_matches_integer_reference():
    vals = [0, 1, 2, 12345, (1 << 63) - 1, 1 << 63, (1 << 64) - 1, 0x0123456789ABCDEF]
    x = torch.tensor([g._to_signed(v) for v in vals], dtype=torch.int64)
    got = [v & ((1 << 64) - 1) for v in g.splitmix64(x).tolist()]
    assert got == [g.splitmix64_int(v) for v in vals]


def test_splitmix64_known_value():
    # splitmix64 seeded with 0: first output 0xE220A8397B1DCDAF (published
    # first value of the reference sequence).
    assert g.splitmix64_int(0) == 0xE220A8397B1DCDAF


def test_slices_regenerate_identically():
    w = g.custom(11, [300, 77], 3, 16)
    full = g.prefill_inputs(w)
    part = g.prefill_inputs(w, t_range=(100, 250), block_tokens=64)
    for name in ("q", "k", "v", "beta", "log_alpha"):
        assert torch.equal(full[name][100:250], part[name]), name


def test_determinism_and_seed_dependence():
    a = g.prefill_inputs(g.custom(3, [64], 2, 8))
    b = g.prefill_inputs(g.custom(3, [64], 2, 8))
    c = g.prefill_inputs(g.custom(4, [64], 2, 8))
    assert torch.equal(a["q"], b["q"]) and not torch.equal(a["q"], c["q"])


def test_distributions_workload1():
    w = g.workload(1)
    d = g.prefill_inputs(w, t_range=(0, 512))
    k = d["k"].double()
    q = d["q"].double()
    assert torch.allclose(k.norm(dim=-1), torch.ones((), dtype=torch.float64), atol=5e-3)
    assert torch.allclose(q.norm(dim=-1), torch.full((), 1 / math.sqrt(128), dtype=torch.float64), atol=5e-4)
    b = d["beta"].double()
    assert 0 < b.min() and b.max() < 1 and abs(b.mean() - 0.5) < 0.02
    la = d["log_alpha"].double()
    assert la.max() <= -0.0005 * (1 - 2 ** -8) and la.min() >= -0.1 * (1 + 2 ** -8)
    v = d["v"].double()
    assert abs(v.mean()) < 0.02 and abs(v.std() - 1) < 0.02
    s = d["initial_state"].double()
    assert abs(s.std() - 0.02) < 1e-3
    assert d["q"].dtype == torch.bfloat16 and d["initial_state"].dtype == torch.float32


def test_workload_shapes():
    w0, w2, w3, w4 = g.workload(0), g.workload(2), g.workload(3), g.workload(4)
    assert (w0.total_tokens, w0.num_heads, w0.d_k, w0.dtype, w0.state_std) == (256, 2, 64, "f32", None)
    assert len(w2.seqlens) == 8 and all(512 <= L <= 16384 for L in w2.seqlens)
    assert (w3.decode_seqs, w3.decode_steps, w3.num_heads) == (256, 64, 32)
    assert w4.total_tokens == 1 << 20 and (w4.la_lo, w4.la_hi) == (0.0001, 0.05)
    d0 = g.prefill_inputs(w0)
    assert d0["initial_state"] is None and d0["q"].dtype == torch.float32


def test_decode_steps_draw_fresh_values():
    w = g.workload(3)
    a = g.decode_inputs(w, 0)
    b = g.decode_inputs(w, 1)
    assert a["q"].shape == (256, 32, 128) and not torch.equal(a["q"], b["q"])
