"""Prefill on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, check_margins, host, max_abs, rel_l2, to_device
from synthetic import custom, prefill_inputs, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


def run_gpu(kda, d, *, final=True, initial=True, stream=None):
    g = to_device(d)
    out, sf, ws = kda.prefill(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["cu_seqlens"],
                              g["initial_state"] if initial else None, want_final_state=final,
                              stream=stream)
    torch.cuda.synchronize()
    return out, sf, ws, g


def run_oracle(d, initial=True, cols=None):
    return oracle.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                          d["initial_state"] if initial else None, cols=cols)


def test_workload0_single_f32_d64(kda):
    w = workload(0)
    d = prefill_inputs(w)
    out, sf, _, _ = run_gpu(kda, d)
    ro, rs = run_oracle(d)
    assert_parity("workload0 T=256 H=2 d=64 fp32", host(out), ro, host(sf), rs, "f32")


def test_workload1_single_bf16_T4096(kda):
    w = workload(1)
    d = prefill_inputs(w)
    out, sf, _, _ = run_gpu(kda, d)
    ro, rs = run_oracle(d)
    assert_parity("workload1 T=4096 H=16", host(out), ro, host(sf), rs, "bf16")


@pytest.mark.parametrize("dtype,dim", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 64)])
def test_ragged_varlen(kda, dtype, dim):
    """Lengths around chunk boundaries, empty and 1-token sequences, several heads."""
    lens = [0, 1, 2, 63, 64, 65, 0, 127, 129, 200]
    w = custom(31 + dim, lens, 3, dim, dtype)
    d = prefill_inputs(w)
    out, sf, _, _ = run_gpu(kda, d)
    ro, rs = run_oracle(d)
    assert_parity(f"ragged {dtype} d{dim}", host(out), ro, host(sf), rs, dtype)
    # an empty sequence hands its initial state straight through
    s0 = d["initial_state"].double().numpy()
    assert np.array_equal(host(sf)[0], s0[0]) and np.array_equal(host(sf)[6], s0[6])


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129])
def test_single_sequence_lengths(kda, T):
    w = custom(100 + T, [T], 2, 128, "bf16")
    d = prefill_inputs(w)
    out, sf, _, _ = run_gpu(kda, d)
    ro, rs = run_oracle(d)
    assert_parity(f"T={T}", host(out), ro, host(sf), rs, "bf16")


def test_null_initial_and_final_state(kda):
    w = custom(7, [130, 64], 2, 128, "bf16")
    d = prefill_inputs(w)
    out, sf, _, _ = run_gpu(kda, d, initial=False)
    ro, rs = run_oracle(d, initial=False)
    assert_parity("zero initial state", host(out), ro, host(sf), rs, "bf16")
    out2, sf2, _, _ = run_gpu(kda, d, initial=False, final=False)
    assert sf2 is None
    assert torch.equal(out2, out)


def test_final_state_aliases_initial_state(kda):
    """In-place continuation: final_state == initial_state pointer."""
    w = custom(8, [100, 37, 256], 2, 128, "bf16")
    d = prefill_inputs(w)
    g = to_device(d)
    st = g["initial_state"].clone()
    out, sf, _ = kda.prefill(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["cu_seqlens"],
                             st, final_state=st)
    torch.cuda.synchronize()
    ro, rs = run_oracle(d)
    assert_parity("aliased state", host(out), ro, host(st), rs, "bf16")


def test_continuation_matches_single_call(kda):
    """Prefix then suffix from the returned state reproduces the uninterrupted run
    (checkpoint semantics): both the split and the single call match the oracle."""
    w = custom(9, [640], 2, 128, "bf16")
    d = prefill_inputs(w)
    g = to_device(d)
    args = lambda a, b: [g[n][a:b] for n in ("q", "k", "v", "log_alpha", "beta")]
    full, sfull, _ = kda.prefill(*args(0, 640), None, g["initial_state"])
    ro, rs = run_oracle(d)
    torch.cuda.synchronize()
    assert_parity("single call", host(full), ro, host(sfull), rs, "bf16")
    for m in (64, 100, 333):
        o1, s1, _ = kda.prefill(*args(0, m), None, g["initial_state"])
        o2, s2, _ = kda.prefill(*args(m, 640), None, s1)
        torch.cuda.synchronize()
        assert_parity(f"split at {m}", host(torch.cat([o1, o2])), ro, host(s2), rs, "bf16")
        assert rel_l2(host(torch.cat([o1, o2])), host(full)) < 1e-2


def test_varlen_isolation_on_gpu(kda):
    """A packed batch equals each sequence run alone (bitwise: chunks restart per sequence)."""
    lens = [77, 0, 150, 64]
    w = custom(12, lens, 2, 128, "bf16")
    d = prefill_inputs(w)
    g = to_device(d)
    out, sf, _ = kda.prefill(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["cu_seqlens"],
                             g["initial_state"])
    cu = d["cu_seqlens"].tolist()
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        if a == b:
            continue
        o1, s1, _ = kda.prefill(*(g[x][a:b] for x in ("q", "k", "v", "log_alpha", "beta")), None,
                                g["initial_state"][n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(o1, out[a:b]) and torch.equal(s1[0], sf[n])


def test_deterministic(kda):
    w = custom(13, [300, 200], 4, 128, "bf16")
    d = prefill_inputs(w)
    o1, s1, _, _ = run_gpu(kda, d)
    o2, s2, _, _ = run_gpu(kda, d)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_bad_cu_seqlens_sets_device_status(kda):
    w = custom(14, [64, 64], 2, 128, "bf16")
    d = prefill_inputs(w)
    g = to_device(d)
    for bad in ([0, 100, 64], [5, 64, 128], [0, 64, 127]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        out, sf, ws = kda.prefill(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], cu, g["initial_state"])
        desc = kda.make_desc(2, 2, 128, 128, 128, torch.bfloat16, ws)
        assert kda.kda_get_device_status(desc) == kda.KDA_ERR_BAD_SEQLENS
    out, sf, ws = kda.prefill(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["cu_seqlens"],
                              g["initial_state"])
    desc = kda.make_desc(2, 2, 128, 128, 128, torch.bfloat16, ws)
    assert kda.kda_get_device_status(desc) == kda.KDA_OK


def test_strong_decay_stress(kda):
    """log alpha ~ -U(0.5, 5): per-chunk cumulative decays far beyond fp32 range
    if formed naively; the result must stay finite and match the oracle."""
    for dtype in ("bf16", "f32"):
        w = custom(15, [200, 64], 2, 128, dtype, la_lo=0.5, la_hi=5.0)
        d = prefill_inputs(w)
        out, sf, _, _ = run_gpu(kda, d)
        ro, rs = run_oracle(d)
        assert_parity(f"strong decay {dtype}", host(out), ro, host(sf), rs, dtype)


def test_workload2_varlen_full_size(kda):
    """The full 8-sequence varlen workload (32 heads, 54,483 tokens), every
    output and state element against the oracle."""
    w = workload(2)
    d = prefill_inputs(w)
    out, sf, _, _ = run_gpu(kda, d)
    ro, rs = run_oracle(d)
    assert_parity("workload2 varlen, all heads and columns", host(out), ro, host(sf), rs, "bf16")


def test_workload4_long_full_size(kda):
    """The 1M-token workload as benchmarked (one sequence of 2^20 tokens, 16
    heads, ten segments of the segment scan), every output and state element
    against the oracle.  The oracle runs one head at a time (heads are
    independent), which keeps its fp64 copies near 5 GB of host memory; the
    errors are accumulated over all heads into whole-tensor figures."""
    w = workload(4)
    d = prefill_inputs(w, device="cuda")
    out, sf, _ = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                             d["initial_state"])
    torch.cuda.synchronize()
    H = w.num_heads
    num_o = den_o = num_s = den_s = 0.0
    max_o = 0.0
    for h in range(H):
        sub = {n: d[n][:, h:h + 1].contiguous().cpu() for n in ("q", "k", "v", "log_alpha", "beta")}
        ro, rs = oracle.prefill(sub["q"], sub["k"], sub["v"], sub["log_alpha"], sub["beta"], None,
                                d["initial_state"][:, h:h + 1].contiguous().cpu())
        go = host(out[:, h:h + 1])
        gs = host(sf[:, h:h + 1])
        assert np.all(np.isfinite(go)) and np.all(np.isfinite(gs)), f"head {h}: non-finite results"
        num_o += float(np.sum((go - ro) ** 2))
        den_o += float(np.sum(ro ** 2))
        num_s += float(np.sum((gs - rs) ** 2))
        den_s += float(np.sum(rs ** 2))
        max_o = max(max_o, max_abs(go, ro))
        del ro, rs, go, gs, sub
    check_margins("workload4 1M tokens, all 16 heads and columns", (num_o / den_o) ** 0.5, max_o,
                  (num_s / den_s) ** 0.5, "bf16")


def test_tensor_core_path_matches_cuda_core_path(kda):
    """The tcgen05 path and the fp32 CUDA-core path agree on the same inputs."""
    w = custom(16, [1000, 37, 640], 4, 128, "bf16")
    d = prefill_inputs(w)
    g = to_device(d)
    args = [g[n] for n in ("q", "k", "v", "log_alpha", "beta")]
    o_tc, s_tc, _ = kda.prefill(*args, g["cu_seqlens"], g["initial_state"])
    o_cc, s_cc, _ = kda.prefill(*args, g["cu_seqlens"], g["initial_state"], flags=kda.KDA_FLAG_CUDA_CORE_PREFILL)
    torch.cuda.synchronize()
    assert rel_l2(host(o_tc), host(o_cc)) < 1e-2
    assert rel_l2(host(s_tc), host(s_cc)) < 1e-2
    ro, rs = run_oracle(d)
    assert_parity("cuda-core path", host(o_cc), ro, host(s_cc), rs, "bf16")


def test_segment_scan_single_long_sequence(kda):
    """A sequence long enough to be split into segments (three segments of 128
    chunks here): the per-segment transitions, their sequential combination and
    the rerun from each segment's start state must reproduce the recurrence."""
    w = custom(17, [24576], 2, 128, "bf16", la_lo=0.0001, la_hi=0.05)
    d = prefill_inputs(w)
    out, sf, _, _ = run_gpu(kda, d)
    ro, rs = run_oracle(d)
    assert_parity("segment scan", host(out), ro, host(sf), rs, "bf16")


def test_segment_scan_mixed_lengths(kda):
    """One sequence split into segments next to short ones that are not."""
    w = custom(18, [20000, 300, 0, 64], 2, 128, "bf16", la_lo=0.0001, la_hi=0.02)
    d = prefill_inputs(w)
    out, sf, _, _ = run_gpu(kda, d)
    ro, rs = run_oracle(d)
    assert_parity("segment scan, mixed", host(out), ro, host(sf), rs, "bf16")


@pytest.mark.parametrize("case", ["no_decay", "no_write", "full_write"])
def test_degenerate_gates(kda, case):
    """The gates' special values: log alpha = 0 (no forgetting: DeltaNet),
    beta = 0 (nothing written: the state only decays), beta = 1 (exact
    overwrite along each key), on the tensor-core and CUDA-core paths."""
    for dtype, dim in (("bf16", 128), ("f32", 64)):
        d = prefill_inputs(custom(130, [150, 64, 1], 2, dim, dtype))
        if case == "no_decay":
            d["log_alpha"] = torch.zeros_like(d["log_alpha"])
        elif case == "no_write":
            d["beta"] = torch.zeros_like(d["beta"])
        else:
            d["beta"] = torch.ones_like(d["beta"])
        out, sf, _, _ = run_gpu(kda, d)
        ro, rs = run_oracle(d)
        assert_parity(f"{case} {dtype} d{dim}", host(out), ro, host(sf), rs, dtype)
        if case == "no_write":
            # nothing written: the final state is the initial state decayed channel by channel
            la = d["log_alpha"].double()
            s0 = d["initial_state"].double()
            cu = d["cu_seqlens"].tolist()
            for n in range(len(cu) - 1):
                decay = torch.exp(la[cu[n]:cu[n + 1]].sum(0))          # [H, d_k]
                ref = (s0[n] * decay[:, :, None]).numpy()
                assert np.abs(host(sf)[n] - ref).max() <= 1e-3 * max(1.0, np.abs(ref).max())


def test_many_sequences(kda):
    """2,500 sequences (more than one pass of the sequence-table kernel's 1,024
    threads), lengths 0..40, including chunk-boundary lengths."""
    lens = [(i * 7919) % 41 for i in range(2500)]
    lens[3], lens[4], lens[5] = 64, 65, 128
    d = prefill_inputs(custom(131, lens, 2, 128, "bf16"))
    out, sf, _, _ = run_gpu(kda, d)
    ro, rs = run_oracle(d)
    assert_parity("2,500 sequences", host(out), ro, host(sf), rs, "bf16")
