"""Reverse mode of the prefill (kda_prefill_backward) on the GPU against the
fp64 oracle's reverse mode, which is itself pinned by finite differences.

Two implementations sit behind the entry point:
  * the tensor-core chunked backward (bf16 inputs, head size 128): bf16
    operands with fp32 accumulation, checked at the operator's bf16
    tolerance, rel-L2 <= 1e-2 on every gradient;
  * the fp32 CUDA-core backward (fp32 inputs, head size 64, or on request
    with KDA_FLAG_CUDA_CORE_PREFILL): fp32 arithmetic against fp64 on the
    same rounded inputs, rel-L2 <= 1e-4.  It is also the tensor-core path's
    fallback for chunks whose decay is too strong for the factorised products.
"""
import pytest
import torch

import oracle
from parity import check_margins, host, rel_l2, to_device
from synthetic import custom, prefill_inputs, workload

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "beta")
TOL_CC = 1e-4      # fp32 arithmetic on the GPU against fp64, on the same (rounded) inputs
TOL_TC = 1e-2      # bf16 tensor-core operands, fp32 accumulation
GRADS = ["dq", "dk", "dv", "dlog_alpha", "dbeta", "d_initial_state"]


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


def _run(kda, d, do, dfin, with_init=True, flags=0):
    g = to_device(d)
    got = kda.prefill_backward(*(g[n] for n in NAMES), g["cu_seqlens"], g["initial_state"], d_out=do.cuda(),
                               d_final_state=None if dfin is None else dfin.cuda(), want_initial_grad=with_init,
                               flags=flags)
    torch.cuda.synchronize()
    return got


def _errors(kda, d, do, dfin, with_init=True, flags=0):
    got = _run(kda, d, do, dfin, with_init, flags)
    ref = oracle.backward(*(d[n] for n in NAMES), d["cu_seqlens"], d["initial_state"], do,
                          None if dfin is None else dfin)
    keys = GRADS if with_init else GRADS[:-1]
    errs = {}
    for key in keys:
        rk = "dinitial_state" if key == "d_initial_state" else key
        errs[key] = rel_l2(host(got[key]), ref[rk])
    return got, errs


def _compare(kda, d, do, dfin, what, with_init=True, flags=0, tol=None):
    tc = d["q"].dtype == torch.bfloat16 and d["q"].shape[2] == 128 and not (flags & kda.KDA_FLAG_CUDA_CORE_PREFILL)
    tol = tol if tol is not None else (TOL_TC if tc else TOL_CC)
    got, errs = _errors(kda, d, do, dfin, with_init, flags)
    for key, err in errs.items():
        assert err <= tol, f"{what}: {key} rel-L2 {err:.3e} > {tol}"
    return got


@pytest.mark.parametrize("dtype,dim", [("f32", 64), ("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_backward_ragged_varlen(kda, dtype, dim):
    lens = [0, 1, 9, 8, 17, 70, 64, 129]
    d = prefill_inputs(custom(110 + dim, lens, 2, dim, dtype))
    do, dfin = _cotangents(d, 1, dtype)
    _compare(kda, d, do, dfin, f"varlen {dtype} d{dim}")


def test_backward_cuda_core_path_on_request(kda):
    """The fp32 CUDA-core backward on bf16 head-size-128 inputs, at the fp32 bound."""
    d = prefill_inputs(custom(111, [0, 1, 9, 70, 129], 2, 128, "bf16"))
    do, dfin = _cotangents(d, 1, "bf16")
    _compare(kda, d, do, dfin, "CUDA-core path", flags=kda.KDA_FLAG_CUDA_CORE_PREFILL)


def test_backward_without_state_gradients(kda):
    d = prefill_inputs(custom(115, [100, 33], 3, 128, "bf16"))
    do, _ = _cotangents(d, 2, "bf16")
    _compare(kda, d, do, None, "no dfinal, no d_initial_state", with_init=False)


def test_backward_zero_initial_state(kda):
    for dtype, dim in (("f32", 64), ("bf16", 128)):
        d = prefill_inputs(custom(116, [130, 64], 2, dim, dtype, state_std=None))
        do, dfin = _cotangents(d, 3, dtype)
        _compare(kda, d, do, dfin, f"zero initial state {dtype} d{dim}")


def test_backward_scalar_gate(kda):
    d = prefill_inputs(custom(117, [50, 0, 77, 200], 2, 128, "bf16", gate="scalar"))
    do, dfin = _cotangents(d, 4, "bf16")
    got = _compare(kda, d, do, dfin, "scalar gate")
    assert tuple(got["dlog_alpha"].shape) == (327, 2)
    _compare(kda, d, do, dfin, "scalar gate, CUDA-core path", flags=kda.KDA_FLAG_CUDA_CORE_PREFILL)


def test_backward_long_sequence(kda):
    """1,000 tokens: sixteen chunks walked in reverse; strong and weak decay."""
    d = prefill_inputs(custom(118, [1000], 2, 128, "bf16", la_lo=0.0001, la_hi=0.3))
    do, dfin = _cotangents(d, 5, "bf16")
    _compare(kda, d, do, dfin, "1000 tokens")


def test_backward_segment_scan_forward(kda):
    """A sequence long enough for the forward's segment scan (whose output
    passes save every chunk's end state for the backward)."""
    d = prefill_inputs(custom(121, [20000, 300], 2, 128, "bf16", la_lo=0.0001, la_hi=0.05))
    do, dfin = _cotangents(d, 8, "bf16")
    _compare(kda, d, do, dfin, "segment-scan forward")


def test_backward_strong_decay_falls_back(kda):
    """log alpha ~ -U(0.5, 5): chunks too strong for the factorised products
    make the tensor-core kernels hand the call to the fp32 CUDA-core backward,
    whose result meets the fp32 bound."""
    d = prefill_inputs(custom(122, [200, 64, 3], 2, 128, "bf16", la_lo=0.5, la_hi=5.0))
    do, dfin = _cotangents(d, 9, "bf16")
    _compare(kda, d, do, dfin, "strong decay (fallback)", tol=TOL_CC)


def test_backward_paths_agree(kda):
    """The tensor-core and CUDA-core backwards agree on the same inputs."""
    d = prefill_inputs(custom(123, [333, 64, 1], 3, 128, "bf16"))
    do, dfin = _cotangents(d, 10, "bf16")
    a = _run(kda, d, do, dfin)
    b = _run(kda, d, do, dfin, flags=kda.KDA_FLAG_CUDA_CORE_PREFILL)
    for key in GRADS:
        assert rel_l2(host(a[key]), host(b[key])) <= TOL_TC, key


def test_backward_workload1_full_size(kda):
    """Workload 1 (4,096 tokens x 16 heads), the benchmarked backward, every
    gradient element against the oracle; the worst rel-L2 is reported."""
    d = prefill_inputs(workload(1))
    do, dfin = _cotangents(d, 11, "bf16")
    _, errs = _errors(kda, d, do, dfin)
    worst = max(errs, key=errs.get)
    check_margins(f"workload1 backward (worst: {worst})", errs[worst], 0.0, None, "bf16")


def test_backward_deterministic(kda):
    d = prefill_inputs(custom(119, [300, 45], 4, 128, "bf16"))
    do, dfin = _cotangents(d, 6, "bf16")
    for flags in (0, kda.KDA_FLAG_CUDA_CORE_PREFILL):
        a = _run(kda, d, do, dfin, flags=flags)
        b = _run(kda, d, do, dfin, flags=flags)
        for key in a:
            assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("nseq,heads", [(10, 2), (20, 2), (4, 2)])
def test_backward_tile_widths(kda, nseq, heads):
    """Sequence x head counts that select 16-, 32- and 8-column tiles of the
    CUDA-core backward (and many short sequences on the tensor-core one)."""
    lens = [(7 * i + 5) % 37 + 1 for i in range(nseq)]
    d = prefill_inputs(custom(120 + nseq, lens, heads, 128, "bf16"))
    do, dfin = _cotangents(d, 7, "bf16")
    _compare(kda, d, do, dfin, f"{nseq} sequences x {heads} heads")
    _compare(kda, d, do, dfin, f"{nseq} sequences x {heads} heads, CUDA-core",
             flags=kda.KDA_FLAG_CUDA_CORE_PREFILL)
