"""Failure handling on the GPU, without faulting it: a bounded wait that can
never complete ends by itself, records KDA_ERR_TIMEOUT in the device status
word, and the context stays usable for the next call."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_gated_delta_chunked_gb300 as m
    return m


def test_wait_that_never_completes_times_out(kda):
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    desc = kda.make_desc(1, 1, 128, 128, 1, torch.bfloat16, ws)
    t = time.perf_counter()
    assert kda.kda_selftest_wait_timeout(desc, 20_000_000) == kda.KDA_OK      # 20 ms limit
    assert kda.kda_get_device_status(desc) == kda.KDA_ERR_TIMEOUT
    assert time.perf_counter() - t < 5.0
    # the context is still healthy: a real prefill on the same workspace succeeds
    from synthetic import custom, prefill_inputs
    d = prefill_inputs(custom(3, [100], 1, 128, "bf16"))
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    out, sf, ws2 = kda.prefill(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["cu_seqlens"],
                               g["initial_state"])
    desc2 = kda.make_desc(1, 1, 128, 128, 100, torch.bfloat16, ws2)
    assert kda.kda_get_device_status(desc2) == kda.KDA_OK
    assert torch.isfinite(out.float()).all()


def test_selftest_rejects_long_limits(kda):
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    desc = kda.make_desc(1, 1, 128, 128, 1, torch.bfloat16, ws)
    assert kda.kda_selftest_wait_timeout(desc, 5_000_000_000) == kda.KDA_ERR_INVALID_ARGUMENT
