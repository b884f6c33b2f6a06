"""The decode's failure path on the GPU, without a fault: a test-only switch
(include/lrkv_testing.h) makes one bounded mbarrier wait of every decode CTA
run out. The call must report LRKV_ERR_TIMEOUT in its status word, every role
of the CTA must leave through the abort path promptly (none waits out its own
~1 s limit), and the next normal call in the same process must still match the
oracle: the context stays usable."""
import pytest
import torch

from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300 import lrkv
from rank_cache_attention_flash_b300.harness import GpuCase
from tests.parity import BF16_TOL, assert_close, oracle_decode_rows

pytestmark = pytest.mark.gpu
TIMEOUT = 5  # LRKV_ERR_TIMEOUT


def _timed_decode(g):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    out = g.decode()
    end.record()
    torch.cuda.synchronize()
    return out, start.elapsed_time(end)


def test_decode_wait_timeout_then_normal_call(cuda_lib):
    case = I.shared_decode(n=600, n_agents=4)
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    g.step_append()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    want = oracle_decode_rows(case, cache="bf16")

    lrkv.testing_set_decode_stall(True)
    try:
        _, ms = _timed_decode(g)
    finally:
        lrkv.testing_set_decode_stall(False)
    assert g.device_status() == TIMEOUT
    # the stalled wait gives up after ~2^20 cycles; every other role follows
    # the abort flag instead of its own 2^31-cycle limit
    assert ms < 100.0, f"stalled decode took {ms:.1f} ms"

    g.status.zero_()
    out, _ = _timed_decode(g)
    assert g.device_status() == 0
    assert_close(out.double().cpu().numpy(), want, BF16_TOL, "decode after a timed-out call")


def test_decode_timeout_is_reported_per_call(cuda_lib):
    """Two stalled calls and a normal one on one status word: the word keeps the
    first error until the caller clears it, and a clean call leaves 0."""
    case = I.shared_decode(n=200, n_agents=2)
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    g.step_append()
    lrkv.testing_set_decode_stall(True)
    try:
        g.decode()
        g.decode()
        torch.cuda.synchronize()
    finally:
        lrkv.testing_set_decode_stall(False)
    assert g.device_status() == TIMEOUT
    g.status.zero_()
    out = g.decode()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    assert_close(out.double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL)
