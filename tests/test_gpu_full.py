"""Full-size parity: the five workloads at their stated sizes, through the same
GpuCase path that bench.py times, every output row compared element by element
with the literal fp64 oracle (each agent's K and V materialised in full, then
textbook softmax attention).

The oracle's cost is one projection of each sequence's hidden states plus the
attention itself, seconds to tens of seconds per workload on the host cores, so
every decode query and every prefill row is checked, not a sample.
LRAgent (arXiv 2602.01053), Abstract, "preserving accuracy": the shared-cache
result must equal each agent's own non-shared result.
"""
import numpy as np
import pytest
import torch

from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300.harness import GpuCase
from tests.parity import assert_close, oracle_decode_rows, oracle_prefill_seq, tol_for, weights64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _run(name):
    case = I.FULL[name]()
    g = GpuCase(case)
    g.setup()
    res = g.step()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    return case, g, res


def _check_all_prefill(case, g, res):
    w64 = weights64(case)
    for p in range(g.n_pre):
        rows, want = oracle_prefill_seq(case, p, w64=w64)
        assert len(rows) == int(case.pre_q_start[p + 1] - case.pre_q_start[p])
        assert_close(res["prefill"][rows].double().cpu().numpy(), want, tol_for(case), f"prefill seq {p}")


def test_full_tiny_fp32_decode(cuda_lib):
    case, g, res = _run("tiny_fp32_decode")
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case), tol_for(case))


def test_full_shared_decode(cuda_lib):
    case, g, res = _run("shared_decode_llama8b")
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case), tol_for(case))


def test_full_long_decode(cuda_lib):
    """All 16 queries, each over its whole 32768-token context."""
    case, g, res = _run("long_decode_ministral8b")
    assert case.dec_q.shape[0] == 16
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case), tol_for(case))


def test_full_prefill(cuda_lib):
    """All 512 rows of each of the 4 agents' chunks over the 16384-token prefix."""
    case, g, res = _run("prefill_chunk_llama8b")
    assert g.n_pre == 4
    _check_all_prefill(case, g, res)


def test_full_mixed(cuda_lib):
    """All 48 decode queries and all 16 prefill chunks of the mixed batch."""
    case, g, res = _run("mixed_batch_qwen3_1p7b")
    assert case.dec_q.shape[0] == 48 and g.n_pre == 16
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case), tol_for(case), "decode")
    _check_all_prefill(case, g, res)
