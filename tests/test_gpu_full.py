"""Full-size parity: the five workloads at their stated sizes, through the same
GpuCase path that bench.py times, compared with the oracle on sampled outputs
(whole queries / chunk rows the oracle computes one by one)."""
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


def test_full_tiny_fp32_decode(cuda_lib):
    case, g, res = _run("tiny_fp32_decode")
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case), tol_for(case))


def test_full_shared_decode(cuda_lib):
    case, g, res = _run("shared_decode_llama8b")
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case), tol_for(case))


def test_full_long_decode_sampled(cuda_lib):
    case, g, res = _run("long_decode_ministral8b")
    rows = [0, 11]
    assert_close(res["decode"][rows].double().cpu().numpy(), oracle_decode_rows(case, rows=rows),
                 tol_for(case))


def test_full_prefill_sampled(cuda_lib):
    case, g, res = _run("prefill_chunk_llama8b")
    w64 = weights64(case)
    for p in (0, 3):
        n = int(case.pre_q_start[p + 1] - case.pre_q_start[p])
        sample = sorted(set([0, 1, 2, n // 3, n // 2, n - 2, n - 1] + list(range(5, n, 97))))
        rows, want = oracle_prefill_seq(case, p, q_rows=sample, w64=w64)
        assert_close(res["prefill"][rows].double().cpu().numpy(), want, tol_for(case), f"agent {p}")


def test_full_mixed_sampled(cuda_lib):
    case, g, res = _run("mixed_batch_qwen3_1p7b")
    rows = [0, 17, 47]
    assert_close(res["decode"][rows].double().cpu().numpy(), oracle_decode_rows(case, rows=rows),
                 tol_for(case), "decode")
    w64 = weights64(case)
    for p in (0, 15):
        rows_p, want = oracle_prefill_seq(case, p, q_rows=[0, 1, 128, 254, 255], w64=w64)
        assert_close(res["prefill"][rows_p].double().cpu().numpy(), want, tol_for(case), f"prefill {p}")
