"""GPU checks of lrkv_attn_mixed, the one-call mixed batch (decode queries and
prefill chunks together, as in the batches SARATHI piggybacks decodes on:
Efficient Multi-Adapter LLM Serving via Cross-Model KV-Cache Reuse with
Activated LoRA, "Builds on"; PReCache, Figure 4). Each part must be bitwise
the result of its own call; the oracle parity of the mixed batch itself runs
through GpuCase.step(), which makes this call (test_gpu_parity, test_gpu_full)."""
import pytest
import torch

from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300 import lrkv
from rank_cache_attention_flash_b300.harness import GpuCase

pytestmark = pytest.mark.gpu


def _case():
    g = GpuCase(I.SMALL["mixed_batch_qwen3_1p7b"](), pool_fill=float("nan"))
    g.setup()
    g.step_append()
    torch.cuda.synchronize()
    assert g.n_dec and g.n_pre
    return g


def _separate(g):
    d = g.decode().clone()
    p = g.prefill().clone()
    torch.cuda.synchronize()
    return d, p


def test_mixed_equals_separate_calls_bitwise(cuda_lib):
    g = _case()
    want_d, want_p = _separate(g)
    g.dec_out.fill_(float("nan"))
    g.pre_out.fill_(float("nan"))
    d, p = g.mixed()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    assert torch.equal(d, want_d)
    assert torch.equal(p, want_p)


def test_mixed_with_one_part(cuda_lib):
    g = _case()
    want_d, want_p = _separate(g)
    dec = {"q": g.dec_q, "ctx_q_start": g.dec_q_start, "adapter_ids": g.dec_adapter, "block_tables": g.dec_bt,
           "ctx_lens": g.dec_lens, "max_ctx_len": g.dec_max_len, "max_q_per_ctx": g.dec_max_q}
    pre = {"q": g.pre_q, "q_start": g.pre_q_start, "max_q_len": g.pre_max_q, "seq_lens": g.pre_lens,
           "max_seq_len": g.pre_max_len, "adapter_ids": g.pre_adapter, "block_tables": g.pre_bt}
    d, p = lrkv.attn_mixed(g.cfg, g.base_pool, g.lr_pool, g.attn_B_K, g.B_V, decode=dec, scale=g.scale, status=g.status)
    assert p is None
    d2, p2 = lrkv.attn_mixed(g.cfg, g.base_pool, g.lr_pool, g.attn_B_K, g.B_V, prefill=pre, scale=g.scale, status=g.status)
    assert d2 is None
    torch.cuda.synchronize()
    assert g.device_status() == 0
    assert torch.equal(d, want_d)
    assert torch.equal(p2, want_p)


def test_mixed_bad_part_launches_nothing(cuda_lib):
    """A bad prefill field is refused before the decode part is launched."""
    g = _case()
    g.dec_out.fill_(7.0)
    g.pre_out.fill_(7.0)
    torch.cuda.synchronize()
    dec = {"q": g.dec_q, "ctx_q_start": g.dec_q_start, "adapter_ids": g.dec_adapter, "block_tables": g.dec_bt,
           "ctx_lens": g.dec_lens, "max_ctx_len": g.dec_max_len, "max_q_per_ctx": g.dec_max_q,
           "out": g.dec_out, "workspace": g.dec_ws}
    pre = {"q": g.pre_q, "q_start": g.pre_q_start, "max_q_len": g.pre_max_q, "seq_lens": g.pre_lens,
           "max_seq_len": g.pre_max_q - 1, "adapter_ids": g.pre_adapter, "block_tables": g.pre_bt,
           "out": g.pre_out}
    with pytest.raises(lrkv.LrkvError) as e:
        lrkv.attn_mixed(g.cfg, g.base_pool, g.lr_pool, g.attn_B_K, g.B_V, decode=dec, prefill=pre,
                        status=g.status)
    assert e.value.code == 1
    torch.cuda.synchronize()
    assert bool((g.dec_out == 7.0).all()) and bool((g.pre_out == 7.0).all())


def test_mixed_captured_in_a_graph(cuda_lib):
    """The fork onto the second stream and the join back become graph edges:
    replaying the captured call gives the eager results."""
    g = _case()
    want_d, want_p = _separate(g)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.mixed(stream=s)  # warm-up: the second stream and its events are made outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.mixed(stream=s)
    g.dec_out.fill_(float("nan"))
    g.pre_out.fill_(float("nan"))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    assert torch.equal(g.dec_out, want_d)
    assert torch.equal(g.pre_out, want_p)


def test_decode_does_not_depend_on_earlier_kernels(cuda_lib):
    """Tensor memory is not cleared between kernels: a decode run after a
    prefill (which leaves its own accumulators there) must give the same bits
    as one run before it. G-mode items with fewer rows than the tile's read W
    columns past their last row; those rows are masked before the softmax."""
    g = _case()
    before = g.decode().clone()
    torch.cuda.synchronize()
    for _ in range(3):
        g.prefill()
        after = g.decode().clone()
        torch.cuda.synchronize()
        assert torch.equal(after, before)
