"""The seeded synthetic inputs (the recipe the workloads are built from): the
same seed gives the same bits, a shared prefix occupies the same physical blocks
in every sequence that reads it, block tables are a permutation of distinct
blocks, and the tensors follow the stated distributions. No GPU needed."""
import math

import torch

from rank_cache_attention_flash_b300 import inputs as I


def _same(a, b):
    assert a.dtype == b.dtype and a.shape == b.shape
    assert torch.equal(a, b)


def test_same_seed_same_bits_other_seed_other_bits():
    a, b, c = I.SMALL["prefill_chunk_llama8b"](0), I.SMALL["prefill_chunk_llama8b"](0), I.SMALL["prefill_chunk_llama8b"](1)
    for k in a.weights:
        _same(a.weights[k], b.weights[k])
        assert not torch.equal(a.weights[k], c.weights[k])
    _same(a.pre_q, b.pre_q)
    _same(a.block_tables, b.block_tables)
    _same(a.seq_hidden(0), b.seq_hidden(0))
    assert not torch.equal(a.seq_hidden(0), c.seq_hidden(0))


def test_shared_prefix_is_one_set_of_blocks():
    case = I.prefill_chunk(prefix=64, chunk=40, n_agents=3)
    nb_prefix = 64 // 16
    rows = case.block_tables
    for s in range(1, rows.shape[0]):
        assert torch.equal(rows[s, :nb_prefix], rows[0, :nb_prefix])
    # the prefix hidden states are the same stream for every agent; the chunks differ
    h0, h1 = case.seq_hidden(0), case.seq_hidden(1)
    assert torch.equal(h0[:64], h1[:64])
    assert not torch.equal(h0[64:], h1[64:])


def test_block_tables_hold_distinct_blocks():
    case = I.SMALL["long_decode_ministral8b"]()
    used = case.block_tables[case.block_tables >= 0]
    assert used.numel() == torch.unique(used).numel()  # no two contexts share a block
    assert int(used.max()) < case.num_blocks and int(used.min()) >= 0
    # a seeded permutation, not the identity
    assert not torch.equal(used.sort().values, used)


def test_stated_distributions():
    # X ~ N(0, x_std^2), W ~ N(0, 1/h), A ~ N(0, 1/h), B ~ N(0, 1/r), q ~ N(0, q_std^2), up to sampling error
    case = I.shared_decode(n=256)
    sh = case.shape
    assert math.isclose(sh.w_std, 1 / math.sqrt(sh.hidden), rel_tol=1e-6)
    assert math.isclose(sh.a_std, 1 / math.sqrt(sh.hidden), rel_tol=1e-6)
    assert math.isclose(sh.b_std, 1 / math.sqrt(sh.rank), rel_tol=1e-6)
    for key, std in (("W_K", sh.w_std), ("A_K", sh.a_std), ("B_K", sh.b_std)):
        w = case.weights[key].double()
        assert abs(float(w.mean())) < 0.05 * std
        assert abs(float(w.std()) / std - 1) < 0.02
    x = case.seq_hidden(0).double()
    assert abs(float(x.std()) / sh.x_std - 1) < 0.02
    q = case.dec_q.double()
    assert abs(float(q.std()) / sh.q_std - 1) < 0.05


def test_decode_queries_sorted_by_context():
    case = I.SMALL["mixed_batch_qwen3_1p7b"]()
    qs = case.dec_q_start.tolist()
    assert qs[0] == 0 and qs[-1] == case.dec_q.shape[0]
    assert all(a <= b for a, b in zip(qs, qs[1:]))
    assert len(case.dec_ctx) == len(qs) - 1
