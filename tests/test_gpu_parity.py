"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Small workloads (every layer shape of the five workloads, several tiles and a
ragged tail) and edge cases are compared element by element with the oracle's
bf16-cache variant (the oracle rounds its own fp64 cache components to bf16,
as the stored cache holds them), which isolates the kernels' own error from the
storage format's: on short contexts, or on the Qwen-shaped layer, the bf16
rounding of the cache alone reaches the stated bounds (rel-Frobenius 4.8e-3
measured on the small mixed batch). The five workloads at their stated sizes
are checked against the literal oracle in test_gpu_full.py. Pools are
pre-filled with NaN so that any read of an unwritten slot shows up.
"""
import math

import numpy as np
import pytest
import torch

from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300.harness import GpuCase
from tests.parity import (BF16_TOL, assert_close, oracle_decode_rows, oracle_prefill_seq, tol_for,
                          weights64)

pytestmark = pytest.mark.gpu
NAN = float("nan")


def _run(case, pool_fill=NAN):
    g = GpuCase(case, pool_fill=pool_fill)
    g.setup()
    res = g.step()
    torch.cuda.synchronize()
    return g, res


@pytest.mark.parametrize("name", list(I.SMALL))
def test_small_workload_parity(cuda_lib, name):
    case = I.SMALL[name]()
    g, res = _run(case)
    assert g.device_status() == 0
    tol = tol_for(case)
    cache = None if case.shape.dtype == "fp32" else "bf16"
    if g.n_dec:
        assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache=cache), tol,
                     f"{name} decode")
    w64 = weights64(case)
    for p in range(g.n_pre):
        rows, want = oracle_prefill_seq(case, p, w64=w64, cache=cache)
        assert_close(res["prefill"][rows].double().cpu().numpy(), want, tol, f"{name} prefill seq {p}")


@pytest.mark.parametrize("n", [1, 15, 16, 17, 33, 64, 65, 300])
def test_decode_context_lengths(cuda_lib, n):
    case = I.shared_decode(n=n)
    g, res = _run(case)
    assert g.device_status() == 0
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL, f"n={n}")


@pytest.mark.parametrize("rank", [8, 16, 32, 64])
def test_decode_ranks(cuda_lib, rank):
    case = I.shared_decode(n=200, n_agents=4, rank=rank)
    g, res = _run(case)
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL, f"r={rank}")


@pytest.mark.parametrize("rank", [8, 32, 64])
def test_prefill_ranks(cuda_lib, rank):
    case = I.prefill_chunk(prefix=96, chunk=40, n_agents=2, rank=rank)
    g, res = _run(case)
    w64 = weights64(case)
    for p in range(g.n_pre):
        rows, want = oracle_prefill_seq(case, p, w64=w64, cache="bf16")
        assert_close(res["prefill"][rows].double().cpu().numpy(), want, BF16_TOL, f"r={rank} seq {p}")


@pytest.mark.parametrize("rank", [16, 64])
def test_head_dim_64_prefill_and_decode(cuda_lib, rank):
    """head_dim 64 (one 64-column swizzle atom per K / V row), with a ragged
    chunk: prefill and decode against the oracle."""
    sh = I.Shape(1024, 8, 2, 64, rank, 2, 10000.0, "bf16", 1.0, 1 / math.sqrt(1024), 1 / math.sqrt(1024),
                 1 / math.sqrt(rank), 1.0)
    seqs = [I.Seq(0, 144, 1 + a, 144, 37, a, "prefill") for a in range(2)]
    case = I._build("head_dim_64", sh, 0, seqs, [], [0, 1], False)
    g, res = _run(case)
    assert g.device_status() == 0
    w64 = weights64(case)
    for p in range(g.n_pre):
        rows, want = oracle_prefill_seq(case, p, w64=w64, cache="bf16")
        assert_close(res["prefill"][rows].double().cpu().numpy(), want, BF16_TOL, f"d=64 r={rank} seq {p}")


def test_decode_many_agents_one_context(cuda_lib):
    """More queries on one context than one sweep serves (several query groups),
    with repeated and base-only adapters."""
    case = I.shared_decode(n=500, n_agents=8)
    case.dec_adapter = torch.tensor([3, -1, 3, 0, 7, -1, 1, 3], dtype=torch.int32)
    g, res = _run(case)
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL)


def test_rebuild_mode_with_base_only_queries(cuda_lib):
    """Rank 64, one query per context (the rebuild mode): contexts whose query
    has no adapter (-1) score against K_base alone, in bf16, next to adapted
    ones."""
    case = I.long_decode(n_seqs=4, n=333)
    case.dec_adapter = torch.tensor([-1, 3, -1, 6], dtype=torch.int32)
    for k in range(4):
        case.seqs[k].adapter = int(case.dec_adapter[k])
    g, res = _run(case)
    assert g.device_status() == 0
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL)


def test_decode_many_splits(cuda_lib):
    """One long context on two kv heads: the split plan takes more than 32
    splits of the context (a ragged last tile included), so the combine merges
    in several rounds; base-only and adapter rows together."""
    sh = I.Shape(1024, 8, 2, 64, 16, 2, 10000.0, "bf16", 1.0, 1 / math.sqrt(1024), 1 / math.sqrt(1024),
                 1 / math.sqrt(16), 1.0)
    seqs = [I.Seq(0, 0, 0, 12000, 0, -1, "context")]
    case = I._build("many_splits", sh, 0, seqs, [(0, 0), (0, 1), (0, -1)], [], False)
    g, res = _run(case)
    assert g.device_status() == 0
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL)


@pytest.mark.parametrize("rank", [16, 64])
def test_decode_without_adapter_factors(cuda_lib, rank):
    """B_K = NULL (adapter on V only), then B_V = NULL (adapter on K only); rank
    64 runs the rebuild mode (one query per item), rank 16 the G mode."""
    case = I.shared_decode(n=260, rank=rank)
    g = GpuCase(case, pool_fill=NAN)
    g.setup()
    w64 = weights64(case)
    for drop in ("B_K", "B_V"):
        bk = None if drop == "B_K" else g.B_K
        bv = None if drop == "B_V" else g.B_V
        out = cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, g.dec_adapter, g.dec_bt, g.dec_lens,
                                   g.dec_max_len, g.dec_max_q, g.base_pool, g.lr_pool, bk, bv, g.scale)
        w = dict(w64)
        w[drop] = np.zeros_like(w[drop])
        want = oracle_decode_rows(case, w64=w, cache="bf16")
        assert_close(out.double().cpu().numpy(), want, BF16_TOL, f"without {drop}")


def test_prefill_without_adapter_factors(cuda_lib):
    case = I.prefill_chunk(prefix=64, chunk=33, n_agents=2)
    g = GpuCase(case, pool_fill=NAN)
    g.setup()
    g.step_append()
    w64 = weights64(case)
    for drop in ("B_K", "B_V"):
        bk = None if drop == "B_K" else g.B_K
        bv = None if drop == "B_V" else g.B_V
        out = cuda_lib.attn_prefill(g.cfg, g.pre_q, g.pre_q_start, g.pre_max_q, g.pre_lens, g.pre_max_len,
                                    g.pre_adapter, g.pre_bt, g.base_pool, g.lr_pool, bk, bv, g.scale)
        w = dict(w64)
        w[drop] = np.zeros_like(w[drop])
        for p in range(g.n_pre):
            rows, want = oracle_prefill_seq(case, p, w64=w, cache="bf16")
            assert_close(out[rows].double().cpu().numpy(), want, BF16_TOL, f"without {drop}")


def test_permuted_block_table_is_bitwise_identical(cuda_lib):
    case = I.long_decode(n_seqs=3, n=400)
    g, res = _run(case, pool_fill=0.0)
    out1 = res["decode"].clone()
    perm = torch.randperm(case.num_blocks, generator=torch.Generator().manual_seed(7)).to(g.device)
    base2 = torch.empty_like(g.base_pool)
    lr2 = torch.empty_like(g.lr_pool)
    base2[perm.long()] = g.base_pool
    lr2[perm.long()] = g.lr_pool
    bt2 = torch.where(g.dec_bt >= 0, perm[g.dec_bt.long().clamp(min=0)].int(), g.dec_bt)
    out2 = cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, g.dec_adapter, bt2, g.dec_lens,
                                g.dec_max_len, g.dec_max_q, base2, lr2, g.B_K, g.B_V, g.scale)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_prefill_permuted_block_table_is_bitwise_identical(cuda_lib):
    """Contiguous block tables take the run-of-blocks copies, a permuted pool the
    per-block copies: both must land the same tiles, bit for bit."""
    case = I.prefill_chunk(prefix=304, chunk=70, n_agents=2)
    g, res = _run(case, pool_fill=0.0)
    out1 = res["prefill"].clone()
    perm = torch.randperm(case.num_blocks, generator=torch.Generator().manual_seed(11)).to(g.device)
    base2 = torch.empty_like(g.base_pool)
    lr2 = torch.empty_like(g.lr_pool)
    base2[perm.long()] = g.base_pool
    lr2[perm.long()] = g.lr_pool
    bt2 = torch.where(g.pre_bt >= 0, perm[g.pre_bt.long().clamp(min=0)].int(), g.pre_bt)
    out2 = cuda_lib.attn_prefill(g.cfg, g.pre_q, g.pre_q_start, g.pre_max_q, g.pre_lens, g.pre_max_len,
                                 g.pre_adapter, bt2, base2, lr2, g.B_K, g.B_V, g.scale)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_batched_decode_equals_one_at_a_time(cuda_lib):
    case = I.shared_decode(n=700)
    g, res = _run(case)
    full = res["decode"].float()
    for n in range(g.n_dec):
        one = cuda_lib.attn_decode(g.cfg, g.dec_q[n:n + 1].contiguous(),
                                   torch.tensor([0, 1], dtype=torch.int32, device=g.device),
                                   g.dec_adapter[n:n + 1].contiguous(), g.dec_bt, g.dec_lens,
                                   g.dec_max_len, 1, g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale)
        err = (one.float() - full[n:n + 1]).norm() / full[n:n + 1].norm()
        assert err < 2e-3, float(err)


def test_prefill_last_row_equals_decode(cuda_lib):
    case = I.prefill_chunk(prefix=128, chunk=24, n_agents=2)
    g, res = _run(case)
    pre = res["prefill"].float()
    for p in range(g.n_pre):
        last = int(case.pre_q_start[p + 1]) - 1
        q = g.pre_q[last:last + 1].contiguous()
        out = cuda_lib.attn_decode(g.cfg, q, torch.tensor([0, 1], dtype=torch.int32, device=g.device),
                                   g.pre_adapter[p:p + 1].contiguous(), g.pre_bt[p:p + 1].contiguous(),
                                   g.pre_lens[p:p + 1].contiguous(), int(case.pre_lens()[p]), 1,
                                   g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale)
        err = (out.float() - pre[last:last + 1]).norm() / pre[last:last + 1].norm()
        assert err < 5e-3, float(err)


def test_bad_block_id_is_reported_not_read(cuda_lib):
    case = I.long_decode(n_seqs=2, n=100)
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    bt = g.dec_bt.clone()
    bt[1, 2] = case.num_blocks + 1000
    out = cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, g.dec_adapter, bt, g.dec_lens,
                               g.dec_max_len, g.dec_max_q, g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale,
                               status=g.status)
    torch.cuda.synchronize()
    assert g.device_status() == 4  # LRKV_ERR_INDEX
    assert torch.isfinite(out.float()).all()
    # the untouched context is still exact
    want = oracle_decode_rows(case, rows=[0], cache="bf16")
    assert_close(out[0:1].double().cpu().numpy(), want, BF16_TOL)


def test_bad_adapter_id_gives_zero_and_status(cuda_lib):
    case = I.shared_decode(n=50)
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    ad = g.dec_adapter.clone()
    ad[2] = 99
    out = cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, ad, g.dec_bt, g.dec_lens, g.dec_max_len,
                               g.dec_max_q, g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale, status=g.status)
    torch.cuda.synchronize()
    assert g.device_status() == 4
    assert float(out[2].float().abs().max()) == 0.0
    assert_close(out[0:2].double().cpu().numpy(), oracle_decode_rows(case, rows=[0, 1], cache="bf16"), BF16_TOL)


def test_zero_length_context_gives_zero_and_status(cuda_lib):
    """ctx_lens = 0 is outside [1, max_ctx_len]: LRKV_ERR_INDEX, zero output for
    that context's queries, the other context unaffected."""
    case = I.long_decode(n_seqs=2, n=100)
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    lens = g.dec_lens.clone()
    lens[1] = 0
    out = cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, g.dec_adapter, g.dec_bt, lens, g.dec_max_len,
                               g.dec_max_q, g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale, status=g.status)
    torch.cuda.synchronize()
    assert g.device_status() == 4
    assert float(out[1].float().abs().max()) == 0.0
    assert_close(out[0:1].double().cpu().numpy(), oracle_decode_rows(case, rows=[0], cache="bf16"), BF16_TOL)


def test_more_queries_than_max_q_per_ctx(cuda_lib):
    """max_q_per_ctx smaller than a context's query count: LRKV_ERR_INDEX, the
    query heads past the planned rows get zero output, the planned ones stay
    exact."""
    case = I.shared_decode(n=300, n_agents=8)
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    # rank 16: 16 rows per chunk, g = 4 -> max_q_per_ctx = 4 plans one chunk of 4 queries
    out = cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, g.dec_adapter, g.dec_bt, g.dec_lens,
                               g.dec_max_len, 4, g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale,
                               status=g.status)
    torch.cuda.synchronize()
    assert g.device_status() == 4
    assert float(out[4:].float().abs().max()) == 0.0
    assert_close(out[:4].double().cpu().numpy(), oracle_decode_rows(case, rows=[0, 1, 2, 3], cache="bf16"),
                 BF16_TOL)


def test_query_outside_every_context_range(cuda_lib):
    """ctx_q_start that stops short of num_queries: the uncovered query gets
    LRKV_ERR_INDEX and zero output, the covered ones stay exact."""
    case = I.shared_decode(n=200)
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    qstart = torch.tensor([0, 3], dtype=torch.int32, device=g.device)  # query 3 is in no range
    out = cuda_lib.attn_decode(g.cfg, g.dec_q, qstart, g.dec_adapter, g.dec_bt, g.dec_lens, g.dec_max_len,
                               g.dec_max_q, g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale, status=g.status)
    torch.cuda.synchronize()
    assert g.device_status() == 4
    assert float(out[3].float().abs().max()) == 0.0
    assert_close(out[:3].double().cpu().numpy(), oracle_decode_rows(case, rows=[0, 1, 2], cache="bf16"), BF16_TOL)


def test_rope_base_500000(cuda_lib):
    """A Llama-3-style RoPE base (500000): decode and prefill against the oracle."""
    import dataclasses

    sh = dataclasses.replace(I.shape_llama8b(16, 2), rope_base=500000.0)
    seqs = [I.Seq(0, 272, 1 + a, 272, 77, a, "prefill") for a in range(2)]
    case = I._build("rope_base_500k", sh, 0, seqs, [(0, 0), (0, 1), (0, -1)], [0, 1], False)
    g, res = _run(case)
    assert g.device_status() == 0
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL,
                 "decode")
    w64 = weights64(case)
    for p in range(g.n_pre):
        rows, want = oracle_prefill_seq(case, p, w64=w64, cache="bf16")
        assert_close(res["prefill"][rows].double().cpu().numpy(), want, BF16_TOL, f"prefill seq {p}")


def test_workspace_too_small_is_rejected(cuda_lib):
    case = I.shared_decode(n=64)
    g = GpuCase(case, pool_fill=0.0)
    ws = torch.empty(16, dtype=torch.uint8, device=g.device)
    with pytest.raises(cuda_lib.LrkvError) as e:
        cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, g.dec_adapter, g.dec_bt, g.dec_lens,
                             g.dec_max_len, g.dec_max_q, g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale,
                             workspace=ws)
    assert e.value.code == 6


# ------------------------------------------------------------------ append
def _bits_close(got: torch.Tensor, want: torch.Tensor, ulps: int, abs_slack: float = 0.0):
    """bf16 values within `ulps` units in the last place of the larger magnitude
    (plus an absolute slack for fp32 accumulation noise); +0 and -0 are equal."""
    a = got.float()
    b = want.float()
    big = torch.maximum(a.abs(), b.abs())
    ulp = torch.where(big > 0, torch.exp2(torch.floor(torch.log2(big.clamp(min=1e-30))) - 7),
                      torch.zeros_like(big))
    return bool(((a - b).abs() <= ulps * ulp + abs_slack).all())


@pytest.mark.parametrize("d,r", [(128, 16), (64, 8), (128, 64)])
def test_append_integer_inputs_bit_exact(cuda_lib, d, r):
    """Integer-valued X in {-1, 0, 1} and 0/1 weights: every projection is an exact
    integer below 256 in magnitude, so V_base, L_K, L_V must match bit for bit;
    K_base is the rounded rotation (within 1 bf16 ulp); untouched rows keep the
    0xFFFF sentinel."""
    import oracle

    gen = torch.Generator().manual_seed(3)
    h, Hkv = 256, 2
    cfg = cuda_lib.make_config(h, 4, Hkv, d, r)
    n_seq, max_blocks, num_blocks = 3, 6, 24
    bt = torch.randperm(num_blocks, generator=gen)[: n_seq * max_blocks].view(n_seq, max_blocks).int()
    T = 70
    seq = torch.randint(0, n_seq, (T,), generator=gen).int()
    pos = torch.randperm(max_blocks * 16, generator=gen)[:T].int()  # distinct positions
    seq = seq  # distinct (seq, pos) pairs follow from distinct positions
    X = torch.randint(-1, 2, (T, h), generator=gen).to(torch.bfloat16)
    W = {k: torch.randint(0, 2, (h, n), generator=gen).to(torch.bfloat16)
         for k, n in (("W_K", Hkv * d), ("W_V", Hkv * d), ("A_K", r), ("A_V", r))}
    dev = torch.device("cuda")
    base, lr = cuda_lib.new_pools(cfg, num_blocks, dev)
    base.view(torch.int16).fill_(-1)
    lr.view(torch.int16).fill_(-1)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cuda_lib.append(cfg, X.to(dev), pos.to(dev), seq.to(dev), bt.to(dev),
                    cuda_lib.pack_w_cat(W["W_K"], W["W_V"], W["A_K"], W["A_V"]).to(dev), base, lr, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    eb = np.full((num_blocks, 2, Hkv, 16, d), np.nan)
    el = np.full((num_blocks, 2, 16, r), np.nan)
    oracle.append_pools(eb, el, X.double().numpy(), pos.numpy(), seq.numpy(), bt.numpy(),
                        *(W[k].double().numpy() for k in ("W_K", "W_V", "A_K", "A_V")), Hkv, d, 10000.0)
    written = torch.from_numpy(~np.isnan(el[:, 0, :, 0]))  # [blocks, 16]
    gb, gl = base.cpu(), lr.cpu()
    wb = torch.from_numpy(np.nan_to_num(eb)).to(torch.bfloat16)
    wl = torch.from_numpy(np.nan_to_num(el)).to(torch.bfloat16)
    m = written
    assert torch.equal(gb[:, 1][m.unsqueeze(1).expand(-1, Hkv, -1)].view(torch.int16),
                       wb[:, 1][m.unsqueeze(1).expand(-1, Hkv, -1)].view(torch.int16)), "V_base"
    assert torch.equal(gl[m.unsqueeze(1).expand(-1, 2, -1)].view(torch.int16),
                       wl[m.unsqueeze(1).expand(-1, 2, -1)].view(torch.int16)), "L_K/L_V"
    kb_g = gb[:, 0][m.unsqueeze(1).expand(-1, Hkv, -1)]
    kb_w = wb[:, 0][m.unsqueeze(1).expand(-1, Hkv, -1)]
    assert _bits_close(kb_g, kb_w, 1), "K_base beyond 1 ulp"
    # untouched rows keep the sentinel
    um = ~m
    assert (gb.permute(0, 3, 1, 2, 4)[um].view(torch.int16) == -1).all()
    assert (gl.permute(0, 2, 1, 3)[um].view(torch.int16) == -1).all()


def test_append_random_inputs_within_one_ulp(cuda_lib):
    import oracle

    case = I.long_decode(n_seqs=2, n=150)
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    torch.cuda.synchronize()
    sh = case.shape
    eb = np.zeros((case.num_blocks, 2, sh.n_kv_heads, 16, sh.head_dim))
    el = np.zeros((case.num_blocks, 2, 16, sh.rank))
    w = weights64(case)
    for s, a, b in case.setup_appends():
        X = case.seq_hidden(s, a, b).double().numpy()
        oracle.append_pools(eb, el, X, np.arange(a, b), np.full(b - a, s), case.block_tables.numpy(),
                            w["W_K"], w["W_V"], w["A_K"], w["A_V"], sh.n_kv_heads, sh.head_dim, sh.rope_base)
    # fp32 accumulation over h = 4096 adds ~1e-5 of noise before the bf16 rounding
    assert _bits_close(g.base_pool.cpu(), torch.from_numpy(eb).to(torch.bfloat16), 1, 1e-4)
    assert _bits_close(g.lr_pool.cpu(), torch.from_numpy(el).to(torch.bfloat16), 1, 1e-4)


def test_append_fp32(cuda_lib):
    import oracle

    case = I.tiny_fp32_decode()
    g = GpuCase(case, pool_fill=0.0)
    g.setup()
    torch.cuda.synchronize()
    sh = case.shape
    eb = np.zeros((case.num_blocks, 2, sh.n_kv_heads, 16, sh.head_dim))
    el = np.zeros((case.num_blocks, 2, 16, sh.rank))
    w = weights64(case)
    X = case.seq_hidden(0).double().numpy()
    oracle.append_pools(eb, el, X, np.arange(X.shape[0]), np.zeros(X.shape[0], dtype=int),
                        case.block_tables.numpy(), w["W_K"], w["W_V"], w["A_K"], w["A_V"],
                        sh.n_kv_heads, sh.head_dim, sh.rope_base)
    assert np.abs(g.base_pool.double().cpu().numpy() - eb).max() < 1e-5
    assert np.abs(g.lr_pool.double().cpu().numpy() - el).max() < 1e-5


def test_append_bad_indices_are_skipped(cuda_lib):
    case = I.shared_decode(n=32)
    g = GpuCase(case, pool_fill=0.0)
    dev = g.device
    X = case.seq_hidden(0, 0, 4).to(dev)
    pos = torch.tensor([0, 1, 10 ** 6, 3], dtype=torch.int32, device=dev)  # position beyond the table
    rows = torch.tensor([0, 5, 0, 0], dtype=torch.int32, device=dev)      # row 5 does not exist
    cuda_lib.append(g.cfg, X, pos, rows, g.block_tables, g.W_cat, g.base_pool, g.lr_pool, g.status)
    torch.cuda.synchronize()
    assert g.device_status() == 4
    assert float(g.base_pool[0, :, :, 1].float().abs().max()) == 0.0  # token 1 skipped
    assert float(g.base_pool[0, 1, :, 0].float().abs().max()) > 0.0   # token 0 written
