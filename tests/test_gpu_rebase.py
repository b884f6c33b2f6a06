"""GPU parity of the re-based cache (PReCache, Abstract and Figure 1,
ReBaseShared): lrkv_append_rebase writes the base part of the cache from
adapter-free hidden states and the low-rank part from the adapted ones, in one
launch ("DB": both paths together) or as a base-only pass after an agent's turn
("LP"); attention then runs over the re-based cache unchanged. Checked against
the oracle's rebase_pools / agent_kv_rebased."""
import numpy as np
import pytest
import torch

import oracle
from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300 import lrkv
from rank_cache_attention_flash_b300.harness import GpuCase
from tests.parity import BF16_TOL, assert_close, weights64

pytestmark = pytest.mark.gpu
NAN = float("nan")


def _bits_close(got: torch.Tensor, want: torch.Tensor, ulps: int, abs_slack: float = 0.0):
    """Within `ulps` bf16 ulps of the larger magnitude, plus an absolute slack."""
    a, b = got.float(), want.float()
    big = torch.maximum(a.abs(), b.abs())
    ulp = torch.where(big > 0, torch.exp2(torch.floor(torch.log2(big.clamp(min=1e-30))) - 7),
                      torch.zeros_like(big))
    return bool(((a - b).abs() <= ulps * ulp + abs_slack).all())


# K_base is the fp32 rotation of integer projections |y| <= 256 (h = 256): the
# rotation's fp32 cos/sin carry an absolute error near 2^-21, so a K value
# whose exact rotation nearly cancels to 0 lands within 256 * 2^-21 ~ 1.2e-4 of
# it rather than within one bf16 ulp of a tiny number.
K_ABS_SLACK = 3e-4


@pytest.mark.parametrize("mode", ["both", "base_only", "lowrank_only"])
def test_append_rebase_integer_sources(cuda_lib, mode):
    """Integer hidden states and 0/1 weights: V_base, L_K, L_V exact, K_base
    within 1 bf16 ulp; the part whose source is NULL keeps its sentinel."""
    gen = torch.Generator().manual_seed(5)
    h, Hkv, d, r = 256, 2, 128, 16
    cfg = cuda_lib.make_config(h, 4, Hkv, d, r)
    n_seq, max_blocks, num_blocks = 2, 8, 20
    bt = torch.randperm(num_blocks, generator=gen)[: n_seq * max_blocks].view(n_seq, max_blocks).int()
    T = 150  # two token tiles, ragged; distinct (sequence, position) slots
    slot = torch.randperm(n_seq * max_blocks * 16, generator=gen)[:T]
    seq = (slot // (max_blocks * 16)).int()
    pos = (slot % (max_blocks * 16)).int()
    Xb = torch.randint(-1, 2, (T, h), generator=gen).to(torch.bfloat16)
    Xl = torch.randint(-1, 2, (T, h), generator=gen).to(torch.bfloat16)
    W = {k: torch.randint(0, 2, (h, n), generator=gen).to(torch.bfloat16)
         for k, n in (("W_K", Hkv * d), ("W_V", Hkv * d), ("A_K", r), ("A_V", r))}
    dev = torch.device("cuda")
    base, lr = cuda_lib.new_pools(cfg, num_blocks, dev)
    base.view(torch.int16).fill_(-1)
    lr.view(torch.int16).fill_(-1)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    xb = None if mode == "lowrank_only" else Xb
    xl = None if mode == "base_only" else Xl
    cuda_lib.append_rebase(cfg, None if xb is None else xb.to(dev), None if xl is None else xl.to(dev),
                           pos.to(dev), seq.to(dev), bt.to(dev),
                           cuda_lib.pack_w_cat(W["W_K"], W["W_V"], W["A_K"], W["A_V"]).to(dev), base, lr, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    eb = np.full((num_blocks, 2, Hkv, 16, d), np.nan)
    el = np.full((num_blocks, 2, 16, r), np.nan)
    oracle.rebase_pools(eb, el, None if xb is None else xb.double().numpy(),
                        None if xl is None else xl.double().numpy(), pos.numpy(), seq.numpy(), bt.numpy(),
                        *(W[k].double().numpy() for k in ("W_K", "W_V", "A_K", "A_V")), Hkv, d, 10000.0)
    gb, gl = base.cpu(), lr.cpu()
    for got, exp, is_base in ((gb, eb, True), (gl, el, False)):
        written = torch.from_numpy(~np.isnan(exp))
        sentinel = got.view(torch.int16) == -1
        assert bool(sentinel[~written].all()), "a part with no source was written"
        want = torch.from_numpy(np.nan_to_num(exp)).to(torch.bfloat16)
        if not bool(written.any()):
            continue
        if is_base:
            vm = written[:, 1]
            assert torch.equal(got[:, 1][vm].view(torch.int16), want[:, 1][vm].view(torch.int16)), "V_base"
            km = written[:, 0]
            assert _bits_close(got[:, 0][km], want[:, 0][km], 1, K_ABS_SLACK), "K_base beyond 1 ulp"
        else:
            assert torch.equal(got[written].view(torch.int16), want[written].view(torch.int16)), "L_K / L_V"


def test_lazy_rebase_equals_batched_rebase(cuda_lib):
    """LP scheduling (the ordinary append during the turn, then a base-only
    re-base from the adapter-free states) leaves the same pools, bit for bit,
    as DB scheduling (one launch with both sources)."""
    case = I.prefill_chunk(prefix=96, chunk=50, n_agents=2)
    g1 = GpuCase(case, pool_fill=0.0)
    g2 = GpuCase(case, pool_fill=0.0)
    dev = g1.device
    for s, a, b in list(case.setup_appends()) + list(case.step_appends()):
        Xl = case.seq_hidden(s, a, b).to(dev)
        Xb = case.seq_hidden_neutral(s, a, b).to(dev)
        pos = torch.arange(a, b, dtype=torch.int32, device=dev)
        rows = torch.full((b - a,), s, dtype=torch.int32, device=dev)
        cuda_lib.append(g1.cfg, Xl, pos, rows, g1.block_tables, g1.W_cat, g1.base_pool, g1.lr_pool, g1.status)
        cuda_lib.append_rebase(g1.cfg, Xb, None, pos, rows, g1.block_tables, g1.W_cat, g1.base_pool,
                               g1.lr_pool, g1.status)
        cuda_lib.append_rebase(g2.cfg, Xb, Xl, pos, rows, g2.block_tables, g2.W_cat, g2.base_pool,
                               g2.lr_pool, g2.status)
    torch.cuda.synchronize()
    assert g1.device_status() == 0 and g2.device_status() == 0
    assert torch.equal(g1.base_pool.view(torch.int16), g2.base_pool.view(torch.int16))
    assert torch.equal(g1.lr_pool.view(torch.int16), g2.lr_pool.view(torch.int16))


def _rebased(case):
    """GpuCase whose every append is re-based: base part from the adapter-free
    states, low-rank part from the adapted states (one launch per append)."""
    g = GpuCase(case, pool_fill=NAN)
    dev = g.device
    for s, a, b in list(case.setup_appends()) + list(case.step_appends()):
        Xl = case.seq_hidden(s, a, b).to(dev)
        Xb = case.seq_hidden_neutral(s, a, b).to(dev)
        pos = torch.arange(a, b, dtype=torch.int32, device=dev)
        rows = torch.full((b - a,), s, dtype=torch.int32, device=dev)
        lrkv.append_rebase(g.cfg, Xb, Xl, pos, rows, g.block_tables, g.W_cat, g.base_pool, g.lr_pool, g.status)
    return g


def test_rebased_cache_decode(cuda_lib):
    case = I.shared_decode(n=700)
    g = _rebased(case)
    out = g.decode()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    sh = case.shape
    w64 = weights64(case)
    Xl = case.seq_hidden(0).double().numpy()
    Xb = case.seq_hidden_neutral(0).double().numpy()
    want = oracle.decode(Xb, case.dec_q.double().numpy(), case.dec_adapter.numpy(), w64, sh.n_kv_heads,
                         sh.head_dim, sh.rope_base, 1 / np.sqrt(sh.head_dim), "bf16", X_lr=Xl)
    assert_close(out.double().cpu().numpy(), want, BF16_TOL, "re-based decode")
    # the re-base changes the result (the base part really comes from the other states)
    plain = oracle.decode(Xl, case.dec_q.double().numpy(), case.dec_adapter.numpy(), w64, sh.n_kv_heads,
                          sh.head_dim, sh.rope_base, 1 / np.sqrt(sh.head_dim), "bf16")
    assert np.abs(plain - want).max() > 0.1


def test_rebased_cache_prefill(cuda_lib):
    case = I.prefill_chunk(prefix=272, chunk=77, n_agents=2)
    g = _rebased(case)
    out = g.prefill()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    sh = case.shape
    w64 = weights64(case)
    for p in range(g.n_pre):
        s = case.pre_seq[p]
        a, b = int(case.pre_q_start[p]), int(case.pre_q_start[p + 1])
        want = oracle.prefill(case.seq_hidden_neutral(s).double().numpy(), case.pre_q[a:b].double().numpy(),
                              int(case.pre_adapter[p]), w64, sh.n_kv_heads, sh.head_dim, sh.rope_base,
                              1 / np.sqrt(sh.head_dim), "bf16", X_lr=case.seq_hidden(s).double().numpy())
        assert_close(out[a:b].double().cpu().numpy(), want, BF16_TOL, f"re-based prefill seq {p}")
