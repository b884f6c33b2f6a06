"""GPU parity of agent-specific low-rank caches (PReCache, Abstract and
Figure 1, PreLRShared): every agent a has its own A_K,a and A_V,a; one append
computes all agents' low-rank rows side by side (lr_groups = G groups of r
columns), and attention reads the agent's own group while the base part stays
shared. Checked against the oracle with A of shape [G, h, r]."""
import math

import numpy as np
import pytest
import torch

import oracle
from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300.harness import GpuCase
from tests.parity import BF16_TOL, FP32_TOL, assert_close, oracle_decode_rows, oracle_prefill_seq, weights64

pytestmark = pytest.mark.gpu
NAN = float("nan")


def _run(case, pool_fill=NAN):
    g = GpuCase(case, pool_fill=pool_fill)
    g.setup()
    res = g.step()
    torch.cuda.synchronize()
    return g, res


@pytest.mark.parametrize("G,r", [(3, 16), (8, 64), (2, 8)])
def test_prelr_append_integer_inputs_bit_exact(cuda_lib, G, r):
    """Integer hidden states, 0/1 base weights, A_g in {-1, 0, 1}: every group's
    L_K, L_V columns exact (one low-rank tile for 2 G r <= 256 columns, several
    for G = 8, r = 64)."""
    gen = torch.Generator().manual_seed(7)
    h, Hkv, d = 256, 2, 128
    cfg = cuda_lib.make_config(h, 4, Hkv, d, r, lr_groups=G)
    n_seq, max_blocks, num_blocks = 2, 6, 16
    bt = torch.randperm(num_blocks, generator=gen)[: n_seq * max_blocks].view(n_seq, max_blocks).int()
    T = 140
    slot = torch.randperm(n_seq * max_blocks * 16, generator=gen)[:T]
    seq = (slot // (max_blocks * 16)).int()
    pos = (slot % (max_blocks * 16)).int()
    X = torch.randint(-1, 2, (T, h), generator=gen).to(torch.bfloat16)
    WK = torch.randint(0, 2, (h, Hkv * d), generator=gen).to(torch.bfloat16)
    WV = torch.randint(0, 2, (h, Hkv * d), generator=gen).to(torch.bfloat16)
    AK = torch.randint(-1, 2, (G, h, r), generator=gen).to(torch.bfloat16)
    AV = torch.randint(-1, 2, (G, h, r), generator=gen).to(torch.bfloat16)
    dev = torch.device("cuda")
    base, lr = cuda_lib.new_pools(cfg, num_blocks, dev)
    assert lr.shape[-1] == G * r
    base.view(torch.int16).fill_(-1)
    lr.view(torch.int16).fill_(-1)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cuda_lib.append(cfg, X.to(dev), pos.to(dev), seq.to(dev), bt.to(dev),
                    cuda_lib.pack_w_cat(WK, WV, AK, AV).to(dev), base, lr, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    eb = np.full((num_blocks, 2, Hkv, 16, d), np.nan)
    el = np.full((num_blocks, 2, 16, G * r), np.nan)
    oracle.append_pools(eb, el, X.double().numpy(), pos.numpy(), seq.numpy(), bt.numpy(), WK.double().numpy(),
                        WV.double().numpy(), AK.double().numpy(), AV.double().numpy(), Hkv, d, 10000.0)
    written = torch.from_numpy(~np.isnan(el))
    got = lr.cpu()
    want = torch.from_numpy(np.nan_to_num(el)).to(torch.bfloat16)
    assert torch.equal(got[written].view(torch.int16), want[written].view(torch.int16)), "L_K / L_V groups"
    assert bool((got.view(torch.int16)[~written] == -1).all()), "untouched rows keep their sentinel"
    vm = torch.from_numpy(~np.isnan(eb[:, 1]))
    assert torch.equal(base.cpu()[:, 1][vm].view(torch.int16),
                       torch.from_numpy(np.nan_to_num(eb[:, 1])).to(torch.bfloat16)[vm].view(torch.int16)), "V_base"


def test_prelr_decode_agents_on_one_context(cuda_lib):
    """Four agents with their own A on one context (rank 16: items hold one
    query each, so each reads one low-rank group), with a base-only query."""
    case = I.shared_decode(n=600, n_agents=4, lr_groups=4)
    case.dec_adapter = torch.tensor([2, 0, -1, 3], dtype=torch.int32)
    g, res = _run(case)
    assert g.device_status() == 0
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL)
    # the groups really differ: the shared-A result of the same queries is far off
    w = weights64(case)
    w["A_K"], w["A_V"] = w["A_K"][0], w["A_V"][0]
    shared = oracle_decode_rows(case, w64=w, cache="bf16")
    assert np.abs(shared[0] - res["decode"][0].double().cpu().numpy()).max() > 0.05


def test_prelr_decode_rank64_rebuild_mode(cuda_lib):
    """Rank 64, one query per context (the rebuild-mode kernel), eight agents
    with their own A."""
    case = I.long_decode(n_seqs=3, n=450, lr_groups=8)
    g, res = _run(case)
    assert g.device_status() == 0
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case, cache="bf16"), BF16_TOL)


@pytest.mark.parametrize("rank", [16, 8])
def test_prelr_prefill(cuda_lib, rank):
    """Each agent's chunk over the shared prefix, reading its own low-rank group
    (rank 8: the 16-column tile reaches into the next group's columns, whose
    products meet zero B rows)."""
    case = I.prefill_chunk(prefix=96, chunk=45, n_agents=3, rank=rank, lr_groups=3)
    g, res = _run(case)
    assert g.device_status() == 0
    w64 = weights64(case)
    for p in range(g.n_pre):
        rows, want = oracle_prefill_seq(case, p, w64=w64, cache="bf16")
        assert_close(res["prefill"][rows].double().cpu().numpy(), want, BF16_TOL, f"r={rank} seq {p}")


def test_prelr_fp32(cuda_lib):
    """The fp32 path with two agents' own A (tolerance of the fp32 workload)."""
    case = I.tiny_fp32_decode(lr_groups=2)
    g, res = _run(case)
    assert g.device_status() == 0
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case), FP32_TOL)


def test_prelr_adapter_beyond_groups_rejected(cuda_lib):
    """More adapters than low-rank groups cannot be served: refused on the host."""
    case = I.shared_decode(n=64, n_agents=4, lr_groups=2)
    g = GpuCase(case, pool_fill=0.0)
    with pytest.raises(cuda_lib.LrkvError) as e:
        cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, g.dec_adapter, g.dec_bt, g.dec_lens, g.dec_max_len,
                             g.dec_max_q, g.base_pool, g.lr_pool, g.B_K, g.B_V, 1 / math.sqrt(128))
    assert e.value.code == 1
