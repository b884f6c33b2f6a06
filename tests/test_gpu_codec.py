"""GPU parity of the compressed base pool (PolyKV codec, the abstract printed at
the end of the PReCache page: q8_0 keys, Walsh-Hadamard rotated 3-bit values)
against the codec oracle (oracle/polykv.py): the append's codes, and decode
over the compressed pool at every rank and both head dims."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import polykv
from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300.harness import GpuCase
from tests.parity import BF16_TOL, _hidden, assert_close, oracle_decode_rows, oracle_prefill_seq, weights64

pytestmark = pytest.mark.gpu
NAN = float("nan")


def _append_case(cuda_lib, gen, T, Hkv, d, r, positions, integer):
    h = 256
    cfg = cuda_lib.make_config(h, 2 * Hkv, Hkv, d, r, kv_codec=cuda_lib.CODEC_POLYKV)
    if integer:
        X = torch.randint(-1, 2, (T, h), generator=gen).to(torch.bfloat16)
        W = [torch.randint(0, 2, s, generator=gen).to(torch.bfloat16)
             for s in ((h, Hkv * d), (h, Hkv * d), (h, r), (h, r))]
    else:
        X = torch.randn(T, h, generator=gen).to(torch.bfloat16)
        W = [(torch.randn(*s, generator=gen) / 16).to(torch.bfloat16)
             for s in ((h, Hkv * d), (h, Hkv * d), (h, r), (h, r))]
    # one sequence per token: block table row t holds block perm[t]
    num_blocks = T + 5
    perm = torch.randperm(num_blocks, generator=gen)[:T].int()
    bt = perm.view(T, 1).repeat(1, 8).contiguous()  # positions < 16: block column 0
    seq = torch.arange(T, dtype=torch.int32)
    pos = torch.as_tensor(positions, dtype=torch.int32)
    dev = torch.device("cuda")
    base, lr = cuda_lib.new_pools(cfg, num_blocks, dev, fill=NAN)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cuda_lib.append(cfg, X.to(dev), pos.to(dev), seq.to(dev), bt.to(dev), cuda_lib.pack_w_cat(*W).to(dev),
                    base, lr, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = cuda_lib.unpack_codec_pool(cfg, base)
    pool = {"Kq": np.zeros((num_blocks, Hkv, 16, d), np.int8), "Ks": np.zeros((num_blocks, Hkv, 16, d // 32), np.float16),
            "Vq": np.zeros((num_blocks, Hkv, 16, d), np.uint8), "Vn": np.zeros((num_blocks, Hkv, 16), np.float32)}
    lp = np.full((num_blocks, 2, 16, r), np.nan)
    polykv.append_pools_codec(pool, lp, X.double().numpy(), pos.numpy(), seq.numpy(), bt.numpy(),
                              *[w.double().numpy() for w in W], Hkv, d, 10000.0)
    rows = [(int(perm[t]), int(pos[t]) % 16) for t in range(T)]
    blks, rws = (np.array(x) for x in zip(*rows))

    def at(a):  # token t's rows of a [num_blocks, Hkv, 16, ...] array -> [T, Hkv, ...]
        return a[blks, :, rws]
    return got, pool, at, base, lr, lp, rows, num_blocks


@pytest.mark.parametrize("d", [128, 64])
def test_codec_append_integer_inputs(cuda_lib, d):
    """Integer hidden states and 0/1 weights at position 0: K_base is integer
    and unrotated, so the q8_0 codes and scales are bit-exact; the value codes
    are decided from the exact integer V rows (a code may differ only where the
    rotated coordinate lies within rounding of a threshold); the norms agree to
    fp32 rounding; untouched rows keep their 0xFF bytes."""
    gen = torch.Generator().manual_seed(11)
    T, Hkv, r = 130, 3, 16
    got, want, at, base, lr, lp, rows, nb = _append_case(cuda_lib, gen, T, Hkv, d, r, [0] * T, True)
    assert np.array_equal(at(got["Kq"]), at(want["Kq"])), "q8_0 codes"
    assert np.array_equal(at(got["Ks"]).view(np.uint16), at(want["Ks"]).view(np.uint16)), "q8_0 scales"
    np.testing.assert_allclose(at(got["Vn"]), at(want["Vn"]), rtol=2e-7)
    diff = at(got["Vq"]).astype(int) - at(want["Vq"]).astype(int)
    assert (np.abs(diff) <= 1).all() and (diff != 0).sum() <= 4, f"value codes differ at {(diff != 0).sum()} places"
    lrg = lr.float().cpu().numpy()
    for (blk, row), t in zip(rows, range(T)):
        assert np.array_equal(lrg[blk, :, row], lp[blk, :, row])
    used = np.zeros(nb, bool)
    used[[b for b, _ in rows]] = True
    raw = base.cpu().numpy().reshape(nb, Hkv, -1)
    assert (raw[~used] == 255).all(), "blocks no token maps to are untouched"


def test_codec_append_random_positions(cuda_lib):
    """Random data at positions 0-15: the GPU rotates K in fp32 and the oracle in
    fp64, so a q8_0 code may differ by one where x / s lies within rounding of
    a half; every other code and every scale agrees."""
    gen = torch.Generator().manual_seed(12)
    T, Hkv, d, r = 96, 4, 128, 8
    pos = torch.randint(0, 16, (T,), generator=gen).tolist()
    got, want, at, *_ = _append_case(cuda_lib, gen, T, Hkv, d, r, pos, False)
    dk = at(got["Kq"]).astype(int) - at(want["Kq"]).astype(int)
    assert (np.abs(dk) <= 1).all() and (dk != 0).mean() < 1e-3
    np.testing.assert_allclose(at(got["Ks"]).astype(np.float64), at(want["Ks"]).astype(np.float64), rtol=1e-3)
    dv = at(got["Vq"]).astype(int) - at(want["Vq"]).astype(int)
    assert (np.abs(dv) <= 1).all() and (dv != 0).mean() < 1e-3
    np.testing.assert_allclose(at(got["Vn"]), at(want["Vn"]), rtol=1e-5)


CASES = {
    # rank 64, one query per context (the long decode's item shape), ragged last context
    "r64_one_query": dict(rank=64, n_ctx=3, q_per_ctx=1, n=700),
    # rank 16, four agents on one context (g = 4: one query's heads per item)
    "r16_shared": dict(rank=16, n_ctx=1, n=900),
    # rank 8, g = 2, three queries per context: two rows per item
    "r8_g2": dict(rank=8, n_ctx=2, q_per_ctx=3, n=500, n_q_heads=16, n_kv_heads=8),
    # d = 64, rank 32
    "d64_r32": dict(rank=32, n_ctx=2, q_per_ctx=2, n=600, head_dim=64),
    # g = 8: two items per query
    "r16_g8": dict(rank=16, n_ctx=1, q_per_ctx=2, n=400, n_q_heads=32, n_kv_heads=4),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_codec_decode(cuda_lib, name):
    case = I.codec_decode(**CASES[name])
    g = GpuCase(case, pool_fill=NAN)
    g.setup()
    res = g.step()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    got = res["decode"].double().cpu().numpy()
    assert_close(got, oracle_decode_rows(case, cache="bf16"), BF16_TOL, name)
    # the compressed pool really is read: the uncompressed result differs by the codec's error
    sh = case.shape
    w64 = weights64(case)
    X, _ = _hidden(case, case.dec_ctx[0])
    n0 = int(case.dec_q_start[1])
    ref = oracle.decode(X, case.dec_q[:n0].double().numpy(), case.dec_adapter[:n0].numpy(), w64,
                        sh.n_kv_heads, sh.head_dim, sh.rope_base, 1 / math.sqrt(sh.head_dim))
    rel = np.linalg.norm(got[:n0] - ref) / np.linalg.norm(ref)
    assert rel > 1e-3, "decode over the compressed pool matches the uncompressed cache too closely"


@pytest.mark.parametrize("rank", [16, 64])
def test_codec_decode_without_adapter_factors(cuda_lib, rank):
    """B_K = NULL (no rebuild: the expanded K^ is scored directly), then B_V = NULL."""
    case = I.codec_decode(rank=rank, n_ctx=2, q_per_ctx=2, n=300)
    g = GpuCase(case, pool_fill=NAN)
    g.setup()
    w64 = weights64(case)
    for drop in ("B_K", "B_V"):
        bk = None if drop == "B_K" else g.B_K
        bv = None if drop == "B_V" else g.B_V
        out = cuda_lib.attn_decode(g.cfg, g.dec_q, g.dec_q_start, g.dec_adapter, g.dec_bt, g.dec_lens,
                                   g.dec_max_len, g.dec_max_q, g.base_pool, g.lr_pool, bk, bv, g.scale)
        torch.cuda.synchronize()
        w = dict(w64)
        w[drop] = np.zeros_like(w[drop])
        assert_close(out.double().cpu().numpy(), oracle_decode_rows(case, w64=w, cache="bf16"), BF16_TOL,
                     f"without {drop}")


@pytest.mark.parametrize("rank,d", [(16, 128), (64, 128), (8, 64), (32, 64)])
def test_codec_prefill(cuda_lib, rank, d):
    """Each agent's chunk over the shared prefix plus its own chunk, read from a
    compressed pool: keys and values expanded in the rebuild warpgroup, the
    output rotated back in the epilogue. Every row against the codec oracle."""
    case = I.codec_prefill(prefix=160, chunk=45, n_agents=3, rank=rank, head_dim=d)
    g = GpuCase(case, pool_fill=NAN)
    g.setup()
    res = g.step()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    got, want = [], []
    for p in range(g.n_pre):
        rows, w = oracle_prefill_seq(case, p, cache="bf16")
        got.append(res["prefill"][rows].double().cpu().numpy())
        want.append(w)
    assert_close(np.concatenate([x.reshape(-1) for x in got]), np.concatenate([x.reshape(-1) for x in want]),
                 BF16_TOL, f"r={rank} d={d}")


def test_codec_prefill_without_adapter_factors(cuda_lib):
    """B_K = NULL: no rebuild; the expanded K^ is scored directly (fp16)."""
    case = I.codec_prefill(prefix=64, chunk=33, n_agents=2, rank=16)
    g = GpuCase(case, pool_fill=NAN)
    g.setup()
    g.step_append()  # the chunks' own tokens
    w64 = weights64(case)
    out = cuda_lib.attn_prefill(g.cfg, g.pre_q, g.pre_q_start, g.pre_max_q, g.pre_lens, g.pre_max_len,
                                g.pre_adapter, g.pre_bt, g.base_pool, g.lr_pool, None, g.B_V, g.scale)
    torch.cuda.synchronize()
    w = dict(w64)
    w["B_K"] = np.zeros_like(w["B_K"])
    got, want = [], []
    for p in range(g.n_pre):
        rows, ww = oracle_prefill_seq(case, p, w64=w, cache="bf16")
        got.append(out[rows].double().cpu().numpy())
        want.append(ww)
    assert_close(np.concatenate([x.reshape(-1) for x in got]), np.concatenate([x.reshape(-1) for x in want]),
                 BF16_TOL, "without B_K")


def test_codec_prefill_last_row_equals_decode(cuda_lib):
    """The last row of a prefill chunk and a decode query at the same position
    over the same compressed context agree (both read the same codes)."""
    case = I.codec_prefill(prefix=208, chunk=17, n_agents=2, rank=16)
    g = GpuCase(case, pool_fill=NAN)
    g.setup()
    res = g.step()
    torch.cuda.synchronize()
    for p in range(g.n_pre):
        a, b = int(case.pre_q_start[p]), int(case.pre_q_start[p + 1])
        q = case.pre_q[b - 1:b].to("cuda")
        s = case.pre_seq[p]
        L = case.seqs[s].total_len
        dec = cuda_lib.attn_decode(g.cfg, q, torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                                   case.pre_adapter[p:p + 1].to("cuda"), g.pre_bt[p:p + 1].contiguous(),
                                   torch.tensor([L], dtype=torch.int32, device="cuda"), L, 1,
                                   g.base_pool, g.lr_pool, g.B_K, g.B_V, g.scale)
        torch.cuda.synchronize()
        assert_close(dec.double().cpu().numpy(), res["prefill"][b - 1:b].double().cpu().numpy(), BF16_TOL,
                     f"sequence {p}")
