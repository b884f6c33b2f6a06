"""Full-size parity: the five workloads at their stated sizes, through the same
GpuCase path that bench.py times, every output row compared element by element
with the literal fp64 oracle (each agent's K and V materialised in full, then
textbook softmax attention).

The oracle's cost is one projection of each sequence's hidden states plus the
attention itself, seconds to tens of seconds per workload on the host cores, so
every decode query and every prefill row is checked, not a sample.
LRAgent (arXiv 2602.01053), Abstract, "preserving accuracy": the shared-cache
result must equal each agent's own non-shared result.

Gates, per workload ("config"):
  * every element within max(2e-2, one bf16 ulp of the oracle value);
  * relative Frobenius error <= 5e-3 over the workload's whole output (its
    decode rows and prefill rows together);
  * per sequence, the relative Frobenius error is within 5e-3 as well; where it
    is not (on some sequences the bf16 storage format alone, the exact result
    passed through a bf16 cache and a bf16 output, already exceeds 5e-3), the
    sequence must instead match the oracle's bf16-cache variant (the oracle's
    own fp64 cache components rounded to bf16, as the stored cache holds them)
    within the same tolerances: the kernels' own error stays inside the bound.
"""
import numpy as np
import pytest
import torch

import oracle
from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300.harness import GpuCase
from tests.parity import (assert_close, errors, oracle_decode_rows, oracle_prefill_seq, tol_for,
                          weights64)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _run(name):
    case = I.FULL[name]()
    g = GpuCase(case)
    g.setup()
    res = g.step()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    return case, g, res


def _per_sequence(got, want, case, what, cache_ref=None):
    """Per-sequence gate (see the module docstring). cache_ref() gives the
    oracle's bf16-cache variant of the same rows."""
    rf = errors(got, want)[1]
    if rf <= 5e-3 or case.shape.dtype == "fp32":
        return rf
    assert cache_ref is not None, f"{what}: rel_fro {rf:.3e}"
    ref = cache_ref()
    rf_fmt = errors(oracle.round_bf16(ref), want)[1]
    mx_c, rf_c = assert_close(got, ref, tol_for(case), f"{what} (against the bf16-cache oracle)")
    print(f"{what}: rel_fro {rf:.3e} (bf16 cache + bf16 output alone: {rf_fmt:.3e}); "
          f"against the bf16-cache oracle: max_abs {mx_c:.3e} rel_fro {rf_c:.3e}")
    return rf


def _prefill_all(case, g, res, w64):
    got_all, want_all = [], []
    for p in range(g.n_pre):
        rows, want = oracle_prefill_seq(case, p, w64=w64)
        assert len(rows) == int(case.pre_q_start[p + 1] - case.pre_q_start[p])
        got = res["prefill"][rows].double().cpu().numpy()
        _per_sequence(got, want, case, f"prefill seq {p}",
                      lambda p=p: oracle_prefill_seq(case, p, w64=w64, cache="bf16")[1])
        got_all.append(got)
        want_all.append(want)
    return got_all, want_all


def _whole(parts_got, parts_want, case, what):
    got = np.concatenate([x.reshape(-1) for x in parts_got])
    want = np.concatenate([x.reshape(-1) for x in parts_want])
    mx, rf = assert_close(got, want, tol_for(case), what)
    print(f"{what}: max_abs {mx:.3e} rel_fro {rf:.3e}")


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
    w64 = weights64(case)
    got = res["decode"].double().cpu().numpy()
    want = oracle_decode_rows(case, w64=w64)
    for n in range(16):
        _per_sequence(got[n], want[n], case, f"query {n}",
                      lambda n=n: oracle_decode_rows(case, rows=[n], w64=w64, cache="bf16")[0])
    _whole([got], [want], case, "long decode")


def test_full_prefill(cuda_lib):
    """All 512 rows of each of the 4 agents' chunks over the 16384-token prefix."""
    case, g, res = _run("prefill_chunk_llama8b")
    assert g.n_pre == 4
    got, want = _prefill_all(case, g, res, weights64(case))
    _whole(got, want, case, "prefill")


def test_full_mixed(cuda_lib):
    """All 48 decode queries and all 16 prefill chunks of the mixed batch."""
    case, g, res = _run("mixed_batch_qwen3_1p7b")
    assert case.dec_q.shape[0] == 48 and g.n_pre == 16
    w64 = weights64(case)
    dec_got = res["decode"].double().cpu().numpy()
    dec_want = oracle_decode_rows(case, w64=w64)
    for n in range(48):
        _per_sequence(dec_got[n], dec_want[n], case, f"decode query {n}",
                      lambda n=n: oracle_decode_rows(case, rows=[n], w64=w64, cache="bf16")[0])
    got, want = _prefill_all(case, g, res, w64)
    _whole([dec_got] + got, [dec_want] + want, case, "mixed batch")


def test_full_prelr_decode(cuda_lib):
    """The shared-context decode with agent-specific A (each agent its own
    low-rank group), all 4 queries against the literal oracle."""
    case, g, res = _run("prelr_decode_llama8b")
    assert case.shape.lr_groups == 4
    assert_close(res["decode"].double().cpu().numpy(), oracle_decode_rows(case), tol_for(case))


def test_full_rebase_prefill(cuda_lib):
    """The prefill workload over a re-based cache (base part from the
    adapter-free states), all rows against the literal oracle's
    K_i = RoPE(X_base W_K + X_lr A_K B_K,i)."""
    case, g, res = _run("rebase_prefill_llama8b")
    assert case.rebase
    got, want = _prefill_all(case, g, res, weights64(case))
    _whole(got, want, case, "re-based prefill")


def test_full_codec_long_decode(cuda_lib):
    """The long decode over a compressed base pool (PolyKV codec): all 16 queries,
    each over its whole 32768-token context, against the codec oracle (which
    encodes its own exact base part). Gated per configuration: whole-output
    relative Frobenius error <= 5e-3 and the per-element bound. Per query the
    error is reported, not gated: a code decided at a rounding boundary may
    differ by one step between the GPU's fp32 projections and the oracle's
    exact ones (test_full_codec_codes checks every such code), and when the
    token holding it dominates a head, that one step moves the head by a few
    tenths of a percent to a few percent."""
    case, g, res = _run("long_decode_codec_ministral8b")
    assert case.shape.kv_codec == 1 and case.dec_q.shape[0] == 16
    w64 = weights64(case)
    got = res["decode"].double().cpu().numpy()
    want = oracle_decode_rows(case, w64=w64)
    for n in range(16):
        mx, rf = errors(got[n], want[n])
        print(f"query {n}: max_abs {mx:.3e} rel_fro {rf:.3e}")
    _whole([got], [want], case, "compressed long decode")


def test_full_codec_prefill(cuda_lib):
    """The prefill-chunk workload over a compressed base pool: all 512 rows of
    each of the 4 agents' chunks against the codec oracle, gated per
    configuration like the compressed long decode (per-sequence errors
    reported)."""
    case, g, res = _run("prefill_chunk_codec_llama8b")
    assert case.shape.kv_codec == 1 and g.n_pre == 4
    w64 = weights64(case)
    got, want = [], []
    for p in range(g.n_pre):
        rows, w = oracle_prefill_seq(case, p, w64=w64)
        got.append(res["prefill"][rows].double().cpu().numpy())
        want.append(w)
        mx, rf = errors(got[-1], want[-1])
        print(f"prefill seq {p}: max_abs {mx:.3e} rel_fro {rf:.3e}")
    _whole(got, want, case, "compressed prefill")


def test_full_codec_codes(cuda_lib):
    """Every code of one 32768-token context of the compressed long decode
    against the codec oracle: keys and values, scales and norms. Codes are
    bit-exact except where the oracle's exact value lies within the GPU's rounding
    of a decision boundary (q8_0: x / s within the fast RoPE's error of a half;
    values: u within 1e-5 of a threshold), and there they differ by one step."""
    import oracle.lrkv_oracle as OL
    from oracle import polykv
    from tests.parity import _hidden
    case = I.codec_long_decode(n_seqs=4)
    g = GpuCase(case)
    g.setup()
    torch.cuda.synchronize()
    assert g.device_status() == 0
    pool = cuda_lib.unpack_codec_pool(g.cfg, g.base_pool)
    sh = case.shape
    w64 = weights64(case)
    ctx = case.dec_ctx[3]
    X, _ = _hidden(case, ctx)
    L = X.shape[0]
    pos = np.arange(L)
    bt = case.block_tables.numpy()[ctx]
    blk, row = bt[pos // 16], pos % 16
    kb, vb, _, _ = OL.base_and_lowrank(X, pos, w64["W_K"], w64["W_V"], w64["A_K"], w64["A_V"], sh.n_kv_heads,
                                      sh.head_dim, sh.rope_base)
    kq, ks = polykv.q8_0_encode(kb)
    vq, vn = polykv.tq3_encode(vb)
    gk, gks = pool["Kq"][blk, :, row], pool["Ks"][blk, :, row]
    gv, gvn = pool["Vq"][blk, :, row], pool["Vn"][blk, :, row]
    np.testing.assert_allclose(gks.astype(np.float64), ks.astype(np.float64), rtol=2 ** -10)
    np.testing.assert_allclose(gvn, vn, rtol=1e-5)
    dk = gk.astype(int) - kq.astype(int)
    # the decision is x / s with s = max |x| / 127 (unrounded); the GPU's keys carry
    # the fast RoPE's absolute error (<= 3e-4, as in the append tests), which moves
    # x / s by up to about 6e-4 / s (the key and the block's maximum both move)
    s_ex = np.repeat(np.abs(kb).reshape(kb.shape[:-1] + (-1, 32)).max(-1) / 127.0, 32, axis=-1)
    ratio = kb / np.where(s_ex > 0, s_ex, 1)
    frac = np.abs(np.abs(ratio) % 1 - 0.5)
    slack = 6e-4 / np.where(s_ex > 0, s_ex, 1) * (1 + np.abs(ratio) / 127)
    assert (np.abs(dk) <= 1).all() and (frac[dk != 0] < slack[dk != 0]).all() and (dk != 0).mean() < 1e-3
    dv = gv.astype(int) - vq.astype(int)
    _, t = polykv.centroids_thresholds()
    u = polykv.rotate(vb) * np.sqrt(sh.head_dim) / np.linalg.norm(vb, axis=-1, keepdims=True)
    dist = np.min(np.abs(u[..., None] - t), axis=-1)
    assert (np.abs(dv) <= 1).all() and (dist[dv != 0] < 1e-5).all() and (dv != 0).mean() < 1e-4
    print(f"key codes differing at a boundary: {(dk != 0).mean():.2e}; value codes: {(dv != 0).mean():.2e}")
