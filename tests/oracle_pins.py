"""Pins for the fp64 oracle: checks against facts fixed outside the oracle itself.

Each ``pin_*`` takes a namespace ``O`` that provides the oracle's functions, so
the mutation tests can hand in a deliberately broken copy and confirm that some
pin fails. Pins use: hand-derived closed forms, a library routine
(``torch.nn.functional.scaled_dot_product_attention`` in float64), brute force
with Python floats/ints on tiny inputs, and algebraic invariants.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- RoPE pins
def pin_rope_closed_form(O):
    """d = 4, base = 100, t = 3, x = [1, 2, 3, 4]: theta = [1, 0.1]; pairs (0, 2)
    and (1, 3) (rotate-half). Values written out by hand."""
    x = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    got = O.apply_rope(x, np.array([3]), 100.0)[0, 0]
    a0, a1 = 3.0 * 1.0, 3.0 * 0.1
    want = [1 * math.cos(a0) - 3 * math.sin(a0),
            2 * math.cos(a1) - 4 * math.sin(a1),
            3 * math.cos(a0) + 1 * math.sin(a0),
            4 * math.cos(a1) + 2 * math.sin(a1)]
    assert np.allclose(got, want, rtol=0, atol=1e-14), (got, want)


def pin_rope_frequencies(O):
    """theta_j = base^(-2j/d): for d = 8, base = 10000 -> 1, 0.1, 0.01, 0.001."""
    got = O.rope_inv_freq(8, 10000.0)
    assert np.allclose(got, [1.0, 0.1, 0.01, 0.001], rtol=1e-15, atol=0)


def pin_rope_invariants(O):
    r = _rng(1)
    x = r.standard_normal((5, 3, 64))
    pos = np.array([0, 1, 7, 4095, 32767])
    y = O.apply_rope(x, pos, 10000.0)
    assert np.array_equal(y[0], x[0])                     # position 0: identity
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    # scores depend on the position difference only
    q = r.standard_normal((1, 1, 64))
    k = r.standard_normal((1, 1, 64))
    for p, t, c in [(5, 2, 32768 - 5), (100, 0, 1000), (17, 16, 12345)]:
        s1 = float(np.sum(O.apply_rope(q, np.array([p]), 10000.0) * O.apply_rope(k, np.array([t]), 10000.0)))
        s2 = float(np.sum(O.apply_rope(q, np.array([p + c]), 10000.0) * O.apply_rope(k, np.array([t + c]), 10000.0)))
        assert abs(s1 - s2) < 1e-9, (s1, s2)


# ----------------------------------------------------------- attention pins
def _sdpa(q, K, V, causal):
    """Library routine: torch SDPA in float64 on CPU, GQA handled by torch."""
    qt = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))[None]   # [1, Hq, N, d]
    kt = torch.from_numpy(np.ascontiguousarray(K.transpose(1, 0, 2)))[None]
    vt = torch.from_numpy(np.ascontiguousarray(V.transpose(1, 0, 2)))[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal,
                                                         enable_gqa=True)
    return o[0].numpy().transpose(1, 0, 2)


def pin_attention_sdpa_decode(O):
    """One query at the last position sees every key: plain SDPA, no mask."""
    r = _rng(2)
    L, Hq, Hkv, d = 37, 8, 2, 16
    K = r.standard_normal((L, Hkv, d))
    V = r.standard_normal((L, Hkv, d))
    q = r.standard_normal((1, Hq, d))
    got = O.gqa_attention(q, [L - 1], K, V, 1 / math.sqrt(d))
    want = _sdpa(q, K, V, causal=False)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-13)


def pin_attention_sdpa_prefill(O):
    """Full-length causal prefill (queries = keys, square mask) against SDPA's
    is_causal; then a trailing chunk must equal the last rows of the full run
    (bottom-right alignment)."""
    r = _rng(3)
    L, Hq, Hkv, d = 29, 6, 3, 8
    K = r.standard_normal((L, Hkv, d))
    V = r.standard_normal((L, Hkv, d))
    q = r.standard_normal((L, Hq, d))
    full = O.gqa_attention(q, np.arange(L), K, V, 1 / math.sqrt(d))
    assert np.allclose(full, _sdpa(q, K, V, causal=True), rtol=1e-12, atol=1e-13)
    n = 9
    chunk = O.gqa_attention(q[-n:], np.arange(L - n, L), K, V, 1 / math.sqrt(d))
    assert np.allclose(chunk, full[-n:], rtol=1e-13, atol=1e-14)


def pin_attention_brute_force(O):
    """Python floats and math.exp, one loop per term, on a tiny GQA case."""
    r = _rng(4)
    L, Hq, Hkv, d = 5, 4, 2, 3
    K = r.standard_normal((L, Hkv, d))
    V = r.standard_normal((L, Hkv, d))
    q = r.standard_normal((2, Hq, d))
    pos = [2, 4]
    scale = 0.7
    got = O.gqa_attention(q, pos, K, V, scale)
    for n in range(2):
        for m in range(Hq):
            kv = m // (Hq // Hkv)
            sc = [scale * sum(q[n, m, j] * K[t, kv, j] for j in range(d)) for t in range(pos[n] + 1)]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            z = sum(w)
            for j in range(d):
                o = sum(w[t] * V[t, kv, j] for t in range(pos[n] + 1)) / z
                assert abs(got[n, m, j] - o) < 1e-13


def pin_attention_special_cases(O):
    r = _rng(5)
    Hq, Hkv, d = 4, 2, 8
    # one key: the output is that key's value
    K = r.standard_normal((1, Hkv, d))
    V = r.standard_normal((1, Hkv, d))
    q = r.standard_normal((1, Hq, d))
    o = O.gqa_attention(q, [0], K, V, 1.0)
    assert np.allclose(o[0], np.repeat(V[0], Hq // Hkv, axis=0), atol=1e-15)
    # zero query: the mean of the visible values
    L = 11
    K = r.standard_normal((L, Hkv, d))
    V = r.standard_normal((L, Hkv, d))
    o = O.gqa_attention(np.zeros((1, Hq, d)), [6], K, V, 1.0)
    assert np.allclose(o[0], np.repeat(V[:7].mean(axis=0), Hq // Hkv, axis=0), atol=1e-14)
    # one dominant key: its value
    K = np.zeros((L, Hkv, d))
    K[3, :, 0] = 1000.0
    q = np.zeros((1, Hq, d))
    q[0, :, 0] = 1.0
    o = O.gqa_attention(q, [L - 1], K, V, 1.0)
    assert np.allclose(o[0], np.repeat(V[3], Hq // Hkv, axis=0), atol=1e-12)


# -------------------------------------------------------- LoRA / cache pins
def pin_lora_closed_form(O):
    """h = 1, one kv head, d = 2, r = 1, two tokens X = [[1], [2]] at positions 0, 1.
    W_K = [[1, 0]], A_K = [[1]], B_K = [[0, 1]] -> K_pre[t] = X[t] * [1, 1];
    W_V = [[0, 1]], A_V = [[2]], B_V = [[1, 0]] -> V[t] = X[t] * [2, 1].
    base = 1 so theta_0 = 1. Query q = [1, 0] at position 1, scale 1:
      K[0] = [1, 1]; K[1] = RoPE_1([2, 2]) = [2cos1 - 2sin1, 2cos1 + 2sin1]
      s0 = 1, s1 = 2cos1 - 2sin1; o = (e^s0 V[0] + e^s1 V[1]) / (e^s0 + e^s1)."""
    w = {"W_K": np.array([[1.0, 0.0]]), "W_V": np.array([[0.0, 1.0]]),
         "A_K": np.array([[1.0]]), "A_V": np.array([[2.0]]),
         "B_K": np.array([[[0.0, 1.0]]]), "B_V": np.array([[[1.0, 0.0]]])}
    X = np.array([[1.0], [2.0]])
    q = np.array([[[1.0, 0.0]]])
    got = O.attend(X, 0, q, [1], w, 1, 2, 1.0, 1.0)[0, 0]
    s0, s1 = 1.0, 2 * math.cos(1.0) - 2 * math.sin(1.0)
    e0, e1 = math.exp(s0), math.exp(s1)
    want = [(e0 * 2 + e1 * 4) / (e0 + e1), (e0 * 1 + e1 * 2) / (e0 + e1)]
    assert np.allclose(got, want, rtol=0, atol=1e-14), (got, want)
    # adapter -1: B = 0 -> K = [1, 0] * X, V = [0, 1] * X
    got0 = O.attend(X, -1, q, [1], w, 1, 2, 1.0, 1.0)[0, 0]
    s1b = 2 * math.cos(1.0)
    e0, e1 = math.exp(1.0), math.exp(s1b)
    want0 = [0.0, (e0 * 1 + e1 * 2) / (e0 + e1)]
    assert np.allclose(got0, want0, rtol=0, atol=1e-14), (got0, want0)


def _small_weights(r, h=24, Hkv=2, d=8, rank=3, na=3):
    return {"W_K": r.standard_normal((h, Hkv * d)), "W_V": r.standard_normal((h, Hkv * d)),
            "A_K": r.standard_normal((h, rank)), "A_V": r.standard_normal((h, rank)),
            "B_K": r.standard_normal((na, rank, Hkv * d)),
            "B_V": r.standard_normal((na, rank, Hkv * d))}


def pin_merged_weights(O):
    """Dense per-agent recomputation with merged weights W + A·B_i (one GEMM per
    projection, the "non-shared" cache of that agent) equals the factored form."""
    r = _rng(6)
    w = _small_weights(r)
    X = r.standard_normal((13, 24))
    pos = np.arange(13) + 5
    for i in range(3):
        k1, v1 = O.agent_kv(X, pos, w["W_K"], w["W_V"], w["A_K"], w["A_V"], w["B_K"][i],
                            w["B_V"][i], 2, 8, 10000.0)
        WK = w["W_K"] + w["A_K"] @ w["B_K"][i]
        WV = w["W_V"] + w["A_V"] @ w["B_V"][i]
        k2, v2 = O.agent_kv(X, pos, WK, WV, w["A_K"], w["A_V"], None, None, 2, 8, 10000.0)
        assert np.allclose(k1, k2, rtol=1e-12, atol=1e-12)
        assert np.allclose(v1, v2, rtol=1e-12, atol=1e-12)


def pin_reordered_equals_materialised(O):
    """The reordered evaluation (what the kernels do) equals the materialised one:
    K_i = K_base + RoPE(L_K·B_K,i) and P·V_i = P·V_base + (P·L_V)·B_V,i."""
    r = _rng(7)
    h, Hq, Hkv, d, rank = 24, 4, 2, 8, 3
    w = _small_weights(r, h, Hkv, d, rank)
    L = 21
    X = r.standard_normal((L, h))
    pos = np.arange(L)
    kb, vb, lk, lv = O.base_and_lowrank(X, pos, w["W_K"], w["W_V"], w["A_K"], w["A_V"],
                                        Hkv, d, 10000.0)
    q = r.standard_normal((1, Hq, d))
    scale = 1 / math.sqrt(d)
    for i in range(3):
        want = O.attend(X, i, q, [L - 1], w, Hkv, d, 10000.0, scale)[0]
        adapter_k = O.apply_rope((lk @ w["B_K"][i]).reshape(L, Hkv, d), pos, 10000.0)
        Ki = kb + adapter_k
        for m in range(Hq):
            kv = m // (Hq // Hkv)
            s = Ki[:, kv, :] @ q[0, m] * scale
            p = np.exp(s - s.max())
            p /= p.sum()
            o = p @ vb[:, kv, :] + (p @ lv) @ w["B_V"][i][:, kv * d:(kv + 1) * d]
            assert np.allclose(o, want[m], rtol=1e-12, atol=1e-12)


def pin_base_equals_ordinary_attention(O):
    """B = 0 (adapter -1): attend() is ordinary GQA attention over K = RoPE(X·W_K),
    V = X·W_V, checked against SDPA."""
    r = _rng(8)
    h, Hq, Hkv, d = 16, 4, 2, 8
    w = _small_weights(r, h, Hkv, d, 3)
    L = 19
    X = r.standard_normal((L, h))
    q = r.standard_normal((1, Hq, d))
    got = O.attend(X, -1, q, [L - 1], w, Hkv, d, 10000.0, 1 / math.sqrt(d))
    K = O.apply_rope((X @ w["W_K"]).reshape(L, Hkv, d), np.arange(L), 10000.0)
    V = (X @ w["W_V"]).reshape(L, Hkv, d)
    assert np.allclose(got, _sdpa(q, K, V, causal=False), rtol=1e-12, atol=1e-13)


def pin_append_integer_bruteforce(O):
    """Integer-valued X and 0/1 weights: the projections are exact integer sums,
    recomputed with Python ints; position 0 rotation is the identity, so K_base
    there is exact too. Pool rows land at block_tables[s][p // 16], row p % 16."""
    r = _rng(9)
    h, Hkv, d, rank = 12, 2, 4, 2
    X = r.integers(-3, 4, size=(5, h)).astype(np.float64)
    WK = r.integers(0, 2, size=(h, Hkv * d)).astype(np.float64)
    WV = r.integers(0, 2, size=(h, Hkv * d)).astype(np.float64)
    AK = r.integers(0, 2, size=(h, rank)).astype(np.float64)
    AV = r.integers(0, 2, size=(h, rank)).astype(np.float64)
    pos = np.array([0, 17, 3, 40, 0])
    seqs = np.array([0, 0, 1, 1, 1])
    bt = np.array([[4, 2, 9], [7, 0, 5]])
    nb = 10
    bp = np.full((nb, 2, Hkv, 16, d), np.nan)
    lp = np.full((nb, 2, 16, rank), np.nan)
    O.append_pools(bp, lp, X, pos, seqs, bt, WK, WV, AK, AV, Hkv, d, 10000.0)

    def isum(row, W, col):
        return sum(int(X[row, k]) * int(W[k, col]) for k in range(h))

    written = set()
    for n in range(5):
        blk = {(0, 0): 4, (0, 1): 2, (1, 0): 7, (1, 2): 5}[(int(seqs[n]), int(pos[n]) // 16)]
        row = int(pos[n]) % 16
        written.add((blk, row))
        for hh in range(Hkv):
            for j in range(d):
                assert bp[blk, 1, hh, row, j] == isum(n, WV, hh * d + j)
                if pos[n] == 0:
                    assert bp[blk, 0, hh, row, j] == isum(n, WK, hh * d + j)
        for k in range(rank):
            assert lp[blk, 0, row, k] == isum(n, AK, k)
            assert lp[blk, 1, row, k] == isum(n, AV, k)
    for blk in range(nb):
        for row in range(16):
            if (blk, row) not in written:
                assert np.isnan(bp[blk, :, :, row]).all() and np.isnan(lp[blk, :, row]).all()


def pin_prefill_last_row_equals_decode(O):
    r = _rng(10)
    h, Hq, Hkv, d = 16, 4, 2, 8
    w = _small_weights(r, h, Hkv, d, 3)
    L = 23
    X = r.standard_normal((L, h))
    qc = r.standard_normal((6, Hq, d))
    pre = O.prefill(X, qc, 1, w, Hkv, d, 10000.0, 0.3)
    dec = O.decode(X, qc[-1:], [1], w, Hkv, d, 10000.0, 0.3)
    assert np.allclose(pre[-1], dec[0], rtol=1e-13, atol=1e-14)


def pin_multi_agent_batch(O):
    """Several agents' queries on one context equal the same queries one at a time."""
    r = _rng(11)
    h, Hq, Hkv, d = 16, 4, 2, 8
    w = _small_weights(r, h, Hkv, d, 3)
    L = 15
    X = r.standard_normal((L, h))
    q = r.standard_normal((4, Hq, d))
    ad = [2, -1, 0, 2]
    both = O.decode(X, q, ad, w, Hkv, d, 10000.0, 0.5)
    for n in range(4):
        one = O.attend(X, ad[n], q[n:n + 1], [L - 1], w, Hkv, d, 10000.0, 0.5)
        assert np.allclose(both[n], one[0], rtol=1e-14, atol=1e-15)
    # and adapters really change the result
    assert not np.allclose(both[0], O.attend(X, -1, q[0:1], [L - 1], w, Hkv, d, 10000.0, 0.5)[0])


def pin_round_bf16_matches_library(O):
    """round_bf16 against torch's float32 -> bfloat16 conversion (round to
    nearest, ties to even), on random values and hand-picked ties."""
    r = _rng(12)
    x = np.concatenate([r.standard_normal(4000) * 10.0 ** r.integers(-6, 6, 4000),
                        [1.00390625, 1.01171875, -1.00390625, 3.0, 0.0, 65504.0, 1e-30]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.round_bf16(x), want)
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    assert O.round_bf16(np.array([1.00390625]))[0] == 1.0
    assert O.round_bf16(np.array([1.01171875]))[0] == 1.015625


def pin_bf16_cache_variant_is_exact_on_representable_data(O):
    """When every cache component is exactly representable in bf16 (small
    integers), the bf16-cache variant equals the exact materialisation."""
    r = _rng(13)
    h, Hkv, d, rank = 16, 2, 8, 2
    X = r.integers(-2, 3, size=(9, h)).astype(np.float64)
    W = {k: r.integers(0, 2, size=(h, n)).astype(np.float64)
         for k, n in (("W_K", Hkv * d), ("W_V", Hkv * d), ("A_K", rank), ("A_V", rank))}
    BK = r.standard_normal((rank, Hkv * d))
    BV = r.standard_normal((rank, Hkv * d))
    pos = np.zeros(9, dtype=int)  # position 0: the rotation is the identity, K_base stays integer
    k1, v1 = O.agent_kv(X, pos, W["W_K"], W["W_V"], W["A_K"], W["A_V"], BK, BV, Hkv, d, 10000.0)
    k2, v2 = O.agent_kv_from_cache(X, pos, W["W_K"], W["W_V"], W["A_K"], W["A_V"], BK, BV, Hkv, d, 10000.0)
    assert np.allclose(k1, k2, rtol=1e-13, atol=1e-13) and np.allclose(v1, v2, rtol=1e-13, atol=1e-13)
    # and on general data the two differ by about the bf16 spacing
    Xg = r.standard_normal((9, h))
    pg = np.arange(9)
    k1, _ = O.agent_kv(Xg, pg, W["W_K"], W["W_V"], W["A_K"], W["A_V"], BK, BV, Hkv, d, 10000.0)
    k2, _ = O.agent_kv_from_cache(Xg, pg, W["W_K"], W["W_V"], W["A_K"], W["A_V"], BK, BV, Hkv, d, 10000.0)
    rel = np.abs(k1 - k2).max() / np.abs(k1).max()
    assert 1e-5 < rel < 2 ** -7, rel


# ------------------------------------------------------ re-based cache pins
def pin_rebase_integer_bruteforce(O):
    """ReBaseShared append: base rows from one integer source, low-rank rows from
    another, recomputed with Python ints; a source of None leaves its part of
    the pools untouched (NaN sentinels)."""
    r = _rng(14)
    h, Hkv, d, rank = 10, 2, 4, 2
    Xb = r.integers(-3, 4, size=(4, h)).astype(np.float64)
    Xl = r.integers(-3, 4, size=(4, h)).astype(np.float64)
    W = {k: r.integers(0, 2, size=(h, n)).astype(np.float64)
         for k, n in (("W_K", Hkv * d), ("W_V", Hkv * d), ("A_K", rank), ("A_V", rank))}
    pos = np.array([0, 0, 16, 0])
    seqs = np.array([0, 1, 1, 2])
    bt = np.array([[3, 1], [0, 6], [5, 2]])
    slot = {0: (3, 0), 1: (0, 0), 2: (6, 0), 3: (5, 0)}

    def isum(X, n, M, col):
        return sum(int(X[n, k]) * int(M[k, col]) for k in range(h))

    for xb, xl in ((Xb, Xl), (Xb, None), (None, Xl)):
        bp = np.full((8, 2, Hkv, 16, d), np.nan)
        lp = np.full((8, 2, 16, rank), np.nan)
        O.rebase_pools(bp, lp, xb, xl, pos, seqs, bt, W["W_K"], W["W_V"], W["A_K"], W["A_V"], Hkv, d, 10000.0)
        for n in range(4):
            blk, row = slot[n]
            for hh in range(Hkv):
                for j in range(d):
                    if xb is None:
                        assert np.isnan(bp[blk, :, hh, row, j]).all()
                        continue
                    assert bp[blk, 1, hh, row, j] == isum(Xb, n, W["W_V"], hh * d + j)
                    if pos[n] == 0:
                        assert bp[blk, 0, hh, row, j] == isum(Xb, n, W["W_K"], hh * d + j)
            for k in range(rank):
                if xl is None:
                    assert np.isnan(lp[blk, :, row, k]).all()
                    continue
                assert lp[blk, 0, row, k] == isum(Xl, n, W["A_K"], k)
                assert lp[blk, 1, row, k] == isum(Xl, n, W["A_V"], k)


def pin_rebased_kv_stacked_weights(O):
    """A re-based agent's keys and values are one projection of the two sources
    side by side, [X_base | X_lr] times the stacked weights [W; A·B_i], before
    the rotation; with X_base = X_lr they are the ordinary agent_kv."""
    r = _rng(15)
    h, Hkv, d, rank = 12, 2, 8, 3
    w = _small_weights(r, h, Hkv, d, rank)
    T = 11
    Xb = r.standard_normal((T, h))
    Xl = r.standard_normal((T, h))
    pos = np.arange(T) + 3
    for i in range(3):
        k, v = O.agent_kv_rebased(Xb, Xl, pos, w["W_K"], w["W_V"], w["A_K"], w["A_V"], w["B_K"][i],
                                  w["B_V"][i], Hkv, d, 10000.0)
        XX = np.hstack([Xb, Xl])
        k_pre = XX @ np.vstack([w["W_K"], w["A_K"] @ w["B_K"][i]])
        v_want = XX @ np.vstack([w["W_V"], w["A_V"] @ w["B_V"][i]])
        assert np.allclose(k, O.apply_rope(k_pre.reshape(T, Hkv, d), pos, 10000.0), rtol=1e-12, atol=1e-12)
        assert np.allclose(v, v_want.reshape(T, Hkv, d), rtol=1e-12, atol=1e-12)
        k1, v1 = O.agent_kv(Xb, pos, w["W_K"], w["W_V"], w["A_K"], w["A_V"], w["B_K"][i], w["B_V"][i],
                            Hkv, d, 10000.0)
        k2, v2 = O.agent_kv_rebased(Xb, Xb, pos, w["W_K"], w["W_V"], w["A_K"], w["A_V"], w["B_K"][i],
                                    w["B_V"][i], Hkv, d, 10000.0)
        assert np.allclose(k1, k2, rtol=1e-13, atol=1e-13) and np.allclose(v1, v2, rtol=1e-13, atol=1e-13)
    # attention over the re-based cache: a query over K_i, V_i as defined above
    q = r.standard_normal((1, 4, d))
    got = O.attend(Xb, 1, q, [T - 1], w, Hkv, d, 10000.0, 0.4, X_lr=Xl)
    k, v = O.agent_kv_rebased(Xb, Xl, np.arange(T), w["W_K"], w["W_V"], w["A_K"], w["A_V"], w["B_K"][1],
                              w["B_V"][1], Hkv, d, 10000.0)
    assert np.allclose(got, _sdpa(q * 0.4 * math.sqrt(d), k, v, causal=False), rtol=1e-12, atol=1e-13)
    # the bf16-stored variant is exact when every component is bf16-representable
    Xi = r.integers(-2, 3, size=(T, h)).astype(np.float64)
    Xj = r.integers(-2, 3, size=(T, h)).astype(np.float64)
    Wi = {k_: r.integers(0, 2, size=x.shape).astype(np.float64) for k_, x in w.items() if k_[0] in "WA"}
    z = np.zeros(T, dtype=int)
    e1 = O.agent_kv_rebased(Xi, Xj, z, Wi["W_K"], Wi["W_V"], Wi["A_K"], Wi["A_V"], w["B_K"][0], w["B_V"][0],
                            Hkv, d, 10000.0)
    e2 = O.agent_kv_rebased(Xi, Xj, z, Wi["W_K"], Wi["W_V"], Wi["A_K"], Wi["A_V"], w["B_K"][0], w["B_V"][0],
                            Hkv, d, 10000.0, "bf16")
    assert np.allclose(e1[0], e2[0], rtol=1e-13, atol=1e-13) and np.allclose(e1[1], e2[1], rtol=1e-13, atol=1e-13)


# ------------------------------------------------ agent-specific A (PreLRShared)
def pin_prelr_merged_weights(O):
    """With agent-specific A_i (weights A_K, A_V of shape [G, h, r]), agent i's
    attention is ordinary attention over its own non-shared cache, one GEMM with
    the merged weights W + A_i B_i per projection (checked against SDPA); the
    agents' results differ; G = 1 equals the shared-A form."""
    r = _rng(16)
    h, Hq, Hkv, d, rank, G = 20, 4, 2, 8, 3, 3
    w = _small_weights(r, h, Hkv, d, rank, G)
    w["A_K"] = r.standard_normal((G, h, rank))
    w["A_V"] = r.standard_normal((G, h, rank))
    L = 17
    X = r.standard_normal((L, h))
    q = r.standard_normal((1, Hq, d))
    scale = 1 / math.sqrt(d)
    outs = []
    for i in range(G):
        got = O.attend(X, i, q, [L - 1], w, Hkv, d, 10000.0, scale)
        K = O.apply_rope((X @ (w["W_K"] + w["A_K"][i] @ w["B_K"][i])).reshape(L, Hkv, d), np.arange(L), 10000.0)
        V = (X @ (w["W_V"] + w["A_V"][i] @ w["B_V"][i])).reshape(L, Hkv, d)
        assert np.allclose(got, _sdpa(q * scale * math.sqrt(d), K, V, causal=False), rtol=1e-12, atol=1e-13)
        outs.append(got)
    assert not np.allclose(outs[0], outs[1])
    # base-only rows ignore A
    got0 = O.attend(X, -1, q, [L - 1], w, Hkv, d, 10000.0, scale)
    K = O.apply_rope((X @ w["W_K"]).reshape(L, Hkv, d), np.arange(L), 10000.0)
    assert np.allclose(got0, _sdpa(q, K, (X @ w["W_V"]).reshape(L, Hkv, d), causal=False), rtol=1e-12, atol=1e-13)
    # one group is the shared-A form
    w1 = dict(w)
    w1["A_K"], w1["A_V"] = w["A_K"][1:2], w["A_V"][1:2]
    w2 = dict(w)
    w2["A_K"], w2["A_V"] = w["A_K"][1], w["A_V"][1]
    assert np.allclose(O.attend(X, 0, q, [L - 1], w1, Hkv, d, 10000.0, scale),
                       O.attend(X, 0, q, [L - 1], w2, Hkv, d, 10000.0, scale), rtol=1e-14, atol=1e-15)


def pin_prelr_pool_bruteforce(O):
    """PreLRShared append on integer data: every agent's low-rank rows, side by
    side (group g in columns [g r, (g + 1) r)), recomputed with Python ints."""
    r = _rng(17)
    h, Hkv, d, rank, G = 9, 1, 4, 2, 3
    X = r.integers(-3, 4, size=(3, h)).astype(np.float64)
    WK = r.integers(0, 2, size=(h, Hkv * d)).astype(np.float64)
    WV = r.integers(0, 2, size=(h, Hkv * d)).astype(np.float64)
    AK = r.integers(-1, 2, size=(G, h, rank)).astype(np.float64)
    AV = r.integers(-1, 2, size=(G, h, rank)).astype(np.float64)
    pos = np.array([5, 0, 31])
    seqs = np.array([0, 1, 0])
    bt = np.array([[2, 0], [1, 3]])
    bp = np.full((4, 2, Hkv, 16, d), np.nan)
    lp = np.full((4, 2, 16, G * rank), np.nan)
    O.append_pools(bp, lp, X, pos, seqs, bt, WK, WV, AK, AV, Hkv, d, 10000.0)
    slot = {0: (2, 5), 1: (1, 0), 2: (0, 15)}
    for n in range(3):
        blk, row = slot[n]
        for g in range(G):
            for k in range(rank):
                want_k = sum(int(X[n, j]) * int(AK[g, j, k]) for j in range(h))
                want_v = sum(int(X[n, j]) * int(AV[g, j, k]) for j in range(h))
                assert lp[blk, 0, row, g * rank + k] == want_k
                assert lp[blk, 1, row, g * rank + k] == want_v


ALL_PINS = [
    pin_rope_closed_form, pin_rope_frequencies, pin_rope_invariants,
    pin_attention_sdpa_decode, pin_attention_sdpa_prefill, pin_attention_brute_force,
    pin_attention_special_cases, pin_lora_closed_form, pin_merged_weights,
    pin_reordered_equals_materialised, pin_base_equals_ordinary_attention,
    pin_append_integer_bruteforce, pin_prefill_last_row_equals_decode, pin_multi_agent_batch,
    pin_round_bf16_matches_library, pin_bf16_cache_variant_is_exact_on_representable_data,
    pin_rebase_integer_bruteforce, pin_rebased_kv_stacked_weights,
    pin_prelr_merged_weights, pin_prelr_pool_bruteforce,
]
