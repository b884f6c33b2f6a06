"""The compressed-pool oracle (oracle/polykv.py) against its pins, and planted
mistakes that the pins must catch. CPU only.

Pins come from outside the oracle:
* the published 8-level Lloyd-Max quantiser for N(0, 1) (Max 1960) and its
  optimality conditions, checked by numerical integration;
* the Sylvester-Hadamard matrix from its entry formula (-1)^popcount(i & j);
* q8_0 on hand-worked blocks and the error bound of the format;
* nearest-centroid coding by brute force, and the quantiser's distortion on
  Gaussian vectors;
* attention over a pool whose base part the codec stores losslessly, which
  must equal the uncompressed oracle exactly.
"""
import os
import types

import numpy as np
import pytest

import oracle as O
from oracle import polykv as PK

PK_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "polykv.py")


def _rng(seed):
    return np.random.default_rng(1000 + seed)


# ---------------------------------------------------------------------------
# pins (each takes the module under test)

def pin_lloyd_max_gaussian(M):
    """Max (1960), 8-level quantiser for a unit Gaussian: output levels +-0.2451,
    +-0.7560, +-1.3440, +-2.1520, thresholds 0, +-0.5006, +-1.0500, +-1.7480,
    distortion 0.03455; and Lloyd's two conditions, by integration."""
    from scipy import integrate
    from scipy.stats import norm
    c, t = M.lloyd_max_gaussian()
    assert np.allclose(c[4:], [0.2451, 0.7560, 1.3440, 2.1520], atol=2e-4)
    assert np.allclose(c[:4], -c[4:][::-1], atol=0) and t[3] == 0.0
    assert np.allclose(t[4:], [0.5006, 1.0500, 1.7480], atol=2e-4)
    edges = np.concatenate([[-np.inf], t, [np.inf]])
    mse = 0.0
    for k in range(8):
        a, b = edges[k], edges[k + 1]
        mass = integrate.quad(norm.pdf, a, b)[0]
        mean = integrate.quad(lambda x: x * norm.pdf(x), a, b)[0] / mass
        assert abs(mean - c[k]) < 1e-9, (k, mean, c[k])
        mse += integrate.quad(lambda x, ck=c[k]: (x - ck) ** 2 * norm.pdf(x), a, b)[0]
    for k in range(7):
        assert abs(t[k] - 0.5 * (c[k] + c[k + 1])) < 1e-15
    assert abs(mse - 0.03455) < 1e-4


def pin_rotation_is_sylvester_hadamard(M):
    for d in (8, 64, 128):
        H = np.array([[(-1) ** bin(i & j).count("1") for j in range(d)] for i in range(d)], dtype=np.float64)
        R = M.rotate(np.eye(d))
        assert np.allclose(R * np.sqrt(d), H, atol=1e-12)
        v = _rng(d).standard_normal((3, d))
        assert np.allclose(M.rotate(M.rotate(v)), v, atol=1e-12)  # its own inverse
        assert np.allclose(np.linalg.norm(M.rotate(v), axis=-1), np.linalg.norm(v, axis=-1), rtol=1e-12)


def pin_q8_0_hand_blocks(M):
    """Block 0: max |x| = 127 -> scale 1; 2.5 -> 3 and -2.5 -> -3 (ties away
    from zero), 0.5 -> 1, 1.49 -> 1, -126.6 -> -127. Block 1: all zero -> scale 0,
    codes 0. Block 2: max 254 -> scale 2; 3 -> 1.5 -> 2, -5 -> -2.5 -> -3."""
    x = np.zeros(96)
    x[0:6] = [127, 2.5, -2.5, 0.5, 1.49, -126.6]
    x[64:67] = [254, 3, -5]
    q, s = M.q8_0_encode(x[None])
    q, s = q[0], s[0].astype(np.float64)
    assert s.tolist() == [1.0, 0.0, 2.0]
    assert q[0:6].tolist() == [127, 3, -3, 1, 1, -127] and (q[6:32] == 0).all()
    assert (q[32:64] == 0).all()
    assert q[64:67].tolist() == [127, 2, -3] and (q[67:] == 0).all()
    assert np.array_equal(M.q8_0_decode(q[None], s[None])[0][64:67], [254.0, 4.0, -6.0])
    # the format's error bound on random data: half a step of the fp16 scale,
    # plus 127 times the scale's fp16 rounding
    r = _rng(1)
    x = r.standard_normal((50, 128)) * r.uniform(0.01, 100, size=(50, 1))
    q, s = M.q8_0_encode(x)
    xb = x.reshape(50, 4, 32)
    s_exact = np.max(np.abs(xb), axis=-1) / 127.0
    s16 = s.astype(np.float64)
    err = np.abs(M.q8_0_decode(q, s).reshape(50, 4, 32) - xb)
    bound = 0.5 * s_exact * (1 + 1e-6) + 127 * np.abs(s16 - s_exact)
    assert (err <= bound[..., None] + 1e-12).all()
    assert np.abs(q.astype(np.int64)).max() == 127


def pin_tq3_nearest_centroid(M):
    """Each value code is the nearest of the 8 centroids to the rotated
    coordinate in units of ||v|| / sqrt(d) (brute force, explicit Hadamard
    matrix); decoding rebuilds c[code] * ||v|| / sqrt(d) and rotates back."""
    from scipy.linalg import hadamard
    c, _ = M.lloyd_max_gaussian()
    r = _rng(2)
    d = 64
    v = r.standard_normal((40, d)) * 3.0 + 0.5
    H = hadamard(d).astype(np.float64)
    codes, norms = M.tq3_encode(v)
    for i in range(40):
        y = H @ v[i] / np.sqrt(d)
        n = np.sqrt(np.sum(v[i] ** 2))
        assert abs(float(norms[i]) - n) <= 1e-6 * n
        u = y * np.sqrt(d) / n
        want = [int(np.argmin(np.abs(uj - c))) for uj in u]
        assert codes[i].tolist() == want
        rec = H @ (c[want] * float(norms[i]) / np.sqrt(d)) / np.sqrt(d)
        assert np.allclose(M.tq3_decode(codes[i:i + 1], norms[i:i + 1])[0], rec, atol=1e-12)
    z_codes, z_norm = M.tq3_encode(np.zeros((1, d)))
    assert float(z_norm[0]) == 0.0 and np.array_equal(M.tq3_decode(z_codes, z_norm), np.zeros((1, d)))


def pin_tq3_distortion(M):
    """Gaussian vectors: the rotated coordinates are Gaussian, so the relative
    squared error is the quantiser's distortion, 0.0345 (to sampling error)."""
    v = _rng(3).standard_normal((4000, 128))
    codes, norms = M.tq3_encode(v)
    rel = np.sum((M.tq3_decode(codes, norms) - v) ** 2) / np.sum(v ** 2)
    assert 0.031 < rel < 0.038, rel


def _weights(r, h, Hkv, d, rank, na):
    return {"W_K": r.standard_normal((h, Hkv * d)) / np.sqrt(h), "W_V": r.standard_normal((h, Hkv * d)) / np.sqrt(h),
            "A_K": r.standard_normal((h, rank)) / np.sqrt(h), "A_V": r.standard_normal((h, rank)) / np.sqrt(h),
            "B_K": r.standard_normal((na, rank, Hkv * d)), "B_V": r.standard_normal((na, rank, Hkv * d))}


def pin_codec_lossless_equals_plain(M):
    """With W_K = W_V = 0 the codec stores the base part exactly (all zero), so
    attention over the compressed pool must equal the uncompressed oracle to
    rounding: the adapter terms and their RoPE are untouched by the codec."""
    r = _rng(4)
    h, Hkv, d, rank, L, Hq = 16, 2, 32, 3, 40, 4
    w = _weights(r, h, Hkv, d, rank, 3)
    w["W_K"] = np.zeros_like(w["W_K"])
    w["W_V"] = np.zeros_like(w["W_V"])
    X = r.standard_normal((L, h))
    q = r.standard_normal((3, Hq, d))
    got = M.decode_codec(X, q, [0, 2, -1], w, Hkv, d, 10000.0, 1 / np.sqrt(d))
    want = O.decode(X, q, [0, 2, -1], w, Hkv, d, 10000.0, 1 / np.sqrt(d))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def pin_codec_close_to_plain(M):
    """On Gaussian data the compressed pool's attention stays within the codec's
    error of the uncompressed result (keys ~0.4% per element, values ~19%
    per vector before averaging over the context)."""
    r = _rng(5)
    h, Hkv, d, rank, L, Hq = 64, 2, 64, 4, 300, 4
    w = _weights(r, h, Hkv, d, rank, 2)
    X = r.standard_normal((L, h))
    q = r.standard_normal((2, Hq, d))
    got = M.decode_codec(X, q, [0, 1], w, Hkv, d, 10000.0, 1 / np.sqrt(d))
    want = O.decode(X, q, [0, 1], w, Hkv, d, 10000.0, 1 / np.sqrt(d))
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert 1e-4 < rel < 0.08, rel


def pin_append_codec_routing(M):
    """Compressed append: token n's codes land at block_tables[s][p // 16], row
    p % 16; what lands there is the codec of that token's exact K_base, V_base;
    untouched rows keep their sentinels."""
    r = _rng(6)
    h, Hkv, d, rank = 16, 2, 32, 2
    X = r.integers(-3, 4, size=(5, h)).astype(np.float64)
    W = {k: r.integers(0, 2, size=s).astype(np.float64) for k, s in
         (("WK", (h, Hkv * d)), ("WV", (h, Hkv * d)), ("AK", (h, rank)), ("AV", (h, rank)))}
    pos = np.array([0, 17, 3, 40, 0])
    seqs = np.array([0, 0, 1, 1, 1])
    bt = np.array([[4, 2, 9], [7, 0, 5]])
    nb = 10
    pool = {"Kq": np.full((nb, Hkv, 16, d), -128, np.int8), "Ks": np.full((nb, Hkv, 16, d // 32), np.nan, np.float16),
            "Vq": np.full((nb, Hkv, 16, d), 255, np.uint8), "Vn": np.full((nb, Hkv, 16), np.nan, np.float32)}
    lp = np.full((nb, 2, 16, rank), np.nan)
    M.append_pools_codec(pool, lp, X, pos, seqs, bt, W["WK"], W["WV"], W["AK"], W["AV"], Hkv, d, 10000.0)
    kb, vb, lk, lv = O.base_and_lowrank(X, pos, W["WK"], W["WV"], W["AK"], W["AV"], Hkv, d, 10000.0)
    written = set()
    for n in range(5):
        blk = {(0, 0): 4, (0, 1): 2, (1, 0): 7, (1, 2): 5}[(int(seqs[n]), int(pos[n]) // 16)]
        row = int(pos[n]) % 16
        written.add((blk, row))
        kq, ks = M.q8_0_encode(kb[n])
        vq, vn = M.tq3_encode(vb[n])
        assert np.array_equal(pool["Kq"][blk, :, row], kq) and np.array_equal(pool["Ks"][blk, :, row], ks)
        assert np.array_equal(pool["Vq"][blk, :, row], vq) and np.array_equal(pool["Vn"][blk, :, row], vn)
        assert np.array_equal(lp[blk, 0, row], lk[n]) and np.array_equal(lp[blk, 1, row], lv[n])
        if pos[n] == 0:  # identity rotation: integer keys, one q8_0 step = max / 127
            for hh in range(Hkv):
                for b in range(d // 32):
                    blkv = kb[n, hh, 32 * b: 32 * b + 32]
                    amax = np.max(np.abs(blkv))
                    assert float(pool["Ks"][blk, hh, row, b]) == float(np.float16(np.float32(amax) / np.float32(127)))
    for blk in range(nb):
        for row in range(16):
            if (blk, row) not in written:
                assert (pool["Kq"][blk, :, row] == -128).all() and (pool["Vq"][blk, :, row] == 255).all()


def pin_operand_rounding_bounds(M):
    """The bf16-cache reading changes each expanded key by at most half an fp16
    step and each rotated value by at most half a bf16 step, so the values it
    rotates back move by at most that, in norm (the rotation is orthonormal);
    and the rounded quantities are exactly those a kernel holds: the keys are
    fp16 numbers, the values are bf16 numbers in the rotated domain."""
    r = _rng(7)
    kb = r.standard_normal((20, 2, 64)) * 3
    vb = r.standard_normal((20, 2, 64))
    k0, v0 = M.base_roundtrip(kb, vb)
    k1, v1 = M.base_roundtrip(kb, vb, operand=True)
    assert np.all(np.abs(k1 - k0) <= np.abs(k0) * 2.0 ** -11 + 1e-12) and np.any(k1 != k0)
    vq, vn = M.tq3_encode(vb)
    c, _ = M.lloyd_max_gaussian()
    yhat = c[vq.astype(np.int64)] * (vn.astype(np.float64) / 8.0)[..., None]
    bound = np.linalg.norm(yhat, axis=-1) * 2.0 ** -8  # bf16: 8 significant bits
    assert np.all(np.linalg.norm(v1 - v0, axis=-1) <= bound + 1e-12) and np.any(v1 != v0)
    # what is rounded is what the kernel holds: fp16 keys, and bf16 values in the rotated domain
    assert np.array_equal(k1, k1.astype(np.float16).astype(np.float64))
    y1 = M.rotate(v1)
    assert np.allclose(y1, O.round_bf16(y1), rtol=1e-12, atol=1e-15)


ALL_PINS = [pin_lloyd_max_gaussian, pin_rotation_is_sylvester_hadamard, pin_q8_0_hand_blocks,
            pin_tq3_nearest_centroid, pin_tq3_distortion, pin_codec_lossless_equals_plain,
            pin_codec_close_to_plain, pin_append_codec_routing, pin_operand_rounding_bounds]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_polykv_pin(pin):
    pin(PK)


def _mutant(old: str, new: str) -> types.ModuleType:
    src = open(PK_SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new).replace("from . import lrkv_oracle as O", "import oracle.lrkv_oracle as O")
    mod = types.ModuleType("polykv_mutant")
    exec(compile(src, "polykv_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = {
    "q8_0_divides_by_128": ("amax / np.float32(127.0)", "amax / np.float32(128.0)"),
    "q8_0_blocks_of_16": ("QK = 32 ", "QK = 16 "),
    "q8_0_ties_to_even": ("return np.sign(p) * np.floor(np.abs(p) + 0.5)", "return np.round(p)"),
    "q8_0_truncates": ("return np.sign(p) * np.floor(np.abs(p) + 0.5)", "return np.trunc(p)"),
    "rotate_unnormalised": ("return v @ hadamard(d).astype(np.float64) / np.sqrt(d)",
                            "return v @ hadamard(d).astype(np.float64)"),
    "rotate_transposed_order": ("return v @ hadamard(d).astype(np.float64) / np.sqrt(d)",
                                "return v[..., ::-1] @ hadamard(d).astype(np.float64) / np.sqrt(d)"),
    "lloyd_no_cell_mass": ("new = (norm.pdf(edges[:-1]) - norm.pdf(edges[1:])) / mass",
                           "new = (norm.pdf(edges[:-1]) - norm.pdf(edges[1:]))"),
    "tq3_centroids_reversed": ("yhat = c[codes.astype(np.int64)]", "yhat = c[::-1][codes.astype(np.int64)]"),
    "tq3_scale_without_sqrt_d": ("inv = np.where(n32 > 0, np.float32(np.sqrt(d)) / np.where",
                                 "inv = np.where(n32 > 0, np.float32(1.0) / np.where"),
    "tq3_decode_not_rotated_back": ("    return rotate(yhat)\n", "    return yhat\n"),
    "codec_k_adapter_without_rope": ("k = k + O.apply_rope((lk @ np.asarray(B_K_i, dtype=np.float64)).reshape(T, n_kv_heads, head_dim),\n                             positions, base)",
                                     "k = k + (lk @ np.asarray(B_K_i, dtype=np.float64)).reshape(T, n_kv_heads, head_dim)"),
    "codec_v_adapter_from_lk": ("v = v + (lv @ np.asarray(B_V_i", "v = v + (lk[:, :lv.shape[1]] @ np.asarray(B_V_i"),
    "append_codec_row_shift": ("        row = p % O.BLOCK\n", "        row = (p + 1) % O.BLOCK\n"),
    "operand_rounding_after_rotation": ("        yhat = O.round_bf16(yhat)\n    return rotate(yhat)",
                                        "        return O.round_bf16(rotate(yhat))\n    return rotate(yhat)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_polykv_planted_mistake_is_caught(name):
    mod = _mutant(*MUTATIONS[name])
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception:  # noqa: BLE001 -- any failure of a pin counts
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
