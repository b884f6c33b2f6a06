"""Compressed base pool (PolyKV codec), fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it. It shares no code with the CUDA library.

PolyKV (the abstract printed at the end of the PReCache page): several agents
read one shared, asymmetrically compressed KV pool. The keys are stored as int8
in q8_0 blocks, which keeps the softmax stable. The values are rotated by a
fast Walsh-Hadamard transform, then quantised to 3 bits with Lloyd-Max
centroids for N(0, 1) ("TurboQuant MSE"). Here the codec compresses the shared
base part of the LoRA-KV cache. The low-rank part and the per-agent
reconstruction are unchanged (LRAgent, Abstract):
    K_i = dec(enc(K_base)) + RoPE(L_K B_K,i),   V_i = dec(enc(V_base)) + L_V B_V,i.

Readings where the abstract is silent:
* q8_0 (the llama.cpp block format the abstract names): blocks of 32
  consecutive head dims. Scale s = max|x| / 127, stored as fp16.
  Code q = round(x * (1 / s)), to nearest with ties away from zero, in
  [-127, 127]; s = 0 gives codes 0. Decoded value: q * fp16(s).
* The rotation is the normalised Sylvester-Hadamard matrix H_d / sqrt(d)
  (natural order, no random sign flips), applied to each value vector of d
  dims. It is orthonormal and its own inverse.
* Scale of the 3-bit code: y = rotate(v), n = ||y|| = ||v||. Each coordinate
  is quantised in units of n / sqrt(d), as u_j = y_j * sqrt(d) / n; for a
  Gaussian v that is N(0, 1). Code_j = the number of Lloyd-Max thresholds
  strictly below u_j (0..7), and n = 0 gives u = 0. Stored: the codes and n
  (fp32). Decoded: y^_j = c[code_j] * n / sqrt(d), v^ = rotate(y^).
* Codes (an integer decided by floating point) are decided in fp32, the
  kernel's precision: the inputs to the decision are rounded to fp32 first.
  Everything else is fp64.
"""
from __future__ import annotations

import numpy as np

from . import lrkv_oracle as O

QK = 32       # q8_0 block: head dims per scale
LEVELS = 8    # 3-bit value codes


# ---------------------------------------------------------------------------
# Lloyd-Max quantiser for N(0, 1)

def lloyd_max_gaussian(levels: int = LEVELS, iters: int = 20000, tol: float = 1e-15):
    """Lloyd's algorithm on the standard normal density: alternately set each
    threshold to the midpoint of its two centroids and each centroid to the
    conditional mean of its cell,
        c_k = (phi(t_k) - phi(t_k+1)) / (Phi(t_k+1) - Phi(t_k)),
    with t_0 = -inf and t_levels = +inf. Returns (centroids [levels] ascending,
    thresholds [levels - 1])."""
    from scipy.stats import norm
    c = np.linspace(-2.0, 2.0, levels)
    for _ in range(iters):
        t = 0.5 * (c[1:] + c[:-1])
        edges = np.concatenate([[-np.inf], t, [np.inf]])
        mass = norm.cdf(edges[1:]) - norm.cdf(edges[:-1])
        new = (norm.pdf(edges[:-1]) - norm.pdf(edges[1:])) / mass
        done = np.max(np.abs(new - c)) < tol
        c = new
        if done:
            break
    c = 0.5 * (c - c[::-1])  # the density is even: so is the fixed point (t = 0 in the middle)
    return c, 0.5 * (c[1:] + c[:-1])


_CT = None


def centroids_thresholds():
    """The 8-level quantiser, computed once."""
    global _CT
    if _CT is None:
        _CT = lloyd_max_gaussian()
    return _CT


# ---------------------------------------------------------------------------
# Walsh-Hadamard rotation

def rotate(v) -> np.ndarray:
    """v [..., d] times H_d / sqrt(d) (Sylvester order; H_d is symmetric)."""
    from scipy.linalg import hadamard
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    return v @ hadamard(d).astype(np.float64) / np.sqrt(d)


# ---------------------------------------------------------------------------
# Keys: q8_0

def _round_half_away(p32) -> np.ndarray:
    """Rounds float32 values to the nearest integer, ties away from zero (the
    sum |p| + 0.5 is exact in float64)."""
    p = np.asarray(p32, dtype=np.float32).astype(np.float64)
    return np.sign(p) * np.floor(np.abs(p) + 0.5)


def q8_0_encode(x):
    """x [..., d] (d a multiple of 32) -> (codes int8 [..., d], scales float16 [..., d/32])."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    shp = x32.shape
    b = x32.reshape(shp[:-1] + (shp[-1] // QK, QK))
    amax = np.max(np.abs(b), axis=-1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(s > 0, np.float32(1.0) / np.where(s > 0, s, np.float32(1.0)), np.float32(0.0)).astype(np.float32)
    q = _round_half_away(b * inv[..., None])
    q = np.clip(q, -127, 127).astype(np.int8).reshape(shp)
    return q, s.astype(np.float16)


def q8_0_decode(codes, scales) -> np.ndarray:
    c = np.asarray(codes, dtype=np.float64)
    shp = c.shape
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    return (c.reshape(shp[:-1] + (shp[-1] // QK, QK)) * s[..., None]).reshape(shp)


# ---------------------------------------------------------------------------
# Values: Hadamard rotation + 3-bit Lloyd-Max codes

def tq3_encode(v):
    """v [..., d] -> (codes uint8 [..., d] in 0..7, norms float32 [...])."""
    _, t = centroids_thresholds()
    y = rotate(v)
    d = y.shape[-1]
    y32 = y.astype(np.float32)
    n32 = np.sqrt(np.sum(y * y, axis=-1)).astype(np.float32)
    inv = np.where(n32 > 0, np.float32(np.sqrt(d)) / np.where(n32 > 0, n32, np.float32(1.0)),
                   np.float32(0.0)).astype(np.float32)
    u = (y32 * inv[..., None]).astype(np.float32)
    codes = np.sum(u[..., None] > t.astype(np.float32), axis=-1).astype(np.uint8)
    return codes, n32


def tq3_decode(codes, norms, operand: bool = False) -> np.ndarray:
    """operand=True: the rotated values are rounded to bf16 before rotating back
    (the bf16-cache reading below)."""
    c, _ = centroids_thresholds()
    codes = np.asarray(codes)
    d = codes.shape[-1]
    yhat = c[codes.astype(np.int64)] * (np.asarray(norms, dtype=np.float32).astype(np.float64) / np.sqrt(d))[..., None]
    if operand:
        yhat = O.round_bf16(yhat)
    return rotate(yhat)


def base_roundtrip(kb, vb, operand: bool = False):
    """The base part as the compressed pool returns it: K_base through q8_0,
    V_base through the rotated 3-bit code.

    operand=True is the bf16-cache reading of the oracle (the components a
    kernel holds in 16 bits are rounded as it holds them): for the compressed
    pool those are the expanded keys q * s in fp16 and the expanded rotated
    values c[code] ||v|| / sqrt(d) in bf16, before the rotation back."""
    kq, ks = q8_0_encode(kb)
    vq, vn = tq3_encode(vb)
    k = q8_0_decode(kq, ks)
    if operand:
        k = k.astype(np.float16).astype(np.float64)
    return k, tq3_decode(vq, vn, operand)


# ---------------------------------------------------------------------------
# Attention over the compressed base pool

def agent_kv_codec(X, positions, W_K, W_V, A_K, A_V, B_K_i, B_V_i, n_kv_heads: int,
                   head_dim: int, base: float, lr_dtype=None):
    """One agent's keys and values read from a compressed base pool:
        K_i = dec(enc(K_base)) + RoPE(L_K B_K,i),   V_i = dec(enc(V_base)) + L_V B_V,i,
    K_base = RoPE(X W_K), V_base = X W_V, L_K = X A_K, L_V = X A_V (exact).
    lr_dtype="bf16": L_K, L_V rounded to bf16, as the low-rank pool stores them,
    and the expanded base operands rounded as a kernel holds them (base_roundtrip)."""
    kb, vb, lk, lv = O.base_and_lowrank(X, positions, W_K, W_V, A_K, A_V, n_kv_heads, head_dim, base)
    k, v = base_roundtrip(kb, vb, operand=lr_dtype == "bf16")
    if lr_dtype == "bf16":
        lk, lv = O.round_bf16(lk), O.round_bf16(lv)
    T = k.shape[0]
    if B_K_i is not None:
        k = k + O.apply_rope((lk @ np.asarray(B_K_i, dtype=np.float64)).reshape(T, n_kv_heads, head_dim),
                             positions, base)
    if B_V_i is not None:
        v = v + (lv @ np.asarray(B_V_i, dtype=np.float64)).reshape(T, n_kv_heads, head_dim)
    return k, v


def attend_codec(X_seq, adapter: int, q, q_positions, weights, n_kv_heads: int, head_dim: int,
                 base: float, scale: float, lr_dtype=None) -> np.ndarray:
    """Queries q [N, Hq, d] of one agent over a sequence X_seq [L, h] whose base
    part is read back through the codec."""
    L = np.asarray(X_seq).shape[0]
    B_K, B_V = O._adapter_B(weights, adapter)
    A_K, A_V = O._agent_A(weights, adapter)
    K, V = agent_kv_codec(X_seq, np.arange(L), weights["W_K"], weights["W_V"], A_K, A_V, B_K, B_V,
                          n_kv_heads, head_dim, base, lr_dtype)
    return O.gqa_attention(q, q_positions, K, V, scale)


def decode_codec(X_ctx, q, adapters, weights, n_kv_heads: int, head_dim: int, base: float,
                 scale: float, lr_dtype=None) -> np.ndarray:
    """Decode queries of several agents on one context X_ctx [L, h] (each at
    position L - 1), base part read through the codec."""
    L = np.asarray(X_ctx).shape[0]
    out = np.empty(np.asarray(q).shape, dtype=np.float64)
    for n, a in enumerate(np.asarray(adapters).tolist()):
        out[n: n + 1] = attend_codec(X_ctx, int(a), np.asarray(q)[n: n + 1], [L - 1], weights,
                                     n_kv_heads, head_dim, base, scale, lr_dtype)
    return out


def append_pools_codec(pool, lr_pool, X, positions, seq_rows, block_tables, W_K, W_V, A_K, A_V,
                       n_kv_heads: int, head_dim: int, base: float):
    """Expected contents of a compressed base pool after an append, written in
    place. pool is a dict of arrays over [num_blocks, Hkv, 16]:
        "Kq" int8 [.., d], "Ks" float16 [.., d / 32], "Vq" uint8 [.., d] (codes
        0..7), "Vn" float32 [..].
    lr_pool [num_blocks, 2, 16, G r] as in the uncompressed append. Token n goes
    to block block_tables[seq_rows[n], positions[n] // 16], row positions[n] % 16."""
    kb, vb, lk, lv = O.base_and_lowrank(X, positions, W_K, W_V, A_K, A_V, n_kv_heads, head_dim, base)
    kq, ks = q8_0_encode(kb)
    vq, vn = tq3_encode(vb)
    for n, (p, s) in enumerate(zip(np.asarray(positions).tolist(), np.asarray(seq_rows).tolist())):
        blk = int(block_tables[s][p // O.BLOCK])
        row = p % O.BLOCK
        pool["Kq"][blk, :, row, :] = kq[n]
        pool["Ks"][blk, :, row, :] = ks[n]
        pool["Vq"][blk, :, row, :] = vq[n]
        pool["Vn"][blk, :, row] = vn[n]
        lr_pool[blk, 0, row, :] = lk[n]
        lr_pool[blk, 1, row, :] = lv[n]
    return pool, lr_pool
