"""fp64 CPU oracle for LoRA-KV attention over a shared base + shared-A low-rank cache.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it. It shares no code with the CUDA library.

What it computes is the plain definition of the method's result, every
per-agent key and value materialised in full, then textbook softmax attention:

* LRAgent: Efficient KV Cache Sharing for Multi-LoRA LLM Agents (arXiv
  2602.01053), Abstract: the cache splits into a base part produced by the
  pretrained weights and an adapter part produced by the LoRA weights; with a
  shared A, the low-rank part X·A is common to all agents. Reaching the same
  values as per-agent ("non-shared") caching is the method's accuracy claim, so
  the reference result is each agent's own full K_i, V_i:
      K_i = RoPE(X·W_K + (X·A_K)·B_K,i),  V_i = X·W_V + (X·A_V)·B_V,i.
* PReCache (thelatestinai.com/papers/2609.34054), Abstract and Table 1: the
  base cache comes from the pretrained weights and the low-rank cache is
  produced once, when a context segment is first processed (the "append").

Readings where the pages are silent:
row-vector convention X·W; rotate-half RoPE pairing (j, j + d/2) with
theta_j = base^(-2j/d) and no frequency scaling; LoRA scale folded into B;
softmax scale 1/sqrt(d); q head m reads kv head floor(m / (Hq/Hkv)); query k of
a chunk of q_len queries over L keys sits at position L - q_len + k and sees
keys at positions <= its own; adapter id -1 means B = 0.

All arithmetic is float64. Inputs are the storage-dtype values converted to
float64; nothing is rounded inside, except in the explicitly named bf16-cache
variant (agent_kv_from_cache), which rounds the four stored cache components
to bf16 as a bf16 cache holds them and is used for short-context edge cases
whose outputs are dominated by that storage rounding.
"""
from __future__ import annotations

import numpy as np

BLOCK = 16


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# Rotary position embedding (reading: rotate-half pairing, HF Llama family).

def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """theta_j = base^(-2j/d) for j in [0, d/2)."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * j / head_dim)


def apply_rope(x: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """Rotates x [T, H, d] at integer positions [T].

    For pair (j, j + d/2) at position t with angle a = t * theta_j:
        x'[j]       = x[j] cos a - x[j + d/2] sin a
        x'[j + d/2] = x[j + d/2] cos a + x[j] sin a
    """
    x = _f64(x)
    d = x.shape[-1]
    half = d // 2
    ang = _f64(positions)[:, None] * rope_inv_freq(d, base)[None, :]  # [T, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


# ---------------------------------------------------------------------------
# Cache construction.

def _lowrank(X, A):
    """X·A for a shared A [h, r]; for agent-specific A [G, h, r] the G products
    side by side, group g in columns [g r, (g + 1) r)."""
    A = _f64(A)
    if A.ndim == 2:
        return X @ A
    return np.concatenate([X @ A[g] for g in range(A.shape[0])], axis=1)


def base_and_lowrank(X, positions, W_K, W_V, A_K, A_V, n_kv_heads: int, head_dim: int,
                     base: float):
    """What one append writes for tokens X [T, h] at the given positions.

    LRAgent, Abstract (base component from the pretrained weights; adapter
    component kept in its low-rank form, shared when A is shared):
        K_base = RoPE(X·W_K)  [T, Hkv, d]     V_base = X·W_V  [T, Hkv, d]
        L_K    = X·A_K        [T, r]          L_V    = X·A_V  [T, r]
    PReCache, Abstract and Figure 1 (PreLRShared): with agent-specific
    A_K,g, A_V,g (arrays [G, h, r]) every agent's low-rank cache is produced
    when the segment is first processed: L_K = [X·A_K,0 | ... | X·A_K,G-1]
    [T, G r], likewise L_V.
    """
    X = _f64(X)
    T = X.shape[0]
    k_pre = (X @ _f64(W_K)).reshape(T, n_kv_heads, head_dim)
    v = (X @ _f64(W_V)).reshape(T, n_kv_heads, head_dim)
    return (apply_rope(k_pre, positions, base), v, _lowrank(X, A_K), _lowrank(X, A_V))


def agent_kv(X, positions, W_K, W_V, A_K, A_V, B_K_i, B_V_i, n_kv_heads: int,
             head_dim: int, base: float):
    """One agent's full keys and values, as that agent alone would cache them.

    K_i = RoPE(X·W_K + (X·A_K)·B_K,i),  V_i = X·W_V + (X·A_V)·B_V,i, each
    [T, Hkv, d]. B_K,i / B_V,i of None stand for B = 0 (base model only).
    """
    X = _f64(X)
    T = X.shape[0]
    k_pre = X @ _f64(W_K)
    v = X @ _f64(W_V)
    if B_K_i is not None:
        k_pre = k_pre + (X @ _f64(A_K)) @ _f64(B_K_i)
    if B_V_i is not None:
        v = v + (X @ _f64(A_V)) @ _f64(B_V_i)
    k = apply_rope(k_pre.reshape(T, n_kv_heads, head_dim), positions, base)
    return k, v.reshape(T, n_kv_heads, head_dim)


def round_bf16(x) -> np.ndarray:
    """Rounds to the nearest bfloat16 (ties to even), returned as float64.

    Used only by the bf16-cache reading below: the value is first rounded to
    float32, then the low 16 bits of the float32 pattern are rounded away
    (round half to even on bit 16)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def agent_kv_from_cache(X, positions, W_K, W_V, A_K, A_V, B_K_i, B_V_i, n_kv_heads: int,
                        head_dim: int, base: float, cache_dtype: str = "bf16"):
    """One agent's keys and values when the cache components are STORED in
    bf16: K_base, V_base, L_K, L_V are computed exactly, rounded to bf16 (what a
    bf16 cache holds), then combined exactly as the decomposition defines:
        K_i = K_base + RoPE(L_K B_K,i),   V_i = V_base + L_V B_V,i.
    (LRAgent, Abstract: base component + low-rank adapter component; RoPE is
    linear, so RoPE(X W_K + X A_K B_K) = RoPE(X W_K) + RoPE(X A_K B_K).)"""
    assert cache_dtype == "bf16"
    kb, vb, lk, lv = base_and_lowrank(X, positions, W_K, W_V, A_K, A_V, n_kv_heads, head_dim, base)
    kb, vb, lk, lv = round_bf16(kb), round_bf16(vb), round_bf16(lk), round_bf16(lv)
    T = kb.shape[0]
    k = kb
    v = vb
    if B_K_i is not None:
        k = k + apply_rope((lk @ _f64(B_K_i)).reshape(T, n_kv_heads, head_dim), positions, base)
    if B_V_i is not None:
        v = v + (lv @ _f64(B_V_i)).reshape(T, n_kv_heads, head_dim)
    return k, v


def agent_kv_rebased(X_base, X_lr, positions, W_K, W_V, A_K, A_V, B_K_i, B_V_i, n_kv_heads: int,
                     head_dim: int, base: float, cache_dtype=None):
    """One agent's keys and values over a re-based cache (PReCache, Abstract and
    Figure 1, ReBaseShared): the shared base part is rebuilt from the
    adapter-free hidden states X_base, while the low-rank part stays the one
    computed from X_lr, so
        K_i = RoPE(X_base·W_K + (X_lr·A_K)·B_K,i),  V_i = X_base·W_V + (X_lr·A_V)·B_V,i.
    cache_dtype="bf16": the four stored components are rounded to bf16 first
    (as agent_kv_from_cache does for a single source)."""
    X_base = _f64(X_base)
    X_lr = _f64(X_lr)
    T = X_base.shape[0]
    if cache_dtype is None:
        k_pre = X_base @ _f64(W_K)
        v = X_base @ _f64(W_V)
        if B_K_i is not None:
            k_pre = k_pre + (X_lr @ _f64(A_K)) @ _f64(B_K_i)
        if B_V_i is not None:
            v = v + (X_lr @ _f64(A_V)) @ _f64(B_V_i)
        k = apply_rope(k_pre.reshape(T, n_kv_heads, head_dim), positions, base)
        return k, v.reshape(T, n_kv_heads, head_dim)
    assert cache_dtype == "bf16"
    kb, vb, _, _ = base_and_lowrank(X_base, positions, W_K, W_V, A_K, A_V, n_kv_heads, head_dim, base)
    _, _, lk, lv = base_and_lowrank(X_lr, positions, W_K, W_V, A_K, A_V, n_kv_heads, head_dim, base)
    k, v = round_bf16(kb), round_bf16(vb)
    if B_K_i is not None:
        k = k + apply_rope((round_bf16(lk) @ _f64(B_K_i)).reshape(T, n_kv_heads, head_dim), positions, base)
    if B_V_i is not None:
        v = v + (round_bf16(lv) @ _f64(B_V_i)).reshape(T, n_kv_heads, head_dim)
    return k, v


# ---------------------------------------------------------------------------
# Attention.

def gqa_attention(q, q_positions, K, V, scale: float) -> np.ndarray:
    """Causal grouped-query softmax attention.

    q [N, Hq, d] at positions [N]; K, V [L, Hkv, d] at positions 0..L-1.
    Query head m reads kv head m // (Hq / Hkv); key t is visible iff t <= the
    query's position. Returns [N, Hq, d].
    """
    q = _f64(q)
    K = _f64(K)
    V = _f64(V)
    N, Hq, d = q.shape
    L, Hkv, _ = K.shape
    g = Hq // Hkv
    qp = np.asarray(q_positions, dtype=np.int64)
    visible = np.arange(L)[None, :] <= qp[:, None]  # [N, L]
    out = np.empty((N, Hq, d), dtype=np.float64)
    for m in range(Hq):
        kv = m // g
        s = (q[:, m, :] @ K[:, kv, :].T) * scale          # [N, L]
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, m, :] = p @ V[:, kv, :]
    return out


# ---------------------------------------------------------------------------
# Whole operations, in the library's terms.

def _adapter_B(weights, adapter: int):
    if adapter < 0:
        return None, None
    return weights["B_K"][adapter], weights["B_V"][adapter]


def _agent_A(weights, adapter: int):
    """The A factors agent `adapter` uses: the shared A [h, r], or its own
    A_g [G, h, r] -> A[adapter] (PReCache, PreLRShared); base-only rows
    (adapter -1) use no A."""
    A_K, A_V = weights["A_K"], weights["A_V"]
    if np.ndim(A_K) == 3:
        g = max(adapter, 0)
        return A_K[g], A_V[g]
    return A_K, A_V


def attend(X_seq, adapter: int, q, q_positions, weights, n_kv_heads: int, head_dim: int,
           base: float, scale: float, cache_dtype=None, X_lr=None) -> np.ndarray:
    """Queries q [N, Hq, d] of one agent over a sequence whose hidden states at
    positions 0..L-1 are X_seq [L, h]: materialise the agent's K, V, then attend.
    cache_dtype="bf16" uses the bf16-stored cache components (agent_kv_from_cache).
    X_lr (ReBaseShared): the low-rank part of the cache came from these hidden
    states instead, the base part from X_seq (agent_kv_rebased)."""
    L = np.asarray(X_seq).shape[0]
    B_K, B_V = _adapter_B(weights, adapter)
    A_K, A_V = _agent_A(weights, adapter)
    if X_lr is not None:
        K, V = agent_kv_rebased(X_seq, X_lr, np.arange(L), weights["W_K"], weights["W_V"],
                                A_K, A_V, B_K, B_V, n_kv_heads, head_dim, base, cache_dtype)
        return gqa_attention(q, q_positions, K, V, scale)
    make = agent_kv if cache_dtype is None else agent_kv_from_cache
    K, V = make(X_seq, np.arange(L), weights["W_K"], weights["W_V"], A_K, A_V, B_K, B_V,
                n_kv_heads, head_dim, base)
    return gqa_attention(q, q_positions, K, V, scale)


def decode(X_ctx, q, adapters, weights, n_kv_heads: int, head_dim: int, base: float,
           scale: float, cache_dtype=None, X_lr=None) -> np.ndarray:
    """Decode queries of several agents on one context X_ctx [L, h]: each query
    (one per row of q [N, Hq, d], adapter ids [N]) sits at position L - 1."""
    L = np.asarray(X_ctx).shape[0]
    out = np.empty(np.asarray(q).shape, dtype=np.float64)
    for n, a in enumerate(np.asarray(adapters).tolist()):
        out[n: n + 1] = attend(X_ctx, int(a), np.asarray(q)[n: n + 1], [L - 1], weights,
                               n_kv_heads, head_dim, base, scale, cache_dtype, X_lr)
    return out


def prefill(X_seq, q_chunk, adapter: int, weights, n_kv_heads: int, head_dim: int,
            base: float, scale: float, cache_dtype=None, X_lr=None) -> np.ndarray:
    """A chunk of q_len queries at the end of a sequence of L tokens (the chunk's
    own tokens included): query k sits at position L - q_len + k."""
    L = np.asarray(X_seq).shape[0]
    n = np.asarray(q_chunk).shape[0]
    return attend(X_seq, adapter, q_chunk, np.arange(L - n, L), weights, n_kv_heads,
                  head_dim, base, scale, cache_dtype, X_lr)


def append_pools(base_pool, lr_pool, X, positions, seq_rows, block_tables, W_K, W_V, A_K,
                 A_V, n_kv_heads: int, head_dim: int, base: float):
    """Expected pool contents after an append, written in place.

    base_pool [num_blocks, 2, Hkv, 16, d]: plane 0 = K_base, plane 1 = V_base.
    lr_pool   [num_blocks, 2, 16, G r]:    plane 0 = L_K, plane 1 = L_V (G = 1 for a
                                           shared A; group g in columns [g r, (g+1) r)).
    Token n goes to block block_tables[seq_rows[n], positions[n] // 16], row
    positions[n] % 16 (PagedAttention-style block table).
    """
    kb, vb, lk, lv = base_and_lowrank(X, positions, W_K, W_V, A_K, A_V, n_kv_heads,
                                      head_dim, base)
    for n, (p, s) in enumerate(zip(np.asarray(positions).tolist(), np.asarray(seq_rows).tolist())):
        blk = int(block_tables[s][p // BLOCK])
        row = p % BLOCK
        base_pool[blk, 0, :, row, :] = kb[n]
        base_pool[blk, 1, :, row, :] = vb[n]
        lr_pool[blk, 0, row, :] = lk[n]
        lr_pool[blk, 1, row, :] = lv[n]
    return base_pool, lr_pool


def rebase_pools(base_pool, lr_pool, X_base, X_lr, positions, seq_rows, block_tables, W_K, W_V,
                 A_K, A_V, n_kv_heads: int, head_dim: int, base: float):
    """Expected pool contents after a re-based append (PReCache, Abstract and
    Figure 1, ReBaseShared), written in place: the base rows (K_base, V_base)
    of each token from the adapter-free hidden states X_base, its low-rank rows
    (L_K, L_V) from X_lr. A source of None leaves that part untouched (a
    base-only re-base after an agent's turn keeps the low-rank cache)."""
    kb = vb = lk = lv = None
    if X_base is not None:
        kb, vb, _, _ = base_and_lowrank(X_base, positions, W_K, W_V, A_K, A_V, n_kv_heads,
                                        head_dim, base)
    if X_lr is not None:
        _, _, lk, lv = base_and_lowrank(X_lr, positions, W_K, W_V, A_K, A_V, n_kv_heads,
                                        head_dim, base)
    for n, (p, s) in enumerate(zip(np.asarray(positions).tolist(), np.asarray(seq_rows).tolist())):
        blk = int(block_tables[s][p // BLOCK])
        row = p % BLOCK
        if kb is not None:
            base_pool[blk, 0, :, row, :] = kb[n]
            base_pool[blk, 1, :, row, :] = vb[n]
        if lk is not None:
            lr_pool[blk, 0, row, :] = lk[n]
            lr_pool[blk, 1, row, :] = lv[n]
    return base_pool, lr_pool
