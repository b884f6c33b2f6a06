"""The decode kernel's adapter-score identity, checked in fp64 on the CPU.

The decode kernel never forms the rotated adapter row RoPE_t(B^T l(t)). For a
query row q it builds, once per work item,

    G[k, j]       = q[j] B[k, j] + q[j + d/2] B[k, j + d/2]
    G[k, d/2 + j] = q[j + d/2] B[k, j] - q[j] B[k, j + d/2]      (j < d/2)

and per token uses u(t) = [cos(t theta_j)..., sin(t theta_j)...]:

    q . RoPE_t(B^T l(t)) = sum_k l_k(t) sum_j' u_j'(t) G[k, j'].

These tests evaluate the left side with the oracle's own RoPE (rotate-half
pairing, theta_j = base^(-2j/d)) and the right side with G and u built as
above, so a sign, a swapped half or a wrong pairing in the kernel's
construction would show here, independently of the GPU.
"""
import numpy as np
import pytest

from oracle import lrkv_oracle as O


def _g_matrix(q: np.ndarray, B: np.ndarray) -> np.ndarray:
    """G [r, d] for one query row q [d] and one kv head's slice B [r, d]."""
    half = q.shape[0] // 2
    q1, q2 = q[:half], q[half:]
    b1, b2 = B[:, :half], B[:, half:]
    return np.concatenate([q1 * b1 + q2 * b2, q2 * b1 - q1 * b2], axis=1)


def _u(t: int, d: int, base: float) -> np.ndarray:
    ang = t * O.rope_inv_freq(d, base)
    return np.concatenate([np.cos(ang), np.sin(ang)])


@pytest.mark.parametrize("d,r", [(64, 8), (64, 64), (128, 16), (128, 64)])
def test_adapter_score_identity(d, r):
    rng = np.random.default_rng(1234 + d + r)
    base = 10000.0
    q = rng.standard_normal(d)
    B = rng.standard_normal((r, d)) / np.sqrt(r)
    positions = np.array([0, 1, 15, 16, 127, 128, 4095, 16383, 32767])
    L = rng.standard_normal((positions.size, r))
    # left: rotate the rebuilt row with the oracle's RoPE, then the dot product
    y = L @ B                                                    # [T, d]
    rot = O.apply_rope(y[:, None, :], positions, base)[:, 0, :]  # [T, d]
    lhs = rot @ q
    # right: the kernel's association
    G = _g_matrix(q, B)                                          # [r, d]
    rhs = np.array([L[i] @ (G @ _u(int(t), d, base)) for i, t in enumerate(positions)])
    scale = np.abs(lhs).max()
    assert np.max(np.abs(lhs - rhs)) <= 1e-12 * max(scale, 1.0)


def test_identity_with_base_term_is_the_oracle_score():
    """Full decode score: q . K_a(t) with K_a = RoPE(X W_K + X A_K B_K) from the
    oracle's materialised cache equals q . K_base(t) + sum_k l_k W_k(t)."""
    rng = np.random.default_rng(7)
    h, d, r, T, base = 32, 64, 8, 40, 10000.0
    X = rng.standard_normal((T, h))
    W_K = rng.standard_normal((h, d)) / np.sqrt(h)
    W_V = rng.standard_normal((h, d)) / np.sqrt(h)
    A_K = rng.standard_normal((h, r)) / np.sqrt(h)
    A_V = rng.standard_normal((h, r)) / np.sqrt(h)
    B_K = rng.standard_normal((r, d)) / np.sqrt(r)
    B_V = rng.standard_normal((r, d)) / np.sqrt(r)
    pos = np.arange(T) + 1000
    K_a, _ = O.agent_kv(X, pos, W_K, W_V, A_K, A_V, B_K, B_V, 1, d, base)
    q = rng.standard_normal(d)
    want = K_a.reshape(T, d) @ q
    K_base = O.apply_rope((X @ W_K)[:, None, :], pos, base)[:, 0, :]
    l = X @ A_K
    G = _g_matrix(q, B_K)
    got = K_base @ q + np.array([l[i] @ (G @ _u(int(t), d, base)) for i, t in enumerate(pos)])
    assert np.max(np.abs(got - want)) <= 1e-11 * max(np.abs(want).max(), 1.0)


def test_planted_sign_error_is_caught():
    """A sign flipped in the second half of G (a plausible kernel slip) breaks
    the identity by far more than rounding."""
    rng = np.random.default_rng(3)
    d, r, base = 64, 8, 10000.0
    q = rng.standard_normal(d)
    B = rng.standard_normal((r, d))
    l = rng.standard_normal(r)
    t = 777
    lhs = O.apply_rope((l @ B)[None, None, :], np.array([t]), base)[0, 0] @ q
    G = _g_matrix(q, B)
    G_bad = G.copy()
    G_bad[:, d // 2:] *= -1.0
    good = l @ (G @ _u(t, d, base))
    bad = l @ (G_bad @ _u(t, d, base))
    assert abs(good - lhs) <= 1e-12 * max(abs(lhs), 1.0)
    assert abs(bad - lhs) > 1e-3 * max(abs(lhs), 1.0)
