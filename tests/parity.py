"""Shared helpers for GPU-vs-oracle parity tests (the oracle runs on the CPU in fp64)."""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np
import torch

import oracle
from oracle import polykv

# Tolerances (relative Frobenius and max-abs error against the fp64 oracle).
BF16_TOL = dict(max_abs=2e-2, rel_fro=5e-3)
FP32_TOL = dict(max_abs=1e-4, rel_fro=1e-4)


def tol_for(case):
    return FP32_TOL if case.shape.dtype == "fp32" else BF16_TOL


def weights64(case):
    return {k: v.double().numpy() for k, v in case.weights.items()}


def errors(got: np.ndarray, want: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), "non-finite values in the GPU output"
    d = got - want
    return float(np.abs(d).max()), float(np.linalg.norm(d) / max(np.linalg.norm(want), 1e-30))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (2^(floor(log2|x|) - 7)); 0 at 0."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def assert_close(got, want, tol, what=""):
    """rel_fro <= tol["rel_fro"] and, per element, |got - want| <= max(tol["max_abs"],
    one bf16 ulp of want) for bf16 outputs: an output stored in bf16 cannot be
    closer than its own spacing once any rounding flips, and above |x| = 4 that
    spacing (2^-5) exceeds 2e-2."""
    mx, rf = errors(got, want)
    if tol is BF16_TOL:
        d = np.abs(np.asarray(got, dtype=np.float64) - np.asarray(want, dtype=np.float64))
        bound = np.maximum(tol["max_abs"], bf16_ulp(want))
        worst = float((d / bound).max())
        assert worst <= 1.0 and rf <= tol["rel_fro"], (
            f"{what}: max_abs {mx:.3e} ({worst:.2f} of the per-element bound), rel_fro {rf:.3e} "
            f"(tol {tol['rel_fro']:.1e})")
        return mx, rf
    assert mx <= tol["max_abs"] and rf <= tol["rel_fro"], (
        f"{what}: max_abs {mx:.3e} (tol {tol['max_abs']:.1e}), rel_fro {rf:.3e} (tol {tol['rel_fro']:.1e})")
    return mx, rf


def _hidden(case, s):
    """Hidden states of sequence s as the oracle takes them: (X, None), or for a
    re-based cache (X_base = the adapter-free states, X_lr = the adapted ones)."""
    if case.rebase:
        return case.seq_hidden_neutral(s).double().numpy(), case.seq_hidden(s).double().numpy()
    return case.seq_hidden(s).double().numpy(), None


def oracle_decode_rows(case, rows: Optional[Iterable[int]] = None, w64=None, cache=None):
    """Oracle outputs [n, Hq, d] of the decode queries ``rows`` (default: all).
    cache="bf16": the oracle's cache components rounded to bf16 first."""
    sh = case.shape
    w64 = w64 or weights64(case)
    scale = 1.0 / math.sqrt(sh.head_dim)
    qs = case.dec_q_start.tolist()
    rows = list(range(case.dec_q.shape[0])) if rows is None else list(rows)
    out = {}
    by_ctx = {}
    for r in rows:
        c = next(i for i in range(len(case.dec_ctx)) if qs[i] <= r < qs[i + 1])
        by_ctx.setdefault(c, []).append(r)
    for c, rs in by_ctx.items():
        X, X_lr = _hidden(case, case.dec_ctx[c])
        q = case.dec_q[rs].double().numpy()
        ad = case.dec_adapter[rs].numpy()
        if getattr(sh, "kv_codec", 0):
            # compressed base pool: the oracle encodes its own exact base part
            o = polykv.decode_codec(X, q, ad, w64, sh.n_kv_heads, sh.head_dim, sh.rope_base, scale,
                                    "bf16" if cache == "bf16" else None)
        else:
            o = oracle.decode(X, q, ad, w64, sh.n_kv_heads, sh.head_dim, sh.rope_base, scale, cache, X_lr)
        for i, r in enumerate(rs):
            out[r] = o[i]
    return np.stack([out[r] for r in rows])


def oracle_prefill_seq(case, p: int, q_rows: Optional[Iterable[int]] = None, w64=None, cache=None):
    """Oracle outputs of prefill sequence ``p`` (index into case.pre_seq), for the
    chunk rows ``q_rows`` (default: the whole chunk). Returns (rows, out)."""
    sh = case.shape
    w64 = w64 or weights64(case)
    scale = 1.0 / math.sqrt(sh.head_dim)
    s = case.pre_seq[p]
    X, X_lr = _hidden(case, s)
    a, b = int(case.pre_q_start[p]), int(case.pre_q_start[p + 1])
    n = b - a
    q_rows = list(range(n)) if q_rows is None else list(q_rows)
    L = X.shape[0]
    q = case.pre_q[a:b][q_rows].double().numpy()
    pos = np.array([L - n + k for k in q_rows])
    if getattr(sh, "kv_codec", 0):
        out = polykv.attend_codec(X, int(case.pre_adapter[p]), q, pos, w64, sh.n_kv_heads, sh.head_dim,
                                  sh.rope_base, scale, "bf16" if cache == "bf16" else None)
    else:
        out = oracle.attend(X, int(case.pre_adapter[p]), q, pos, w64, sh.n_kv_heads, sh.head_dim,
                            sh.rope_base, scale, cache, X_lr)
    return [a + k for k in q_rows], out
