"""The fp64 oracle against its pins, and planted mistakes that the pins must catch.

CPU only. The mutation tests load a private copy of the oracle's source with
one deliberate mistake planted in it (a flipped sign, a dropped term, a wrong
index, a swapped operand) and check that at least one pin fails on it.
"""
import importlib.util
import os
import types

import pytest

from tests import oracle_pins as P

import oracle as O

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "lrkv_oracle.py")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(O)


def _mutant(old: str, new: str) -> types.ModuleType:
    src = open(ORACLE_SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = {
    "rope_sign": ("lo * c - hi * s", "lo * c + hi * s"),
    "rope_interleaved_pairs": ("lo, hi = x[..., :half], x[..., half:]",
                               "lo, hi = x[..., 0::2], x[..., 1::2]"),
    "rope_freq_exponent": ("-2.0 * j / head_dim", "-1.0 * j / head_dim"),
    "rope_on_values": ("return k, v.reshape(T, n_kv_heads, head_dim)",
                       "return k, apply_rope(v.reshape(T, n_kv_heads, head_dim), positions, base)"),
    "drop_k_adapter": ("k_pre = k_pre + (X @ _f64(A_K)) @ _f64(B_K_i)", "k_pre = k_pre"),
    "drop_v_adapter": ("v = v + (X @ _f64(A_V)) @ _f64(B_V_i)", "v = v"),
    "swap_A_in_agent_kv": ("k_pre = k_pre + (X @ _f64(A_K)) @ _f64(B_K_i)",
                           "k_pre = k_pre + (X @ _f64(A_V)) @ _f64(B_K_i)"),
    "swap_lowrank_outputs": ("_lowrank(X, A_K), _lowrank(X, A_V))", "_lowrank(X, A_V), _lowrank(X, A_K))"),
    "prelr_groups_reversed": ("np.concatenate([X @ A[g] for g in range(A.shape[0])], axis=1)",
                              "np.concatenate([X @ A[g] for g in reversed(range(A.shape[0]))], axis=1)"),
    "prelr_agent_uses_group_0": ("        g = max(adapter, 0)\n", "        g = 0\n"),
    "prelr_agent_off_by_one": ("        g = max(adapter, 0)\n", "        g = (adapter + 1) % A_K.shape[0]\n"),
    "kv_head_modulo": ("kv = m // g", "kv = m % Hkv"),
    "causal_strict": ("np.arange(L)[None, :] <= qp[:, None]", "np.arange(L)[None, :] < qp[:, None]"),
    "causal_peek_ahead": ("np.arange(L)[None, :] <= qp[:, None]", "np.arange(L)[None, :] <= qp[:, None] + 1"),
    "no_softmax_scale": ("(q[:, m, :] @ K[:, kv, :].T) * scale", "(q[:, m, :] @ K[:, kv, :].T)"),
    "key_positions_shifted": ("make(X_seq, np.arange(L),", "make(X_seq, np.arange(1, L + 1),"),
    "prefill_positions_shifted": ("np.arange(L - n, L)", "np.arange(L - n - 1, L - 1)"),
    "decode_position_shifted": ("np.asarray(q)[n: n + 1], [L - 1]", "np.asarray(q)[n: n + 1], [L - 2]"),
    "append_row_shifted": ("row = p % BLOCK", "row = (p + 1) % BLOCK"),
    "append_block_index": ("blk = int(block_tables[s][p // BLOCK])",
                           "blk = int(block_tables[s][(p // BLOCK + 1) % len(block_tables[s])])"),
    "adapter_off_by_one": ('return weights["B_K"][adapter], weights["B_V"][adapter]',
                           'return weights["B_K"][adapter - 1], weights["B_V"][adapter - 1]'),
    "bf16_truncation": ("u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000", "u = u & 0xFFFF0000"),
    "bf16_ties_away": ("u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000", "u = (u + 0x8000) & 0xFFFF0000"),
    "cache_variant_drops_rope": ("k = k + apply_rope((lk @ _f64(B_K_i)).reshape(T, n_kv_heads, head_dim), positions, base)",
                                 "k = k + (lk @ _f64(B_K_i)).reshape(T, n_kv_heads, head_dim)"),
    "rebase_base_from_lowrank_source": ("kb, vb, _, _ = base_and_lowrank(X_base, positions,",
                                        "kb, vb, _, _ = base_and_lowrank(X_lr if X_lr is not None else X_base, positions,"),
    "rebase_lowrank_from_base_source": ("_, _, lk, lv = base_and_lowrank(X_lr, positions,",
                                        "_, _, lk, lv = base_and_lowrank(X_base if X_base is not None else X_lr, positions,"),
    "rebased_kv_lowrank_from_base": ("k_pre = k_pre + (X_lr @ _f64(A_K)) @ _f64(B_K_i)",
                                     "k_pre = k_pre + (X_base @ _f64(A_K)) @ _f64(B_K_i)"),
    "rebased_v_from_lowrank_source": ("        v = X_base @ _f64(W_V)\n", "        v = X_lr @ _f64(W_V)\n"),
    "swapped_B": ('return weights["B_K"][adapter], weights["B_V"][adapter]',
                  'return weights["B_V"][adapter], weights["B_K"][adapter]'),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    old, new = MUTATIONS[name]
    M = _mutant(old, new)
    failed = []
    for pin in P.ALL_PINS:
        try:
            with __import__("warnings").catch_warnings():
                __import__("warnings").simplefilter("ignore")
                pin(M)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
