"""Host-only checks of the C ABI (no GPU needed): the library loads, exports every
entry point that the headers under include/ declare, and rejects bad arguments
before any launch."""
import ctypes
import glob
import os
import re

import pytest

from rank_cache_attention_flash_b300 import build as B
from rank_cache_attention_flash_b300 import lrkv

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "lrkv.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return lrkv.load()


def declared_functions(headers=None):
    names = set()
    for h in headers or sorted(glob.glob(os.path.join(INCLUDE, "*.h"))):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(lrkv_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions([HEADER])
    for n in ("lrkv_append", "lrkv_append_rebase", "lrkv_attn_decode", "lrkv_attn_prefill",
              "lrkv_decode_workspace_bytes", "lrkv_attn_decode_noalloc", "lrkv_attn_mixed"):
        assert n in names
    assert "lrkv_testing_set_decode_stall" in declared_functions([os.path.join(INCLUDE, "lrkv_testing.h")])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared under include/ but not exported"
    assert set(lrkv.EXPORTS) <= set(declared_functions())


def test_status_strings_and_version(lib):
    for code, name in lrkv.STATUS.items():
        assert lrkv.status_string(code) == name
    assert lrkv.status_string(77) == "LRKV_UNKNOWN_STATUS"
    assert lrkv.version() >= 100


def _cfg(**kw):
    base = dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, rank=8, block_size=16,
                rope_base=10000.0, dtype=0, lr_groups=1, kv_codec=0)
    base.update(kw)
    return lrkv.Config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), 2), (dict(rank=12), 2), (dict(block_size=32), 2), (dict(dtype=5), 2),
    (dict(n_q_heads=5), 1), (dict(hidden=0), 1), (dict(rope_base=0.0), 1), (dict(hidden=100), 2),
    (dict(n_q_heads=64, n_kv_heads=2), 2), (dict(lr_groups=0), 1), (dict(lr_groups=65), 2),
    (dict(kv_codec=2), 1), (dict(kv_codec=-1), 1), (dict(kv_codec=1, dtype=1), 2),
])
def test_bad_config_rejected_before_launch(lib, kw, code):
    cfg = _cfg(**kw)
    r = lib.lrkv_append(ctypes.byref(cfg), 16, 1, 16, 16, 16, 1, 1, 16, 16, 16, 1, None, None)
    assert r == code


def test_null_and_misaligned_pointers_rejected(lib):
    cfg = _cfg()
    P = 1 << 20  # a fake, 16-byte aligned address: never dereferenced on these paths
    # append: null X
    assert lib.lrkv_append(ctypes.byref(cfg), None, 4, P, P, P, 1, 1, P, P, P, 1, None, None) == 1
    # append: misaligned X
    assert lib.lrkv_append(ctypes.byref(cfg), P + 2, 4, P, P, P, 1, 1, P, P, P, 1, None, None) == 1
    # append: T = 0 is a no-op
    assert lib.lrkv_append(ctypes.byref(cfg), None, 0, None, None, None, 0, 0, None, None, None, 0,
                           None, None) == 0
    # append: negative T
    assert lib.lrkv_append(ctypes.byref(cfg), P, -1, P, P, P, 1, 1, P, P, P, 1, None, None) == 1
    # decode: null q
    args = [ctypes.byref(cfg), None, 2, P, 1, P, P, 4, P, 64, 2, P, P, 8, P, P, 2, 0.125, P, P, 1 << 20,
            None, None]
    assert lib.lrkv_attn_decode(*args) == 1
    # decode: no queries is a no-op
    args0 = list(args)
    args0[2] = 0
    assert lib.lrkv_attn_decode(*args0) == 0
    # decode: adapters given but n_adapters == 0
    args2 = list(args)
    args2[1] = P
    args2[16] = 0
    assert lib.lrkv_attn_decode(*args2) == 1
    # decode: max_ctx_len beyond the block table
    args3 = list(args)
    args3[1] = P
    args3[9] = 4 * 16 + 1
    assert lib.lrkv_attn_decode(*args3) == 1
    # prefill: null seq_lens
    pargs = [ctypes.byref(cfg), P, P, 1, 8, 8, None, 64, P, P, 4, P, P, 8, P, P, 2, 0.125, P, None, 0,
             None, None]
    assert lib.lrkv_attn_prefill(*pargs) == 1
    # prefill: max_seq_len < max_q_len
    pargs2 = list(pargs)
    pargs2[6] = P
    pargs2[7] = 4
    assert lib.lrkv_attn_prefill(*pargs2) == 1


def test_mixed_call_checks_both_parts_before_launch(lib):
    """lrkv_attn_mixed: a bad field in either part is refused before anything
    runs (these calls reach no CUDA call), and two empty parts are a no-op."""
    cfg = _cfg()
    P = 1 << 20  # a fake, 16-byte aligned address: never dereferenced on these paths
    dec = lrkv.DecodeBatch(P, 2, P, 1, P, P, 4, P, 64, 2, P, P, 1 << 20)
    pre = lrkv.PrefillBatch(P, P, 1, 8, 8, P, 64, P, P, 4, P)
    call = lambda d, p: lib.lrkv_attn_mixed(ctypes.byref(cfg), d, p, P, P, 8, P, P, 2, 0.125, None, None)
    empty_d = lrkv.DecodeBatch(None, 0, None, 0, None, None, 0, None, 0, 0, None, None, 0)
    empty_p = lrkv.PrefillBatch(None, None, 0, 0, 0, None, 0, None, None, 0, None)
    assert call(None, None) == 0
    assert call(ctypes.byref(empty_d), ctypes.byref(empty_p)) == 0
    bad_d = lrkv.DecodeBatch(None, 2, P, 1, P, P, 4, P, 64, 2, P, P, 1 << 20)  # null q
    assert call(ctypes.byref(bad_d), ctypes.byref(pre)) == 1
    bad_p = lrkv.PrefillBatch(P, P, 1, 8, 8, None, 64, P, P, 4, P)  # null seq_lens
    assert call(None, ctypes.byref(bad_p)) == 1
    bad_p2 = lrkv.PrefillBatch(P, P, 1, 8, 8, P, 4, P, P, 4, P)  # max_seq_len < max_q_len
    assert call(ctypes.byref(empty_d), ctypes.byref(bad_p2)) == 1
    bad_d2 = lrkv.DecodeBatch(P, 2, P, 1, P, P, 4, P, 4 * 16 + 1, 2, P, P, 1 << 20)  # past the block table
    assert call(ctypes.byref(bad_d2), None) == 1
    assert lib.lrkv_attn_mixed(None, None, None, P, P, 8, P, P, 2, 0.125, None, None) == 1


def _header_struct_fields(name):
    """(field, C type) pairs of a struct typedef in lrkv.h, in declaration order."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"typedef struct(?:\s+\w+)?\s*\{([^}]*)\}\s*" + name + r"\s*;", src)
    assert m, name
    out = []
    for decl in m.group(1).split(";"):
        decl = " ".join(decl.split())
        if decl:
            ctype, field = decl.rsplit(" ", 1)
            out.append((field.lstrip("*"), ctype + ("*" if field.startswith("*") else "")))
    return out


def _ctypes_kind(ctype):
    if ctype.endswith("*"):
        return ctypes.c_void_p
    return {"int32_t": ctypes.c_int32, "float": ctypes.c_float, "size_t": ctypes.c_size_t}[ctype]


@pytest.mark.parametrize("cname,pyclass", [("lrkv_config", lrkv.Config), ("lrkv_decode_batch", lrkv.DecodeBatch),
                                           ("lrkv_prefill_batch", lrkv.PrefillBatch)])
def test_binding_structs_match_the_header(cname, pyclass):
    """The ctypes structures the binding passes by pointer have the header's
    fields, in its order, with types of the same size and kind."""
    fields = _header_struct_fields(cname)
    assert [f for f, _ in fields] == [f for f, _ in pyclass._fields_]
    for (f, ctype), (_, pytype) in zip(fields, pyclass._fields_):
        want = _ctypes_kind(ctype)
        assert ctypes.sizeof(pytype) == ctypes.sizeof(want), (cname, f)
        assert (pytype in (ctypes.c_float, ctypes.c_double)) == (want is ctypes.c_float), (cname, f)


def _header_prototypes():
    """name -> list of parameter C types of every function declared in lrkv.h."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(lrkv_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src):
        params = " ".join(m.group(2).split())
        if params in ("", "void"):
            protos[m.group(1)] = []
            continue
        types = []
        for p in params.split(","):
            p = p.strip()
            ptr = "*" in p
            base = p.replace("*", " ").split()
            base = [w for w in base if w != "const"]
            types.append("ptr" if ptr or base[0] == "lrkv_stream_t" else base[0])
        protos[m.group(1)] = types
    return protos


def test_binding_argtypes_match_the_header(lib):
    """Every function the binding types has the header's parameter count, and
    each parameter a ctypes type of the same size and kind (pointer, 32-bit
    int, 64-bit int, size_t, float)."""
    kinds = {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
             "float": ctypes.c_float, "lrkv_status": ctypes.c_int, "ptr": ctypes.c_void_p}
    protos = _header_prototypes()
    checked = 0
    for name, params in protos.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        assert len(fn.argtypes) == len(params), name
        for i, (have, want) in enumerate(zip(fn.argtypes, params)):
            w = kinds[want]
            if w is ctypes.c_void_p:
                assert ctypes.sizeof(have) == ctypes.sizeof(ctypes.c_void_p) and have not in (
                    ctypes.c_int64, ctypes.c_size_t, ctypes.c_double), (name, i)
            else:
                assert ctypes.sizeof(have) == ctypes.sizeof(w), (name, i, have, want)
                assert (have in (ctypes.c_float, ctypes.c_double)) == (w is ctypes.c_float), (name, i)
        checked += 1
    assert checked >= 10


def test_positions_limit_rejected(lib):
    cfg = _cfg()
    P = 1 << 20
    # max_blocks * 16 above 2^20 positions
    r = lib.lrkv_append(ctypes.byref(cfg), P, 4, P, P, P, 1, (1 << 16) + 1, P, P, P, 10, None, None)
    assert r == 2


def test_base_pool_block_bytes(lib):
    """bf16 / fp32 planes: 2 Hkv 16 d elements; compressed: Hkv (23 d + 64) bytes
    (Kq 16 d, Ks 16 d/32 fp16, Vq 16 x 3 x d/8, Vn 16 fp32)."""
    assert lrkv.base_pool_block_bytes(_cfg()) == 2 * 2 * 16 * 64 * 2
    assert lrkv.base_pool_block_bytes(_cfg(dtype=1)) == 2 * 2 * 16 * 64 * 4
    for d in (64, 128):
        want = 2 * (16 * d + 16 * (d // 32) * 2 + 16 * 3 * (d // 8) + 16 * 4)
        assert lrkv.base_pool_block_bytes(_cfg(kv_codec=1, head_dim=d)) == want == 2 * (23 * d + 64)
    assert lrkv.base_pool_block_bytes(_cfg(kv_codec=3)) == 0


def test_compressed_pool_arguments_checked(lib):
    """A compressed pool goes through the same host checks (null seq_lens)."""
    cfg = _cfg(kv_codec=1)
    P = 1 << 20
    pargs = [ctypes.byref(cfg), P, P, 1, 8, 8, None, 64, P, P, 4, P, P, 8, P, P, 2, 0.125, P, None, 0,
             None, None]
    assert lib.lrkv_attn_prefill(*pargs) == 1
