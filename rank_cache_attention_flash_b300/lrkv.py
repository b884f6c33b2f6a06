"""Python binding of liblrkv (ctypes). Argument marshalling only: every step of
the computation runs in the CUDA library; torch provides device memory and
streams. The library must be built (``python -m rank_cache_attention_flash_b300.build``);
nothing here falls back to another implementation.

Entry points mirror the C ABI in ``include/lrkv.h``:
  append, append_rebase, attn_decode, attn_prefill, decode_workspace_bytes,
  prefill_workspace_bytes, status_string, version, attn_decode_noalloc.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

from . import build as _build

LIB_PATH = _build.LIB
BLOCK = 16

STATUS = {0: "LRKV_OK", 1: "LRKV_ERR_INVALID_ARG", 2: "LRKV_ERR_UNSUPPORTED", 3: "LRKV_ERR_CUDA",
          4: "LRKV_ERR_INDEX", 5: "LRKV_ERR_TIMEOUT", 6: "LRKV_ERR_WORKSPACE"}
BF16, FP32 = 0, 1
CODEC_NONE, CODEC_POLYKV = 0, 1

EXPORTS = ("lrkv_append", "lrkv_append_rebase", "lrkv_attn_decode", "lrkv_decode_workspace_bytes", "lrkv_attn_prefill",
           "lrkv_prefill_workspace_bytes", "lrkv_status_string", "lrkv_version",
           "lrkv_attn_decode_noalloc", "lrkv_testing_set_decode_stall", "lrkv_base_pool_block_bytes",
           "lrkv_attn_mixed")
NOALLOC_SCRATCH_BYTES = 16 << 20  # LRKV_NOALLOC_SCRATCH_BYTES in lrkv.h


class LrkvError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where} failed: {STATUS.get(code, code)}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rank", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("rope_base", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("lr_groups", ctypes.c_int32), ("kv_codec", ctypes.c_int32)]

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == BF16 else torch.float32

    @property
    def lr_width(self) -> int:
        """Columns of a low-rank pool row: every group's r columns side by side."""
        return max(1, self.lr_groups) * self.rank

    @property
    def codec_chunk_bytes(self) -> int:
        """Bytes of one (block, kv head) chunk of a compressed base pool."""
        return 23 * self.head_dim + 64

    @property
    def n_cols(self) -> int:
        return 2 * self.n_kv_heads * self.head_dim + 2 * self.lr_width


class DecodeBatch(ctypes.Structure):
    """lrkv_decode_batch: the decode part of a mixed call."""
    _fields_ = [("q", ctypes.c_void_p), ("num_queries", ctypes.c_int32), ("ctx_q_start", ctypes.c_void_p),
                ("num_ctx", ctypes.c_int32), ("adapter_ids", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p), ("max_blocks", ctypes.c_int32),
                ("ctx_lens", ctypes.c_void_p), ("max_ctx_len", ctypes.c_int32),
                ("max_q_per_ctx", ctypes.c_int32), ("out", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


class PrefillBatch(ctypes.Structure):
    """lrkv_prefill_batch: the prefill part of a mixed call."""
    _fields_ = [("q", ctypes.c_void_p), ("q_start", ctypes.c_void_p), ("num_seqs", ctypes.c_int32),
                ("total_q", ctypes.c_int32), ("max_q_len", ctypes.c_int32), ("seq_lens", ctypes.c_void_p),
                ("max_seq_len", ctypes.c_int32), ("adapter_ids", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p), ("max_blocks", ctypes.c_int32), ("out", ctypes.c_void_p)]


def make_config(hidden: int, n_q_heads: int, n_kv_heads: int, head_dim: int, rank: int,
                rope_base: float = 10000.0, dtype: torch.dtype = torch.bfloat16,
                lr_groups: int = 1, kv_codec: int = 0) -> Config:
    """lr_groups = 1: one A shared by every agent; lr_groups = n: agent a has its
    own A_a and reads low-rank group a (PreLRShared). kv_codec = CODEC_POLYKV:
    the base pool is compressed (q8_0 keys, rotated 3-bit values)."""
    return Config(hidden, n_q_heads, n_kv_heads, head_dim, rank, BLOCK, rope_base,
                  BF16 if dtype == torch.bfloat16 else FP32, lr_groups, kv_codec)


_lib = None
_P, _I32, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


def load() -> ctypes.CDLL:
    """Loads liblrkv.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m rank_cache_attention_flash_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    cfgp = ctypes.POINTER(Config)
    lib.lrkv_append.argtypes = [cfgp, _P, _I32, _P, _P, _P, _I32, _I32, _P, _P, _P, _I64, _P, _P]
    lib.lrkv_append.restype = ctypes.c_int
    lib.lrkv_append_rebase.argtypes = [cfgp, _P, _P, _I32, _P, _P, _P, _I32, _I32, _P, _P, _P, _I64, _P, _P]
    lib.lrkv_append_rebase.restype = ctypes.c_int
    lib.lrkv_attn_decode.argtypes = [cfgp, _P, _I32, _P, _I32, _P, _P, _I32, _P, _I32, _I32, _P, _P,
                                     _I64, _P, _P, _I32, _F, _P, _P, _SZ, _P, _P]
    lib.lrkv_attn_decode.restype = ctypes.c_int
    lib.lrkv_decode_workspace_bytes.argtypes = [cfgp, _I32, _I32, _I32, _I32]
    lib.lrkv_decode_workspace_bytes.restype = _SZ
    lib.lrkv_attn_prefill.argtypes = [cfgp, _P, _P, _I32, _I32, _I32, _P, _I32, _P, _P, _I32, _P,
                                      _P, _I64, _P, _P, _I32, _F, _P, _P, _SZ, _P, _P]
    lib.lrkv_attn_prefill.restype = ctypes.c_int
    lib.lrkv_prefill_workspace_bytes.argtypes = [cfgp, _I32, _I32, _I32, _I32]
    lib.lrkv_prefill_workspace_bytes.restype = _SZ
    lib.lrkv_attn_decode_noalloc.argtypes = [cfgp, _P, _I32, _P, _I32, _P, _P, _I32, _P, _I32, _I32,
                                             _P, _P, _I64, _P, _P, _I32, _F, _P, _P, _P]
    lib.lrkv_attn_decode_noalloc.restype = ctypes.c_int
    lib.lrkv_attn_mixed.argtypes = [cfgp, ctypes.POINTER(DecodeBatch), ctypes.POINTER(PrefillBatch), _P, _P,
                                    _I64, _P, _P, _I32, _F, _P, _P]
    lib.lrkv_attn_mixed.restype = ctypes.c_int
    lib.lrkv_status_string.argtypes = [ctypes.c_int]
    lib.lrkv_status_string.restype = ctypes.c_char_p
    lib.lrkv_version.argtypes = []
    lib.lrkv_version.restype = ctypes.c_int32
    lib.lrkv_base_pool_block_bytes.argtypes = [ctypes.POINTER(Config)]
    lib.lrkv_base_pool_block_bytes.restype = _SZ
    lib.lrkv_testing_set_decode_stall.argtypes = [_I32]
    lib.lrkv_testing_set_decode_stall.restype = None
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(t: Optional[torch.Tensor], name: str, dtype=None, device=None):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must live on {device}")


def _raise(code: int, where: str):
    if code != 0:
        raise LrkvError(code, where)


def status_string(code: int) -> str:
    return load().lrkv_status_string(code).decode()


def version() -> int:
    return load().lrkv_version()


def testing_set_decode_stall(enable: bool) -> None:
    """Test only (include/lrkv_testing.h): while enabled, every G-mode decode
    launch makes one bounded wait run out, reports LRKV_ERR_TIMEOUT in its
    status word and returns through its abort path."""
    load().lrkv_testing_set_decode_stall(1 if enable else 0)


# ------------------------------------------------------------------ helpers
def pack_w_cat(W_K: torch.Tensor, W_V: torch.Tensor, A_K: torch.Tensor, A_V: torch.Tensor) -> torch.Tensor:
    """One-time weight layout for append: [N, h] rows = output columns
    (nn.Linear layout), in the order K | V | A_K | A_V. Agent-specific factors
    A_K, A_V of shape [G, h, r] contribute their groups in order (group g's r
    rows after group g-1's)."""
    def rows(A):
        return A.t() if A.dim() == 2 else A.permute(0, 2, 1).reshape(-1, A.shape[1])
    return torch.cat([W_K.t(), W_V.t(), rows(A_K), rows(A_V)], 0).contiguous()


def new_pools(cfg: Config, num_blocks: int, device, fill: Optional[float] = None
              ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Allocates (base_pool, lr_pool) for ``num_blocks`` blocks. A compressed
    base pool is bytes [num_blocks][Hkv][23 d + 64]; ``fill`` then fills only
    the low-rank pool (the base pool's bytes are set to 0xFF)."""
    dt = cfg.torch_dtype
    if cfg.kv_codec == CODEC_POLYKV:
        base = torch.empty(num_blocks, cfg.n_kv_heads, cfg.codec_chunk_bytes, dtype=torch.uint8, device=device)
    else:
        base = torch.empty(num_blocks, 2, cfg.n_kv_heads, BLOCK, cfg.head_dim, dtype=dt, device=device)
    lr = torch.empty(num_blocks, 2, BLOCK, cfg.lr_width, dtype=dt, device=device)
    if fill is not None:
        if cfg.kv_codec == CODEC_POLYKV:
            base.fill_(255)
        else:
            base.fill_(fill)
        lr.fill_(fill)
    return base, lr


def base_pool_block_bytes(cfg: Config) -> int:
    return int(load().lrkv_base_pool_block_bytes(ctypes.byref(cfg)))


def unpack_codec_pool(cfg: Config, base: torch.Tensor):
    """Host-side view of a compressed base pool: dict of CPU arrays over
    [num_blocks, Hkv, 16]: Kq int8 [.., d], Ks fp16 [.., d/32], Vq uint8 codes
    0..7 [.., d] (from the three bit planes), Vn fp32 [..]."""
    import numpy as np
    d = cfg.head_dim
    b = base.cpu().numpy()
    nb, hkv = b.shape[0], b.shape[1]
    o_ks, o_vq, o_vn = 16 * d, 17 * d, 23 * d
    Kq = b[:, :, :o_ks].view(np.int8).reshape(nb, hkv, BLOCK, d)
    Ks = np.ascontiguousarray(b[:, :, o_ks:o_vq]).view(np.float16).reshape(nb, hkv, BLOCK, d // 32)
    planes = b[:, :, o_vq:o_vn].reshape(nb, hkv, BLOCK, 3, d // 8)
    bits = np.unpackbits(planes, axis=-1, bitorder="little")  # [.., 3, d]
    Vq = (bits[..., 0, :] | (bits[..., 1, :] << 1) | (bits[..., 2, :] << 2)).astype(np.uint8)
    Vn = np.ascontiguousarray(b[:, :, o_vn:o_vn + 64]).view(np.float32).reshape(nb, hkv, BLOCK)
    return {"Kq": Kq, "Ks": Ks, "Vq": Vq, "Vn": Vn}


# ------------------------------------------------------------- entry points
def append(cfg: Config, X: torch.Tensor, positions: torch.Tensor, seq_rows: torch.Tensor,
           block_tables: torch.Tensor, W_cat: torch.Tensor, base_pool: torch.Tensor,
           lr_pool: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None) -> None:
    lib = load()
    dev = base_pool.device
    _check(X, "X", cfg.torch_dtype, dev)
    _check(W_cat, "W_cat", cfg.torch_dtype, dev)
    for t, n in ((positions, "positions"), (seq_rows, "seq_rows"), (block_tables, "block_tables")):
        _check(t, n, torch.int32, dev)
    _check(status, "status", torch.int32, dev)
    T = X.shape[0]
    if X.shape != (T, cfg.hidden) or positions.numel() != T or seq_rows.numel() != T:
        raise ValueError("append: shape mismatch")
    if W_cat.shape != (cfg.n_cols, cfg.hidden):
        raise ValueError("append: W_cat must be [2*Hkv*d + 2*r, h]")
    code = lib.lrkv_append(ctypes.byref(cfg), _ptr(X), T, _ptr(positions), _ptr(seq_rows),
                           _ptr(block_tables), block_tables.shape[0], block_tables.shape[1],
                           _ptr(W_cat), _ptr(base_pool), _ptr(lr_pool), base_pool.shape[0],
                           _ptr(status), _stream(stream))
    _raise(code, "lrkv_append")


def append_rebase(cfg: Config, X_base: Optional[torch.Tensor], X_lr: Optional[torch.Tensor],
                  positions: torch.Tensor, seq_rows: torch.Tensor, block_tables: torch.Tensor,
                  W_cat: torch.Tensor, base_pool: torch.Tensor, lr_pool: torch.Tensor,
                  status: Optional[torch.Tensor] = None, stream=None) -> None:
    """lrkv_append_rebase: base rows from X_base, low-rank rows from X_lr (either
    may be None: that part of the pools is left as it is)."""
    lib = load()
    dev = base_pool.device
    _check(X_base, "X_base", cfg.torch_dtype, dev)
    _check(X_lr, "X_lr", cfg.torch_dtype, dev)
    _check(W_cat, "W_cat", cfg.torch_dtype, dev)
    for t, n in ((positions, "positions"), (seq_rows, "seq_rows"), (block_tables, "block_tables")):
        _check(t, n, torch.int32, dev)
    _check(status, "status", torch.int32, dev)
    T = positions.numel()
    for X in (X_base, X_lr):
        if X is not None and X.shape != (T, cfg.hidden):
            raise ValueError("append_rebase: X must be [T, h]")
    if seq_rows.numel() != T or W_cat.shape != (cfg.n_cols, cfg.hidden):
        raise ValueError("append_rebase: shape mismatch")
    code = lib.lrkv_append_rebase(ctypes.byref(cfg), _ptr(X_base), _ptr(X_lr), T, _ptr(positions),
                                  _ptr(seq_rows), _ptr(block_tables), block_tables.shape[0],
                                  block_tables.shape[1], _ptr(W_cat), _ptr(base_pool), _ptr(lr_pool),
                                  base_pool.shape[0], _ptr(status), _stream(stream))
    _raise(code, "lrkv_append_rebase")


def decode_workspace_bytes(cfg: Config, num_queries: int, num_ctx: int, max_ctx_len: int,
                           max_q_per_ctx: int) -> int:
    return int(load().lrkv_decode_workspace_bytes(ctypes.byref(cfg), num_queries, num_ctx,
                                                   max_ctx_len, max_q_per_ctx))


def prefill_workspace_bytes(cfg: Config, num_seqs: int, total_q: int, max_q_len: int,
                            max_seq_len: int) -> int:
    return int(load().lrkv_prefill_workspace_bytes(ctypes.byref(cfg), num_seqs, total_q, max_q_len,
                                                    max_seq_len))


def attn_decode(cfg: Config, q: torch.Tensor, ctx_q_start: torch.Tensor, adapter_ids: torch.Tensor,
                block_tables: torch.Tensor, ctx_lens: torch.Tensor, max_ctx_len: int,
                max_q_per_ctx: int, base_pool: torch.Tensor, lr_pool: torch.Tensor,
                B_K: Optional[torch.Tensor], B_V: Optional[torch.Tensor],
                scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    lib = load()
    dev = base_pool.device
    _check(q, "q", cfg.torch_dtype, dev)
    for t, n in ((ctx_q_start, "ctx_q_start"), (adapter_ids, "adapter_ids"),
                 (block_tables, "block_tables"), (ctx_lens, "ctx_lens")):
        _check(t, n, torch.int32, dev)
    _check(B_K, "B_K", cfg.torch_dtype, dev)
    _check(B_V, "B_V", cfg.torch_dtype, dev)
    _check(status, "status", torch.int32, dev)
    nq = q.shape[0]
    num_ctx = ctx_lens.numel()
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", cfg.torch_dtype, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(cfg.head_dim)
    if workspace is None:  # a workspace passed in is checked by the library (LRKV_ERR_WORKSPACE)
        need = decode_workspace_bytes(cfg, nq, num_ctx, max_ctx_len, max_q_per_ctx)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    n_adapters = 0 if B_K is None and B_V is None else (B_K if B_K is not None else B_V).shape[0]
    code = lib.lrkv_attn_decode(
        ctypes.byref(cfg), _ptr(q), nq, _ptr(ctx_q_start), num_ctx, _ptr(adapter_ids),
        _ptr(block_tables), block_tables.shape[1], _ptr(ctx_lens), max_ctx_len, max_q_per_ctx,
        _ptr(base_pool), _ptr(lr_pool), base_pool.shape[0], _ptr(B_K), _ptr(B_V), n_adapters,
        float(scale), _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream))
    _raise(code, "lrkv_attn_decode")
    return out


def attn_prefill(cfg: Config, q: torch.Tensor, q_start: torch.Tensor, max_q_len: int,
                 seq_lens: torch.Tensor, max_seq_len: int, adapter_ids: torch.Tensor,
                 block_tables: torch.Tensor, base_pool: torch.Tensor, lr_pool: torch.Tensor,
                 B_K: Optional[torch.Tensor], B_V: Optional[torch.Tensor],
                 scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    lib = load()
    dev = base_pool.device
    _check(q, "q", cfg.torch_dtype, dev)
    for t, n in ((q_start, "q_start"), (seq_lens, "seq_lens"), (adapter_ids, "adapter_ids"),
                 (block_tables, "block_tables")):
        _check(t, n, torch.int32, dev)
    _check(B_K, "B_K", cfg.torch_dtype, dev)
    _check(B_V, "B_V", cfg.torch_dtype, dev)
    _check(status, "status", torch.int32, dev)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", cfg.torch_dtype, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(cfg.head_dim)
    S = seq_lens.numel()
    n_adapters = 0 if B_K is None and B_V is None else (B_K if B_K is not None else B_V).shape[0]
    code = lib.lrkv_attn_prefill(
        ctypes.byref(cfg), _ptr(q), _ptr(q_start), S, q.shape[0], max_q_len, _ptr(seq_lens),
        max_seq_len, _ptr(adapter_ids), _ptr(block_tables), block_tables.shape[1], _ptr(base_pool),
        _ptr(lr_pool), base_pool.shape[0], _ptr(B_K), _ptr(B_V), n_adapters, float(scale), _ptr(out),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _raise(code, "lrkv_attn_prefill")
    return out


def attn_mixed(cfg: Config, base_pool: torch.Tensor, lr_pool: torch.Tensor, B_K: Optional[torch.Tensor],
               B_V: Optional[torch.Tensor], decode: Optional[dict] = None, prefill: Optional[dict] = None,
               scale: Optional[float] = None, status: Optional[torch.Tensor] = None, stream=None):
    """lrkv_attn_mixed: a decode batch and a prefill batch in one call (the two
    run concurrently on the GPU). ``decode`` holds the tensors and sizes of
    attn_decode (q, ctx_q_start, adapter_ids, block_tables, ctx_lens,
    max_ctx_len, max_q_per_ctx, out, workspace), ``prefill`` those of
    attn_prefill (q, q_start, max_q_len, seq_lens, max_seq_len, adapter_ids,
    block_tables, out); outputs and the decode workspace are allocated here
    when missing. Returns (decode out or None, prefill out or None)."""
    lib = load()
    dev = base_pool.device
    _check(B_K, "B_K", cfg.torch_dtype, dev)
    _check(B_V, "B_V", cfg.torch_dtype, dev)
    _check(status, "status", torch.int32, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(cfg.head_dim)
    dref = pref = None
    d_out = p_out = None
    ws = None
    if decode is not None:
        d = decode
        _check(d["q"], "decode q", cfg.torch_dtype, dev)
        for n in ("ctx_q_start", "adapter_ids", "block_tables", "ctx_lens"):
            _check(d[n], "decode " + n, torch.int32, dev)
        nq, num_ctx = d["q"].shape[0], d["ctx_lens"].numel()
        d_out = d.get("out")
        if d_out is None:
            d_out = torch.empty_like(d["q"])
        _check(d_out, "decode out", cfg.torch_dtype, dev)
        ws = d.get("workspace")
        if ws is None:
            need = decode_workspace_bytes(cfg, nq, num_ctx, d["max_ctx_len"], d["max_q_per_ctx"])
            if need > 0:
                ws = torch.empty(need, dtype=torch.uint8, device=dev)
        dref = ctypes.byref(DecodeBatch(
            _ptr(d["q"]), nq, _ptr(d["ctx_q_start"]), num_ctx, _ptr(d["adapter_ids"]), _ptr(d["block_tables"]),
            d["block_tables"].shape[1], _ptr(d["ctx_lens"]), d["max_ctx_len"], d["max_q_per_ctx"], _ptr(d_out),
            _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size()))
    if prefill is not None:
        f = prefill
        _check(f["q"], "prefill q", cfg.torch_dtype, dev)
        for n in ("q_start", "seq_lens", "adapter_ids", "block_tables"):
            _check(f[n], "prefill " + n, torch.int32, dev)
        p_out = f.get("out")
        if p_out is None:
            p_out = torch.empty_like(f["q"])
        _check(p_out, "prefill out", cfg.torch_dtype, dev)
        pref = ctypes.byref(PrefillBatch(
            _ptr(f["q"]), _ptr(f["q_start"]), f["seq_lens"].numel(), f["q"].shape[0], f["max_q_len"],
            _ptr(f["seq_lens"]), f["max_seq_len"], _ptr(f["adapter_ids"]), _ptr(f["block_tables"]),
            f["block_tables"].shape[1], _ptr(p_out)))
    n_adapters = 0 if B_K is None and B_V is None else (B_K if B_K is not None else B_V).shape[0]
    code = lib.lrkv_attn_mixed(ctypes.byref(cfg), dref, pref, _ptr(base_pool), _ptr(lr_pool), base_pool.shape[0],
                               _ptr(B_K), _ptr(B_V), n_adapters, float(scale), _ptr(status), _stream(stream))
    _raise(code, "lrkv_attn_mixed")
    return d_out, p_out


def attn_decode_noalloc(cfg: Config, q: torch.Tensor, ctx_q_start: torch.Tensor,
                        adapter_ids: torch.Tensor, block_tables: torch.Tensor, ctx_lens: torch.Tensor,
                        max_ctx_len: int, max_q_per_ctx: int, base_pool: torch.Tensor,
                        lr_pool: torch.Tensor, B_K: Optional[torch.Tensor], B_V: Optional[torch.Tensor],
                        out: torch.Tensor, scale: Optional[float] = None,
                        status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """lrkv_attn_decode_noalloc: decode without a caller workspace, for callers
    that cannot allocate device memory (the library keeps a fixed scratch array
    of NOALLOC_SCRATCH_BYTES per device). ``out`` is required: this wrapper
    allocates nothing either."""
    lib = load()
    dev = base_pool.device
    _check(q, "q", cfg.torch_dtype, dev)
    for t, n in ((ctx_q_start, "ctx_q_start"), (adapter_ids, "adapter_ids"),
                 (block_tables, "block_tables"), (ctx_lens, "ctx_lens")):
        _check(t, n, torch.int32, dev)
    _check(B_K, "B_K", cfg.torch_dtype, dev)
    _check(B_V, "B_V", cfg.torch_dtype, dev)
    _check(status, "status", torch.int32, dev)
    _check(out, "out", cfg.torch_dtype, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(cfg.head_dim)
    n_adapters = 0 if B_K is None and B_V is None else (B_K if B_K is not None else B_V).shape[0]
    code = lib.lrkv_attn_decode_noalloc(
        ctypes.byref(cfg), _ptr(q), q.shape[0], _ptr(ctx_q_start), ctx_lens.numel(), _ptr(adapter_ids),
        _ptr(block_tables), block_tables.shape[1], _ptr(ctx_lens), max_ctx_len, max_q_per_ctx,
        _ptr(base_pool), _ptr(lr_pool), base_pool.shape[0], _ptr(B_K), _ptr(B_V), n_adapters,
        float(scale), _ptr(out), _ptr(status), _stream(stream))
    _raise(code, "lrkv_attn_decode_noalloc")
    return out
