"""Drives a seeded workload (``inputs.Case``) through the CUDA library.

Uploads the weights and block tables, fills the paged pools with the untimed
setup appends (the context cached before the step), and runs the step: the
append of every new token, then decode and prefill attention. Only argument
preparation happens here; every computation is a library call.
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import torch

from . import inputs as I
from . import lrkv


def _align(n: int, a: int = 256) -> int:
    return (n + a - 1) // a * a


class _Arena:
    """One contiguous byte buffer holding several tensors as views, so that a
    step's inputs (or outputs) move between host and device in one copy."""

    def __init__(self):
        self.parts = []  # (name, offset, dtype, shape)
        self.nbytes = 0

    def add(self, name: str, t: torch.Tensor) -> None:
        self.parts.append((name, self.nbytes, t.dtype, tuple(t.shape), t))
        self.nbytes = _align(self.nbytes + t.numel() * t.element_size())

    def materialise(self, device, fill_from_parts: bool):
        """(device buffer, pinned host buffer or None, {name: device view})."""
        dev_buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device)
        host_buf = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8).pin_memory() \
            if torch.cuda.is_available() else None
        views = {}
        for name, off, dt, shape, src in self.parts:
            n = src.numel() * src.element_size()
            views[name] = dev_buf[off:off + n].view(dt).view(shape)
            if fill_from_parts and host_buf is not None:
                host_buf[off:off + n].view(dt).view(shape).copy_(src)
        if fill_from_parts and host_buf is not None:
            dev_buf.copy_(host_buf)
        return dev_buf, host_buf, views


class GpuCase:
    """A workload on one GPU. The step's per-call inputs (queries, context
    lengths, adapter ids, the new tokens' hidden states and positions) live in
    one input arena and its outputs in one output arena, each with a pinned
    host mirror: ``upload_inputs`` / ``download_outputs`` are then one copy
    each. Pools, weights and block tables stay resident.

    no_bk: pass B_K = NULL to attention (the K adapter term and its rebuild
    are skipped), a diagnostic that isolates the rebuild's cost."""

    def __init__(self, case: I.Case, device="cuda", pool_fill: Optional[float] = None,
                 setup_chunk_tokens: int = 1 << 16, no_bk: bool = False):
        self.case = case
        self.device = torch.device(device)
        sh = case.shape
        self.cfg = lrkv.make_config(sh.hidden, sh.n_q_heads, sh.n_kv_heads, sh.head_dim, sh.rank,
                                    sh.rope_base, sh.torch_dtype, sh.lr_groups, sh.kv_codec)
        dev = self.device
        w = case.weights
        self.W_cat = lrkv.pack_w_cat(w["W_K"], w["W_V"], w["A_K"], w["A_V"]).to(dev)
        self.B_K = w["B_K"].contiguous().to(dev)
        self.B_V = w["B_V"].contiguous().to(dev)
        self.attn_B_K = None if no_bk else self.B_K
        self.block_tables = case.block_tables.to(dev)
        self.base_pool, self.lr_pool = lrkv.new_pools(self.cfg, case.num_blocks, dev, pool_fill)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.scale = 1.0 / math.sqrt(sh.head_dim)
        self.setup_chunk_tokens = setup_chunk_tokens
        ins, outs = _Arena(), _Arena()
        bt = case.block_tables
        # decode arguments
        self.n_dec = int(case.dec_q.shape[0])
        if self.n_dec:
            ins.add("dec_q", case.dec_q)
            ins.add("dec_q_start", case.dec_q_start)
            ins.add("dec_adapter", case.dec_adapter)
            lens = case.dec_lens()
            ins.add("dec_lens", lens)
            outs.add("dec_out", case.dec_q)
            self.dec_bt = bt[torch.tensor(case.dec_ctx, dtype=torch.long)].contiguous().to(dev)
            self.dec_max_len = int(lens.max())
            qs = case.dec_q_start
            self.dec_max_q = int((qs[1:] - qs[:-1]).max())
            self.dec_ws = torch.empty(
                max(1, lrkv.decode_workspace_bytes(self.cfg, self.n_dec, len(case.dec_ctx),
                                                   self.dec_max_len, self.dec_max_q)),
                dtype=torch.uint8, device=dev)
        # prefill arguments
        self.n_pre = len(case.pre_seq)
        if self.n_pre:
            ins.add("pre_q", case.pre_q)
            ins.add("pre_q_start", case.pre_q_start)
            ins.add("pre_adapter", case.pre_adapter)
            lens = case.pre_lens()
            ins.add("pre_lens", lens)
            outs.add("pre_out", case.pre_q)
            self.pre_bt = bt[torch.tensor(case.pre_seq, dtype=torch.long)].contiguous().to(dev)
            self.pre_max_len = int(lens.max())
            qs = case.pre_q_start
            self.pre_max_q = int((qs[1:] - qs[:-1]).max())
        # step append arguments (all new tokens in one call)
        xs, pos, rows = [], [], []
        for s, a, b in case.step_appends():
            xs.append(case.seq_hidden(s, a, b))
            pos.append(torch.arange(a, b, dtype=torch.int32))
            rows.append(torch.full((b - a,), s, dtype=torch.int32))
        self.n_step_tokens = sum(x.shape[0] for x in xs)
        if xs:
            ins.add("step_X", torch.cat(xs))
            ins.add("step_pos", torch.cat(pos))
            ins.add("step_rows", torch.cat(rows))
            if case.rebase:  # the new tokens' adapter-free hidden states (base part)
                ins.add("step_Xb", torch.cat([case.seq_hidden_neutral(s, a, b) for s, a, b in case.step_appends()]))
        self.in_dev, self.in_host, views = ins.materialise(dev, True)
        self.out_dev, self.out_host, oviews = outs.materialise(dev, False)
        self.h2d_bytes = ins.nbytes
        self.d2h_bytes = outs.nbytes
        for k, v in {**views, **oviews}.items():
            setattr(self, k, v)

    # ------------------------------------------------------------------
    def upload_inputs(self) -> None:
        """The step's inputs from pinned host memory: one host-to-device copy on
        the current stream."""
        self.in_dev.copy_(self.in_host, non_blocking=True)

    def download_outputs(self) -> None:
        """The step's outputs to pinned host memory: one device-to-host copy on
        the current stream."""
        self.out_host.copy_(self.out_dev, non_blocking=True)

    def setup(self) -> None:
        """Untimed: append the tokens cached before the step."""
        case, dev = self.case, self.device
        pend_x, pend_p, pend_r, n = [], [], [], 0

        pend_xb = []

        def flush():
            nonlocal pend_x, pend_xb, pend_p, pend_r, n
            if not pend_x:
                return
            X = torch.cat(pend_x).to(dev)
            P = torch.cat(pend_p).to(dev)
            Rw = torch.cat(pend_r).to(dev)
            if case.rebase:
                lrkv.append_rebase(self.cfg, torch.cat(pend_xb).to(dev), X, P, Rw, self.block_tables,
                                   self.W_cat, self.base_pool, self.lr_pool, self.status)
            else:
                lrkv.append(self.cfg, X, P, Rw, self.block_tables, self.W_cat, self.base_pool,
                            self.lr_pool, self.status)
            pend_x, pend_xb, pend_p, pend_r, n = [], [], [], [], 0

        for s, a, b in case.setup_appends():
            for lo in range(a, b, self.setup_chunk_tokens):
                hi = min(b, lo + self.setup_chunk_tokens)
                pend_x.append(case.seq_hidden(s, lo, hi))
                if case.rebase:
                    pend_xb.append(case.seq_hidden_neutral(s, lo, hi))
                pend_p.append(torch.arange(lo, hi, dtype=torch.int32))
                pend_r.append(torch.full((hi - lo,), s, dtype=torch.int32))
                n += hi - lo
                if n >= self.setup_chunk_tokens:
                    flush()
        flush()

    def step_append(self) -> None:
        if not self.n_step_tokens:
            return
        if self.case.rebase:  # one launch, base part from the adapter-free states
            lrkv.append_rebase(self.cfg, self.step_Xb, self.step_X, self.step_pos, self.step_rows,
                               self.block_tables, self.W_cat, self.base_pool, self.lr_pool, self.status)
        else:
            lrkv.append(self.cfg, self.step_X, self.step_pos, self.step_rows, self.block_tables,
                        self.W_cat, self.base_pool, self.lr_pool, self.status)

    def decode(self, stream=None) -> Optional[torch.Tensor]:
        if not self.n_dec:
            return None
        return lrkv.attn_decode(self.cfg, self.dec_q, self.dec_q_start, self.dec_adapter,
                                self.dec_bt, self.dec_lens, self.dec_max_len, self.dec_max_q,
                                self.base_pool, self.lr_pool, self.attn_B_K, self.B_V, self.scale,
                                out=self.dec_out, workspace=self.dec_ws, status=self.status,
                                stream=stream)

    def prefill(self, stream=None) -> Optional[torch.Tensor]:
        if not self.n_pre:
            return None
        return lrkv.attn_prefill(self.cfg, self.pre_q, self.pre_q_start, self.pre_max_q,
                                 self.pre_lens, self.pre_max_len, self.pre_adapter, self.pre_bt,
                                 self.base_pool, self.lr_pool, self.attn_B_K, self.B_V, self.scale,
                                 out=self.pre_out, status=self.status, stream=stream)

    def mixed(self, stream=None):
        """The decode and the prefill of this step in one lrkv_attn_mixed call
        (the two parts run concurrently on the GPU)."""
        dec = pre = None
        if self.n_dec:
            dec = {"q": self.dec_q, "ctx_q_start": self.dec_q_start, "adapter_ids": self.dec_adapter,
                   "block_tables": self.dec_bt, "ctx_lens": self.dec_lens, "max_ctx_len": self.dec_max_len,
                   "max_q_per_ctx": self.dec_max_q, "out": self.dec_out, "workspace": self.dec_ws}
        if self.n_pre:
            pre = {"q": self.pre_q, "q_start": self.pre_q_start, "max_q_len": self.pre_max_q,
                   "seq_lens": self.pre_lens, "max_seq_len": self.pre_max_len, "adapter_ids": self.pre_adapter,
                   "block_tables": self.pre_bt, "out": self.pre_out}
        return lrkv.attn_mixed(self.cfg, self.base_pool, self.lr_pool, self.attn_B_K, self.B_V, decode=dec,
                               prefill=pre, scale=self.scale, status=self.status, stream=stream)

    def step(self) -> Dict[str, Optional[torch.Tensor]]:
        """One pass of the hot path: append the new tokens, then attend."""
        self.step_append()
        if self.n_dec and self.n_pre:
            d, p = self.mixed()
            return {"decode": d, "prefill": p}
        return {"decode": self.decode(), "prefill": self.prefill()}

    def device_status(self) -> int:
        return int(self.status.item())
