"""Seeded synthetic workloads for LoRA-KV attention.

This module only draws random numbers and lays out bookkeeping: shapes, block
tables, token positions, sequence ids, query rows. It holds none of the
method's arithmetic (no projection, no rotation, no attention), so both the
CUDA path and the CPU oracle can read its tensors and compute everything on
their own.

Recipe (every workload):
  * each tensor comes from its own CPU ``torch.Generator`` seeded with
    ``seed * 1_000_003 + stream`` where ``stream`` is a fixed id per tensor, so a
    single sequence's hidden states can be regenerated without drawing the rest;
  * values are fp32 normals scaled by the stated standard deviation, then
    rounded once (round-to-nearest-even) to the storage dtype (bf16, or kept
    fp32 for the tiny fp32 workload);
  * integers (block permutation, context lengths, adapter ids) come from their
    own streams.

Sequence model. A sequence is one row of the block table. Its hidden states at
positions [0, prefix_len) come from a shared "prefix stream" (so several
sequences can share those physical blocks), the rest from its own stream.
``ctx_len`` tokens are already in the cache before the timed step (written by an
untimed append), ``new_len`` tokens are appended inside the step. A decode query
sits at position ``ctx_len + new_len - 1``; a prefill chunk's queries are the
``new_len`` new tokens.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

BLOCK = 16  # tokens per paged block

# stream ids (fixed, one per tensor kind)
_S_WK, _S_WV, _S_AK, _S_AV, _S_BK, _S_BV = 3, 4, 5, 6, 7, 8
_S_QDEC, _S_QPRE, _S_PERM, _S_LENS, _S_ADAPT = 9, 10, 11, 12, 13
_S_XSTREAM = 1000  # + stream index
_S_NEUTRAL = 500_000  # added to a hidden-state stream index: its adapter-free twin


def _gen(seed: int, stream: int) -> torch.Generator:
    return torch.Generator().manual_seed(seed * 1_000_003 + stream)


@dataclasses.dataclass(frozen=True)
class Shape:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    rank: int
    n_adapters: int
    rope_base: float
    dtype: str  # "bf16" | "fp32"
    x_std: float
    w_std: float
    a_std: float
    b_std: float
    q_std: float
    lr_groups: int = 1  # 1: one A shared by every agent; n: agent a has its own A (PreLRShared)
    kv_codec: int = 0   # 1: the base pool is compressed (PolyKV codec: q8_0 keys, rotated 3-bit values)

    @property
    def kv_cols(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def n_cols(self) -> int:  # packed projection width: K | V | A_K | A_V
        return 2 * self.kv_cols + 2 * self.lr_groups * self.rank

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


@dataclasses.dataclass
class Seq:
    prefix_stream: int   # stream id for positions [0, prefix_len)
    prefix_len: int
    own_stream: int      # stream id for positions [prefix_len, ctx_len + new_len)
    ctx_len: int         # tokens cached before the step
    new_len: int         # tokens appended during the step
    adapter: int         # adapter id used by this sequence's prefill chunk (-1: base only)
    role: str            # "decode" | "prefill" | "context"

    @property
    def total_len(self) -> int:
        return self.ctx_len + self.new_len


@dataclasses.dataclass
class Case:
    name: str
    shape: Shape
    seed: int
    seqs: List[Seq]
    num_blocks: int
    block_tables: torch.Tensor          # int32 [S, max_blocks], -1 = unused
    # decode: queries sorted by the sequence (context) they read
    dec_ctx: List[int]                  # context (block-table row) per decode context slot
    dec_q_start: torch.Tensor           # int32 [n_dec_ctx + 1]
    dec_adapter: torch.Tensor           # int32 [Nd]
    dec_q: torch.Tensor                 # [Nd, Hq, d] storage dtype
    # prefill: one chunk per listed sequence
    pre_seq: List[int]
    pre_q_start: torch.Tensor           # int32 [P + 1]
    pre_adapter: torch.Tensor           # int32 [P]
    pre_q: torch.Tensor                 # [Np, Hq, d]
    weights: Dict[str, torch.Tensor]    # W_K, W_V [h, Hkv*d]; A_K, A_V [h, r] or [G, h, r]; B_K, B_V [n_adapters, r, Hkv*d]
    rebase: bool = False                # every append re-based: base part from the adapter-free states
    _xcache: Dict[int, torch.Tensor] = dataclasses.field(default_factory=dict)

    # ----- hidden states -------------------------------------------------
    def stream_rows(self, stream: int, n: int) -> torch.Tensor:
        """First ``n`` rows of a hidden-state stream, [n, h] in storage dtype."""
        cached = self._xcache.get(stream)
        if cached is not None and cached.shape[0] >= n:
            return cached[:n]
        g = _gen(self.seed, _S_XSTREAM + stream)
        x = torch.randn(n, self.shape.hidden, generator=g).mul_(self.shape.x_std)
        x = x.to(self.shape.torch_dtype)
        if n * self.shape.hidden <= (1 << 26):  # keep small streams around
            self._xcache[stream] = x
        return x

    def seq_hidden(self, s: int, start: int = 0, stop: Optional[int] = None) -> torch.Tensor:
        """Hidden states of sequence ``s`` at positions [start, stop)."""
        q = self.seqs[s]
        stop = q.total_len if stop is None else stop
        parts = []
        if start < q.prefix_len:
            e = min(stop, q.prefix_len)
            parts.append(self.stream_rows(q.prefix_stream, e)[start:e])
        if stop > q.prefix_len:
            b = max(start, q.prefix_len) - q.prefix_len
            e = stop - q.prefix_len
            parts.append(self.stream_rows(q.own_stream, e)[b:e])
        if not parts:
            return torch.empty(0, self.shape.hidden, dtype=self.shape.torch_dtype)
        return torch.cat(parts, 0) if len(parts) > 1 else parts[0]

    def seq_hidden_neutral(self, s: int, start: int = 0, stop: Optional[int] = None) -> torch.Tensor:
        """Adapter-free hidden states of sequence ``s`` at positions [start, stop):
        the same layout as ``seq_hidden`` drawn from streams of their own (a
        re-based cache takes its base part from these)."""
        q = self.seqs[s]
        shifted = dataclasses.replace(q, prefix_stream=q.prefix_stream + _S_NEUTRAL,
                                      own_stream=q.own_stream + _S_NEUTRAL)
        saved = self.seqs[s]
        self.seqs[s] = shifted
        try:
            return self.seq_hidden(s, start, stop)
        finally:
            self.seqs[s] = saved

    # ----- append plans --------------------------------------------------
    def setup_appends(self):
        """Untimed appends that fill the cache before the step.

        Yields (seq_row, start_pos, stop_pos). A shared prefix is appended once,
        through the first sequence that uses it.
        """
        done_prefix = set()
        for s, q in enumerate(self.seqs):
            lo = 0
            if q.prefix_len > 0:
                if q.prefix_stream in done_prefix:
                    lo = q.prefix_len
                done_prefix.add(q.prefix_stream)
            if q.ctx_len > lo:
                yield s, lo, q.ctx_len

    def step_appends(self):
        """Appends inside the step: the new tokens of every sequence."""
        for s, q in enumerate(self.seqs):
            if q.new_len > 0:
                yield s, q.ctx_len, q.total_len

    def dec_lens(self) -> torch.Tensor:
        return torch.tensor([self.seqs[s].total_len for s in self.dec_ctx], dtype=torch.int32)

    def pre_lens(self) -> torch.Tensor:
        return torch.tensor([self.seqs[s].total_len for s in self.pre_seq], dtype=torch.int32)

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]


# ---------------------------------------------------------------------------
def _weights(shape: Shape, seed: int) -> Dict[str, torch.Tensor]:
    h, kc, r, na = shape.hidden, shape.kv_cols, shape.rank, shape.n_adapters
    dt = shape.torch_dtype

    def draw(stream, size, std):
        return torch.randn(*size, generator=_gen(seed, stream)).mul_(std).to(dt)

    def draw_a(stream):
        # shared A: [h, r]; agent-specific A: [G, h, r], group g from its own stream
        if shape.lr_groups == 1:
            return draw(stream, (h, r), shape.a_std)
        return torch.stack([draw(stream + 100 * g, (h, r), shape.a_std) for g in range(shape.lr_groups)])

    return {
        "W_K": draw(_S_WK, (h, kc), shape.w_std),
        "W_V": draw(_S_WV, (h, kc), shape.w_std),
        "A_K": draw_a(_S_AK),
        "A_V": draw_a(_S_AV),
        "B_K": draw(_S_BK, (na, r, kc), shape.b_std),
        "B_V": draw(_S_BV, (na, r, kc), shape.b_std),
    }


def _tables(seqs: List[Seq], seed: int, permute: bool):
    """Assigns physical blocks. Sequences sharing a prefix stream share its blocks.

    Logical block ids are handed out in sequence order (a shared prefix once, at
    its first user); a seeded permutation then maps them to physical ids.
    """
    layout = []
    seen: Dict[int, int] = {}
    logical = 0
    for q in seqs:
        nb = -(-q.total_len // BLOCK)
        row = []
        shared = 0
        if q.prefix_len > 0:
            assert q.prefix_len % BLOCK == 0
            shared = q.prefix_len // BLOCK
            if q.prefix_stream not in seen:
                seen[q.prefix_stream] = logical
                logical += shared
            st = seen[q.prefix_stream]
            row.extend(range(st, st + shared))
        row.extend(range(logical, logical + nb - shared))
        logical += nb - shared
        layout.append(row)
    total = logical
    ids = torch.arange(total, dtype=torch.int64)
    if permute:
        ids = ids[torch.randperm(total, generator=_gen(seed, _S_PERM))]
    mb = max(1, max(len(r) for r in layout))
    bt = torch.full((len(seqs), mb), -1, dtype=torch.int32)
    for s, row in enumerate(layout):
        if row:
            bt[s, : len(row)] = ids[torch.tensor(row, dtype=torch.int64)].to(torch.int32)
    return bt, total


def _q(shape: Shape, seed: int, stream: int, n: int, skip: int = 0) -> torch.Tensor:
    """Query rows [skip, skip + n) of a query stream (the rows before ``skip``
    belong to the contexts of other shards)."""
    g = _gen(seed, stream)
    x = torch.randn(skip + n, shape.n_q_heads, shape.head_dim, generator=g)[skip:].mul_(shape.q_std)
    return x.to(shape.torch_dtype)


def _build(name, shape, seed, seqs, dec, pre, permute, q_skip=(0, 0)):
    """dec: list of (ctx_row, adapter) sorted by ctx_row; pre: list of seq rows."""
    bt, nblocks = _tables(seqs, seed, permute)
    dec_ctx = []
    starts = [0]
    adapters = []
    for ctx, a in dec:
        if not dec_ctx or dec_ctx[-1] != ctx:
            if dec_ctx:
                starts.append(len(adapters))
            dec_ctx.append(ctx)
        adapters.append(a)
    starts.append(len(adapters))
    if not dec:
        starts = [0]
    pre_start = [0]
    for s in pre:
        pre_start.append(pre_start[-1] + seqs[s].new_len)
    return Case(
        name=name, shape=shape, seed=seed, seqs=seqs, num_blocks=nblocks, block_tables=bt,
        dec_ctx=dec_ctx, dec_q_start=torch.tensor(starts, dtype=torch.int32),
        dec_adapter=torch.tensor(adapters, dtype=torch.int32),
        dec_q=_q(shape, seed, _S_QDEC, len(adapters), q_skip[0]),
        pre_seq=list(pre), pre_q_start=torch.tensor(pre_start, dtype=torch.int32),
        pre_adapter=torch.tensor([seqs[s].adapter for s in pre], dtype=torch.int32),
        pre_q=_q(shape, seed, _S_QPRE, pre_start[-1], q_skip[1]),
        weights=_weights(shape, seed),
    )


# ---------------------------------------------------------------------------
# The five workloads (full size) and their small parity variants.

def shape_tiny_fp32() -> Shape:
    s = 1.0 / math.sqrt(256)
    return Shape(256, 4, 2, 64, 8, 2, 10000.0, "fp32", s, s, s, 1 / math.sqrt(8), 1.0)


def shape_llama8b(rank: int, n_adapters: int) -> Shape:
    w = 1.0 / math.sqrt(4096)
    return Shape(4096, 32, 8, 128, rank, n_adapters, 10000.0, "bf16", 1.0, w, w, 1 / math.sqrt(rank), 1.0)


def shape_qwen3_1p7b() -> Shape:
    w = 1.0 / math.sqrt(2048)
    return Shape(2048, 16, 8, 128, 8, 8, 10000.0, "bf16", 1.0, w, w, 1 / math.sqrt(8), 1.0)


def tiny_fp32_decode(seed: int = 0, n: int = 128, first: int = 0, lr_groups: int = 1) -> Case:
    """Tiny fp32 decode: 2 agents query one shared n-token context.
    ``first``: global index of this shard's context (see ``shard_range``);
    ``lr_groups``: 1 = shared A, n = each agent its own A (PreLRShared)."""
    shape = dataclasses.replace(shape_tiny_fp32(), lr_groups=lr_groups)
    seqs = [Seq(first, 0, first, n, 0, -1, "context")]
    return _build("tiny_fp32_decode", shape, seed, seqs, [(0, 0), (0, 1)], [], False, (2 * first, 0))


def shared_decode(seed: int = 0, n: int = 8192, n_agents: int = 4, rank: int = 16,
                  first: int = 0, lr_groups: int = 1) -> Case:
    """Llama-3.1-8B-shaped decode: n_agents queries on one shared n-token context,
    identity block table. ``first``: global index of this shard's context;
    ``lr_groups``: 1 = shared A, n = each agent its own A (PreLRShared)."""
    shape = dataclasses.replace(shape_llama8b(rank, n_agents), lr_groups=lr_groups)
    seqs = [Seq(first, 0, first, n, 0, -1, "context")]
    dec = [(0, a) for a in range(n_agents)]
    return _build("shared_decode_llama8b", shape, seed, seqs, dec, [], False, (n_agents * first, 0))


def prefill_chunk(seed: int = 0, prefix: int = 16384, chunk: int = 512, n_agents: int = 4,
                  rank: int = 16, first: int = 0, lr_groups: int = 1) -> Case:
    """Each agent appends a new chunk and attends causally over the shared prefix
    plus its own chunk. The prefix blocks are shared physically. ``first``:
    global index of this shard's shared context (its prefix and chunks use
    hidden-state streams of their own)."""
    shape = dataclasses.replace(shape_llama8b(rank, n_agents), lr_groups=lr_groups)
    base = first * (n_agents + 1)
    seqs = [Seq(base, prefix, base + 1 + a, prefix, chunk, a, "prefill") for a in range(n_agents)]
    return _build("prefill_chunk_llama8b", shape, seed, seqs, [], list(range(n_agents)), False,
                  (0, first * n_agents * chunk))


def long_decode(seed: int = 0, n_seqs: int = 16, n: int = 32768, n_agents: int = 8,
                rank: int = 64, first: int = 0, lr_groups: int = 1) -> Case:
    """Ministral-8B-shaped paged decode: independent sequences, adapter ids uniform
    over the agents, blocks placed by a seeded permutation of the pool.
    ``first``: global index of this shard's first sequence."""
    shape = dataclasses.replace(shape_llama8b(rank, n_agents), lr_groups=lr_groups)
    ad = torch.randint(0, n_agents, (first + n_seqs,), generator=_gen(seed, _S_ADAPT))[first:].tolist()
    seqs = [Seq(0, 0, 1 + first + s, n, 0, ad[s], "context") for s in range(n_seqs)]
    dec = [(s, ad[s]) for s in range(n_seqs)]
    return _build("long_decode_ministral8b", shape, seed, seqs, dec, [], True, (first, 0))


def mixed_batch(seed: int = 0, n_seqs: int = 64, n_decode: int = 48, chunk: int = 256,
                lo: int = 1024, hi: int = 16384, n_agents: int = 8, first: int = 0) -> Case:
    """Qwen3-1.7B-shaped mixed serving batch: ``n_decode`` sequences decode one new
    token, the rest prefill a ``chunk``-token chunk; context lengths uniform in
    [lo, hi] (cached before the step); random block tables. ``first``: global
    index of this shard's batch (its sequences are global sequences
    [first * n_seqs, (first + 1) * n_seqs))."""
    shape = shape_qwen3_1p7b()
    g0 = first * n_seqs
    lens = torch.randint(lo, hi + 1, (g0 + n_seqs,), generator=_gen(seed, _S_LENS))[g0:].tolist()
    ad = torch.randint(0, n_agents, (g0 + n_seqs,), generator=_gen(seed, _S_ADAPT))[g0:].tolist()
    seqs = []
    for s in range(n_seqs):
        dec = s < n_decode
        seqs.append(Seq(0, 0, 1 + g0 + s, lens[s], 1 if dec else chunk, ad[s], "decode" if dec else "prefill"))
    dec = [(s, ad[s]) for s in range(n_decode)]
    pre = list(range(n_decode, n_seqs))
    return _build("mixed_batch_qwen3_1p7b", shape, seed, seqs, dec, pre, True,
                  (first * n_decode, first * (n_seqs - n_decode) * chunk))


def prelr_decode(seed: int = 0, n: int = 8192, n_agents: int = 4, rank: int = 16, first: int = 0) -> Case:
    """The shared-context decode with agent-specific A (PReCache, PreLRShared):
    each of the 4 agents reads its own low-rank group of the cache."""
    case = shared_decode(seed, n, n_agents, rank, first, lr_groups=n_agents)
    case.name = "prelr_decode_llama8b"
    return case


def codec_long_decode(seed: int = 0, n_seqs: int = 16, n: int = 32768, n_agents: int = 8,
                      rank: int = 64, first: int = 0) -> Case:
    """The paged long decode over a compressed base pool (PolyKV, the abstract
    printed at the end of the PReCache page: int8 q8_0 keys, Walsh-Hadamard
    rotated 3-bit values); same sequences, adapters and block placement."""
    case = long_decode(seed, n_seqs, n, n_agents, rank, first)
    case.shape = dataclasses.replace(case.shape, kv_codec=1)
    case.name = "long_decode_codec_ministral8b"
    return case


def codec_decode(seed: int = 0, n: int = 700, n_agents: int = 4, rank: int = 16, n_ctx: int = 1,
                 head_dim: int = 128, n_q_heads: int = 32, n_kv_heads: int = 8, q_per_ctx: int = 0) -> Case:
    """Decode over a compressed base pool at small sizes: n_ctx contexts of n
    tokens (the last one shorter: a ragged tail), q_per_ctx queries on each
    (0: n_agents), adapters cycling over the agents with a base-only query when
    there are more than one."""
    shape = dataclasses.replace(shape_llama8b(rank, n_agents), head_dim=head_dim, n_q_heads=n_q_heads,
                                n_kv_heads=n_kv_heads, kv_codec=1)
    q_per_ctx = q_per_ctx or n_agents
    seqs, dec = [], []
    for c in range(n_ctx):
        L = n if c + 1 < n_ctx else max(1, n - 37 * c - 5)
        seqs.append(Seq(c, 0, c, L, 0, -1, "context"))
        for k in range(q_per_ctx):
            a = (c + k) % n_agents
            dec.append((c, -1 if (q_per_ctx > 1 and k == q_per_ctx - 1) else a))
    case = _build("codec_decode", shape, seed, seqs, dec, [], n_ctx > 1, (0, 0))
    return case


def codec_prefill_chunk(seed: int = 0, prefix: int = 16384, chunk: int = 512, n_agents: int = 4,
                        rank: int = 16, first: int = 0) -> Case:
    """The prefill-chunk workload (4 agents x 512 new tokens over a 16384-token
    shared prefix) over a compressed base pool (PolyKV codec)."""
    case = prefill_chunk(seed, prefix, chunk, n_agents, rank, first)
    case.shape = dataclasses.replace(case.shape, kv_codec=1)
    case.name = "prefill_chunk_codec_llama8b"
    return case


def codec_prefill(seed: int = 0, prefix: int = 96, chunk: int = 45, n_agents: int = 3, rank: int = 16,
                  head_dim: int = 128) -> Case:
    """The prefill-chunk workload at small sizes over a compressed base pool
    (PolyKV codec): each agent's chunk over the shared prefix plus its own
    chunk, the prefix blocks shared physically."""
    shape = dataclasses.replace(shape_llama8b(rank, n_agents), head_dim=head_dim, kv_codec=1)
    seqs = [Seq(0, prefix, 1 + a, prefix, chunk, a, "prefill") for a in range(n_agents)]
    return _build("codec_prefill", shape, seed, seqs, [], list(range(n_agents)), False, (0, 0))


def rebase_prefill(seed: int = 0, prefix: int = 16384, chunk: int = 512, n_agents: int = 4,
                   rank: int = 16, first: int = 0) -> Case:
    """The prefill-chunk workload with a re-based cache (PReCache, ReBaseShared):
    every append writes the base part from the adapter-free hidden states and
    the low-rank part from the adapted ones, in one launch."""
    case = prefill_chunk(seed, prefix, chunk, n_agents, rank, first)
    case.name = "rebase_prefill_llama8b"
    case.rebase = True
    return case


def shard_range(n_global: int, world: int, rank: int) -> range:
    """The contiguous share [lo, hi) of ``n_global`` independent contexts that
    rank ``rank`` of ``world`` owns (sizes differ by at most one)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    q, r = divmod(n_global, world)
    lo = rank * q + min(rank, r)
    return range(lo, lo + q + (1 if rank < r else 0))


# Units of independent work per workload (contexts that share nothing but the
# weights): the weak-scaling job on N GPUs holds N times these, and rank k
# builds the share shard_range(N * units, N, k) through the builders' ``first``.
SHARD_UNITS = {
    "tiny_fp32_decode": 1,
    "shared_decode_llama8b": 1,
    "prefill_chunk_llama8b": 1,
    "long_decode_ministral8b": 16,
    "mixed_batch_qwen3_1p7b": 1,
    "prelr_decode_llama8b": 1,
    "rebase_prefill_llama8b": 1,
    "long_decode_codec_ministral8b": 16,
    "prefill_chunk_codec_llama8b": 1,
}


def build_shard(name: str, world: int = 1, rank: int = 0, seed: int = 0) -> Case:
    """Rank ``rank``'s share of the weak-scaling job of ``world`` GPUs."""
    units = SHARD_UNITS[name]
    share = shard_range(world * units, world, rank)
    if len(share) != units:
        raise AssertionError("weak scaling: every rank holds the same number of contexts")
    first = share.start
    return FULL[name](seed, first)


FULL = {
    "tiny_fp32_decode": lambda seed=0, first=0: tiny_fp32_decode(seed, first=first),
    "shared_decode_llama8b": lambda seed=0, first=0: shared_decode(seed, first=first),
    "prefill_chunk_llama8b": lambda seed=0, first=0: prefill_chunk(seed, first=first),
    "long_decode_ministral8b": lambda seed=0, first=0: long_decode(seed, first=first),
    "mixed_batch_qwen3_1p7b": lambda seed=0, first=0: mixed_batch(seed, first=first),
    "prelr_decode_llama8b": lambda seed=0, first=0: prelr_decode(seed, first=first),
    "rebase_prefill_llama8b": lambda seed=0, first=0: rebase_prefill(seed, first=first),
    "long_decode_codec_ministral8b": lambda seed=0, first=0: codec_long_decode(seed, first=first),
    "prefill_chunk_codec_llama8b": lambda seed=0, first=0: codec_prefill_chunk(seed, first=first),
}

# Small variants: same layer shapes, lengths the oracle finishes in seconds,
# several tiles, ragged tails.
SMALL = {
    "tiny_fp32_decode": lambda seed=0: tiny_fp32_decode(seed, n=128),
    "shared_decode_llama8b": lambda seed=0: shared_decode(seed, n=1000),
    "prefill_chunk_llama8b": lambda seed=0: prefill_chunk(seed, prefix=272, chunk=77),
    "long_decode_ministral8b": lambda seed=0: long_decode(seed, n_seqs=3, n=709),
    "mixed_batch_qwen3_1p7b": lambda seed=0: mixed_batch(seed, n_seqs=6, n_decode=4, chunk=45,
                                                          lo=1024, hi=1400),
}
