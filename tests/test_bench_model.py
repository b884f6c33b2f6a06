"""The algorithmic bytes and flops that bench.py divides by its kernel times
(the roofline numerators), pinned to closed forms written out per workload.

Bytes are what a kernel must move at least once: the cached base part (K and V
per token and kv head), the low-rank part (L_K and L_V per token, once for all
kv heads), each context's distinct adapters' B_K and B_V, and the queries in and
the outputs out. Flops count the score and value products over the visible
(query, key) pairs, the K rebuild once per key, and O_lr B_V once per output row
(LRAgent, Abstract: Flash-LoRA-Attention). No GPU needed."""
import pytest

import bench
from rank_cache_attention_flash_b300 import inputs as I


def model(name):
    return bench.workload_model(I.FULL[name]())


def test_shared_decode_bytes_and_flops():
    # one 8192-token context, Hkv 8, d 128, r 16, 4 agents (4 distinct adapters), Hq 32
    L, Hkv, d, r, Hq, agents, g = 8192, 8, 128, 16, 32, 4, 4
    base = L * Hkv * 2 * d * 2                 # K_base and V_base, bf16
    lowrank = L * 2 * r * 2                    # L_K and L_V, bf16, shared by all kv heads
    adapters = agents * 2 * r * Hkv * d * 2    # B_K and B_V of each distinct adapter
    queries = agents * 2 * Hq * d * 2          # q in, out out
    m = model("shared_decode_llama8b")["decode"]
    assert m["bytes"] == base + lowrank + adapters + queries == 34_406_400
    rows = agents * g
    flops = L * Hkv * (agents * 2 * r * d + rows * (4 * d + 2 * r)) + agents * Hq * 2 * r * d
    assert m["flops"] == flops
    assert m["units"] == agents


def test_long_decode_bytes():
    # 16 contexts of 32768 tokens, rank 64, one query (one adapter) per context
    n, L, Hkv, d, r, Hq = 16, 32768, 8, 128, 64, 32
    per_ctx = L * (Hkv * 2 * d * 2 + 2 * r * 2) + 2 * r * Hkv * d * 2 + 2 * Hq * d * 2
    assert model("long_decode_ministral8b")["decode"]["bytes"] == n * per_ctx == 2_286_157_824


def test_compressed_pool_long_decode_bytes():
    # the base part as PolyKV chunks: per 16 tokens and kv head 16 d (int8 keys) +
    # 2 d / 32 * 16 (fp16 scales) + 6 d (3 bit planes) + 64 (fp32 norms) = 23 d + 64 bytes
    n, L, Hkv, d, r, Hq = 16, 32768, 8, 128, 64, 32
    chunk = 16 * d + 16 * (d // 32) * 2 + 16 * 3 * (d // 8) + 16 * 4
    assert chunk == 23 * d + 64
    per_ctx = L * (Hkv * chunk // 16 + 2 * r * 2) + 2 * r * Hkv * d * 2 + 2 * Hq * d * 2
    m = model("long_decode_codec_ministral8b")["decode"]
    assert m["bytes"] == n * per_ctx == 927_203_328
    # same arithmetic as the bf16 pool
    assert m["flops"] == model("long_decode_ministral8b")["decode"]["flops"]


def test_agent_specific_a_reads_each_agents_group():
    # PreLRShared: each of the 4 agents reads its own low-rank group (4 x 2 r columns per token)
    L, Hkv, d, r, Hq, agents = 8192, 8, 128, 16, 32, 4
    nbytes = L * Hkv * 2 * d * 2 + L * 2 * r * agents * 2 + agents * 2 * r * Hkv * d * 2 + agents * 2 * Hq * d * 2
    assert model("prelr_decode_llama8b")["decode"]["bytes"] == nbytes == 35_979_264


@pytest.mark.parametrize("name,chunk_bytes", [("prefill_chunk_llama8b", None),
                                              ("prefill_chunk_codec_llama8b", 23 * 128 + 64)])
def test_prefill_flops_and_bytes(name, chunk_bytes):
    # 4 sequences of a 16384-token prefix + a 512-token chunk, causal (bottom-right)
    seqs, P, n, Hkv, d, r, Hq = 4, 16384, 512, 8, 128, 16, 32
    L = P + n
    visible = n * P + n * (n + 1) // 2
    flops = Hq * visible * (4 * d + 2 * r) + Hkv * L * 2 * r * d + n * Hq * 2 * r * d
    base_tok = Hkv * 2 * d * 2 if chunk_bytes is None else Hkv * chunk_bytes // 16
    nbytes = L * (base_tok + 2 * r * 2) + 2 * n * Hq * d * 2
    m = model(name)["prefill"]
    assert m["flops"] == seqs * flops == 595_743_211_520
    assert m["bytes"] == seqs * nbytes
    assert m["pairs"] == seqs * visible


@pytest.mark.parametrize("name,sources", [("prefill_chunk_llama8b", 1), ("rebase_prefill_llama8b", 2)])
def test_append_flops_and_bytes(name, sources):
    # T = 4 x 512 new tokens through W_cat (N = 2 Hkv d + 2 r columns, h = 4096)
    T, h, Hkv, d, r = 2048, 4096, 8, 128, 16
    N = 2 * Hkv * d + 2 * r
    m = model(name)["append"]
    assert m["flops"] == 2 * T * h * N == 34_896_609_280
    assert m["bytes"] == (sources * T * h + N * h + T * N) * 2  # X (one or two sources), W_cat, pool rows


def test_mixed_batch_append_flops():
    # 48 decode tokens + 16 chunks of 256, h 2048, Hkv 8, d 128, r 8
    T, h, N = 48 + 16 * 256, 2048, 2 * 8 * 128 + 2 * 8
    m = model("mixed_batch_qwen3_1p7b")
    assert m["append"]["flops"] == 2 * T * h * N == 35_033_972_736
    assert m["decode"]["units"] == 48 and m["prefill"]["units"] == 16 * 256
