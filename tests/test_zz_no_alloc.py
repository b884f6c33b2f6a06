"""lrkv_attn_decode_noalloc: decode for callers that cannot allocate device
memory (a runtime whose device memory is reserved once at start-up, or a
serving loop where allocation is forbidden). The entry point uses a fixed
scratch array inside the library instead of a caller workspace; its output must
match lrkv_attn_decode's on the same inputs, call after call, although every
call reuses (and leaves behind) the same scratch contents.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import pytest
import torch

from rank_cache_attention_flash_b300 import inputs as I
from rank_cache_attention_flash_b300 import lrkv
from rank_cache_attention_flash_b300.harness import GpuCase
from tests.parity import BF16_TOL, assert_close

pytestmark = pytest.mark.gpu


def _decode_pair(cuda_lib, g, q):
    """(existing entry point with its own workspace, no-alloc entry point)."""
    ref = cuda_lib.attn_decode(g.cfg, q, g.dec_q_start, g.dec_adapter, g.dec_bt, g.dec_lens,
                               g.dec_max_len, g.dec_max_q, g.base_pool, g.lr_pool, g.B_K, g.B_V,
                               g.scale, status=g.status)
    out = torch.full_like(q, float("nan"))
    cuda_lib.attn_decode_noalloc(g.cfg, q, g.dec_q_start, g.dec_adapter, g.dec_bt, g.dec_lens,
                                 g.dec_max_len, g.dec_max_q, g.base_pool, g.lr_pool, g.B_K, g.B_V,
                                 out, g.scale, status=g.status)
    torch.cuda.synchronize()
    return ref, out


@pytest.mark.parametrize("name", ["shared_decode_llama8b", "long_decode_ministral8b"])
def test_noalloc_matches_workspace_decode_twice(cuda_lib, name):
    case = I.FULL[name]() if name == "shared_decode_llama8b" else I.SMALL[name]()
    g = GpuCase(case)
    g.setup()
    need = lrkv.decode_workspace_bytes(g.cfg, g.n_dec, len(case.dec_ctx), g.dec_max_len, g.dec_max_q)
    assert 0 < need <= lrkv.NOALLOC_SCRATCH_BYTES
    # two calls in a row; the second with other queries, so that the scratch
    # holds the first call's partials when it starts
    for q in (g.dec_q, (-0.5 * g.dec_q.float()).to(g.dec_q.dtype).flip(0).contiguous()):
        ref, out = _decode_pair(cuda_lib, g, q)
        assert g.device_status() == 0
        assert_close(out.double().cpu().numpy(), ref.double().cpu().numpy(), BF16_TOL, name)


def test_noalloc_rejects_sizes_beyond_the_scratch(cuda_lib):
    case = I.SMALL["shared_decode_llama8b"]()
    g = GpuCase(case)
    g.setup()
    # many queries on one long context: split partials beyond the fixed array
    max_len = 8192
    nq = next(n for n in (64, 128, 256, 512, 1024, 2048)
              if lrkv.decode_workspace_bytes(g.cfg, n, 1, max_len, n) > lrkv.NOALLOC_SCRATCH_BYTES)
    dev = g.base_pool.device
    q = torch.zeros(nq, g.cfg.n_q_heads, g.cfg.head_dim, dtype=torch.bfloat16, device=dev)
    out = torch.full_like(q, 7.0)
    starts = torch.tensor([0, nq], dtype=torch.int32, device=dev)
    ads = torch.zeros(nq, dtype=torch.int32, device=dev)
    bt = torch.zeros(1, max_len // 16, dtype=torch.int32, device=dev)
    lens = torch.tensor([max_len], dtype=torch.int32, device=dev)
    with pytest.raises(lrkv.LrkvError) as e:
        cuda_lib.attn_decode_noalloc(g.cfg, q, starts, ads, bt, lens, max_len, nq, g.base_pool,
                                     g.lr_pool, g.B_K, g.B_V, out)
    assert e.value.code == 6  # LRKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # rejected before any launch
