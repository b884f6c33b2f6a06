"""fp64 CPU oracle (test infrastructure only; never on the product path)."""
from .lrkv_oracle import (  # noqa: F401
    BLOCK,
    agent_kv,
    agent_kv_from_cache,
    agent_kv_rebased,
    append_pools,
    apply_rope,
    attend,
    base_and_lowrank,
    decode,
    gqa_attention,
    prefill,
    rebase_pools,
    rope_inv_freq,
    round_bf16,
)
