"""kvx for GB300 (sm_103a): non-uniform paged KV decode attention and the
coalesced KV gather, as a C-ABI library (libkvx.so) with a thin binding.

    from paged_non_uniform_gb300 import kvx
    plan = kvx.kvx_plan_create(...); kvx.kvx_plan_upload(plan)
    kvx.kvx_decode_attn(plan, q, k_pools, v_pools, ...)
    kvx.kvx_gather_coalesce(block_table, num_blocks, ...)

Importing `kvx` raises ImportError if the library is not built; nothing falls
back to another implementation.
"""
__version__ = "0.1.0"
