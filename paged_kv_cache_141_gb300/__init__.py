"""GB300-native paged KV cache: the KV write and the PagedAttention decode
step as hand-written sm_103a CUDA kernels behind a C ABI (include/pagedkv.h).

    from paged_kv_cache_141_gb300 import binding as pagedkv
    pagedkv.reshape_and_cache(key, value, k_cache, v_cache, slot_mapping)
    pagedkv.decode_auto(out, query, k_cache, v_cache, block_tables, context_lens,
                        max_context_len, scale)
"""
