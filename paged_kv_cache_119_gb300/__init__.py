"""paged_kv_cache_119_gb300 -- PagedAttention decode over a paged KV cache on GB300.

A CUDA library (``libpa.so``, C ABI in ``include/pa.h``) with three operations,
each one hand-written sm_103a kernel launch (plus a merge pass for split
contexts), and this thin binding that passes PyTorch tensors to it:

    pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping)
    pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
              num_kv_heads, block_size)
    pa_copy_blocks(k_caches, v_caches, src_dst_pairs)
    pa_chunk_attention(out, q, k_cache, v_cache, block_tables, context_lens,
                       query_start, scale, num_kv_heads, block_size, max_query_len)

``workloads`` builds seeded synthetic inputs.  The binding is imported lazily
so the input generator works on machines without the built library; any call
into the library raises if ``libpa.so`` is missing.
"""
__version__ = "0.1.0"

_API = ("pa_decode", "pa_decode_noalloc", "pa_decode_fp8", "pa_reshape_and_cache",
        "pa_reshape_and_cache_fp8", "pa_copy_blocks", "pa_decode_workspace_bytes",
        "pa_chunk_attention", "pa_chunk_workspace_bytes", "pa_decode_partition_tokens",
        "pa_decode_orders_sequences",
        "pa_chunk_partition_tokens", "pa_swap_blocks", "pa_chunk_attention_fp8",
        "pa_decode_kernel_name", "pa_chunk_kernel_name", "pa_stream_read", "pa_stream_read_runs",
        "pa_get_device_error", "pa_version")

__all__ = list(_API) + ["workloads", "build"]


def __getattr__(name):
    if name in _API:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
