"""paged_gqa_decode_kv_gb300 -- paged GQA decode attention and KV append for
GB300 (sm_103a), behind the C ABI declared in include/pgd.h.

The compute path runs only in the CUDA library ``libpgd.so``; this package is
argument marshalling over it.  Importing the package does not load the
library; the first call does, and fails loudly if it was not built.
"""
from .inputs import (WORKLOADS, Workload, PagedBatch, make_batch, make_workload,  # noqa: F401
                     tile_pool, untile_pool, pool_shape, pack_pool8, unpack_pool8, pool_shape8)
from ._native import (  # noqa: F401
    PGDError, BlockAllocator, kv_append, paged_decode_attention,
    paged_decode_attention_noalloc, append_decode_attention, decode_step, copy_blocks,
    kv_append_fp8, paged_decode_attention_fp8, append_decode_attention_fp8,
    cascade_decode_attention, cascade_workspace_size, kv_append_tokens, paged_verify_attention,
    append_verify_attention, verify_step, verify_workspace_size, mla_append, mla_decode_attention,
    mla_append_decode_attention, mla_step, mla_workspace_size, device_errors,
    workspace_size, make_workspace, attention_grid, validate_tables, read_stream, set_wait_limit_ns,
    wait_limit_ns, set_short_context_tokens, uses_short_path, PreparedCall, prepare, lib,
    library_path)

__all__ = ["WORKLOADS", "Workload", "PagedBatch", "make_batch", "make_workload", "tile_pool",
           "untile_pool", "pool_shape", "pack_pool8", "unpack_pool8", "pool_shape8", "PGDError",
           "BlockAllocator", "kv_append", "paged_decode_attention",
           "paged_decode_attention_noalloc", "append_decode_attention", "decode_step",
           "copy_blocks", "kv_append_fp8", "paged_decode_attention_fp8",
           "append_decode_attention_fp8", "cascade_decode_attention", "cascade_workspace_size",
           "kv_append_tokens", "paged_verify_attention", "append_verify_attention",
           "verify_step", "verify_workspace_size",
           "mla_append", "mla_decode_attention", "mla_append_decode_attention", "mla_step",
           "mla_workspace_size",
           "device_errors", "workspace_size", "make_workspace", "attention_grid",
           "validate_tables", "read_stream", "set_wait_limit_ns", "wait_limit_ns",
           "set_short_context_tokens", "uses_short_path", "PreparedCall", "prepare", "lib",
           "library_path"]
