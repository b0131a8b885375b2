"""GB300-native sparse KV residency for long-context MLA decode.

The hot path (top-K selection, hot-cache resolve, LRU victims, gather and
bf16 dequant) and the session block store/restore run in the CUDA kernels of ``libkvo.so`` behind the C ABI in
``include/kvo.h``; ``gather_radix_top_gb300.kvo`` is its Python binding.
"""
from .kvo import (Context, KvoError, kvo_append_rows, kvo_create, kvo_debug_dump_layer, kvo_decode_step,  # noqa: F401
                  kvo_debug_evictions, kvo_debug_record_evictions, kvo_destroy, kvo_get_stats,
                  kvo_history_length, kvo_probe_host_read, kvo_resolve_gather, kvo_resolve_gather_multi, kvo_select_topk,
                  kvo_sync, lib, library_path)
from .kvo import (Pool, kvo_pool_alloc, kvo_pool_create, kvo_pool_destroy, kvo_pool_read,  # noqa: F401
                  kvo_pool_release, kvo_pool_write, kvo_restore_blocks, kvo_store_blocks, kvo_tier_blocks)
