"""GB300-native paged KV-cache hot path: slot mapping (paged and range), KV
write (alone or fused with the slot mapping), block-table gather and
kernel-block expansion, as hand-written CUDA kernels for sm_103a behind the C
ABI of ``include/kvpaged.h``.

The Python layer only marshals tensors into that ABI (``ops``); the seeded
synthetic workloads live in ``workloads``.
"""
from ._lib import (ERR_BITS, KV_EINVAL, KV_EUNSUPPORTED, KV_ECUDA, KV_OK, KVError,
                   MAX_GATHER_REQS, MAX_RANGES_PER_REQ, MAX_TOKENS, NULL_BLOCK_ID, PAD_SLOT_ID,
                   load)
from .ops import (Prepared, kv_cache_gather, kv_cache_gather_range, kv_cache_write, kv_copy_blocks,
                  kv_expand_kernel_blocks, kv_slot_mapping_paged, kv_slot_mapping_paged_cp,
                  kv_slot_mapping_paged_write, kv_slot_mapping_range,
                  kv_slot_mapping_range_write, kv_table_from_ranges, new_error_word)

__all__ = [
    "ERR_BITS", "KV_EINVAL", "KV_EUNSUPPORTED", "KV_ECUDA", "KV_OK", "KVError",
    "MAX_GATHER_REQS", "MAX_RANGES_PER_REQ", "MAX_TOKENS", "NULL_BLOCK_ID", "PAD_SLOT_ID", "load",
    "kv_cache_gather", "kv_cache_write", "kv_expand_kernel_blocks", "kv_slot_mapping_paged",
    "kv_slot_mapping_range", "new_error_word", "kv_table_from_ranges", "kv_cache_gather_range",
    "kv_copy_blocks", "kv_slot_mapping_paged_cp", "kv_slot_mapping_paged_write",
    "kv_slot_mapping_range_write", "Prepared",
]
