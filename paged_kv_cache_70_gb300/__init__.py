"""Paged KV-cache attention for one NVIDIA GB300 (sm_103a).

The computation runs in hand-written CUDA kernels behind the C ABI of
``libpagedkv.so`` (``include/pagedkv.h``); this package is its thin Python
binding.  Importing it does not load the library; the first call does, and
raises if the library has not been built.
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    PKV_ERR_NO_SPACE,
    BlockManager,
    paged_copy_blocks,
    LIB_PATH,
    PKV_BF16,
    PKV_F32,
    PKV_FLAG_BAD_BLOCK,
    PKV_FLAG_BAD_LENGTH,
    PKV_FLAG_BAD_SEQ,
    PKV_FLAG_BAD_SLOT,
    PKV_FLAG_TIMEOUT,
    Geom,
    PagedKVError,
    geom_of,
    load_library,
    paged_build_slot_mapping,
    paged_decode,
    paged_decode_append,
    paged_decode_noalloc,
    paged_mixed_step,
    paged_decode_shared_prefix,
    paged_decode_workspace_size,
    paged_error_flags,
    paged_kv_write,
    paged_kv_write_positions,
    paged_varlen_prefill,
    paged_varlen_prefill_workspace_size,
)
