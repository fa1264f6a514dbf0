"""Paged KV attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libpagedattn.so`` (hand-written CUDA,
declared in ``include/pagedattn.h``); this package is its thin Python binding.
Importing the package does not load the library; the first call does, and
fails loudly if the library has not been built.
"""
from ._binding import (  # noqa: F401
    PagedAttnError,
    copy_blocks,
    count_chunk_kv_tokens,
    decode_partition,
    decode_workspace_bytes,
    library_path,
    load_library,
    paged_attention_decode,
    paged_attention_decode_fp8,
    paged_attention_prefill,
    paged_attention_prefill_fp8,
    paged_kv_gather,
    paged_kv_write,
    paged_kv_write_fp8,
    prefill_fp8_workspace_bytes,
    prefill_workspace_bytes,
    selftest_wait_timeout,
    slot_mapping,
    device_error,
)
from .block_manager import BlockManager, BlockManagerError  # noqa: F401,E402
