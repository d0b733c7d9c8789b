"""paged_gqa_decode_pa_gb300: paged grouped-query decode attention for GB300.

The compute lives in libpagedgqa.so (hand-written CUDA for sm_103a, C ABI in
include/pagedgqa.h); this package is its thin ctypes binding.  The library is
loaded on first use and every entry point raises LibraryNotBuilt when it is
missing -- there is no other implementation to fall back to.
"""
from ._binding import (  # noqa: F401
    EXPORTS, LIB_PATH, LibraryNotBuilt, PagedGQAError, alloc_workspace, lib, options,
    pa_cache_append, pa_decode, pa_decode_append, pa_decode_merge, pa_decode_noalloc,
    pa_decode_split, pa_options,
    pa_plan_merge, pa_plan_pieces, pa_launch_plan, pa_read_status, pa_shape, pa_version, pa_workspace_size,
    shape_of, status_string,
    BlockManager, pa_bm_create, pa_bm_destroy, pa_bm_allocate, pa_bm_free_sequence,
    pa_bm_share_prefix, pa_bm_copy_on_write, pa_bm_reserve_slot, pa_bm_block_table, pa_bm_query,
    pa_copy_blocks, pa_decode_multi, pa_workspace_size_multi, alloc_workspace_multi,
    shape_multi, pa_decode_host, pa_workspace_size_host, alloc_workspace_host,
    pa_decode_multi_host, pa_workspace_size_multi_host, alloc_workspace_multi_host,
    bind_decode, bind_decode_multi, bind_decode_append, bind_decode_host, bind_decode_multi_host,
    pa_workspace_size_host_async,
    alloc_workspace_host_async, pa_workspace_size_multi_host_async,
    alloc_workspace_multi_host_async, bind_decode_host_async, bind_decode_multi_host_async,
    PA_MAX_QUERY_TOKENS, PA_MAX_BATCH, PA_STATIC_SCRATCH_BYTES, PA_PHASE_BOTH, PA_PHASE_SPLIT, PA_PHASE_MERGE, PA_ERR_STATE, PA_ERR_NO_BLOCKS, PA_BM_FREE_BLOCKS, PA_BM_REF_COUNT,
    PA_BM_SEQ_BLOCKS,
    PA_OK, PA_ERR_NULL, PA_ERR_SHAPE, PA_ERR_ALIGN, PA_ERR_WORKSPACE, PA_ERR_CUDA,
    PA_ERR_OPTION, PA_ERR_SCRATCH_LIMIT, PA_STATUS_BAD_BLOCK, PA_STATUS_BAD_SEQLEN, PA_STATUS_TIMEOUT,
    PA_STATUS_NO_SLOT, PA_F16, PA_BF16,
)
