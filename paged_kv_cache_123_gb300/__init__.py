"""paged_kv_cache_123_gb300 — PagedAttention's decode hot path on GB300.

The KV cache lives in fixed-size blocks anywhere in a physical pool and each
sequence reaches its blocks only through a block table. The work runs in
hand-written CUDA kernels for sm_103a behind the C ABI of libpagedattn.so
(include/pagedattn.h); this package is the thin Python binding (same names
as the C entry points), the host-side block bookkeeping and the seeded input
generators.
"""
from .ops import (  # noqa: F401
    pa_compute_slot_mapping, pa_reshape_and_cache, pa_decode_workspace_bytes,
    pa_decode_partitioning, pa_decode_attention, pa_copy_blocks, pa_get_device_error,
    pa_map_to_kernel_blocks, pa_multi_query_attention, pa_multi_query_workspace_bytes,
    pa_reshape_and_cache_fp8, pa_decode_attention_fp8, pa_decode_window_workspace_bytes,
    pa_decode_attention_window, pa_decode_attention_fp8_window, pa_selftest_bounded_wait,
    pa_decode_window_partitioning, pa_decode_fp8_partitioning, pa_reshape_and_cache_fp8_scaled,
    pa_decode_attention_fp8_scaled, pa_decode_fp8_workspace_bytes, pa_decode_even_ctas,
)
from ._lib import PagedAttnError, LIB_PATH, lib  # noqa: F401
from .block_pool import BlockPool  # noqa: F401
