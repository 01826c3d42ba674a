"""CPU oracle for the paged-KV decode hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product package imports, calls or
links anything under this directory; only the test-suite, the smoke check and
the benchmark's CPU-baseline / reference arm do. It is a plain, slow,
obviously-correct restatement of what the pages say the method computes, in
fp64 for the attention arithmetic and exact integers/bytes for the indexing and
copies. It shares no code with the CUDA path.

Sources, by page title:
  [P1] "PagedAttention 核心创新深度分析" (openeuler.csdn.net)
  [P2] "Visual reading: paged-attention-kv-cache" (blog.vllbc.top)
  [P3] "vLLM 的 PagedAttention：显存管理如何撑起大模型推理" (deepsonar.com.cn)
  [P4] "Infra: PagedAttention" (pufanyi.com)

Every function is pinned by tests under tests/ to values the pages print,
closed forms, special cases and an independent library routine; see the
test files named test_oracle_*.py.
"""
from .paged_attention import (  # noqa: F401
    upcast, slot_mapping, reshape_and_cache, copy_blocks, gather_kv,
    decode_attention, decode_attention_one, decode_step, blocks_needed,
    slots_allocated,
    fragmentation, kv_bytes_per_token, sharing_saving, map_to_kernel_blocks,
    multi_query_attention, e4m3_decode, e4m3_encode, quantize_e4m3, reshape_and_cache_fp8,
    decode_attention_fp8, window_start, skipped_blocks, block_scale_e4m3,
    reshape_and_cache_fp8_block_scaled, decode_attention_fp8_block_scaled,
)
from .block_manager import OracleBlockManager  # noqa: F401
