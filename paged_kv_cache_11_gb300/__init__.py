"""paged_kv_cache_11_gb300 -- the decode hot path of a paged KV cache on one
GB300 GPU (sm_103a): block write, paged decode attention (GQA grouping, split-K
with a log-sum-exp merge, shared-prefix groups read once) and the
copy-on-write block copy, as hand-written
CUDA behind the C ABI in ``include/pagedkv.h``.

``binding`` exposes the C ABI calls by the same names; ``block_manager`` is the
host-side fork/append/free bookkeeping that produces block tables, slot
mappings and copy-on-write pairs; ``workload`` builds seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    PKV_BF16, PKV_FP16, PKV_FP32, CacheDesc, PagedKVError, cache_desc, check_device_error, compact_tokens, copy_blocks,
    launch_count, paged_attention_append_decode, paged_attention_append_decode_grouped, paged_attention_decode,
    paged_attention_decode_grouped,
    paged_attention_decode_static, paged_attention_grouped_workspace_bytes, paged_attention_partition_size,
    paged_attention_plan, paged_attention_workspace_bytes, paged_kv_append, status_string, swap_blocks, version,
    wait_selftest,
)
from .block_manager import BlockManager, OutOfBlocks  # noqa: F401
