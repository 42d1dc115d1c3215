"""paged_kv_cache_11_gb300 -- the decode hot path of a paged KV cache on one
GB300 GPU (sm_103a).  ``block_manager`` is the host-side fork/append/free
bookkeeping; ``workload`` builds seeded synthetic inputs."""
from .block_manager import BlockManager, OutOfBlocks  # noqa: F401
