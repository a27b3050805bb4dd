"""Test infrastructure: the fp64 CPU oracle for the paged KV-cache read.

Only the test suite, the smoke check and the bench's CPU-baseline leg may
import this package.  The product path (the CUDA library and its binding)
never calls it and shares no code with it.
"""

from .paged_attention import (  # noqa: F401
    kv_head_of,
    token_address,
    gather_history,
    attend,
    paged_decode,
    paged_decode_one,
    split_ranges,
    splitkv_partials,
    merge_partials,
    cache_append,
    paged_decode_chunk,
    chunk_splitkv_partials,
)
