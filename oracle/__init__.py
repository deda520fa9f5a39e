"""Float64 CPU oracle for paged decode attention, cache writes and block copies.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library in
``paged_kv_cache_122_gb300`` never imports it and shares no code with it; the
two meet only through the seeded inputs of ``paged_kv_cache_122_gb300.workloads``.

Every function states the passage of the source pages it follows.  The pages are:

* "PagedAttention from First Principles" (chrisgmartin)
* "vLLM PagedAttention" (chenyuan1125)
* "vLLM — PagedAttention" (hungchun0201 agentic-AI survey)
* "How vLLM and PagedAttention Actually Work" (binarydose)
* "PagedAttention Explained: How vLLM Pages the KV Cache to Stop Memory Waste" (sevydevy)

Pinned functions (see tests/test_oracle_pins.py): all of them.  None is
"parity unpinned".
"""

from .paged_ref import (  # noqa: F401
    bf16_bits_to_f64,
    num_logical_blocks,
    last_block_fill,
    token_slot,
    gather_sequence,
    softmax_attention,
    paged_decode_attention,
    paged_multi_query_attention,
    partial_attention,
    merge_partials,
    reshape_and_cache,
    copy_blocks,
    swap_blocks,
    kv_bytes_per_token,
    kv_bytes_per_block,
    block_table_bytes,
)
from .block_manager import CowBlockManager  # noqa: F401
