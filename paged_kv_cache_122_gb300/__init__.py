"""GB300-native paged KV-cache decode path: a C-ABI CUDA library and its binding.

The calls follow the pages' statement of the problem:

* ``paged_attention_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, block_size)``
* ``reshape_and_cache(k, v, k_cache, v_cache, slot_mapping)``
* ``copy_blocks(k_cache, v_cache, src_dst_pairs)``

All work runs in the library's sm_103a kernels (``csrc/``); PyTorch supplies
device memory and streams.  ``BlockManager`` is the library's host-side C++
block manager (free list, block tables, copy-on-write) that produces the
slot mapping, copy pairs and tables of a decode step.  Importing the package does not load the library;
the first call does, and fails loudly if it has not been built.
"""
from .api import (  # noqa: F401
    LayerPointers,
    copy_blocks,
    new_workspace,
    paged_attention_decode,
    paged_attention_multi_query,
    pk_paged_attention_multi_query,
    pk_copy_blocks,
    pk_copy_blocks_layers,
    pk_decode_workspace_bytes,
    pk_gather_kv,
    pk_get_device_error,
    pk_paged_attention_decode,
    pk_reshape_and_cache,
    pk_reshape_and_cache_layers,
    pk_selftest_decode_wait_timeout,
    pk_selftest_decode_stale_lengths,
    pk_set_decode_path,
    pk_swap_blocks,
    reshape_and_cache,
    swap_blocks,
)
from ._native import PagedKVError, load as load_library  # noqa: F401
from .block_manager import BlockManager  # noqa: F401
