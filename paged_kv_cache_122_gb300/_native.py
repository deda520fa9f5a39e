"""ctypes declarations of the C ABI in ``include/pagedkv.h``.

Loading fails loudly when the compiled library is missing: there is no CPU
fallback for any operation.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_int, c_float, c_size_t, c_void_p, c_uint = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_uint

# name -> (restype, argtypes), in the header's order.
SIGNATURES = {
    "pk_status_string": (ctypes.c_char_p, [c_int]),
    "pk_version": (c_int, []),
    "pk_decode_workspace_bytes": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "pk_paged_attention_decode": (c_int, [
        c_void_p, c_int, c_void_p,             # out, out_dtype, q
        c_void_p, c_void_p,                    # k_cache, v_cache
        c_void_p, c_int,                       # block_tables, max_blocks_per_seq
        c_void_p, c_int,                       # seq_lens, max_seq_len
        c_int, c_int, c_int, c_int,            # num_seqs, num_heads, num_kv_heads, head_dim
        c_int, c_int, c_float,                 # num_blocks, block_size, scale
        c_void_p, c_size_t, c_void_p]),        # workspace, workspace_bytes, stream
    "pk_paged_attention_decode_noalloc": (c_int, [
        c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int,
        c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_void_p]),
    "pk_selftest_decode_wait_timeout": (c_int, [
        c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int,
        c_int, c_int, c_int, c_int, c_int, c_int, c_float,
        c_void_p, c_size_t, c_int, c_uint, c_void_p]),   # workspace, bytes, stall_tile, wait_limit_us, stream
    "pk_selftest_decode_stale_lengths": (c_int, [
        c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int,
        c_int, c_int, c_int, c_int, c_int, c_int, c_float,
        c_void_p, c_void_p, c_size_t, c_void_p]),       # stale_seq_lens, workspace, bytes, stream
    "pk_paged_attention_multi_query": (c_int, [
        c_void_p, c_int, c_void_p, c_int,      # out, out_dtype, q, total_q
        c_void_p, c_int,                       # cu_q_lens, max_q_len
        c_void_p, c_void_p, c_void_p, c_int,   # k_cache, v_cache, block_tables, max_blocks_per_seq
        c_void_p, c_int,                       # seq_lens, max_seq_len
        c_int, c_int, c_int, c_int,            # num_seqs, num_heads, num_kv_heads, head_dim
        c_int, c_int, c_float,                 # num_blocks, block_size, scale
        c_void_p, c_size_t, c_void_p]),        # workspace, workspace_bytes, stream
    "pk_reshape_and_cache": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
        c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "pk_copy_blocks": (c_int, [
        c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "pk_reshape_and_cache_layers": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
        c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "pk_copy_blocks_layers": (c_int, [
        c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "pk_swap_blocks": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "pk_gather_kv": (c_int, [
        c_void_p, c_void_p, c_void_p, c_void_p,
        c_void_p, c_int, c_void_p, c_void_p, c_int,
        c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "pk_get_device_error": (c_int, [ctypes.POINTER(c_uint), c_void_p]),
    "pk_set_decode_path": (c_int, [c_int]),
    # include/pagedkv_block_manager.h
    "pk_bm_create": (c_void_p, [c_int, c_int]),
    "pk_bm_destroy": (None, [c_void_p]),
    "pk_bm_add_sequence": (c_int, [c_void_p, ctypes.c_int64]),
    "pk_bm_append_slots": (c_int, [c_void_p, c_void_p, c_int, c_void_p]),
    "pk_bm_fork": (c_int, [c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]),
    "pk_bm_free_sequence": (c_int, [c_void_p, ctypes.c_int64]),
    "pk_bm_num_pending_copies": (c_int, [c_void_p]),
    "pk_bm_take_copies": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(c_int)]),
    "pk_bm_export": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p]),
    "pk_bm_sequence_info": (c_int, [c_void_p, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(c_int)]),
    "pk_bm_num_free_blocks": (c_int, [c_void_p]),
    "pk_bm_blocks_in_use": (c_int, [c_void_p]),
}

PK_OK = 0
PK_BF16, PK_FP32 = 0, 1
STATUS_NAMES = {
    0: "PK_OK", -1: "PK_ERR_NULL", -2: "PK_ERR_SHAPE", -3: "PK_ERR_UNSUPPORTED",
    -4: "PK_ERR_WORKSPACE", -5: "PK_ERR_CUDA", -6: "PK_ERR_ALIGNMENT", -7: "PK_ERR_NO_DEVICE",
    -8: "PK_ERR_NO_BLOCKS", -9: "PK_ERR_UNKNOWN_SEQUENCE", -10: "PK_ERR_SEQUENCE_EXISTS",
    -11: "PK_ERR_HOST_MEMORY",
}
PK_ERR_NO_BLOCKS, PK_ERR_UNKNOWN_SEQUENCE, PK_ERR_SEQUENCE_EXISTS = -8, -9, -10
DEVERR_BLOCK_ID, DEVERR_SLOT, DEVERR_PAIR, DEVERR_SEQ_LEN, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10
DEVERR_POINTER = 0x20
PATH_AUTO, PATH_CUDA_CORE, PATH_TENSOR_CORE = 0, 1, 2

_lib = None


def library_path() -> str:
    return _build.LIBPATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (once) and declare the library."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise ImportError(
            f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()'); "
            "this package has no CPU fallback")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = load().pk_status_string(status).decode()
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)} ({msg})")


def check(fn: str, status: int) -> None:
    if status != PK_OK:
        raise PagedKVError(fn, status)
