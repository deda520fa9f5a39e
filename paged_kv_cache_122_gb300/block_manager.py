"""Python binding of the host block manager (``include/pagedkv_block_manager.h``).

Argument marshalling only: the free list, tables, reference counts and
copy-on-write decisions live in the library's C++ code.  Sequence ids are
Python ints (int64).  Batch calls take and return numpy arrays in the layouts
the decode-step calls consume: int64 slots for ``reshape_and_cache``, int64
``[n, 2]`` pairs for ``copy_blocks``, int32 ``[n, max_blocks]`` tables (-1
padded) and int32 lengths for ``paged_attention_decode``.
"""
from __future__ import annotations

import ctypes
from typing import Iterable, Optional, Tuple

import numpy as np

from ._native import PagedKVError, check, load


def _ids(seq_ids) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64).reshape(-1))
    return a


class BlockManager:
    """Free list, block tables and copy-on-write for one KV-cache pool."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load()
        self._h = self._lib.pk_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError(f"pk_bm_create({num_blocks}, {block_size}) failed")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.pk_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- sequence operations ------------------------------------------------
    def add_sequence(self, seq_id: int) -> None:
        check("pk_bm_add_sequence", self._lib.pk_bm_add_sequence(self._h, int(seq_id)))

    def append_slots(self, seq_ids: Iterable[int]) -> np.ndarray:
        """One more token for each id (in order); returns their flat slots."""
        ids = _ids(seq_ids)
        out = np.empty(ids.shape[0], dtype=np.int64)
        if ids.shape[0]:
            check("pk_bm_append_slots", self._lib.pk_bm_append_slots(
                self._h, ids.ctypes.data, ids.shape[0], out.ctypes.data))
        return out

    def fork(self, parent: int, child: int, num_tokens: Optional[int] = None) -> None:
        n = -1 if num_tokens is None else int(num_tokens)
        check("pk_bm_fork", self._lib.pk_bm_fork(self._h, int(parent), int(child), n))

    def free_sequence(self, seq_id: int) -> None:
        check("pk_bm_free_sequence", self._lib.pk_bm_free_sequence(self._h, int(seq_id)))

    # -- outputs ------------------------------------------------------------
    def take_copies(self) -> np.ndarray:
        """The queued (src, dst) pairs, in decision order, as int64 [k, 2]."""
        k = self._lib.pk_bm_num_pending_copies(self._h)
        out = np.empty((max(k, 0), 2), dtype=np.int64)
        got = ctypes.c_int(0)
        check("pk_bm_take_copies", self._lib.pk_bm_take_copies(
            self._h, out.ctypes.data if k else None, k, ctypes.byref(got)))
        return out[:got.value]

    def export(self, seq_ids: Iterable[int], max_blocks: int,
               tables_out: Optional[np.ndarray] = None,
               lens_out: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
        """Block tables (int32 [n, max_blocks], -1 padded) and lengths (int32 [n]).

        ``tables_out`` / ``lens_out`` may be given (e.g. pinned host tensors'
        numpy views) to be filled in place.
        """
        ids = _ids(seq_ids)
        n = ids.shape[0]
        tables = tables_out if tables_out is not None else np.empty((n, max_blocks), dtype=np.int32)
        lens = lens_out if lens_out is not None else np.empty(n, dtype=np.int32)
        if tables.dtype != np.int32 or tables.shape != (n, max_blocks) or not tables.flags.c_contiguous:
            raise ValueError("tables_out must be a contiguous int32 [n, max_blocks] array")
        if lens.dtype != np.int32 or lens.shape != (n,) or not lens.flags.c_contiguous:
            raise ValueError("lens_out must be a contiguous int32 [n] array")
        if n:
            check("pk_bm_export", self._lib.pk_bm_export(
                self._h, ids.ctypes.data, n, tables.ctypes.data if max_blocks else None, int(max_blocks),
                lens.ctypes.data))
        return tables, lens

    # -- queries ------------------------------------------------------------
    def sequence_info(self, seq_id: int) -> Tuple[int, int]:
        """(length in tokens, number of blocks) of one sequence."""
        length = ctypes.c_int64(0)
        nb = ctypes.c_int(0)
        check("pk_bm_sequence_info", self._lib.pk_bm_sequence_info(
            self._h, int(seq_id), ctypes.byref(length), ctypes.byref(nb)))
        return length.value, nb.value

    def num_free_blocks(self) -> int:
        return int(self._lib.pk_bm_num_free_blocks(self._h))

    def blocks_in_use(self) -> int:
        return int(self._lib.pk_bm_blocks_in_use(self._h))


__all__ = ["BlockManager", "PagedKVError"]
