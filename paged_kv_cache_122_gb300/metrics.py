"""Useful-byte accounting of a decode step (the roofline numerator).

Useful bytes are the bytes the step must move at least once:
* attention: every attended token's K and V row of every KV head
  (L_s * Hkv * D * 2 tensors * 2 bytes), plus Q and the output;
* cache write: each new token's K and V read once and written once;
* block copies: each copied block's K and V read once and written once.
Block-table entries, sequence lengths and split-K partials are not counted.
"""
from __future__ import annotations

from typing import Dict

from .workloads import Workload

BF16 = 2


def useful_bytes(w: Workload, out_bytes: int = BF16) -> Dict[str, int]:
    Hkv, D, H, N = w.num_kv_heads, w.head_dim, w.num_heads, w.num_seqs
    tokens = int(w.seq_lens.astype("int64").sum())
    kv = tokens * Hkv * D * 2 * BF16
    q = N * H * D * BF16
    o = N * H * D * out_bytes
    append = w.num_new_tokens * Hkv * D * 2 * BF16 * 2
    copies = int(w.copy_pairs.shape[0]) * w.block_size * Hkv * D * 2 * BF16 * 2
    # Unique K/V bytes: each physical block counted once however many
    # sequences read it (differs from kv only when blocks are shared).
    seen = set()
    unique_tokens = 0
    for s in range(N):
        L = int(w.seq_lens[s])
        nb = -(-L // w.block_size)
        for i in range(nb):
            b = int(w.block_tables[s, i])
            if b not in seen:
                seen.add(b)
                unique_tokens += min(w.block_size, L - i * w.block_size)
    return {
        "attention": kv + q + o,
        "kv": kv,
        "kv_unique": unique_tokens * Hkv * D * 2 * BF16,
        "q_o": q + o,
        "append": append,
        "copies": copies,
        "step": kv + q + o + append + copies,
        "tokens": tokens,
    }
