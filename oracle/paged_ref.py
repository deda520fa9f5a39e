"""Plain float64 restatement of what the paged decode path computes.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product library never
imports this module.

Conventions shared with the pages and fixed here:

* Caches are ``[num_blocks, block_size, num_kv_heads, head_dim]`` arrays of raw
  bf16 bit patterns (``uint16``).  This is the layout of the conceptual kernel
  signature in "vLLM — PagedAttention", section "Fused CUDA Kernels", and of the
  prose in "PagedAttention from First Principles" §7 ("all 16 tokens of a block
  live side-by-side, all heads of one token live side-by-side, all elements of
  one head live side-by-side").
* bf16 values enter the arithmetic by exact widening to float64; nothing is
  rounded on the way in.
* Query head ``h`` reads KV head ``h // G`` with ``G = num_heads // num_kv_heads``
  (contiguous groups; the pages only say that several query heads share one KV
  head: "PagedAttention Explained", section on bytes per token).
"""

from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np


# ----------------------------------------------------------------------------
# bf16 bit patterns
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns as float64.

    A bf16 number is the upper half of an IEEE binary32 number, so shifting the
    16 bits into the top of a 32-bit word gives the float32 with the same value,
    and float32 -> float64 is exact.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Block arithmetic
# ----------------------------------------------------------------------------

def num_logical_blocks(seq_len: int, block_size: int) -> int:
    """Number of blocks a sequence of ``seq_len`` tokens occupies.

    "PagedAttention from First Principles" §5, pseudocode: the number of blocks
    is the ceiling of context_len / BLOCK_SIZE.  "PagedAttention Explained",
    blocks section: a 900-token chat holds 57 blocks of 16.
    """
    if seq_len < 0 or block_size <= 0:
        raise ValueError("seq_len must be >= 0 and block_size > 0")
    return -(-seq_len // block_size)


def last_block_fill(seq_len: int, block_size: int) -> int:
    """Tokens held by the last block (0 for an empty sequence).

    "PagedAttention from First Principles" §5, tail handling: the last block
    holds min(B, L - i*B) valid tokens.
    """
    n = num_logical_blocks(seq_len, block_size)
    if n == 0:
        return 0
    return seq_len - (n - 1) * block_size


def token_slot(block_table_row: Sequence[int], pos: int, block_size: int) -> int:
    """Flat physical slot ``phys * B + pos % B`` of logical token ``pos``.

    "PagedAttention from First Principles" §5: every block read goes through
    ``block_table[i]``; logical block ``i = pos // B`` lives at physical block
    ``block_table[i]``, and the token sits at offset ``pos % B`` inside it.
    """
    phys = int(block_table_row[pos // block_size])
    return phys * block_size + pos % block_size


def gather_sequence(cache_bits: np.ndarray, block_table_row: Sequence[int],
                    seq_len: int, block_size: int, kv_head: int) -> np.ndarray:
    """Raw bits ``[seq_len, head_dim]`` of one KV head of one sequence.

    "PagedAttention from First Principles" §5: for logical block ``i`` the
    kernel reads ``k_cache[block_table[i]]`` and keeps its first ``valid``
    tokens.  Table entries at or beyond ``ceil(L/B)`` are never read (§6: the
    sentinel in unused slots is never dereferenced).
    """
    num_blocks = cache_bits.shape[0]
    pos = np.arange(seq_len, dtype=np.int64)
    row = np.asarray(block_table_row, dtype=np.int64)
    nb = num_logical_blocks(seq_len, block_size)
    if nb > row.shape[0]:
        raise ValueError("block table row shorter than ceil(seq_len / block_size)")
    used = row[:nb]
    if nb and (used.min() < 0 or used.max() >= num_blocks):
        raise ValueError("block table names a physical block outside the pool")
    phys = row[pos // block_size]
    off = pos % block_size
    return cache_bits[phys, off, kv_head, :]


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Textbook single-query attention, float64.

    "How vLLM and PagedAttention Actually Work" §5: softmax(Q K^T / sqrt(d_k)) V,
    with the scale passed in.  ``q`` is ``[G, D]`` (the query heads that share
    this K/V), ``K`` and ``V`` are ``[L, D]``.  Returns ``(o [G, D], lse [G])``
    where ``lse`` is the natural log of the softmax denominator including the
    max shift, i.e. ``log(sum_j exp(z_j))``.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    z = scale * (q @ K.T)                       # [G, L] scores
    m = z.max(axis=1, keepdims=True)            # max shift: exact, avoids overflow
    e = np.exp(z - m)
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom                               # attention weights
    o = p @ V
    lse = (m + np.log(denom))[:, 0]
    return o, lse


def paged_decode_attention(q_bits: np.ndarray, k_cache_bits: np.ndarray,
                           v_cache_bits: np.ndarray, block_tables: np.ndarray,
                           seq_lens: Sequence[int], scale: float, block_size: int,
                           seqs: Iterable[int] | None = None) -> np.ndarray:
    """Decode attention through block tables; ``out [N, H, D]`` float64.

    "vLLM — PagedAttention", Mathematical Formulation (Equation 4): the
    attention of query ``i`` over key blocks ``K_j`` fetched through the block
    table is the same softmax as over the contiguous keys; "PagedAttention from
    First Principles" §18: the math of attention is unchanged by paging.  So the
    oracle gathers each sequence through its table and runs textbook attention,
    with no online softmax and no splitting.

    A sequence of length 0 yields zeros (the pages are silent; this is the
    reading adopted for an empty context).  ``seqs`` restricts the work to some
    sequences (the rest of ``out`` stays zero); it is used for sampled checks.
    """
    N, H, D = q_bits.shape
    Hkv = k_cache_bits.shape[2]
    if H % Hkv:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    G = H // Hkv
    out = np.zeros((N, H, D), dtype=np.float64)
    for s in (range(N) if seqs is None else seqs):
        L = int(seq_lens[s])
        if L == 0:
            continue
        for kvh in range(Hkv):
            K = bf16_bits_to_f64(gather_sequence(k_cache_bits, block_tables[s], L, block_size, kvh))
            V = bf16_bits_to_f64(gather_sequence(v_cache_bits, block_tables[s], L, block_size, kvh))
            q = bf16_bits_to_f64(q_bits[s, kvh * G:(kvh + 1) * G, :])
            o, _ = softmax_attention(q, K, V, scale)
            out[s, kvh * G:(kvh + 1) * G, :] = o
    return out


def paged_multi_query_attention(q_bits: np.ndarray, k_cache_bits: np.ndarray,
                                v_cache_bits: np.ndarray, block_tables: np.ndarray,
                                seq_lens: Sequence[int], cu_q_lens: Sequence[int], scale: float,
                                block_size: int, seqs: Iterable[int] | None = None) -> np.ndarray:
    """Several new query tokens per sequence over the paged cache, causal
    among them; ``out [total_q, H, D]`` float64.

    "PagedAttention from First Principles" §12 (chunked prefill: a chunk of a
    prompt is processed over the cache in one pass) and §14 (speculative
    decoding: the verifier checks several appended tokens in one forward
    pass over the paged cache).  Sequence ``s`` owns query rows
    ``cu_q_lens[s] .. cu_q_lens[s+1]-1``: its ``q_s`` newest tokens, already
    appended, so its context has ``L = seq_lens[s]`` tokens and query ``r``
    sits at position ``L - q_s + r``.  Causal reading (the plainest one the
    pages support: a token never sees tokens after it): query ``r`` attends
    keys ``0 .. L - q_s + r``.  Everything else is the decode definition.
    """
    Tq, H, D = q_bits.shape
    Hkv = k_cache_bits.shape[2]
    if H % Hkv:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    G = H // Hkv
    N = len(seq_lens)
    if len(cu_q_lens) != N + 1 or cu_q_lens[0] != 0 or cu_q_lens[N] != Tq:
        raise ValueError("cu_q_lens must be [0, ..., total_q] with one entry per sequence plus one")
    out = np.zeros((Tq, H, D), dtype=np.float64)
    for s in (range(N) if seqs is None else seqs):
        L = int(seq_lens[s])
        q0, q1 = int(cu_q_lens[s]), int(cu_q_lens[s + 1])
        qs = q1 - q0
        if qs < 0 or qs > L:
            raise ValueError("a sequence has more queries than context tokens")
        if qs == 0:
            continue
        for kvh in range(Hkv):
            K = bf16_bits_to_f64(gather_sequence(k_cache_bits, block_tables[s], L, block_size, kvh))
            V = bf16_bits_to_f64(gather_sequence(v_cache_bits, block_tables[s], L, block_size, kvh))
            for r in range(qs):
                last = L - qs + r            # the query's own position
                q = bf16_bits_to_f64(q_bits[q0 + r, kvh * G:(kvh + 1) * G, :])
                o, _ = softmax_attention(q, K[:last + 1], V[:last + 1], scale)
                out[q0 + r, kvh * G:(kvh + 1) * G, :] = o
    return out


def partial_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Attention restricted to a contiguous token range: ``(lse [G], o [G, D])``.

    "PagedAttention from First Principles" §17: the partitioned kernel computes
    partial softmax results over parts of one sequence and a reduce step
    combines them.  A part's result is the plain definition applied to its own
    tokens: its normalised output and the log of its softmax denominator.
    An empty range has ``lse = -inf`` and ``o = 0``.
    """
    G, D = np.asarray(q).shape
    if np.asarray(K).shape[0] == 0:
        return np.full(G, -np.inf), np.zeros((G, D))
    o, lse = softmax_attention(q, K, V, scale)
    return lse, o


def merge_partials(lses: Sequence[np.ndarray], outs: Sequence[np.ndarray]):
    """Combine part results into the result over the union of the parts.

    Each part's softmax denominator is ``exp(lse_p)``; the union's denominator
    is their sum and the union's output is the denominator-weighted mean of the
    part outputs.  This is the reduce step named in "PagedAttention from First
    Principles" §17, written from the definition of softmax.
    """
    lse = np.stack([np.asarray(x, dtype=np.float64) for x in lses])      # [P, G]
    o = np.stack([np.asarray(x, dtype=np.float64) for x in outs])        # [P, G, D]
    M = lse.max(axis=0)                                                   # [G]
    safe_M = np.where(np.isfinite(M), M, 0.0)
    w = np.exp(lse - safe_M)                                              # [P, G]
    tot = w.sum(axis=0)
    merged = np.einsum('pg,pgd->gd', w, o) / np.where(tot > 0, tot, 1.0)[:, None]
    with np.errstate(divide='ignore'):
        merged_lse = safe_M + np.log(tot)
    return merged_lse, merged


# ----------------------------------------------------------------------------
# Cache writes and block copies (bitwise)
# ----------------------------------------------------------------------------

def reshape_and_cache(k_bits: np.ndarray, v_bits: np.ndarray, k_cache_bits: np.ndarray,
                      v_cache_bits: np.ndarray, slot_mapping: Sequence[int], block_size: int):
    """Return copies of the caches with each new token written to its slot.

    "vLLM — PagedAttention", Fused CUDA Kernels (1): new K/V are saved at the
    positions the block table specifies; "PagedAttention from First Principles"
    §2: the cache is append-only, one new K and V per token and layer.  Token
    ``t`` with flat slot ``s = slot_mapping[t]`` goes to
    ``cache[s // B, s % B, :, :]``.  A negative slot marks a padding token and
    writes nothing.  Tokens are applied in order, so a repeated slot keeps the
    last writer.
    """
    kc = np.array(k_cache_bits, copy=True)
    vc = np.array(v_cache_bits, copy=True)
    P = kc.shape[0]
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        if blk >= P:
            raise ValueError("slot outside the pool")
        kc[blk, off] = k_bits[t]
        vc[blk, off] = v_bits[t]
    return kc, vc


def copy_blocks(k_cache_bits: np.ndarray, v_cache_bits: np.ndarray,
                pairs: Sequence[Sequence[int]]):
    """Return copies of the caches with ``cache[dst] = cache[src]`` per pair.

    "vLLM — PagedAttention", Copy-on-Write Logic and Fused CUDA Kernels (3): a
    shared block is copied to a fresh physical block before a sequence writes
    into it, and all pending copies of a step go into one launch.  Every pair
    reads the caches as they were before the call (the pairs of one step never
    write a block another pair reads).
    """
    kc = np.array(k_cache_bits, copy=True)
    vc = np.array(v_cache_bits, copy=True)
    P = kc.shape[0]
    for src, dst in pairs:
        src, dst = int(src), int(dst)
        if not (0 <= src < P and 0 <= dst < P):
            raise ValueError("block id outside the pool")
        kc[dst] = k_cache_bits[src]
        vc[dst] = v_cache_bits[src]
    return kc, vc


def swap_blocks(src_k_bits: np.ndarray, src_v_bits: np.ndarray, dst_k_bits: np.ndarray,
                dst_v_bits: np.ndarray, pairs: Sequence[Sequence[int]]):
    """Return copies of the destination pool with ``dst[d] = src[s]`` per pair.

    "PagedAttention from First Principles" §15 (KV-cache offloading): a block
    that is swapped out is copied to host RAM and its HBM slot freed; swapping
    in copies it back.  "PagedAttention Explained" (preemption): swapping
    copies all of an evicted request's blocks, in both directions.  The two
    pools may have different sizes; block contents move unchanged.
    """
    kd = np.array(dst_k_bits, copy=True)
    vd = np.array(dst_v_bits, copy=True)
    for src, dst in pairs:
        src, dst = int(src), int(dst)
        if not (0 <= src < src_k_bits.shape[0] and 0 <= dst < kd.shape[0]):
            raise ValueError("block id outside its pool")
        kd[dst] = src_k_bits[src]
        vd[dst] = src_v_bits[src]
    return kd, vd


# ----------------------------------------------------------------------------
# Byte counts
# ----------------------------------------------------------------------------

def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                       dtype_bytes: int) -> int:
    """K and V bytes one token occupies across all layers.

    "PagedAttention from First Principles" §1 and "How vLLM and PagedAttention
    Actually Work" §2: 2 (K and V) x layers x KV heads x head dim x bytes.
    """
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes


def kv_bytes_per_block(block_size: int, num_kv_heads: int, head_dim: int,
                       dtype_bytes: int, num_layers: int = 1) -> int:
    """Bytes of one physical block (K and V) for ``num_layers`` layers.

    "PagedAttention from First Principles" §6: block_size x KV heads x head dim
    x 2 (K+V) x bytes, per layer.
    """
    return block_size * kv_bytes_per_token(num_layers, num_kv_heads, head_dim, dtype_bytes)


def block_table_bytes(num_seqs: int, max_model_len: int, block_size: int,
                      entry_bytes: int = 4) -> int:
    """Bytes of an int32 block-table tensor ``[N, ceil(max_len / B)]``.

    "PagedAttention from First Principles" §6, the block table byte by byte.
    """
    return num_seqs * num_logical_blocks(max_model_len, block_size) * entry_bytes


def logsumexp(z: Iterable[float]) -> float:
    """log(sum(exp(z))) computed with a max shift; used by tests only."""
    z = list(z)
    if not z:
        return -math.inf
    m = max(z)
    return m + math.log(math.fsum(math.exp(x - m) for x in z))
