"""Seeded synthetic decode-step workloads.

This module builds inputs only: sequence lengths, a shuffled physical pool,
block tables, the slots new tokens go to, copy-on-write pairs, and N(0,1)
values rounded to bf16.  It holds none of the attention arithmetic.  The same
objects feed the CUDA library (tests, bench) and the float64 oracle (tests).

One decode step of a workload is, in this order:
  1. copy_blocks(copy_pairs)                  (only the prefix-sharing workload)
  2. reshape_and_cache(k_new, v_new, slot_mapping)
  3. paged_attention_decode(q, caches, block_tables, seq_lens, scale, block_size)
``seq_lens`` are the lengths attended in step 3, i.e. after the appends.

Workloads (sizes are the ones the step is measured on):
  tiny         4 seqs, 8 q / 8 kv heads, d 64, B 16, L ~ U{1..128} before the
               append, pool of 64 blocks, random distinct block ids, +1 token each
  l3-8b        64 seqs, 32 q / 8 kv heads, d 128, B 16, L ~ U{512..2048},
               pool = blocks needed + 10 %, shuffled
  l3-70b       256 seqs, 64 q / 8 kv heads, d 128, B 16,
               L ~ round(lognormal(ln 600, 1)) clipped to [16, 8192] before the
               append, +1 token each, pool = needed + 10 %, shuffled
  long         8 seqs, 32 q / 8 kv heads, d 128, B 16, L ~ U{32768..131072},
               pool = needed + 10 %, shuffled
  prefix-bB    B in {8, 16, 32}: 4 groups x 32 seqs, 32 q / 8 kv heads, d 128;
               each group shares one 1,030-token prefix (its last block holds
               6 tokens); each seq owns p ~ U{0..512} private tokens and appends
               one more.  In the step, the first 31 seqs of a group clone the
               shared partial block (copy-on-write, the 32nd writes in place),
               then every seq writes the tokens that fall inside that block
               (its first private tokens) plus its new token.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seq_lens: np.ndarray                 # int32 [N], attended lengths (after appends)
    block_tables: np.ndarray             # int32 [N, MB], -1 past each sequence's blocks
    slot_mapping: np.ndarray             # int64 [T], slots written in the step
    copy_pairs: np.ndarray               # int64 [n, 2], (src, dst)
    seed: int
    scale: float = field(default=0.0)
    notes: Dict[str, object] = field(default_factory=dict)

    def __post_init__(self):
        if not self.scale:
            self.scale = 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def num_new_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads


def _ceil_div(a, b):
    return -(-a // b)


def _tables(rng, nblocks_per_seq, pool):
    """Assign ``nblocks_per_seq[s]`` ids to each sequence from a shuffled pool."""
    perm = rng.permutation(pool).astype(np.int32)
    MB = max(1, int(max(nblocks_per_seq)))
    bt = np.full((len(nblocks_per_seq), MB), -1, dtype=np.int32)
    k = 0
    for s, nb in enumerate(nblocks_per_seq):
        bt[s, :nb] = perm[k:k + nb]
        k += nb
    return bt


def _append_slots(bt, lens_before, B):
    """Slot of the token at position ``lens_before[s]`` of every sequence."""
    out = np.empty(len(lens_before), dtype=np.int64)
    for s, L in enumerate(lens_before):
        out[s] = int(bt[s, L // B]) * B + L % B
    return out


def _decode_with_append(name, seed, rng, N, H, Hkv, D, B, lens_before, pool=None, spare=0.10):
    lens = lens_before.astype(np.int64) + 1
    nbs = [_ceil_div(int(L), B) for L in lens]
    need = sum(nbs)
    P = pool if pool is not None else int(math.ceil(need * (1.0 + spare)))
    if P < need:
        raise ValueError("pool too small")
    bt = _tables(rng, nbs, P)
    slots = _append_slots(bt, lens_before, B)
    return Workload(name, N, H, Hkv, D, B, P, lens.astype(np.int32), bt, slots,
                    np.zeros((0, 2), dtype=np.int64), seed)


def _decode_no_append(name, seed, rng, N, H, Hkv, D, B, lens, spare=0.10):
    nbs = [_ceil_div(int(L), B) for L in lens]
    P = int(math.ceil(sum(nbs) * (1.0 + spare)))
    bt = _tables(rng, nbs, P)
    return Workload(name, N, H, Hkv, D, B, P, lens.astype(np.int32), bt,
                    np.zeros((0,), dtype=np.int64), np.zeros((0, 2), dtype=np.int64), seed)


def tiny(seed: int = 0) -> Workload:
    rng = np.random.default_rng([seed, 1])
    lens_before = rng.integers(1, 129, size=4)
    return _decode_with_append("tiny", seed, rng, 4, 8, 8, 64, 16, lens_before, pool=64)


def llama3_8b(seed: int = 0) -> Workload:
    rng = np.random.default_rng([seed, 2])
    lens = rng.integers(512, 2049, size=64)
    return _decode_no_append("l3-8b", seed, rng, 64, 32, 8, 128, 16, lens)


def llama3_70b(seed: int = 0) -> Workload:
    rng = np.random.default_rng([seed, 3])
    raw = rng.lognormal(mean=math.log(600.0), sigma=1.0, size=256)
    lens_before = np.clip(np.rint(raw), 16, 8192).astype(np.int64)
    return _decode_with_append("l3-70b", seed, rng, 256, 64, 8, 128, 16, lens_before)


def long_context(seed: int = 0) -> Workload:
    rng = np.random.default_rng([seed, 4])
    lens = rng.integers(32768, 131073, size=8)
    return _decode_no_append("long", seed, rng, 8, 32, 8, 128, 16, lens)


PREFIX_TOKENS = 1030
PREFIX_GROUPS = 4
PREFIX_SEQS_PER_GROUP = 32


def prefix_cow(seed: int = 0, block_size: int = 16) -> Workload:
    B = block_size
    rng = np.random.default_rng([seed, 5, B])
    G_, S_ = PREFIX_GROUPS, PREFIX_SEQS_PER_GROUP
    N = G_ * S_
    private = rng.integers(0, 513, size=N)
    lens = PREFIX_TOKENS + private + 1                      # attended lengths
    nb_shared = _ceil_div(PREFIX_TOKENS, B)
    boundary = nb_shared * B                                # end of the shared partial block
    nbs = [_ceil_div(int(L), B) for L in lens]
    clones = G_ * (S_ - 1)
    need = G_ * nb_shared + clones + sum(nb - nb_shared for nb in nbs)
    P = int(math.ceil(need * 1.10))
    perm = rng.permutation(P).astype(np.int64)
    nxt = 0

    def take(n):
        nonlocal nxt
        ids = perm[nxt:nxt + n]
        nxt += n
        return ids

    MB = max(nbs)
    bt = np.full((N, MB), -1, dtype=np.int32)
    pairs, slots = [], []
    for g in range(G_):
        shared = take(nb_shared)
        for j in range(S_):
            s = g * S_ + j
            bt[s, :nb_shared] = shared
            if j < S_ - 1:                                  # copy-on-write target
                dst = int(take(1)[0])
                pairs.append((int(shared[-1]), dst))
                bt[s, nb_shared - 1] = dst
            bt[s, nb_shared:nbs[s]] = take(nbs[s] - nb_shared)
            L = int(lens[s])
            write_pos = list(range(PREFIX_TOKENS, min(L, boundary)))
            if L - 1 >= boundary:
                write_pos.append(L - 1)
            for pos in write_pos:
                slots.append(int(bt[s, pos // B]) * B + pos % B)
    assert nxt == need
    w = Workload(f"prefix-b{B}", N, 32, 8, 128, B, P, lens.astype(np.int32), bt,
                 np.array(slots, dtype=np.int64), np.array(pairs, dtype=np.int64).reshape(-1, 2), seed)
    w.notes.update(prefix_tokens=PREFIX_TOKENS, groups=G_, seqs_per_group=S_,
                   shared_blocks_per_group=nb_shared)
    return w


def custom(seed: int, lens, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
           spare: float = 0.25, pad: str = "neg1", extra_table_cols: int = 2) -> Workload:
    """A decode batch with given lengths (no appends) for edge-case tests.

    ``pad`` fills the table entries past each sequence's blocks: "neg1" with -1,
    "garbage" with ids far outside the pool (they must never be read).
    """
    rng = np.random.default_rng([seed, 6])
    lens = np.asarray(lens, dtype=np.int64)
    nbs = [_ceil_div(int(L), block_size) for L in lens]
    P = max(1, int(math.ceil(sum(nbs) * (1.0 + spare))))
    bt = _tables(rng, nbs, P)
    bt = np.concatenate([bt, np.full((len(lens), extra_table_cols), -1, dtype=np.int32)], axis=1)
    if pad == "garbage":
        for s, nb in enumerate(nbs):
            bt[s, nb:] = rng.integers(P + 1000, 2 ** 31 - 1, size=bt.shape[1] - nb)
    return Workload(f"custom-g{num_heads // num_kv_heads}-d{head_dim}-b{block_size}", len(lens), num_heads,
                    num_kv_heads, head_dim, block_size, P, lens.astype(np.int32), bt,
                    np.zeros((0,), dtype=np.int64), np.zeros((0, 2), dtype=np.int64), seed)


def get(name: str, seed: int = 0) -> Workload:
    if name == "tiny":
        return tiny(seed)
    if name == "l3-8b":
        return llama3_8b(seed)
    if name == "l3-70b":
        return llama3_70b(seed)
    if name == "long":
        return long_context(seed)
    if name.startswith("prefix-b"):
        return prefix_cow(seed, int(name[len("prefix-b"):]))
    raise KeyError(name)


NAMES = ("tiny", "l3-8b", "l3-70b", "long", "prefix-b8", "prefix-b16", "prefix-b32")


# ---------------------------------------------------------------------------
# Tensor values
# ---------------------------------------------------------------------------

def _randn_bf16(shape, gen: torch.Generator, device, chunk=1 << 26) -> torch.Tensor:
    """N(0,1) float32 draws rounded to bf16 (round-to-nearest-even), chunked."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        flat[i:i + m] = torch.randn(m, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_tensors(w: Workload, device="cpu") -> Dict[str, torch.Tensor]:
    """Materialise a workload's tensors on ``device`` from its seed.

    The K/V pool covers every block, used or not, with N(0,1) values, so a
    read of a wrong block or an unmasked tail changes the result.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.seed) * 1_000_003 + 17)
    N, H, Hkv, D, B, P = w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks
    T = w.num_new_tokens
    t = {
        "q": _randn_bf16((N, H, D), gen, device),
        "k_new": _randn_bf16((T, Hkv, D), gen, device),
        "v_new": _randn_bf16((T, Hkv, D), gen, device),
        "k_cache": _randn_bf16((P, B, Hkv, D), gen, device),
        "v_cache": _randn_bf16((P, B, Hkv, D), gen, device),
        "block_tables": torch.from_numpy(w.block_tables).to(device),
        "seq_lens": torch.from_numpy(w.seq_lens).to(device),
        "slot_mapping": torch.from_numpy(w.slot_mapping).to(device),
        "copy_pairs": torch.from_numpy(w.copy_pairs).to(device),
    }
    return t


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a uint16 numpy array (on the host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
