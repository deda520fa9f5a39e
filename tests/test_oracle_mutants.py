"""The pins must catch plausible mistakes in the oracle.

Each case below plants one mistake in one oracle function (a small edit of its
source, compiled afresh and patched into the module for the duration of the
case) and runs every pin of ``test_oracle_pins``; at least one pin has to fail.
The unmodified oracle passes all of them.  CPU only; nothing here touches the
CUDA path.

Edits that cannot change a result on valid input are left out: for instance a
block copy that reads the partly updated pool instead of the pool as it was
differs only when one pair's source is another pair's destination, which the
operation's contract excludes.
"""
import __future__
import inspect
import textwrap

import numpy as np
import pytest

import oracle
from oracle import block_manager as bm_mod
from oracle import paged_ref as ref

import test_oracle_pins as pins

# (name, owner, function, [(old, new), ...]): each ``old`` must occur exactly
# once in the function's source.
MUTANTS = [
    # bf16 and block arithmetic
    ("bf16_shift_15", ref, "bf16_bits_to_f64", [("<< np.uint32(16)", "<< np.uint32(15)")]),
    ("blocks_floor", ref, "num_logical_blocks", [("-(-seq_len // block_size)", "seq_len // block_size")]),
    ("last_fill_mod", ref, "last_block_fill", [("seq_len - (n - 1) * block_size", "seq_len % block_size")]),
    ("slot_offset_from_block", ref, "token_slot",
     [("phys * block_size + pos % block_size", "phys * block_size + pos // block_size")]),
    # the table walk
    ("gather_offset_reversed", ref, "gather_sequence",
     [("off = pos % block_size", "off = block_size - 1 - pos % block_size")]),
    ("gather_ignores_kv_head", ref, "gather_sequence",
     [("cache_bits[phys, off, kv_head, :]", "cache_bits[phys, off, 0, :]")]),
    ("gather_unmasked_tail", ref, "gather_sequence",
     [("pos = np.arange(seq_len, dtype=np.int64)",
       "pos = np.arange(num_logical_blocks(seq_len, block_size) * block_size, dtype=np.int64)")]),
    ("gather_sentinel_unchecked", ref, "gather_sequence",
     [("if nb and (used.min() < 0 or used.max() >= num_blocks):", "if False:")]),
    # the softmax
    ("softmax_dropped_scale", ref, "softmax_attention", [("z = scale * (q @ K.T)", "z = q @ K.T")]),
    ("softmax_sign", ref, "softmax_attention", [("z = scale * (q @ K.T)", "z = -scale * (q @ K.T)")]),
    ("softmax_k_v_swapped", ref, "softmax_attention",
     [("z = scale * (q @ K.T)", "z = scale * (q @ V.T)"), ("o = p @ V", "o = p @ K")]),
    ("softmax_wrong_axis", ref, "softmax_attention",
     [("denom = e.sum(axis=1, keepdims=True)", "denom = e.sum(axis=0, keepdims=True)")]),
    ("softmax_unnormalised", ref, "softmax_attention", [("p = e / denom", "p = e")]),
    ("lse_without_max", ref, "softmax_attention",
     [("lse = (m + np.log(denom))[:, 0]", "lse = np.log(denom)[:, 0]")]),
    # decode through block tables
    ("gqa_interleaved", ref, "paged_decode_attention",
     [("q_bits[s, kvh * G:(kvh + 1) * G, :]", "q_bits[s, kvh::Hkv, :]"),
      ("out[s, kvh * G:(kvh + 1) * G, :] = o", "out[s, kvh::Hkv, :] = o")]),
    ("decode_context_short_by_one", ref, "paged_decode_attention",
     [("L = int(seq_lens[s])", "L = int(seq_lens[s]) - 1")]),
    ("decode_v_from_k_cache", ref, "paged_decode_attention",
     [("V = bf16_bits_to_f64(gather_sequence(v_cache_bits,", "V = bf16_bits_to_f64(gather_sequence(k_cache_bits,")]),
    # several queries per sequence
    ("causal_off_by_one", ref, "paged_multi_query_attention",
     [("last = L - qs + r ", "last = L - qs + r - 1 ")]),
    ("not_causal", ref, "paged_multi_query_attention", [("last = L - qs + r ", "last = L - 1 ")]),
    ("positions_from_chunk_start", ref, "paged_multi_query_attention", [("last = L - qs + r ", "last = r ")]),
    ("mq_gqa_interleaved", ref, "paged_multi_query_attention",
     [("q_bits[q0 + r, kvh * G:(kvh + 1) * G, :]", "q_bits[q0 + r, kvh::Hkv, :]"),
      ("out[q0 + r, kvh * G:(kvh + 1) * G, :] = o", "out[q0 + r, kvh::Hkv, :] = o")]),
    # partial results and their merge
    ("partial_empty_lse_zero", ref, "partial_attention",
     [("return np.full(G, -np.inf), np.zeros((G, D))", "return np.zeros(G), np.zeros((G, D))")]),
    ("merge_equal_weights", ref, "merge_partials", [("w = np.exp(lse - safe_M)", "w = np.ones_like(lse)")]),
    ("merge_unnormalised", ref, "merge_partials",
     [("merged = np.einsum('pg,pgd->gd', w, o) / np.where(tot > 0, tot, 1.0)[:, None]",
       "merged = np.einsum('pg,pgd->gd', w, o)")]),
    ("merge_lse_is_max", ref, "merge_partials", [("merged_lse = safe_M + np.log(tot)", "merged_lse = safe_M")]),
    # cache writes and block copies
    ("append_negative_slot_written", ref, "reshape_and_cache",
     [("if slot < 0:\n            continue", "if slot < -(10 ** 9):\n            continue")]),
    ("append_slot_split_swapped", ref, "reshape_and_cache",
     [("blk, off = divmod(slot, block_size)", "off, blk = divmod(slot, block_size)")]),
    ("append_k_into_v", ref, "reshape_and_cache", [("vc[blk, off] = v_bits[t]", "vc[blk, off] = k_bits[t]")]),
    ("copy_direction_reversed", ref, "copy_blocks",
     [("kc[dst] = k_cache_bits[src]", "kc[src] = k_cache_bits[dst]"),
      ("vc[dst] = v_cache_bits[src]", "vc[src] = v_cache_bits[dst]")]),
    ("copy_skips_v", ref, "copy_blocks", [("vc[dst] = v_cache_bits[src]", "vc[dst] = v_cache_bits[dst]")]),
    ("swap_reads_destination_pool", ref, "swap_blocks", [("kd[dst] = src_k_bits[src]", "kd[dst] = dst_k_bits[src]")]),
    ("swap_skips_v", ref, "swap_blocks", [("vd[dst] = src_v_bits[src]", "vd[dst] = dst_v_bits[dst]")]),
    ("swap_bounds_from_source_pool", ref, "swap_blocks",
     [("0 <= dst < kd.shape[0]", "0 <= dst < src_k_bits.shape[0]")]),
    # byte counts
    ("bytes_without_k_and_v", ref, "kv_bytes_per_token",
     [("2 * num_layers * num_kv_heads", "num_layers * num_kv_heads")]),
    ("block_bytes_one_layer", ref, "kv_bytes_per_block",
     [("kv_bytes_per_token(num_layers,", "kv_bytes_per_token(1,")]),
    ("table_bytes_floor", ref, "block_table_bytes",
     [("num_logical_blocks(max_model_len, block_size)", "(max_model_len // block_size)")]),
    ("logsumexp_without_max", ref, "logsumexp", [("return m + math.log(", "return math.log(")]),
    # the block manager
    ("take_from_back", bm_mod.CowBlockManager, "_take", [("self.free.pop(0)", "self.free.pop()")]),
    ("freed_block_to_front", bm_mod.CowBlockManager, "_drop", [("self.free.append(b)", "self.free.insert(0, b)")]),
    ("cow_threshold_two", bm_mod.CowBlockManager, "append_slot",
     [("elif self.ref[table[-1]] > 1:", "elif self.ref[table[-1]] > 2:")]),
    ("cow_keeps_reference", bm_mod.CowBlockManager, "append_slot",
     [("self.ref[old] -= 1          # still > 0: another sequence holds it", "pass")]),
    ("cow_copy_reversed", bm_mod.CowBlockManager, "append_slot",
     [("self.pending_copies.append((old, new))", "self.pending_copies.append((new, old))")]),
    ("cow_without_copy", bm_mod.CowBlockManager, "append_slot",
     [("self.pending_copies.append((old, new))", "pass")]),
    ("fork_without_reference", bm_mod.CowBlockManager, "fork", [("self.ref[b] += 1", "pass")]),
    ("fork_drops_partial_block", bm_mod.CowBlockManager, "fork",
     [("nb = len(self.tables[parent])", "nb = num_tokens // self.block_size")]),
    ("fork_accepts_partial_prefix", bm_mod.CowBlockManager, "fork",
     [("if num_tokens % self.block_size:", "if False:")]),
    ("free_never_returns", bm_mod.CowBlockManager, "free_sequence", [("self._drop(b)", "self.ref[b] -= 1")]),
    ("in_use_counts_zero_refs", bm_mod.CowBlockManager, "blocks_in_use", [("if c > 0", "if c >= 0")]),
]


def _pins():
    return [(n, getattr(pins, n)) for n in sorted(dir(pins)) if n.startswith("test_")]


def _mutated(owner, name, edits):
    fn = getattr(owner, name)
    src = textwrap.dedent(inspect.getsource(fn))
    for old, new in edits:
        assert src.count(old) == 1, f"{name}: {old!r} occurs {src.count(old)} times"
        src = src.replace(old, new)
    module = inspect.getmodule(fn)
    code = compile(src, f"<mutant of {name}>", "exec", flags=__future__.annotations.compiler_flag,
                   dont_inherit=True)
    scope = {}
    exec(code, module.__dict__, scope)      # globals: the oracle module, so helpers resolve live
    return scope[name]


def _failing_pins():
    failed = []
    for n, f in _pins():
        try:
            with np.errstate(all="ignore"):      # a mutant may divide by zero
                f()
        except (Exception, pytest.fail.Exception):
            failed.append(n)
    return failed


def test_unmodified_oracle_passes_every_pin():
    assert len(_pins()) >= 25
    assert _failing_pins() == []


def test_mutant_names_are_unique():
    names = [m[0] for m in MUTANTS]
    assert len(names) == len(set(names))


@pytest.mark.parametrize("name,owner,func,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, name, owner, func, edits):
    monkeypatch.setattr(owner, func, _mutated(owner, func, edits))
    assert oracle.CowBlockManager is bm_mod.CowBlockManager
    failed = _failing_pins()
    assert failed, f"mutant {name} of {func} passes every pin"
