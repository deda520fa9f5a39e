"""The library's C++ host block manager against the pages' printed outcomes and,
op by op, against the oracle's block manager (integer work: exact).

No GPU: the block manager is host code in the same shared library.
"""
import copy
import ctypes
import json
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN
from paged_kv_cache_122_gb300 import BlockManager, PagedKVError
from paged_kv_cache_122_gb300 import _native


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _table(bm, sid):
    _, nb = bm.sequence_info(sid)
    t, _ = bm.export([sid], max(nb, 1))
    return [int(x) for x in t[0][:nb]]


# ---------------------------------------------------------------------------
# The pages' printed examples, through the native manager
# ---------------------------------------------------------------------------

def test_cow_sim_printed_results_native():
    g = _golden("cow_and_sharing.json")["cow_sim"]
    B = g["block_size"]
    bm = BlockManager(g["pool_blocks"], B)
    bm.add_sequence(0)
    bm.append_slots([0] * g["prompt_tokens"])
    prompt = _table(bm, 0)
    assert len(prompt) == 63
    samples = list(range(1, g["samples"] + 1))
    for s in samples:
        bm.fork(0, s)
    bm.free_sequence(0)
    for _ in range(g["tokens_per_sample"]):
        bm.append_slots(samples)
    assert bm.blocks_in_use() == g["blocks_in_use"]
    tables = [_table(bm, s) for s in samples]
    assert sum(t[0] == prompt[0] for t in tables) == g["first_block_shared_by"]
    assert [t[len(prompt) - 1] for t in tables] == g["last_prompt_block_per_sample"]
    assert bm.take_copies().tolist() == [[62, 63], [62, 64], [62, 65]]


def test_blueprint_allocation_printed_native():
    g = _golden("cow_and_sharing.json")["blueprint"]
    bm = BlockManager(g["pool_blocks"], g["block_size"])
    bm.add_sequence(7)
    grew = []
    for t in range(g["tokens"]):
        before = bm.sequence_info(7)[1]
        bm.append_slots([7])
        if bm.sequence_info(7)[1] > before:
            grew.append(t)
    assert grew == g["new_block_at_tokens"]
    assert _table(bm, 7) == g["table"]
    bm.free_sequence(7)
    assert bm.blocks_in_use() == 0 and bm.num_free_blocks() == g["pool_blocks"]


def test_system_prompt_full_block_sharing_native():
    g = _golden("cow_and_sharing.json")["system_prompt"]
    B = g["block_size"]
    bm = BlockManager(10_000, B)
    bm.add_sequence(-1)
    bm.append_slots([-1] * g["prompt_tokens"])
    full = (g["prompt_tokens"] // B) * B
    for c in range(g["chats"]):
        bm.fork(-1, c, num_tokens=full)
        bm.append_slots([c] * (g["prompt_tokens"] - full))
    bm.free_sequence(-1)
    assert bm.take_copies().shape == (0, 2)
    assert bm.blocks_in_use() == g["blocks_with_sharing"]


# ---------------------------------------------------------------------------
# Differential test against the oracle, op by op
# ---------------------------------------------------------------------------

def _run_random(seed, num_blocks, B, n_ops):
    rng = np.random.default_rng(seed)
    ref = oracle.CowBlockManager(num_blocks, B)
    bm = BlockManager(num_blocks, B)
    live = []
    next_id = 0
    n_no_blocks = 0
    for _ in range(n_ops):
        op = rng.choice(["add", "append", "append", "append", "fork", "fork_prefix", "free"])
        if op == "add" or not live:
            sid = next_id
            next_id += 1
            ref.new_sequence(str(sid))
            bm.add_sequence(sid)
            live.append(sid)
        elif op == "append":
            ids = [int(x) for x in rng.choice(live, size=int(rng.integers(1, 6)))]
            saved = copy.deepcopy(ref)
            try:
                want = [ref.append_slot(str(i)) for i in ids]
            except MemoryError:
                ref = saved                      # the native batch is all or nothing
                want = None
            if want is None:
                with pytest.raises(PagedKVError) as e:
                    bm.append_slots(ids)
                assert e.value.status == _native.PK_ERR_NO_BLOCKS
                n_no_blocks += 1
            else:
                assert bm.append_slots(ids).tolist() == want
        elif op in ("fork", "fork_prefix"):
            parent = int(rng.choice(live))
            child = next_id
            next_id += 1
            if op == "fork":
                ref.fork(str(parent), str(child))
                bm.fork(parent, child)
            else:
                full = ref.lengths[str(parent)] // B
                k = int(rng.integers(0, full + 1)) * B
                ref.fork(str(parent), str(child), num_tokens=k)
                bm.fork(parent, child, num_tokens=k)
            live.append(child)
        else:
            sid = int(rng.choice(live))
            live.remove(sid)
            ref.free_sequence(str(sid))
            bm.free_sequence(sid)
        # Same state after every op.
        assert bm.take_copies().tolist() == [list(p) for p in ref.take_copies()]
        assert bm.num_free_blocks() == len(ref.free)
        assert bm.blocks_in_use() == ref.blocks_in_use()
        for sid in live:
            length, nb = bm.sequence_info(sid)
            assert length == ref.lengths[str(sid)]
            assert _table(bm, sid) == ref.tables[str(sid)]
    return n_no_blocks


@pytest.mark.parametrize("seed,num_blocks,B", [(0, 48, 4), (1, 32, 1), (2, 200, 16), (3, 24, 8)])
def test_random_ops_match_oracle(seed, num_blocks, B):
    _run_random(seed, num_blocks, B, 600)


def test_random_ops_exercise_pool_exhaustion():
    # A tiny pool makes the all-or-nothing failure path common.
    assert _run_random(11, 12, 2, 800) > 0


# ---------------------------------------------------------------------------
# Batches, errors and the C edge cases
# ---------------------------------------------------------------------------

def test_failed_batch_leaves_state_unchanged():
    bm = BlockManager(3, 2)
    for s in (1, 2):
        bm.add_sequence(s)
    bm.append_slots([1, 1, 1])              # seq 1: blocks 0, 1 (3 tokens)
    bm.fork(1, 3)                            # shares 0, 1; block 1 is partial
    before = (bm.export([1, 2, 3], 4), bm.num_free_blocks(), bm.blocks_in_use())
    # 3 -> copy-on-write of block 1 (takes block 2), then 2 needs a block: none left.
    with pytest.raises(PagedKVError) as e:
        bm.append_slots([3, 2])
    assert e.value.status == _native.PK_ERR_NO_BLOCKS
    after = (bm.export([1, 2, 3], 4), bm.num_free_blocks(), bm.blocks_in_use())
    for x, y in zip(before[0], after[0]):
        assert np.array_equal(x, y)
    assert before[1:] == after[1:]
    assert bm.take_copies().shape == (0, 2)
    # The undone block went back to the front: the next taker gets block 2.
    assert bm.append_slots([2]).tolist() == [4]


def test_repeated_id_in_one_batch_appends_in_order():
    bm = BlockManager(8, 2)
    bm.add_sequence(5)
    assert bm.append_slots([5, 5, 5]).tolist() == [0, 1, 2]
    assert bm.sequence_info(5) == (3, 2)


def test_errors():
    bm = BlockManager(4, 4)
    bm.add_sequence(1)
    with pytest.raises(PagedKVError) as e:
        bm.add_sequence(1)
    assert e.value.status == _native.PK_ERR_SEQUENCE_EXISTS
    for fn in (lambda: bm.append_slots([2]), lambda: bm.free_sequence(2), lambda: bm.fork(2, 3),
               lambda: bm.sequence_info(2), lambda: bm.export([2], 1)):
        with pytest.raises(PagedKVError) as e:
            fn()
        assert e.value.status == _native.PK_ERR_UNKNOWN_SEQUENCE
    bm.append_slots([1] * 6)
    with pytest.raises(PagedKVError) as e:
        bm.fork(1, 9, num_tokens=3)          # only whole blocks can be shared by prefix
    assert e.value.status == -2
    with pytest.raises(PagedKVError) as e:
        bm.fork(1, 9, num_tokens=8)          # longer than the parent
    assert e.value.status == -2
    with pytest.raises(PagedKVError) as e:
        bm.export([1], 1)                    # two blocks do not fit one column
    assert e.value.status == -2
    assert BlockManager(1, 1).num_free_blocks() == 1
    with pytest.raises(ValueError):
        BlockManager(0, 16)


def test_take_copies_reports_needed_room():
    lib = _native.load()
    bm = BlockManager(8, 4)
    bm.add_sequence(1)
    bm.append_slots([1, 1])
    bm.fork(1, 2)
    bm.fork(1, 3)
    bm.append_slots([2, 3])                 # two copy-on-write copies
    got = ctypes.c_int(-1)
    buf = np.zeros((1, 2), dtype=np.int64)
    assert lib.pk_bm_take_copies(bm._h, buf.ctypes.data, 1, ctypes.byref(got)) == -2
    assert got.value == 2 and lib.pk_bm_num_pending_copies(bm._h) == 2
    assert bm.take_copies().tolist() == [[0, 1], [0, 2]]


def test_export_pads_with_minus_one_and_fills_given_buffers():
    bm = BlockManager(16, 4)
    for s in (3, 4):
        bm.add_sequence(s)
    bm.append_slots([3] * 9 + [4])
    tables = np.full((2, 5), 77, dtype=np.int32)
    lens = np.zeros(2, dtype=np.int32)
    bm.export([4, 3], 5, tables_out=tables, lens_out=lens)
    assert tables.tolist() == [[3, -1, -1, -1, -1], [0, 1, 2, -1, -1]]
    assert lens.tolist() == [1, 9]


@pytest.mark.parametrize("B", [8, 16, 32])
def test_prefix_workload_driven_by_native_manager(B):
    """Config 5 (shared prefix + copy-on-write) built by the native manager:
    its slot mapping, copy pairs and tables equal the workload's, up to one
    relabelling of physical ids."""
    from paged_kv_cache_122_gb300 import workloads as W
    w = W.prefix_cow(0, B)
    nb_shared = oracle.num_logical_blocks(W.PREFIX_TOKENS, B)
    S = W.PREFIX_SEQS_PER_GROUP
    bm = BlockManager(10 ** 5, B)
    slots, pairs = [], []
    for g in range(W.PREFIX_GROUPS):
        parent = 10 ** 6 + g
        bm.add_sequence(parent)
        bm.append_slots([parent] * W.PREFIX_TOKENS)
        for j in range(S):
            bm.fork(parent, g * S + j)
        bm.free_sequence(parent)
        for j in range(S):
            s = g * S + j
            L = int(w.seq_lens[s])
            got = bm.append_slots([s] * (L - W.PREFIX_TOKENS))
            for pos, slot in zip(range(W.PREFIX_TOKENS, L), got.tolist()):
                if pos < nb_shared * B or pos == L - 1:
                    slots.append(slot)
            pairs.extend(tuple(p) for p in bm.take_copies().tolist())
    MB = w.block_tables.shape[1]
    tables, lens = bm.export(list(range(w.num_seqs)), MB)
    assert np.array_equal(lens, w.seq_lens)
    relabel = {}
    for s in range(w.num_seqs):
        nb = oracle.num_logical_blocks(int(w.seq_lens[s]), B)
        assert (tables[s, nb:] == -1).all()
        for a, b in zip(tables[s, :nb].tolist(), w.block_tables[s, :nb].tolist()):
            assert relabel.setdefault(a, b) == b
    assert len(set(relabel.values())) == len(relabel)
    assert [(relabel[a], relabel[b]) for a, b in pairs] == [tuple(p) for p in w.copy_pairs.tolist()]
    assert [relabel[x // B] * B + x % B for x in slots] == w.slot_mapping.tolist()
