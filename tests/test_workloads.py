"""The seeded workloads follow their recipes.  CPU only."""
import math

import numpy as np
import pytest

import oracle
from paged_kv_cache_122_gb300 import workloads as W


def _check_tables(w):
    used = []
    for s in range(w.num_seqs):
        nb = oracle.num_logical_blocks(int(w.seq_lens[s]), w.block_size)
        row = w.block_tables[s]
        assert np.all(row[:nb] >= 0) and np.all(row[:nb] < w.num_blocks)
        assert np.all(row[nb:] == -1)
        used.extend(row[:nb].tolist())
    return used


@pytest.mark.parametrize("name", ["tiny", "l3-8b", "l3-70b", "long"])
def test_plain_workloads_follow_recipe(name):
    w = W.get(name, seed=0)
    used = _check_tables(w)
    assert len(used) == len(set(used)), "no sharing outside the prefix workload"
    spec = {"tiny": (4, 8, 8, 64, 16), "l3-8b": (64, 32, 8, 128, 16), "l3-70b": (256, 64, 8, 128, 16),
            "long": (8, 32, 8, 128, 16)}[name]
    assert (w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size) == spec
    L = w.seq_lens.astype(np.int64)
    if name == "tiny":
        assert w.num_blocks == 64 and L.min() >= 2 and L.max() <= 129 and w.num_new_tokens == 4
    elif name == "l3-8b":
        assert L.min() >= 512 and L.max() <= 2048 and w.num_new_tokens == 0
        assert w.num_blocks == math.ceil(len(used) * 1.1)
    elif name == "l3-70b":
        assert L.min() >= 17 and L.max() <= 8193 and w.num_new_tokens == 256
        assert 500 <= np.median(L) <= 720          # lognormal median 600
        assert w.num_blocks == math.ceil(len(used) * 1.1)
    else:
        assert L.min() >= 32768 and L.max() <= 131072 and w.num_new_tokens == 0
    if w.num_new_tokens:
        # Each appended token is the last position of its sequence.
        for s in range(w.num_seqs):
            assert w.slot_mapping[s] == oracle.token_slot(w.block_tables[s], int(L[s]) - 1, w.block_size)


def test_workloads_are_deterministic_per_seed():
    a, b, c = W.get("l3-70b", 0), W.get("l3-70b", 0), W.get("l3-70b", 1)
    assert np.array_equal(a.block_tables, b.block_tables) and np.array_equal(a.seq_lens, b.seq_lens)
    assert not np.array_equal(a.seq_lens, c.seq_lens)


@pytest.mark.parametrize("B", [8, 16, 32])
def test_prefix_workload_matches_block_manager_rules(B):
    """Tables and copy pairs equal the reference block manager's, up to relabelling."""
    w = W.prefix_cow(0, B)
    nb_shared = oracle.num_logical_blocks(W.PREFIX_TOKENS, B)
    assert oracle.last_block_fill(W.PREFIX_TOKENS, B) == 6
    assert nb_shared == {8: 129, 16: 65, 32: 33}[B]
    bm = oracle.CowBlockManager(10 ** 6, B)
    S = W.PREFIX_SEQS_PER_GROUP
    slots_ref, pairs_ref = [], []
    for g in range(W.PREFIX_GROUPS):
        bm.new_sequence(f"p{g}")
        for _ in range(W.PREFIX_TOKENS):
            bm.append_slot(f"p{g}")
        for j in range(S):
            bm.fork(f"p{g}", f"s{g * S + j}")
        bm.free_sequence(f"p{g}")
        for j in range(S):
            s = g * S + j
            # Setup: private tokens up to the end of the shared block are written
            # in the step, the rest already lie in private blocks.
            L = int(w.seq_lens[s])
            for pos in range(W.PREFIX_TOKENS, L):
                slot = bm.append_slot(f"s{s}")
                if pos < nb_shared * B or pos == L - 1:
                    slots_ref.append(slot)
            pairs_ref.extend(bm.take_copies())
    assert len(pairs_ref) == len(w.copy_pairs) == W.PREFIX_GROUPS * (S - 1)
    # One relabelling of physical ids maps the manager's tables onto the workload's.
    relabel = {}
    for s in range(w.num_seqs):
        mine = bm.tables[f"s{s}"]
        nb = oracle.num_logical_blocks(int(w.seq_lens[s]), B)
        assert len(mine) == nb
        for a, b in zip(mine, w.block_tables[s, :nb].tolist()):
            assert relabel.setdefault(a, b) == b
    assert len(set(relabel.values())) == len(relabel)
    assert [(relabel[a], relabel[b]) for a, b in pairs_ref] == [tuple(p) for p in w.copy_pairs.tolist()]
    mapped = [relabel[x // B] * B + x % B for x in slots_ref]
    assert mapped == w.slot_mapping.tolist()
    assert max(relabel.values()) < w.num_blocks


def test_tensor_values_are_seeded_bf16_normal():
    w = W.tiny(0)
    t1, t2 = W.make_tensors(w, "cpu"), W.make_tensors(w, "cpu")
    for k in ("q", "k_new", "k_cache", "v_cache"):
        assert t1[k].dtype.is_floating_point and str(t1[k].dtype) == "torch.bfloat16"
        assert np.array_equal(W.bits(t1[k]), W.bits(t2[k]))
    x = t1["k_cache"].float().numpy().ravel()
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1.0) < 0.05
