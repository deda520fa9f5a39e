"""Pins for the float64 oracle: values the pages print, closed forms,
invariants and brute force on tiny inputs.  CPU only.

Each test targets a mistake the oracle could plausibly contain (a dropped
scale, swapped K and V, a wrong sign in the exponent, a transposed index in the
table walk, an unmasked tail, a wrong GQA head mapping) so that such a mistake
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import paged_ref as ref
from conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(x):
    """Round float32 to bf16 bits (nearest-even); test-side helper."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def _rand_bits(rng, shape, scale=1.0):
    return _bf16_bits(rng.standard_normal(shape).astype(np.float32) * scale)


# ---------------------------------------------------------------------------
# Printed examples
# ---------------------------------------------------------------------------

def test_block_counts_printed_on_pages():
    g = _golden("block_math.json")
    for c in g["cases"]:
        assert ref.num_logical_blocks(c["seq_len"], c["block_size"]) == c["num_blocks"], c["cite"]
        assert ref.last_block_fill(c["seq_len"], c["block_size"]) == c["last_fill"], c["cite"]
        assert c["seq_len"] // c["block_size"] == c["full_blocks"], c["cite"]


def test_block_table_walk_printed_example():
    ex = _golden("block_math.json")["block_table_example"]
    B = ex["block_size"]
    for tok, phys in ex["token_to_physical_block"].items():
        slot = ref.token_slot(ex["block_table"], int(tok), B)
        assert slot // B == phys
        assert slot % B == int(tok) % B


def test_gather_follows_printed_block_table():
    # 50 tokens through [7, 23, 4, 19]: token t must come from physical block
    # table[t // 16] at offset t % 16.  Pool rows carry their own coordinates.
    ex = _golden("block_math.json")["block_table_example"]
    P, B, D = 32, 16, 2
    cache = np.zeros((P, B, 1, D), dtype=np.uint16)
    for b in range(P):
        for o in range(B):
            cache[b, o, 0] = (b, o)
    got = ref.gather_sequence(cache, ex["block_table"], ex["seq_len"], B, 0)
    for tok, phys in ex["token_to_physical_block"].items():
        assert tuple(got[int(tok)]) == (phys, int(tok) % B)


def test_byte_counts_printed_on_pages():
    g = _golden("byte_counts.json")
    for c in g["per_token"]:
        assert ref.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["dtype_bytes"]) == c["bytes"], c["cite"]
    for c in g["per_block"]:
        assert ref.kv_bytes_per_block(c["block_size"], c["kv_heads"], c["head_dim"], c["dtype_bytes"],
                                      c["layers"]) == c["bytes"], c["cite"]
    for c in g["pools"]:
        assert c["pool_bytes"] // c["block_bytes"] == c["blocks"], c["cite"]
        assert c["blocks"] * c["block_size"] == c["tokens"], c["cite"]
    pb = ref.kv_bytes_per_block(16, 8, 128, 2, 80)
    assert pb == g["pools"][0]["block_bytes"]
    pb = ref.kv_bytes_per_block(16, 8, 128, 2, 32)
    assert pb == g["pools"][1]["block_bytes"]
    for c in g["per_request"]:
        assert c["tokens"] * ref.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"],
                                                    c["dtype_bytes"]) == c["bytes"], c["cite"]
    for c in g["block_tables"]:
        assert ref.block_table_bytes(c["num_seqs"], c["max_model_len"], c["block_size"],
                                     c["entry_bytes"]) == c["bytes"], c["cite"]
        assert c["num_seqs"] * ref.num_logical_blocks(c["max_model_len"], c["block_size"]) == c["numel"]


def test_block_table_has_room_for_a_ragged_longest_sequence():
    # "PagedAttention from First Principles" §6: a row holds one entry per block
    # of the longest allowed sequence, the last block partly filled included.
    assert ref.block_table_bytes(1, 17, 16) == 8          # 17 tokens: 2 blocks of 16
    assert ref.block_table_bytes(2, 1, 16) == 8           # 1 token: 1 block per sequence
    assert ref.block_table_bytes(200, 8193, 16) == 410_400  # 513 entries of 4 bytes
    # A row of that many entries is exactly long enough for the gather.
    cache = np.zeros((4, 16, 1, 2), dtype=np.uint16)
    row = [3, 1]
    assert len(row) * 4 == ref.block_table_bytes(1, 17, 16)
    assert ref.gather_sequence(cache, row, 17, 16, 0).shape == (17, 2)
    with pytest.raises(ValueError):
        ref.gather_sequence(cache, row[:1], 17, 16, 0)


# ---------------------------------------------------------------------------
# Block manager: copy-on-write and sharing examples
# ---------------------------------------------------------------------------

def test_cow_sim_printed_results():
    g = _golden("cow_and_sharing.json")["cow_sim"]
    B = g["block_size"]
    bm = oracle.CowBlockManager(g["pool_blocks"], B)
    bm.new_sequence("prompt")
    for _ in range(g["prompt_tokens"]):
        bm.append_slot("prompt")
    assert len(bm.tables["prompt"]) == ref.num_logical_blocks(g["prompt_tokens"], B) == 63
    names = [f"s{i}" for i in range(g["samples"])]
    for n in names:
        bm.fork("prompt", n)
    first = bm.tables["prompt"][0]
    last_prompt_idx = len(bm.tables["prompt"]) - 1
    bm.free_sequence("prompt")
    for _ in range(g["tokens_per_sample"]):
        for n in names:
            bm.append_slot(n)
    assert bm.blocks_in_use() == g["blocks_in_use"]
    assert bm.ref[first] == g["first_block_shared_by"]
    assert [bm.tables[n][last_prompt_idx] for n in names] == g["last_prompt_block_per_sample"]
    # Without sharing every sample owns ceil(1200 / 16) blocks.
    per = ref.num_logical_blocks(g["prompt_tokens"] + g["tokens_per_sample"], B)
    assert per * g["samples"] == g["blocks_without_sharing"]
    assert round(100 * (1 - g["blocks_in_use"] / g["blocks_without_sharing"])) == g["saving_percent"]
    # The copies the rule decided: the shared partial prompt block (62) went to
    # three fresh blocks, the last writer kept it.
    copies = bm.take_copies()
    assert copies == [(62, 63), (62, 64), (62, 65)]


def test_blueprint_allocation_printed():
    g = _golden("cow_and_sharing.json")["blueprint"]
    bm = oracle.CowBlockManager(g["pool_blocks"], g["block_size"])
    bm.new_sequence("req-1")
    grew = []
    for t in range(g["tokens"]):
        before = len(bm.tables["req-1"])
        bm.append_slot("req-1")
        if len(bm.tables["req-1"]) > before:
            grew.append(t)
    assert grew == g["new_block_at_tokens"]
    assert bm.tables["req-1"] == g["table"]
    bm.free_sequence("req-1")
    assert bm.blocks_in_use() == 0
    assert sorted(bm.free) == list(range(g["pool_blocks"]))


def test_system_prompt_full_block_sharing():
    g = _golden("cow_and_sharing.json")["system_prompt"]
    B = g["block_size"]
    bm = oracle.CowBlockManager(10_000, B)
    bm.new_sequence("sys")
    for _ in range(g["prompt_tokens"]):
        bm.append_slot("sys")
    full = (g["prompt_tokens"] // B) * B
    assert full // B == g["shared_full_blocks"]
    for c in range(g["chats"]):
        bm.fork("sys", f"chat{c}", num_tokens=full)
        for _ in range(g["prompt_tokens"] - full):
            bm.append_slot(f"chat{c}")
    bm.free_sequence("sys")
    assert bm.take_copies() == []        # only whole, never-written blocks are shared
    assert bm.blocks_in_use() == g["blocks_with_sharing"]
    assert g["chats"] * ref.num_logical_blocks(g["prompt_tokens"], B) == g["blocks_without_sharing"]


def test_block_manager_rejects_partial_prefix_share_and_runs_dry():
    bm = oracle.CowBlockManager(2, 4)
    bm.new_sequence("a")
    for _ in range(6):
        bm.append_slot("a")
    with pytest.raises(ValueError):
        bm.fork("a", "b", num_tokens=3)
    for _ in range(2):
        bm.append_slot("a")
    with pytest.raises(MemoryError):
        bm.append_slot("a")


def test_freed_blocks_join_the_back_of_the_free_list():
    # "How vLLM and PagedAttention Actually Work" §6 (Python blueprint): a new
    # block is the front id of the free list, and a block whose count drops to
    # zero is appended to the list.  Pool of 4 blocks of 2 tokens, worked by hand:
    # a -> 0, b -> 1; freeing a leaves [2, 3, 0]; then c -> 2, d -> 3, e -> 0.
    bm = oracle.CowBlockManager(4, 2)
    for seq in ("a", "b"):
        bm.new_sequence(seq)
        for _ in range(2):
            bm.append_slot(seq)
    bm.free_sequence("a")
    assert bm.free == [2, 3, 0]
    for seq in ("c", "d", "e"):
        bm.new_sequence(seq)
        bm.append_slot(seq)
    assert (bm.tables["c"], bm.tables["d"], bm.tables["e"]) == ([2], [3], [0])
    with pytest.raises(MemoryError):
        bm.new_sequence("f")
        bm.append_slot("f")


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x0001, 0x3FC0, 0x4049], dtype=np.uint16)
    got = ref.bf16_bits_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 0.0
    assert math.copysign(1.0, got[3]) == -1.0
    assert math.isinf(got[4]) and got[4] > 0
    assert got[5] == 2.0 ** -133
    assert got[6] == 1.5
    assert got[7] == 3.140625


def test_two_token_closed_form():
    # D = 4, scale = 1/sqrt(4).  q = (2,0,0,0), k0 = (1,0,0,0), k1 = (-1,0,0,0):
    # scores z0 = +1, z1 = -1, so p0 = 1/(1+e^-2), p1 = 1 - p0, p0 - p1 = tanh(1).
    # With v0 = (1,2,3,4), v1 = (-1,0,1,0):  o = (tanh 1, 2 p0, 3 p0 + p1, 4 p0).
    q = np.array([[2.0, 0, 0, 0]])
    K = np.array([[1.0, 0, 0, 0], [-1.0, 0, 0, 0]])
    V = np.array([[1.0, 2, 3, 4], [-1.0, 0, 1, 0]])
    o, lse = ref.softmax_attention(q, K, V, 1 / math.sqrt(4))
    p0 = 1.0 / (1.0 + math.exp(-2.0))
    want = [math.tanh(1.0), 2 * p0, 3 * p0 + (1 - p0), 4 * p0]
    assert np.allclose(o[0], want, rtol=0, atol=1e-15)
    assert abs(lse[0] - math.log(math.e + math.exp(-1.0))) < 1e-15


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(3)
    P, B, Hkv, D, H = 8, 16, 2, 64, 4
    kc = _rand_bits(rng, (P, B, Hkv, D))
    vc = _rand_bits(rng, (P, B, Hkv, D))
    q = _rand_bits(rng, (1, H, D), 5.0)
    bt = np.array([[5, -1]], dtype=np.int32)
    out = ref.paged_decode_attention(q, kc, vc, bt, [1], 0.125, B)
    for h in range(H):
        assert np.array_equal(out[0, h], ref.bf16_bits_to_f64(vc[5, 0, h // 2]))


def test_zero_query_and_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(4)
    L, D = 37, 16
    V = rng.standard_normal((L, D))
    K = rng.standard_normal((L, D))
    o, lse = ref.softmax_attention(np.zeros((1, D)), K, V, 0.3)
    assert np.allclose(o[0], V.mean(axis=0), atol=1e-14)
    assert abs(lse[0] - math.log(L)) < 1e-13
    Keq = np.tile(rng.standard_normal((1, D)), (L, 1))
    o2, _ = ref.softmax_attention(rng.standard_normal((2, D)), Keq, V, 0.3)
    assert np.allclose(o2, np.tile(V.mean(axis=0), (2, 1)), atol=1e-14)


def test_spike_selects_its_value():
    rng = np.random.default_rng(5)
    L, D = 20, 8
    K = rng.standard_normal((L, D)) * 0.01
    V = rng.standard_normal((L, D))
    q = np.zeros((1, D)); q[0, 0] = 1.0
    K[7, 0] = 1000.0
    o, lse = ref.softmax_attention(q, K, V, 1.0)
    assert np.allclose(o[0], V[7], atol=1e-12)
    assert abs(lse[0] - 1000.0) < 1e-9


def test_shift_of_all_scores_leaves_output_unchanged():
    # Append one coordinate: q' = (q, c/scale), k'_j = (k_j, 1)  =>  z'_j = z_j + c.
    rng = np.random.default_rng(6)
    L, D, scale = 50, 8, 0.35
    q = rng.standard_normal((3, D)); K = rng.standard_normal((L, D)); V = rng.standard_normal((L, D))
    o, lse = ref.softmax_attention(q, K, V, scale)
    for c in (-700.0, 5.0, 700.0):
        q2 = np.concatenate([q, np.full((3, 1), c / scale)], axis=1)
        K2 = np.concatenate([K, np.ones((L, 1))], axis=1)
        o2, lse2 = ref.softmax_attention(q2, K2, V, scale)
        assert np.allclose(o2, o, atol=1e-12)
        assert np.allclose(lse2, lse + c, atol=1e-9)


def test_weights_sum_to_one_via_constant_values():
    rng = np.random.default_rng(7)
    L, D = 64, 8
    K = rng.standard_normal((L, D)) * 3
    V = np.full((L, D), 2.5)
    o, _ = ref.softmax_attention(rng.standard_normal((4, D)), K, V, 1.0)
    assert np.allclose(o, 2.5, atol=1e-14)


# ---------------------------------------------------------------------------
# Brute force and invariances of the paged path
# ---------------------------------------------------------------------------

def _brute_force_contiguous(q64, K64, V64, scale):
    """Independent restatement with scalar loops and fsum: one query row."""
    z = [scale * math.fsum(float(a) * float(b) for a, b in zip(q64, k)) for k in K64]
    m = max(z)
    e = [math.exp(x - m) for x in z]
    den = math.fsum(e)
    return [math.fsum(e[j] * float(V64[j][d]) for j in range(len(z))) / den for d in range(len(V64[0]))]


def _make_paged_case(rng, N, H, Hkv, D, B, lens, pool, spare_tail_value=None):
    MB = max(ref.num_logical_blocks(L, B) for L in lens) + 2
    need = sum(ref.num_logical_blocks(L, B) for L in lens)
    ids = rng.permutation(pool)[:need]
    bt = np.full((N, MB), -1, dtype=np.int32)
    k = 0
    for s, L in enumerate(lens):
        nb = ref.num_logical_blocks(L, B)
        bt[s, :nb] = ids[k:k + nb]
        k += nb
    kc = _rand_bits(rng, (pool, B, Hkv, D))
    vc = _rand_bits(rng, (pool, B, Hkv, D))
    if spare_tail_value is not None:
        # Unused slots of each last block hold huge values; they must be masked.
        for s, L in enumerate(lens):
            nb = ref.num_logical_blocks(L, B)
            fill = ref.last_block_fill(L, B)
            if nb and fill < B:
                kc[bt[s, nb - 1], fill:] = _bf16_bits(np.float32(spare_tail_value))
                vc[bt[s, nb - 1], fill:] = _bf16_bits(np.float32(-spare_tail_value))
    q = _rand_bits(rng, (N, H, D))
    return q, kc, vc, bt


def test_paged_equals_brute_force_contiguous():
    rng = np.random.default_rng(11)
    N, H, Hkv, D, B = 3, 4, 2, 8, 4
    lens = [1, 7, 13]
    q, kc, vc, bt = _make_paged_case(rng, N, H, Hkv, D, B, lens, pool=16, spare_tail_value=3.0e4)
    scale = 1 / math.sqrt(D)
    out = ref.paged_decode_attention(q, kc, vc, bt, lens, scale, B)
    G = H // Hkv
    for s, L in enumerate(lens):
        for h in range(H):
            # Contiguous K/V built by walking positions one by one.
            Kc, Vc = [], []
            for pos in range(L):
                blk = bt[s][pos // B]
                Kc.append(ref.bf16_bits_to_f64(kc[blk, pos % B, h // G]))
                Vc.append(ref.bf16_bits_to_f64(vc[blk, pos % B, h // G]))
            want = _brute_force_contiguous(ref.bf16_bits_to_f64(q[s, h]), Kc, Vc, scale)
            assert np.allclose(out[s, h], want, rtol=0, atol=1e-13)


def test_gqa_maps_consecutive_query_heads_to_one_kv_head():
    # KV head 0 has V = +1, KV head 1 has V = -1: query heads 0,1 -> +1, 2,3 -> -1.
    rng = np.random.default_rng(12)
    P, B, Hkv, D, H = 4, 4, 2, 8, 4
    kc = _rand_bits(rng, (P, B, Hkv, D))
    vc = np.zeros((P, B, Hkv, D), dtype=np.uint16)
    vc[:, :, 0, :] = 0x3F80
    vc[:, :, 1, :] = 0xBF80
    q = _rand_bits(rng, (1, H, D))
    bt = np.array([[2, 0]], dtype=np.int32)
    out = ref.paged_decode_attention(q, kc, vc, bt, [6], 0.5, B)
    assert np.allclose(out[0, 0], 1) and np.allclose(out[0, 1], 1)
    assert np.allclose(out[0, 2], -1) and np.allclose(out[0, 3], -1)


def test_output_invariant_under_physical_relabelling():
    rng = np.random.default_rng(13)
    N, H, Hkv, D, B, P = 4, 8, 2, 16, 8, 40
    lens = [3, 17, 40, 64]
    q, kc, vc, bt = _make_paged_case(rng, N, H, Hkv, D, B, lens, pool=P)
    scale = 0.25
    base = ref.paged_decode_attention(q, kc, vc, bt, lens, scale, B)
    for trial in range(3):
        perm = rng.permutation(P)                # new id of old block b is perm[b]
        kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
        kc2[perm] = kc; vc2[perm] = vc
        bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
        got = ref.paged_decode_attention(q, kc2, vc2, bt2, lens, scale, B)
        assert np.allclose(got, base, rtol=0, atol=1e-12)


def test_output_invariant_under_block_size():
    rng = np.random.default_rng(14)
    N, H, Hkv, D = 3, 4, 1, 16
    lens = [5, 33, 70]
    # One logical K/V stream per sequence, laid out in pools of three block sizes.
    Ks = [_rand_bits(rng, (L, Hkv, D)) for L in lens]
    Vs = [_rand_bits(rng, (L, Hkv, D)) for L in lens]
    q = _rand_bits(rng, (N, H, D))
    outs = []
    for B in (8, 16, 32):
        nbs = [ref.num_logical_blocks(L, B) for L in lens]
        P = sum(nbs) + 3
        ids = rng.permutation(P)
        kc = _rand_bits(rng, (P, B, Hkv, D)); vc = _rand_bits(rng, (P, B, Hkv, D))
        bt = np.full((N, max(nbs)), -1, dtype=np.int32)
        k = 0
        for s, L in enumerate(lens):
            bt[s, :nbs[s]] = ids[k:k + nbs[s]]
            k += nbs[s]
            for pos in range(L):
                kc[bt[s, pos // B], pos % B] = Ks[s][pos]
                vc[bt[s, pos // B], pos % B] = Vs[s][pos]
        outs.append(ref.paged_decode_attention(q, kc, vc, bt, lens, 0.2, B))
    assert np.allclose(outs[0], outs[1], rtol=0, atol=1e-12)
    assert np.allclose(outs[0], outs[2], rtol=0, atol=1e-12)


def test_empty_sequence_gives_zeros_and_sentinels_are_not_read():
    rng = np.random.default_rng(15)
    P, B, Hkv, D, H = 4, 4, 1, 8, 2
    kc = _rand_bits(rng, (P, B, Hkv, D)); vc = _rand_bits(rng, (P, B, Hkv, D))
    q = _rand_bits(rng, (2, H, D))
    bt = np.array([[-1, -1], [1, 10 ** 6]], dtype=np.int32)   # row 1: sentinel past ceil(L/B)
    out = ref.paged_decode_attention(q, kc, vc, bt, [0, 3], 0.5, B)
    assert np.all(out[0] == 0)
    with pytest.raises(ValueError):
        ref.paged_decode_attention(q, kc, vc, bt, [0, 5], 0.5, B)   # would need the sentinel


def test_merge_of_any_partition_equals_whole():
    rng = np.random.default_rng(16)
    L, D, G = 301, 16, 4
    q = rng.standard_normal((G, D)) * 2; K = rng.standard_normal((L, D)); V = rng.standard_normal((L, D))
    o, lse = ref.softmax_attention(q, K, V, 0.4)
    for cuts in ([], [1], [100, 200], sorted(rng.choice(np.arange(1, L), 20, replace=False)), [0, 0, 150, L]):
        edges = [0] + list(cuts) + [L]
        parts = [ref.partial_attention(q, K[a:b], V[a:b], 0.4) for a, b in zip(edges[:-1], edges[1:])]
        mlse, mo = ref.merge_partials([p[0] for p in parts], [p[1] for p in parts])
        assert np.allclose(mo, o, rtol=0, atol=1e-12)
        assert np.allclose(mlse, lse, rtol=0, atol=1e-11)


def test_logsumexp_helper_matches_softmax_denominator():
    z = [0.5, -3.0, 2.25, 700.0]
    assert abs(ref.logsumexp(z) - (700.0 + math.log1p(sum(math.exp(x - 700.0) for x in z[:3])))) < 1e-12


# ---------------------------------------------------------------------------
# Cache writes and copies: bitwise
# ---------------------------------------------------------------------------

def test_reshape_and_cache_writes_only_target_slots():
    rng = np.random.default_rng(21)
    P, B, Hkv, D, T = 10, 8, 2, 16, 6
    kc = rng.integers(0, 65536, (P, B, Hkv, D), dtype=np.uint16)
    vc = rng.integers(0, 65536, (P, B, Hkv, D), dtype=np.uint16)
    k = rng.integers(0, 65536, (T, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 65536, (T, Hkv, D), dtype=np.uint16)
    slots = np.array([0, 79, -1, 17, 40, 41], dtype=np.int64)
    kc2, vc2 = ref.reshape_and_cache(k, v, kc, vc, slots, B)
    touched = np.zeros((P, B), dtype=bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(kc2[s // B, s % B], k[t]) and np.array_equal(vc2[s // B, s % B], v[t])
        touched[s // B, s % B] = True
    assert np.array_equal(kc2[~touched], kc[~touched]) and np.array_equal(vc2[~touched], vc[~touched])
    # The skipped token's data appears nowhere it was not already.
    assert kc2.tobytes().count(k[2].tobytes()) == kc.tobytes().count(k[2].tobytes())


def test_reshape_then_gather_reads_back_the_appended_token():
    rng = np.random.default_rng(22)
    P, B, Hkv, D = 12, 4, 2, 8
    kc = rng.integers(0, 65536, (P, B, Hkv, D), dtype=np.uint16); vc = kc.copy()
    table = [9, 2, 7]
    L = 9                                  # next position 9 -> block 2 (phys 7), offset 1
    slot = ref.token_slot(table, L, B)
    assert slot == 7 * B + 1
    k = rng.integers(0, 65536, (1, Hkv, D), dtype=np.uint16)
    kc2, _ = ref.reshape_and_cache(k, k, kc, vc, [slot], B)
    got = ref.gather_sequence(kc2, table, L + 1, B, 1)
    assert np.array_equal(got[L], k[0, 1])
    assert np.array_equal(got[:L], ref.gather_sequence(kc, table, L, B, 1))


def test_copy_blocks_clones_whole_blocks_only():
    rng = np.random.default_rng(23)
    P, B, Hkv, D = 12, 8, 2, 8
    kc = rng.integers(0, 65536, (P, B, Hkv, D), dtype=np.uint16)
    vc = rng.integers(0, 65536, (P, B, Hkv, D), dtype=np.uint16)
    pairs = [(62 % P, 3), (2, 4), (2, 5)]
    kc2, vc2 = ref.copy_blocks(kc, vc, pairs)
    for src, dst in pairs:
        assert np.array_equal(kc2[dst], kc[src]) and np.array_equal(vc2[dst], vc[src])
    untouched = [b for b in range(P) if b not in {d for _, d in pairs}]
    assert np.array_equal(kc2[untouched], kc[untouched]) and np.array_equal(vc2[untouched], vc[untouched])
    with pytest.raises(ValueError):
        ref.copy_blocks(kc, vc, [(0, P)])


def test_swap_blocks_within_one_pool_is_copy_blocks_and_round_trips():
    rng = np.random.default_rng(24)
    P, H, B, Hkv, D = 10, 6, 4, 2, 8
    kd = rng.integers(0, 65536, (P, B, Hkv, D), dtype=np.uint16)
    vd = rng.integers(0, 65536, (P, B, Hkv, D), dtype=np.uint16)
    kh = rng.integers(0, 65536, (H, B, Hkv, D), dtype=np.uint16)
    vh = rng.integers(0, 65536, (H, B, Hkv, D), dtype=np.uint16)
    # Inside one pool the swap is exactly the copy-on-write block copy.
    pairs = [(1, 7), (4, 8)]
    a = ref.swap_blocks(kd, vd, kd, vd, pairs)
    b = ref.copy_blocks(kd, vd, pairs)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # Out to the host pool and back into other device blocks: the blocks come back unchanged.
    out = [(2, 0), (5, 3), (9, 5)]
    kh2, vh2 = ref.swap_blocks(kd, vd, kh, vh, out)
    back = [(d, s) for s, d in out]
    kd2, vd2 = ref.swap_blocks(kh2, vh2, np.zeros_like(kd), np.zeros_like(vd), back)
    for s, _ in out:
        assert np.array_equal(kd2[s], kd[s]) and np.array_equal(vd2[s], vd[s])
    # Host blocks not named keep their bits.
    keep = [b for b in range(H) if b not in {d for _, d in out}]
    assert np.array_equal(kh2[keep], kh[keep]) and np.array_equal(vh2[keep], vh[keep])
    with pytest.raises(ValueError):
        ref.swap_blocks(kd, vd, kh, vh, [(0, H)])


# ---------------------------------------------------------------------------
# Multi-query (causal) paged attention
# ---------------------------------------------------------------------------

def _mq_case(seed, lens, qlens, H=4, Hkv=2, D=8, B=4, extra=3):
    rng = np.random.default_rng(seed)
    nb = [ref.num_logical_blocks(L, B) for L in lens]
    P = sum(nb) + extra
    perm = rng.permutation(P)
    bt = np.full((len(lens), max(nb)), -1, dtype=np.int32)
    k = 0
    for s, n in enumerate(nb):
        bt[s, :n] = perm[k:k + n]
        k += n
    kc = ref_bits(rng, (P, B, Hkv, D))
    vc = ref_bits(rng, (P, B, Hkv, D))
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int64)
    q = ref_bits(rng, (int(cu[-1]), H, D))
    return q, kc, vc, bt, cu, B


def ref_bits(rng, shape):
    # bf16 bit patterns of N(0, 1) draws (round to nearest even), like the workloads.
    x = rng.standard_normal(shape).astype(np.float32).view(np.uint32)
    return ((x + 0x7FFF + ((x >> 16) & 1)) >> 16).astype(np.uint16)


def test_multi_query_with_one_query_is_decode():
    lens = [1, 9, 23]
    q, kc, vc, bt, cu, B = _mq_case(30, lens, [1, 1, 1])
    a = ref.paged_multi_query_attention(q, kc, vc, bt, lens, cu, 0.35, B)
    b = ref.paged_decode_attention(q, kc, vc, bt, lens, 0.35, B)
    assert np.array_equal(a, b)


def test_multi_query_full_prefill_matches_brute_force_causal_attention():
    # Every token of the sequence is a query: masked attention written out
    # with explicit loops and math.fsum, on the contiguous gather.
    L, H, Hkv, D = 7, 4, 2, 8
    q, kc, vc, bt, cu, B = _mq_case(31, [L], [L], H=H, Hkv=Hkv, D=D)
    got = ref.paged_multi_query_attention(q, kc, vc, bt, [L], cu, 0.4, B)
    G = H // Hkv
    for h in range(H):
        K = ref.bf16_bits_to_f64(ref.gather_sequence(kc, bt[0], L, B, h // G))
        V = ref.bf16_bits_to_f64(ref.gather_sequence(vc, bt[0], L, B, h // G))
        for i in range(L):
            qi = ref.bf16_bits_to_f64(q[i, h])
            z = [0.4 * math.fsum(qi[d] * K[j, d] for d in range(D)) if j <= i else -math.inf for j in range(L)]
            m = max(z)
            w = [math.exp(x - m) if x != -math.inf else 0.0 for x in z]
            den = math.fsum(w)
            want = [math.fsum(w[j] * V[j, d] for j in range(L)) / den for d in range(D)]
            assert np.allclose(got[i, h], want, rtol=0, atol=1e-12)


def test_multi_query_is_causal_and_equals_truncated_decode():
    lens, qlens = [12, 5], [4, 5]
    q, kc, vc, bt, cu, B = _mq_case(32, lens, qlens)
    out = ref.paged_multi_query_attention(q, kc, vc, bt, lens, cu, 0.3, B)
    # Query r of sequence s equals decode over the first L - q_s + r + 1 tokens.
    for s, (L, qs) in enumerate(zip(lens, qlens)):
        for r in range(qs):
            n = L - qs + r + 1
            one = ref.paged_decode_attention(q[cu[s] + r][None], kc, vc, bt[s:s + 1], [n], 0.3, B)
            assert np.array_equal(out[cu[s] + r], one[0])
    # Changing a later token's K/V leaves earlier queries unchanged.
    pos = lens[0] - 1                                   # the last token of sequence 0
    blk, off = bt[0, pos // B], pos % B
    kc2 = kc.copy(); kc2[blk, off] ^= 0x0100
    out2 = ref.paged_multi_query_attention(q, kc2, vc, bt, lens, cu, 0.3, B)
    assert np.array_equal(out2[:cu[1] - 1], out[:cu[1] - 1])
    assert not np.array_equal(out2[cu[1] - 1], out[cu[1] - 1])
    with pytest.raises(ValueError):
        ref.paged_multi_query_attention(q, kc, vc, bt, [3, 5], cu, 0.3, B)   # 4 queries, 3 tokens
