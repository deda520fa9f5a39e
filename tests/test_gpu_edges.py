"""GPU edge cases: lengths at block and partition boundaries, every supported
group size / head dim / block size, sentinels, invariances, determinism,
guard bytes, and the device error word for bad data (no GPU fault: every
bad index below is one the kernels check and skip)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import assert_close, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PATHS = ["cuda_core", "tensor_core"]


@pytest.fixture
def decode_path(request):
    prev = pk.pk_set_decode_path(request.param)
    yield request.param
    pk.pk_set_decode_path(prev)

EDGE_LENS = [0, 1, 2, 7, 8, 15, 16, 17, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1023, 1024, 1025, 2047, 4103]


def _attend(w, t, out_dtype=torch.float32, max_seq_len=None, out=None):
    return pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                     w.scale, w.block_size, out_dtype=out_dtype, out=out,
                                     max_seq_len=max_seq_len if max_seq_len is not None else w.max_seq_len)


def _ref(w, t):
    return oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                         w.block_tables, w.seq_lens, w.scale, w.block_size)


@pytest.mark.parametrize("decode_path", PATHS, indirect=True)
@pytest.mark.parametrize("pad", ["neg1", "garbage"])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_boundary_lengths(B, pad, decode_path):
    w = W.custom(3, EDGE_LENS, 32, 8, 128, B, pad=pad)
    t = W.make_tensors(w, DEV)
    for dt in (torch.float32, torch.bfloat16):
        out = _attend(w, t, dt)
        ref = _ref(w, t)
        assert_close(out.float().cpu().numpy(), ref, dt == torch.bfloat16, f"B={B} pad={pad}")
        assert torch.all(out[0] == 0)          # empty sequence writes zeros
    assert pk.pk_get_device_error() == 0


@pytest.mark.parametrize("decode_path", PATHS, indirect=True)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_group_and_head_dim(G, D, decode_path):
    Hkv = 2
    w = W.custom(4, [1, 40, 700, 1500], G * Hkv, Hkv, D, 16)
    t = W.make_tensors(w, DEV)
    out = _attend(w, t)
    assert_close(out.cpu().numpy(), _ref(w, t), False, f"G={G} D={D}")


@pytest.mark.parametrize("decode_path", PATHS, indirect=True)
@pytest.mark.parametrize("G,B", [(4, 8), (8, 8), (4, 32), (8, 32)])
def test_head_dim_64_with_small_and_large_blocks(G, B, decode_path):
    # A 64-element head is one swizzle half: each page lands as B / 8 blocks
    # of [8 rows][64], for the blocks sizes other than the default too.
    Hkv = 2
    w = W.custom(6, [1, 9, 130, 700, 1500], G * Hkv, Hkv, 64, B)
    t = W.make_tensors(w, DEV)
    out = _attend(w, t)
    assert_close(out.cpu().numpy(), _ref(w, t), False, f"G={G} D=64 B={B}")
    assert pk.pk_get_device_error() == 0


@pytest.mark.parametrize("decode_path", PATHS, indirect=True)
@pytest.mark.parametrize("Hkv,G", [(1, 4), (3, 2), (8, 1), (8, 4), (8, 8), (6, 16)])
def test_head_dim_64_head_pairs_and_odd_kv_head_counts(Hkv, G, decode_path):
    # At head dim 64 the tensor-core kernel reads two adjacent KV heads per
    # tile when the KV head count is even and G <= 8; an odd count, or G = 16,
    # keeps one head per tile.  Both must give the oracle's result, with
    # sequences cut across CTAs.
    w = W.custom(8, [1, 17, 129, 700, 2100, 4097], G * Hkv, Hkv, 64, 16)
    t = W.make_tensors(w, DEV)
    for dt in (torch.float32, torch.bfloat16):
        out = _attend(w, t, dt)
        assert_close(out.float().cpu().numpy(), _ref(w, t), dt == torch.bfloat16, f"Hkv={Hkv} G={G} D=64")
    assert pk.pk_get_device_error() == 0


@pytest.mark.parametrize("decode_path", PATHS, indirect=True)
def test_physical_relabelling_gives_identical_bits(decode_path):
    w = W.custom(5, [3, 300, 1000, 2500], 32, 8, 128, 16)
    t = W.make_tensors(w, DEV)
    base = _attend(w, t, torch.bfloat16).clone()
    g = torch.Generator().manual_seed(0)
    perm = torch.randperm(w.num_blocks, generator=g).to(DEV)          # old id b -> new id perm[b]
    t2 = dict(t)
    t2["k_cache"] = torch.empty_like(t["k_cache"]); t2["k_cache"][perm] = t["k_cache"]
    t2["v_cache"] = torch.empty_like(t["v_cache"]); t2["v_cache"][perm] = t["v_cache"]
    bt = t["block_tables"].long()
    t2["block_tables"] = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int()
    again = _attend(w, t2, torch.bfloat16)
    assert torch.equal(base, again)


def test_block_size_invariance():
    lens = [5, 130, 777, 3000]
    outs = []
    ws = {B: W.custom(6, lens, 32, 8, 128, B) for B in (8, 16, 32)}
    base = W.make_tensors(ws[16], DEV)
    # Lay the same logical K/V stream out in pools of three block sizes.
    gk, gv, cu = pk.pk_gather_kv(base["k_cache"], base["v_cache"], base["block_tables"], base["seq_lens"], lens)
    ref_k, ref_v = host_bits(gk), host_bits(gv)
    cu = cu.cpu().numpy()
    for B, w in ws.items():
        t = W.make_tensors(w, DEV)
        t["q"] = base["q"]
        kc, vc = host_bits(t["k_cache"]).copy(), host_bits(t["v_cache"]).copy()
        for s, L in enumerate(lens):
            for pos in range(L):
                blk = w.block_tables[s, pos // B]
                kc[blk, pos % B] = ref_k[cu[s] + pos]
                vc[blk, pos % B] = ref_v[cu[s] + pos]
        t["k_cache"] = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16).to(DEV)
        t["v_cache"] = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16).to(DEV)
        outs.append(_attend(w, t).cpu().numpy())
        if B == 16:
            ref = _ref(w, t)
    # Same logical K/V, three block sizes (and, on tensor cores, different
    # kernels): every result is within the parity bound of the same oracle.
    for B, o in zip(ws, outs):
        assert_close(o, ref, False, f"block size {B}")


@pytest.mark.parametrize("decode_path", PATHS, indirect=True)
def test_deterministic_and_guard_bytes_untouched(decode_path):
    w = W.get("l3-8b", 0)
    t = W.make_tensors(w, DEV)
    N, H, D = w.num_seqs, w.num_heads, w.head_dim
    guard = torch.full((N * H * D + 2 * 4096,), -7.0, dtype=torch.float32, device=DEV)
    out = guard[4096:4096 + N * H * D].view(N, H, D)
    a = _attend(w, t, torch.float32, out=out).clone()
    b = _attend(w, t, torch.float32).clone()
    assert torch.equal(a, b)
    assert torch.all(guard[:4096] == -7.0) and torch.all(guard[-4096:] == -7.0)


def test_non_default_stream():
    w = W.get("tiny", 0)
    t = W.make_tensors(w, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = _attend(w, t)
    s.synchronize()
    assert_close(out.cpu().numpy(), _ref(w, t), False, "stream")


@pytest.mark.parametrize("decode_path", PATHS, indirect=True)
@pytest.mark.parametrize("kv_heads", [2, 8])
def test_bad_block_id_is_reported_not_faulted(decode_path, kv_heads):
    w = W.custom(7, [40, 40], 4 * kv_heads, kv_heads, 64, 16)
    t = W.make_tensors(w, DEV)
    pk.pk_get_device_error()
    bt = t["block_tables"].clone()
    bt[1, 1] = w.num_blocks + 5                    # inside ceil(L/B): read would be out of bounds
    t["block_tables"] = bt
    out = _attend(w, t)
    code = pk.pk_get_device_error()
    assert code & 0x1
    assert torch.isfinite(out).all()
    assert pk.pk_get_device_error() == 0            # read clears


def test_bad_slot_pair_and_length_are_reported():
    w = W.custom(8, [20, 20], 8, 2, 64, 16)
    t = W.make_tensors(w, DEV)
    pk.pk_get_device_error()
    before = host_bits(t["k_cache"]).copy()
    k = torch.ones(3, 2, 64, dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([-1, w.num_blocks * 16 + 3, 5], dtype=torch.int64, device=DEV)
    pk.reshape_and_cache(k, k, t["k_cache"], t["v_cache"], slots)
    assert pk.pk_get_device_error() & 0x2
    after = host_bits(t["k_cache"])
    changed = np.argwhere(np.any(after != before, axis=(2, 3)))
    assert changed.tolist() == [[0, 5]]              # only the valid slot 5 was written
    pairs = torch.tensor([[0, w.num_blocks]], dtype=torch.int64, device=DEV)
    pk.copy_blocks(t["k_cache"], t["v_cache"], pairs)
    assert pk.pk_get_device_error() & 0x4
    sl = t["seq_lens"].clone()
    sl[0] = 10 ** 6
    t["seq_lens"] = sl
    out = _attend(w, t, max_seq_len=20)
    assert pk.pk_get_device_error() & 0x8
    assert torch.isfinite(out).all()


def test_copy_blocks_bitwise_on_gpu():
    w = W.get("prefix-b16", 0)
    t = W.make_tensors(w, DEV)
    kb, vb = host_bits(t["k_cache"]), host_bits(t["v_cache"])
    pk.copy_blocks(t["k_cache"], t["v_cache"], t["copy_pairs"])
    kr, vr = oracle.copy_blocks(kb, vb, w.copy_pairs.tolist())
    assert np.array_equal(host_bits(t["k_cache"]), kr) and np.array_equal(host_bits(t["v_cache"]), vr)


@pytest.mark.parametrize("decode_path", PATHS, indirect=True)
@pytest.mark.parametrize("scale", [0.0, -0.09, 0.3])
def test_any_finite_scale(decode_path, scale):
    # The scale multiplies q.k before the softmax whatever its sign: 0 gives
    # the plain mean of V over the context, a negative scale favours the
    # keys least aligned with q.
    w = W.custom(23, [1, 16, 130, 600, 1500], 32, 8, 128, 16)
    t = W.make_tensors(w, DEV)
    out = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                    scale, w.block_size, out_dtype=torch.float32, max_seq_len=w.max_seq_len)
    ref = oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                        w.block_tables, w.seq_lens, scale, w.block_size)
    assert_close(out.cpu().numpy(), ref, False, f"{decode_path} scale={scale}")
    assert pk.pk_get_device_error() == 0
