"""The tensor-core decode kernel plans its range before the programmatic wait
and plans again when the lengths read after the wait differ.

pk_selftest_decode_stale_lengths makes the first read come from another
array, so the second plan always runs when the two differ.  Its output must
equal a normal call's bit for bit (the same final plan), report no error
(out-of-range values in the stale array are never reported), and match the
float64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import assert_close, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _stale(kind, w):
    n, cap = w.num_seqs, w.max_seq_len
    rng = np.random.default_rng(7)
    if kind == "zeros":
        v = np.zeros(n)
    elif kind == "reversed":
        v = w.seq_lens[::-1]
    elif kind == "out_of_range":
        v = rng.integers(-5, 2 * cap + 2, n)
    else:                                   # the true lengths: no second plan
        v = w.seq_lens
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).to(DEV)


def _workload(name):
    if name == "d64-g4":
        base = W.get("l3-8b", 1)
        return W.custom(1, base.seq_lens, 32, 8, 64, 16)
    return W.get(name, 0)


@pytest.mark.parametrize("name", ["l3-8b", "prefix-b16", "d64-g4", "l3-70b"])
@pytest.mark.parametrize("kind", ["zeros", "reversed", "out_of_range", "same"])
def test_stale_lengths_give_the_normal_result(name, kind):
    w = _workload(name)
    t = W.make_tensors(w, DEV)
    ws = pk.new_workspace(pk.pk_decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                       w.max_seq_len), DEV)
    prev = pk.pk_set_decode_path("tensor_core")
    try:
        normal = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                           w.scale, w.block_size, out_dtype=torch.float32,
                                           max_seq_len=w.max_seq_len, workspace=ws)
    finally:
        pk.pk_set_decode_path(prev)
    out = torch.full_like(normal, float("nan"))
    assert pk.pk_get_device_error() == 0
    st = pk.pk_selftest_decode_stale_lengths(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                             t["seq_lens"], w.scale, w.max_seq_len, _stale(kind, w), ws)
    assert st == 0
    torch.cuda.synchronize()
    assert pk.pk_get_device_error() == 0
    assert torch.equal(out, normal)
    if name == "l3-8b" and kind == "reversed":
        ref = oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                            w.block_tables, w.seq_lens, w.scale, w.block_size)
        assert_close(out.cpu().numpy(), ref, False, "decode planned from stale lengths")


@pytest.mark.parametrize("stale", ["ones", "reversed"])
def test_lengths_written_by_the_previous_kernel(stale):
    """The kernel before the decode call writes the lengths: here
    reshape_and_cache, whose cache rows alias the lengths array (one KV head
    of 64 elements = 32 int32 per slot), itself delayed behind a long fill.
    The decode grid is launched as that kernel's programmatic dependent, so
    it may read the lengths before they are written; its result must be that
    of the new lengths."""
    w = W.get("l3-8b", 2)
    t = W.make_tensors(w, DEV)
    n = w.num_seqs
    rows = (n * 4 + 127) // 128                       # 128-byte slots holding the lengths
    lens_cache = torch.zeros((1, 16, 1, 64), dtype=torch.bfloat16, device=DEV)
    dummy_v = torch.zeros_like(lens_cache)
    lens_view = lens_cache.view(-1).view(torch.int32)[:n]
    old = w.seq_lens.astype(np.int32)
    lens_view.copy_(torch.from_numpy(np.ones(n, np.int32) if stale == "ones" else np.ascontiguousarray(old[::-1])))
    new_rows = np.zeros(rows * 32, np.int32)
    new_rows[:n] = old
    k_new = torch.from_numpy(new_rows.view(np.int16).copy()).view(torch.bfloat16).view(rows, 1, 64).to(DEV)
    v_new = torch.zeros_like(k_new)
    slots = torch.arange(rows, dtype=torch.int64, device=DEV)
    ws = pk.new_workspace(pk.pk_decode_workspace_bytes(n, w.num_heads, w.num_kv_heads, w.head_dim, w.max_seq_len), DEV)
    big = torch.empty(1 << 30, dtype=torch.uint8, device=DEV)
    ref = oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                        w.block_tables, w.seq_lens, w.scale, w.block_size)
    torch.cuda.synchronize()
    for _ in range(3):
        lens_view.copy_(torch.from_numpy(np.ones(n, np.int32) if stale == "ones" else np.ascontiguousarray(old[::-1])))
        torch.cuda.synchronize()
        big.fill_(1)                                   # keeps the append waiting
        pk.reshape_and_cache(k_new, v_new, lens_cache, dummy_v, slots)
        got = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], lens_view,
                                        w.scale, w.block_size, out_dtype=torch.float32,
                                        max_seq_len=w.max_seq_len, workspace=ws)
        torch.cuda.synchronize()
        assert pk.pk_get_device_error() == 0
        assert np.array_equal(lens_view.cpu().numpy(), old)
        assert_close(got.cpu().numpy(), ref, False, "decode after the lengths were written by the previous kernel")
