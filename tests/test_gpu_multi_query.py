"""Multi-query paged attention (several newest tokens per sequence, causal
among them) on the tensor cores against the float64 oracle, and one query
per sequence against the decode call bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import assert_close, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(seed, lens, qlens, G, Hkv, D, B):
    w = W.custom(seed, lens, G * Hkv, Hkv, D, B)
    t = W.make_tensors(w, DEV)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed + 100)
    q = torch.randn(int(cu[-1]), G * Hkv, D, generator=g).to(torch.bfloat16).to(DEV)
    return w, t, q, cu


def _run(w, t, q, cu, qmax, out_dtype=torch.float32):
    return pk.paged_attention_multi_query(q, torch.from_numpy(cu).to(DEV), qmax, t["k_cache"], t["v_cache"],
                                          t["block_tables"], t["seq_lens"], w.scale, out_dtype=out_dtype,
                                          max_seq_len=w.max_seq_len)


def _ref(w, t, q, cu):
    return oracle.paged_multi_query_attention(host_bits(q), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                              w.block_tables, w.seq_lens, cu.tolist(), w.scale, w.block_size)


@pytest.mark.parametrize("G,qmax", [(8, 2), (4, 4), (2, 8), (1, 16), (16, 1), (4, 3), (1, 5)])
@pytest.mark.parametrize("D,B", [(128, 16), (64, 8), (128, 32)])
def test_multi_query_matches_oracle(G, qmax, D, B):
    Hkv = 2
    rng = np.random.default_rng(G * 100 + qmax + D + B)
    lens = [1, 2, 17, 128, 129, 300, 700, 1500]
    qlens = [min(L, int(rng.integers(1, qmax + 1))) for L in lens]
    qlens[-1] = qmax                                      # the widest case occurs
    w, t, q, cu = _case(7, lens, qlens, G, Hkv, D, B)
    out = _run(w, t, q, cu, qmax)
    assert_close(out.cpu().numpy(), _ref(w, t, q, cu), False, f"G={G} q={qmax} D={D} B={B}")
    assert pk.pk_get_device_error() == 0


def test_multi_query_bf16_out_and_full_prefill_of_short_sequences():
    # q = L: every token of the sequence is a query (a whole prompt chunk).
    lens = [1, 3, 8, 16]
    w, t, q, cu = _case(11, lens, lens, 1, 4, 128, 16)
    out = _run(w, t, q, cu, 16, torch.bfloat16)
    assert_close(out.float().cpu().numpy(), _ref(w, t, q, cu), True, "full prefill")


def test_one_query_per_sequence_equals_decode_bit_for_bit():
    lens = [5, 130, 900, 2049]
    G, Hkv = 8, 2
    w, t, q, cu = _case(13, lens, [1] * len(lens), G, Hkv, 128, 16)
    prev = pk.pk_set_decode_path("tensor_core")
    try:
        dec = pk.paged_attention_decode(q, t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                        w.scale, w.block_size, out_dtype=torch.float32,
                                        max_seq_len=w.max_seq_len)
    finally:
        pk.pk_set_decode_path(prev)
    mq = _run(w, t, q, cu, 1)
    assert torch.equal(dec, mq)


@pytest.mark.parametrize("G,qmax", [(8, 3), (8, 64), (4, 100), (1, 300), (16, 40), (2, 129)])
@pytest.mark.parametrize("D,B", [(128, 16), (64, 32), (128, 8), (64, 8)])
def test_wide_query_blocks_match_oracle(G, qmax, D, B):
    # Prompt chunks: 128 / G query tokens x G heads per CTA over the key tiles.
    Hkv = 2
    rng = np.random.default_rng(G * 1000 + qmax + D + B)
    lens = [1, 5, 130, 300, 700, 1111]
    qlens = [min(L, int(rng.integers(1, qmax + 1))) for L in lens]
    qlens[-1] = qmax
    qlens[2] = 130                                       # a whole prompt as one chunk
    qmax = max(qlens)
    w, t, q, cu = _case(17, lens, qlens, G, Hkv, D, B)
    out = _run(w, t, q, cu, qmax)
    assert_close(out.cpu().numpy(), _ref(w, t, q, cu), False, f"wide G={G} q={qmax} D={D} B={B}")
    assert pk.pk_get_device_error() == 0


def test_wide_block_bf16_out_with_garbage_table_padding():
    lens = [40, 513, 1024]
    w = W.custom(19, lens, 16, 2, 128, 16, pad="garbage")
    t = W.make_tensors(w, DEV)
    qlens = [40, 200, 512]
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    g = torch.Generator().manual_seed(5)
    q = torch.randn(int(cu[-1]), 16, 128, generator=g).to(torch.bfloat16).to(DEV)
    out = _run(w, t, q, cu, 512, torch.bfloat16)
    assert_close(out.float().cpu().numpy(), _ref(w, t, q, cu), True, "wide bf16")
    assert pk.pk_get_device_error() == 0


@pytest.mark.parametrize("scale", [0.0, -0.09])
@pytest.mark.parametrize("qmax", [2, 200])
def test_multi_query_any_finite_scale(scale, qmax):
    # Zero and negative scales on both kernels (narrow: 2 tokens x G = 8;
    # wide: prompt chunks): the prefill softmax takes the row MIN of the raw
    # scores when the scale is negative.
    lens = [5, 130, 700, 1111]
    qlens = [min(L, qmax) for L in lens]
    w, t, q, cu = _case(29, lens, qlens, 8, 2, 128, 16)
    out = pk.paged_attention_multi_query(q, torch.from_numpy(cu).to(DEV), max(qlens), t["k_cache"], t["v_cache"],
                                         t["block_tables"], t["seq_lens"], scale, out_dtype=torch.float32,
                                         max_seq_len=w.max_seq_len)
    ref = oracle.paged_multi_query_attention(host_bits(q), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                             w.block_tables, w.seq_lens, cu.tolist(), scale, w.block_size)
    assert_close(out.cpu().numpy(), ref, False, f"scale={scale} q={qmax}")
    assert pk.pk_get_device_error() == 0


def test_output_not_16_byte_aligned_is_refused_before_any_launch():
    # Device pointers must be 16-byte aligned (the TMA store and the vector
    # stores rely on it): a bf16 output 2 bytes into an allocation is
    # refused on the host and left untouched.
    lens = [300, 700]
    qlens = [256, 300]
    w, t, q, cu = _case(31, lens, qlens, 8, 2, 128, 16)
    n = q.numel()
    buf = torch.full((n + 8,), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[1:1 + n].view(q.shape)
    assert out.data_ptr() % 16 != 0
    with pytest.raises(pk.PagedKVError, match="ALIGNMENT"):
        pk.paged_attention_multi_query(q, torch.from_numpy(cu).to(DEV), max(qlens), t["k_cache"], t["v_cache"],
                                       t["block_tables"], t["seq_lens"], w.scale, out=out,
                                       max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    assert (buf.float().cpu().numpy() == 7.0).all()
    assert pk.pk_get_device_error() == 0
