"""Batches around the tensor-core kernel's shared-memory length cache (2,048
sequences): at or below it the kernel plans its range before the
programmatic wait from a copy of the lengths; above it, after the wait from
the lengths in device memory.  Both against the float64 oracle, for the
per-head tiles (head dim 128) and the head pairs (head dim 64), and for two
query tokens per sequence."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import assert_close, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _lens(n, seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 300, n)
    lens[::97] = 0                                   # some empty sequences
    lens[5::211] = 900                               # some cut across CTAs
    return lens


@pytest.mark.parametrize("n", [2048, 2049, 3000])
@pytest.mark.parametrize("D", [128, 64])
def test_large_batches_match_oracle(n, D):
    w = W.custom(60 + n % 7, _lens(n, n), 32, 8, D, 16)
    t = W.make_tensors(w, DEV)
    prev = pk.pk_set_decode_path("tensor_core")
    try:
        got = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                        w.scale, w.block_size, out_dtype=torch.float32, max_seq_len=w.max_seq_len)
    finally:
        pk.pk_set_decode_path(prev)
    torch.cuda.synchronize()
    assert pk.pk_get_device_error() == 0
    ref = oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                        w.block_tables, w.seq_lens, w.scale, w.block_size)
    assert_close(got.cpu().numpy(), ref, False, f"decode, {n} sequences, head dim {D}")


@pytest.mark.parametrize("n", [2048, 2300])
def test_large_batches_two_queries_match_oracle(n):
    lens = np.maximum(_lens(n, n + 1), 2)            # room for two query tokens
    w = W.custom(70, lens, 32, 8, 128, 16)
    t = W.make_tensors(w, DEV)
    cu = np.arange(n + 1, dtype=np.int32) * 2
    g = torch.Generator().manual_seed(71)
    q = torch.randn(2 * n, 32, 128, generator=g).to(torch.bfloat16).to(DEV)
    got = pk.paged_attention_multi_query(q, torch.from_numpy(cu).to(DEV), 2, t["k_cache"], t["v_cache"],
                                         t["block_tables"], t["seq_lens"], w.scale, out_dtype=torch.float32,
                                         max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    assert pk.pk_get_device_error() == 0
    ref = oracle.paged_multi_query_attention(host_bits(q), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                             w.block_tables, w.seq_lens, cu.tolist(), w.scale, w.block_size)
    assert_close(got.cpu().numpy(), ref, False, f"two queries, {n} sequences")
