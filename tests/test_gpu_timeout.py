"""The bounded waits of the tensor-core decode kernel give up cleanly.

Every wait of a CTA on its own pipeline barriers has a time limit; when it
runs out the kernel sets PK_DEVERR_TIMEOUT, lets its own copies and MMAs land,
frees its tensor memory and returns.  pk_selftest_decode_wait_timeout makes
that happen without any fault: CTA 0's copy producer stops before one tile,
so nothing ever arrives on that tile's barriers, and the limit is a few
milliseconds.  The test checks the error bit, that the call ends, and that
the next call on the same context and workspace matches the float64 oracle.
"""
import time

import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import _native
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import assert_close, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("stall_tile", [1, 5])
def test_wait_runs_out_and_the_next_call_is_correct(stall_tile):
    w = W.get("l3-8b", 0)                 # ~34 tiles per CTA, sequences cut across CTAs
    t = W.make_tensors(w, DEV)
    ws = pk.new_workspace(pk.pk_decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                       w.max_seq_len), DEV)
    out = torch.zeros((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float32, device=DEV)
    assert pk.pk_get_device_error() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = pk.pk_selftest_decode_wait_timeout(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                            t["seq_lens"], w.scale, w.max_seq_len, ws, stall_tile, 5000)
    assert st == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert pk.pk_get_device_error() & _native.DEVERR_TIMEOUT
    assert elapsed < 5.0                  # a few 5 ms limits, not the 1 s default

    ref = oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                        w.block_tables, w.seq_lens, w.scale, w.block_size)
    for _ in range(2):
        got = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                        w.scale, w.block_size, out_dtype=torch.float32,
                                        max_seq_len=w.max_seq_len, workspace=ws)
        torch.cuda.synchronize()
        assert_close(got.cpu().numpy(), ref, False, "decode after a timed-out call")
        assert pk.pk_get_device_error() == 0
