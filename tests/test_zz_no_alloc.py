"""The allocation-free decode entry point gives the results of the regular one.

pk_paged_attention_decode_noalloc serves callers that cannot allocate device
memory (a host program that owns all of it, a plugin without an allocator, a
loop that cannot afford cudaMalloc's device synchronisation): it keeps its
scratch in a fixed array inside the library instead of a caller workspace.
Every call leaves that array's contents behind, so each workload is run
through it twice in a row, and two workloads of different shapes follow each
other; every output must match the regular entry point's within the parity
tolerance.  The file name puts it last in collection order, so a failure here
comes after every other test has run.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import _native
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, out, t, w):
    return lib.pk_paged_attention_decode_noalloc(
        _p(out), _native.PK_FP32, _p(t["q"]), _p(t["k_cache"]), _p(t["v_cache"]), _p(t["block_tables"]),
        w.max_blocks_per_seq, _p(t["seq_lens"]), w.max_seq_len, w.num_seqs, w.num_heads, w.num_kv_heads,
        w.head_dim, w.num_blocks, w.block_size, w.scale, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_regular_entry_point_on_calls_in_a_row():
    lib = _native.load()
    pk.pk_get_device_error()
    for name in ("l3-8b", "prefix-b16"):          # many sequences span several CTAs in both
        w = W.get(name, 0)
        t = W.make_tensors(w, DEV)
        ref = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                        w.scale, w.block_size, out_dtype=torch.float32, max_seq_len=w.max_seq_len)
        for call in range(2):
            out = torch.full_like(ref, float("nan"))
            assert _noalloc(lib, out, t, w) == 0
            torch.cuda.synchronize()
            err = (out - ref).abs()
            assert torch.isfinite(out).all(), f"{name} call {call}"
            assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, f"{name} call {call}"
        assert pk.pk_get_device_error() == 0


def test_noalloc_rejects_bad_arguments_before_launch():
    lib = _native.load()
    w = W.get("tiny", 0)
    t = W.make_tensors(w, DEV)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float32, device=DEV)
    args = [_p(out), _native.PK_FP32, _p(t["q"]), _p(t["k_cache"]), _p(t["v_cache"]), _p(t["block_tables"]),
            w.max_blocks_per_seq, _p(t["seq_lens"]), w.max_seq_len, w.num_seqs, w.num_heads, w.num_kv_heads,
            w.head_dim, w.num_blocks, w.block_size, w.scale, None]
    bad_group = list(args); bad_group[10] = 24; bad_group[11] = 8       # G = 3
    assert lib.pk_paged_attention_decode_noalloc(*bad_group) == -3
    too_long = list(args); too_long[8] = w.max_blocks_per_seq * w.block_size + 1
    assert lib.pk_paged_attention_decode_noalloc(*too_long) == -2
    no_out = list(args); no_out[0] = None
    assert lib.pk_paged_attention_decode_noalloc(*no_out) == -1
