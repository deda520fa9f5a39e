"""The allocation-free decode entry point gives the results of the regular one.

pk_paged_attention_decode_noalloc serves callers that cannot allocate device
memory (a host program that owns all of it, a plugin without an allocator, a
loop that cannot afford cudaMalloc's device synchronisation): it keeps its
scratch in a fixed array inside the library instead of a caller workspace.
Every call leaves that array's contents behind, so each workload is run
through it twice in a row, and workloads of different shapes follow each
other; every output must match the regular entry point's within the parity
tolerance, and the float64 oracle's too.  The workloads cover head dim 64 and
128, group sizes 1 to 8, bf16 and fp32 outputs, and a long-context batch
whose sequences each span many CTAs.  The file name puts it last in
collection order, so a failure here comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import _native
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import MAX_ABS, MEAN_ABS, assert_close, half_ulp_bf16, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, out, t, w, out_dtype):
    code = _native.PK_FP32 if out_dtype == torch.float32 else _native.PK_BF16
    return lib.pk_paged_attention_decode_noalloc(
        _p(out), code, _p(t["q"]), _p(t["k_cache"]), _p(t["v_cache"]), _p(t["block_tables"]),
        w.max_blocks_per_seq, _p(t["seq_lens"]), w.max_seq_len, w.num_seqs, w.num_heads, w.num_kv_heads,
        w.head_dim, w.num_blocks, w.block_size, w.scale, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    ("l3-8b", torch.float32),             # G = 4, D = 128: many sequences span two CTAs
    ("prefix-b16", torch.bfloat16),       # shared prefixes, bf16 output
    ("d64-g2", torch.bfloat16),           # head dim 64
    ("long-g8", torch.float32),           # each sequence spans dozens of CTAs
    ("g1-b8", torch.bfloat16),            # one query head per KV head, block size 8
]


def _workload(name):
    if name == "d64-g2":
        return W.custom(21, [1, 130, 700, 2500, 4097, 33, 900, 129], 16, 8, 64, 16)
    if name == "long-g8":
        return W.custom(22, [20000, 9000, 31000], 16, 2, 128, 16)
    if name == "g1-b8":
        return W.custom(23, [3000, 17, 1200, 640, 5, 2049], 8, 8, 128, 8)
    return W.get(name, 0)


def test_noalloc_matches_regular_entry_point_on_calls_in_a_row():
    lib = _native.load()
    pk.pk_get_device_error()
    # Set-up call: the first call on a device looks up the scratch array's
    # address, and the driver loads the library code that holds the array on
    # first use (the array then stays resident until the process exits).
    # Device memory is compared only across the calls that follow it.
    w0 = W.custom(20, [5, 300], 8, 2, 128, 16)       # one sequence longer than a 128-token tile
    t0 = W.make_tensors(w0, DEV)
    assert _noalloc(lib, torch.empty(w0.num_seqs, w0.num_heads, w0.head_dim, device=DEV), t0, w0,
                    torch.float32) == 0
    torch.cuda.synchronize()
    for name, out_dtype in CASES:
        w = _workload(name)
        t = W.make_tensors(w, DEV)
        ref = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                        w.scale, w.block_size, out_dtype=out_dtype, max_seq_len=w.max_seq_len)
        want = oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                             w.block_tables, w.seq_lens, w.scale, w.block_size)
        outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        alloc0 = torch.cuda.memory_allocated()
        for call in range(2):
            assert _noalloc(lib, outs[call], t, w, out_dtype) == 0
        torch.cuda.synchronize()
        # Neither call allocated device memory.
        assert torch.cuda.mem_get_info()[0] == free0 and torch.cuda.memory_allocated() == alloc0, name
        bf16 = out_dtype == torch.bfloat16
        for call, out in enumerate(outs):
            assert torch.isfinite(out).all(), f"{name} call {call}"
            got, base = out.float().cpu().numpy(), ref.float().cpu().numpy()
            err = np.abs(got - base)
            tol = MAX_ABS + (half_ulp_bf16(base) if bf16 else 0.0)
            assert np.all(err <= tol) and err.mean() <= MEAN_ABS, f"{name} call {call}"
            assert_close(out.float().cpu().numpy(), want, bf16, f"{name} call {call} vs oracle")
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
    many_heads = list(args); many_heads[10] = 40000; many_heads[11] = 40000   # the regular call's bound too
    assert lib.pk_paged_attention_decode_noalloc(*many_heads) == -2
    no_out = list(args); no_out[0] = None
    assert lib.pk_paged_attention_decode_noalloc(*no_out) == -1
