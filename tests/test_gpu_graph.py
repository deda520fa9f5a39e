"""Every call is asynchronous on the caller's stream with no host
synchronisation, so a whole step can be captured in a CUDA graph and
replayed: the replay must give the eager result bit for bit, and follow
new inputs written into the captured buffers."""
import numpy as np
import pytest
import torch

import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _capture(fn):
    # Warm up on a side stream (first calls set kernel attributes), then capture.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_step_replays_in_a_cuda_graph():
    # Copy-on-write clones, appends and the tensor-core decode (GQA 4, long
    # sequences cut across CTAs and merged) of the prefix-sharing batch.
    w = W.get("prefix-b16", 0)
    t = W.make_tensors(w, DEV)
    assert t["copy_pairs"].shape[0] > 0 and w.num_new_tokens > 0
    ws = pk.new_workspace((pk.pk_decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                         w.max_seq_len)), DEV)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.bfloat16, device=DEV)

    def step():
        pk.copy_blocks(t["k_cache"], t["v_cache"], t["copy_pairs"])
        pk.reshape_and_cache(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
        pk.pk_paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                     w.scale, w.block_size, w.max_seq_len, ws)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    g = _capture(step)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)

    # New queries in the captured buffer: the replay follows them.
    gen = torch.Generator(device=DEV).manual_seed(3)
    t["q"].copy_(torch.randn(t["q"].shape, generator=gen, device=DEV).to(torch.bfloat16))
    step()
    torch.cuda.synchronize()
    eager2 = out.clone()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager2)
    assert not torch.equal(eager, eager2)
    assert pk.pk_get_device_error() == 0


def test_head_pair_decode_and_verification_replay_in_a_cuda_graph():
    # Head dim 64 (tiles of two KV heads) and two newest tokens per sequence
    # as causal queries on the decode kernel's columns, both with sequences
    # cut across CTAs, captured together and replayed.
    w = W.custom(43, [5, 300, 1500, 4000, 129, 2200], 32, 8, 64, 16)
    t = W.make_tensors(w, DEV)
    ws = pk.new_workspace(pk.pk_decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                       w.max_seq_len), DEV)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float32, device=DEV)
    N = w.num_seqs
    cu = torch.arange(N + 1, dtype=torch.int32, device=DEV) * 2
    gen = torch.Generator(device=DEV).manual_seed(11)
    q2 = torch.randn(2 * N, w.num_heads, w.head_dim, generator=gen, device=DEV).to(torch.bfloat16)
    out2 = torch.empty_like(q2)
    ws2 = pk.new_workspace(pk.pk_decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                        w.max_seq_len), DEV)

    def step():
        pk.pk_paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                     w.scale, w.block_size, w.max_seq_len, ws)
        pk.paged_attention_multi_query(q2, cu, 2, t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                       w.scale, out=out2, max_seq_len=w.max_seq_len, workspace=ws2)

    step()
    torch.cuda.synchronize()
    eager, eager2 = out.clone(), out2.clone()
    g = _capture(step)
    out.zero_()
    out2.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager) and torch.equal(out2, eager2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager) and torch.equal(out2, eager2)
    assert pk.pk_get_device_error() == 0


def test_prompt_chunk_replays_in_a_cuda_graph():
    # The prefill kernel (two query tiles per CTA) under capture.
    lens = [300, 1111]
    w = W.custom(41, lens, 16, 2, 128, 16)
    t = W.make_tensors(w, DEV)
    qlens = [200, 513]
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)).to(DEV)
    gen = torch.Generator(device=DEV).manual_seed(7)
    q = torch.randn(sum(qlens), 16, 128, generator=gen, device=DEV).to(torch.bfloat16)
    out = torch.empty_like(q)

    def chunk():
        pk.paged_attention_multi_query(q, cu, max(qlens), t["k_cache"], t["v_cache"], t["block_tables"],
                                       t["seq_lens"], w.scale, out=out, max_seq_len=w.max_seq_len)

    chunk()
    torch.cuda.synchronize()
    eager = out.clone()
    g = _capture(chunk)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert pk.pk_get_device_error() == 0
