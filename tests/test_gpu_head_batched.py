"""GPU parity of the head-batched tensor-core kernel (8 KV heads, tiles of 16
tokens x all heads) against the float64 oracle: every group size and head dim
it serves, both block sizes, lengths around tile boundaries, batches with fewer
tiles than CTAs, batches where many sequences are cut across CTAs and merged,
and a workspace full of stale bytes (the merge tickets are tagged per call)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import assert_close, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _tensor_cores():
    prev = pk.pk_set_decode_path("tensor_core_head_batched")
    yield
    pk.pk_set_decode_path(prev)


def _run(w, out_dtype=torch.float32, workspace=None):
    t = W.make_tensors(w, DEV)
    out = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], w.scale,
                                    w.block_size, out_dtype=out_dtype, max_seq_len=w.max_seq_len, workspace=workspace)
    ref = oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                        w.block_tables, w.seq_lens, w.scale, w.block_size)
    return out, ref


@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_groups_dims_blocks(G, D, B):
    w = W.custom(11, [0, 1, 15, 16, 17, 31, 33, 250, 1000, 2049], 8 * G, 8, D, B)
    out, ref = _run(w)
    assert_close(out.cpu().numpy(), ref, False, f"G={G} D={D} B={B}")
    assert torch.all(out[0] == 0)
    assert pk.pk_get_device_error() == 0


@pytest.mark.parametrize("lens", [[5], [300], [16, 16, 16], [7, 40, 100]])
def test_fewer_tiles_than_ctas(lens):
    w = W.custom(12, lens, 64, 8, 128, 16)
    out, ref = _run(w, torch.bfloat16)
    assert_close(out.float().cpu().numpy(), ref, True, f"lens={lens}")


def test_many_cut_sequences_merge():
    # 40 sequences of ~3000 tokens: ~7,500 tiles over the CTAs, so most CTA
    # boundaries cut a sequence; one very long sequence spans many CTAs.
    rng = np.random.default_rng(13)
    lens = list(rng.integers(2500, 3500, size=40)) + [60000]
    w = W.custom(13, lens, 32, 8, 128, 16)
    out, ref = _run(w)
    assert_close(out.cpu().numpy(), ref, False, "cuts")
    assert pk.pk_get_device_error() == 0


def test_stale_workspace_and_repeated_calls():
    w = W.custom(14, [900, 4000, 17, 2500], 64, 8, 128, 16)
    nbytes = pk.pk_decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.max_seq_len)
    g = torch.Generator(device=DEV).manual_seed(5)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=DEV, generator=g)
    t = W.make_tensors(w, DEV)
    ref = oracle.paged_decode_attention(host_bits(t["q"]), host_bits(t["k_cache"]), host_bits(t["v_cache"]),
                                        w.block_tables, w.seq_lens, w.scale, w.block_size)
    outs = []
    for _ in range(3):
        out = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                        w.scale, w.block_size, out_dtype=torch.float32, max_seq_len=w.max_seq_len,
                                        workspace=ws)
        outs.append(out.clone())
        assert_close(out.cpu().numpy(), ref, False, "stale workspace")
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_matches_per_head_kernel():
    w = W.get("l3-70b", 0)
    t = W.make_tensors(w, DEV)
    a = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], w.scale,
                                  w.block_size, out_dtype=torch.float32, max_seq_len=w.max_seq_len).clone()
    pk.pk_set_decode_path("tensor_core")
    b = pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], w.scale,
                                  w.block_size, out_dtype=torch.float32, max_seq_len=w.max_seq_len)
    assert (a - b).abs().max().item() < 5e-3
