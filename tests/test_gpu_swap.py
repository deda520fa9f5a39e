"""Block swap between the device pool and a pinned host pool, one launch per
direction, bit for bit against the oracle; a bad pair is skipped and
reported (the kernel checks ids before any access)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import _native
from paritylib import host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pool(g, P, B, Hkv, D, pinned):
    x = torch.randn(P, B, Hkv, D, generator=g).to(torch.bfloat16)
    return x.pin_memory() if pinned else x.to(DEV)


@pytest.mark.parametrize("B,Hkv,D", [(16, 8, 128), (8, 2, 64), (32, 4, 128)])
def test_swap_out_and_in_match_oracle(B, Hkv, D):
    g = torch.Generator().manual_seed(B + D)
    dk, dv = _pool(g, 48, B, Hkv, D, False), _pool(g, 48, B, Hkv, D, False)
    hk, hv = _pool(g, 20, B, Hkv, D, True), _pool(g, 20, B, Hkv, D, True)
    out_pairs = np.array([[3, 0], [17, 4], [40, 19], [5, 7]], dtype=np.int64)
    pre = (host_bits(dk), host_bits(dv), hk.view(torch.int16).numpy().view(np.uint16).copy(),
           hv.view(torch.int16).numpy().view(np.uint16).copy())
    pk.swap_blocks(hk, hv, dk, dv, torch.from_numpy(out_pairs).to(DEV))          # swap out
    torch.cuda.synchronize()
    want_k, want_v = oracle.swap_blocks(pre[0], pre[1], pre[2], pre[3], out_pairs.tolist())
    assert np.array_equal(hk.view(torch.int16).numpy().view(np.uint16), want_k)
    assert np.array_equal(hv.view(torch.int16).numpy().view(np.uint16), want_v)
    in_pairs = np.array([[0, 30], [4, 31], [19, 2], [7, 47]], dtype=np.int64)
    pk.swap_blocks(dk, dv, hk, hv, torch.from_numpy(in_pairs).to(DEV))           # swap in
    torch.cuda.synchronize()
    want_dk, want_dv = oracle.swap_blocks(want_k, want_v, pre[0], pre[1], in_pairs.tolist())
    assert np.array_equal(host_bits(dk), want_dk) and np.array_equal(host_bits(dv), want_dv)
    # Round trip: the swapped-in copies equal the blocks that were swapped out.
    for (src, mid), (mid2, dst) in zip(out_pairs.tolist(), in_pairs.tolist()):
        assert mid == mid2 and torch.equal(dk[dst], torch.from_numpy(pre[0][src]).view(torch.bfloat16).to(DEV))
    assert pk.pk_get_device_error() == 0


def test_swap_device_to_device_equals_copy_blocks_and_bad_pair_is_skipped():
    g = torch.Generator().manual_seed(3)
    a_k, a_v = _pool(g, 16, 16, 8, 128, False), _pool(g, 16, 16, 8, 128, False)
    b_k, b_v = _pool(g, 8, 16, 8, 128, False), _pool(g, 8, 16, 8, 128, False)
    before = host_bits(b_k)
    pairs = torch.tensor([[1, 2], [15, 7], [3, 8]], dtype=torch.int64, device=DEV)   # last dst is outside b
    pk.swap_blocks(b_k, b_v, a_k, a_v, pairs)
    assert pk.pk_get_device_error() & _native.DEVERR_PAIR
    assert torch.equal(b_k[2], a_k[1]) and torch.equal(b_v[7], a_v[15])
    keep = [i for i in range(8) if i not in (2, 7)]
    assert np.array_equal(host_bits(b_k)[keep], before[keep])
