"""Multi-layer append and block copy (one launch for every layer) against the
oracle, bit for bit, per layer; and a bad per-layer pointer, which only the
GPU can see, is skipped and reported through the error word (checked before
any access: no fault)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import _native
from paritylib import host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _layers(seed, L, P, B, Hkv, D, T):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16).to(DEV)
    kc = [mk(P, B, Hkv, D) for _ in range(L)]
    vc = [mk(P, B, Hkv, D) for _ in range(L)]
    kn = [mk(T, Hkv, D) for _ in range(L)]
    vn = [mk(T, Hkv, D) for _ in range(L)]
    return kc, vc, kn, vn


@pytest.mark.parametrize("B,D,Hkv", [(16, 128, 8), (8, 64, 2), (32, 128, 4)])
def test_layers_match_oracle_per_layer(B, D, Hkv):
    L, P, T = 5, 40, 37
    kc, vc, kn, vn = _layers(1, L, P, B, Hkv, D, T)
    rng = np.random.default_rng(2)
    slots = rng.choice(P * B, size=T, replace=False).astype(np.int64)
    slots[[3, 17]] = -1                                   # padding tokens write nothing
    src = rng.choice(P // 2, size=6, replace=False)
    dst = P // 2 + rng.choice(P // 2, size=6, replace=False)
    pairs = np.stack([src, dst], 1).astype(np.int64)
    pre = [(host_bits(kc[l]), host_bits(vc[l]), host_bits(kn[l]), host_bits(vn[l])) for l in range(L)]
    lk, lv = pk.LayerPointers(kc), pk.LayerPointers(vc)
    pk.pk_copy_blocks_layers(lk, lv, torch.from_numpy(pairs).to(DEV))
    pk.pk_reshape_and_cache_layers(kn, vn, lk, lv, torch.from_numpy(slots).to(DEV))
    torch.cuda.synchronize()
    for l in range(L):
        k0, v0, knb, vnb = pre[l]
        k1, v1 = oracle.copy_blocks(k0, v0, pairs.tolist())
        k2, v2 = oracle.reshape_and_cache(knb, vnb, k1, v1, slots.tolist(), B)
        assert np.array_equal(host_bits(kc[l]), k2), f"layer {l} K"
        assert np.array_equal(host_bits(vc[l]), v2), f"layer {l} V"
    assert pk.pk_get_device_error() == 0


def test_layers_equal_one_layer_calls():
    L, P, B, Hkv, D, T = 3, 24, 16, 8, 128, 20
    kc, vc, kn, vn = _layers(5, L, P, B, Hkv, D, T)
    kc2 = [x.clone() for x in kc]
    vc2 = [x.clone() for x in vc]
    slots = torch.arange(T, dtype=torch.int64, device=DEV) * 7
    pairs = torch.tensor([[0, 20], [3, 21]], dtype=torch.int64, device=DEV)
    pk.pk_copy_blocks_layers(kc, vc, pairs)
    pk.pk_reshape_and_cache_layers(kn, vn, kc, vc, slots)
    for l in range(L):
        pk.copy_blocks(kc2[l], vc2[l], pairs)
        pk.reshape_and_cache(kn[l], vn[l], kc2[l], vc2[l], slots)
    torch.cuda.synchronize()
    for l in range(L):
        assert torch.equal(kc[l], kc2[l]) and torch.equal(vc[l], vc2[l])


def test_bad_layer_pointer_is_skipped_and_reported():
    L, P, B, Hkv, D, T = 4, 16, 16, 2, 64, 8
    kc, vc, kn, vn = _layers(7, L, P, B, Hkv, D, T)
    before = [host_bits(x) for x in kc]
    lk, lv = pk.LayerPointers(kc), pk.LayerPointers(vc)
    bad = pk.LayerPointers(kc)
    bad.ptrs[1] = 0                                       # NULL for layer 1
    bad.ptrs[2] = kc[2].data_ptr() + 2                    # not 16-byte aligned for layer 2
    slots = torch.arange(T, dtype=torch.int64, device=DEV)
    assert pk.pk_get_device_error() == 0
    pk.pk_reshape_and_cache_layers(kn, vn, bad, lv, slots)
    code = pk.pk_get_device_error()
    assert code & _native.DEVERR_POINTER
    # Layers 1 and 2 are skipped entirely (their K is untouched); 0 and 3 are written.
    for l in (1, 2):
        assert np.array_equal(host_bits(kc[l]), before[l])
    for l in (0, 3):
        assert torch.equal(kc[l].view(-1, Hkv, D)[:T], kn[l])
    # Block copies: a NULL V cache pointer for layer 3.
    badv = pk.LayerPointers(vc)
    badv.ptrs[3] = 0
    pk.pk_copy_blocks_layers(lk, badv, torch.tensor([[0, 9]], dtype=torch.int64, device=DEV))
    assert pk.pk_get_device_error() & _native.DEVERR_POINTER
    assert torch.equal(kc[3][9], kc[3][0])
