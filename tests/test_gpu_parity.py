"""GPU parity: every workload's decode step through the C ABI against the
float64 oracle on the same seeded inputs.

Every workload, the Llama-3-70B-shaped batch and the long-context batch
included, runs at full size in the launch configuration the bench times, and
its output is compared with the oracle element by element over every
sequence; seeds 1 and 2 repeat that on every workload.  The cache writes are
checked bit for bit over the whole pool.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_122_gb300 import workloads as W
from paritylib import assert_close, gpu_step, oracle_step, pre_step_host, host_bits

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run(name, seed, out_dtype):
    w = W.get(name, seed)
    t = W.make_tensors(w, DEV)
    pre = pre_step_host(t)
    out = gpu_step(w, t, out_dtype)
    torch.cuda.synchronize()
    ref, kc, vc = oracle_step(w, pre)
    g = out.float().cpu().numpy()
    err = assert_close(g, ref, out_dtype == torch.bfloat16, f"{name} seed {seed}")
    # The caches after the step equal the oracle's, bit for bit, over the whole pool.
    assert np.array_equal(host_bits(t["k_cache"]), kc)
    assert np.array_equal(host_bits(t["v_cache"]), vc)
    import paged_kv_cache_122_gb300 as pk
    assert pk.pk_get_device_error() == 0
    return err


ALL = ["tiny", "l3-8b", "l3-70b", "long", "prefix-b8", "prefix-b16", "prefix-b32"]


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("name", ALL)
def test_full_parity(name, out_dtype):
    _run(name, 0, out_dtype)


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("name", ALL)
def test_full_parity_more_seeds(name, seed):
    _run(name, seed, torch.bfloat16 if seed == 1 else torch.float32)


@pytest.mark.parametrize("name", ["tiny", "prefix-b8", "prefix-b32"])
def test_gather_is_bit_exact(name):
    import paged_kv_cache_122_gb300 as pk
    w = W.get(name, 0)
    t = W.make_tensors(w, DEV)
    ok, ov, cu = pk.pk_gather_kv(t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"], w.seq_lens)
    kb, vb = host_bits(t["k_cache"]), host_bits(t["v_cache"])
    gk, gv = host_bits(ok), host_bits(ov)
    cu = cu.cpu().numpy()
    for s in range(w.num_seqs):
        L = int(w.seq_lens[s])
        for h in range(w.num_kv_heads):
            assert np.array_equal(gk[cu[s]:cu[s] + L, h], oracle.gather_sequence(kb, w.block_tables[s], L, w.block_size, h))
            assert np.array_equal(gv[cu[s]:cu[s] + L, h], oracle.gather_sequence(vb, w.block_tables[s], L, w.block_size, h))
    assert pk.pk_get_device_error() == 0
