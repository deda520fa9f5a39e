"""Helpers shared by the GPU parity tests: run a decode step through the C ABI
and the same step through the oracle, and compare.

Tolerances (attention against the float64 oracle):
* fp32 output: max-abs <= 1e-2 and mean-abs <= 1e-3.
* bf16 output: the kernel rounds its fp32 result to nearest-even bf16, which
  adds up to half a bf16 ulp of the value; so each element may differ by
  1e-2 + half_ulp(|ref|), and the mean-abs bound stays 1e-3.
Cache writes, block copies and the gather are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_122_gb300 as pk
from paged_kv_cache_122_gb300 import workloads as W

MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126)
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def assert_close(gpu: np.ndarray, ref: np.ndarray, bf16_out: bool, what: str = ""):
    gpu = np.asarray(gpu, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    tol = MAX_ABS + (half_ulp_bf16(ref) if bf16_out else 0.0)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert np.all(err <= tol), (f"{what}: max-abs {err.max():.3e} at {worst} "
                                f"(gpu {gpu[worst]:.6f}, ref {ref[worst]:.6f}, tol {tol if np.isscalar(tol) else tol[worst]:.3e})")
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def host_bits(t):
    return W.bits(t)


def gpu_step(w: W.Workload, t: dict, out_dtype=torch.bfloat16, max_seq_len=None):
    """copy_blocks -> reshape_and_cache -> paged_attention_decode, in place on t."""
    if w.copy_pairs.shape[0]:
        pk.copy_blocks(t["k_cache"], t["v_cache"], t["copy_pairs"])
    if w.num_new_tokens:
        pk.reshape_and_cache(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    return pk.paged_attention_decode(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                     w.scale, w.block_size, out_dtype=out_dtype,
                                     max_seq_len=max_seq_len if max_seq_len is not None else w.max_seq_len)


def oracle_step(w: W.Workload, pre: dict, seqs=None):
    """The same step in float64 on host copies of the pre-step inputs."""
    kc, vc = pre["k_cache"], pre["v_cache"]
    if w.copy_pairs.shape[0]:
        kc, vc = oracle.copy_blocks(kc, vc, w.copy_pairs.tolist())
    if w.num_new_tokens:
        kc, vc = oracle.reshape_and_cache(pre["k_new"], pre["v_new"], kc, vc, w.slot_mapping.tolist(),
                                          w.block_size)
    out = oracle.paged_decode_attention(pre["q"], kc, vc, w.block_tables, w.seq_lens, w.scale,
                                        w.block_size, seqs=seqs)
    return out, kc, vc


def pre_step_host(t: dict) -> dict:
    return {k: host_bits(t[k]) for k in ("q", "k_new", "v_new", "k_cache", "v_cache")}
