"""Decode-step benchmark: paged decode attention HBM GB/s on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload l3-70b] [--impl ours|reference]

One step = one pass of the whole hot path over one batch: reshape_and_cache of
the step's new tokens, copy_blocks of its copy-on-write pairs (prefix
workloads only), then paged_attention_decode.  ``value`` is the step's useful
bytes (attended K/V + Q + O + appended K/V read and written + copied blocks)
over its device time, all inputs resident in HBM.  When a step's K/V is at
least twice the L2 (the Llama-3-70B batch reads 1.1 GB, 8.6x the L2), the K
timed steps run back to back as in serving, alternating between two separate
copies of the cache so that no step finds the previous step's reads in L2,
with one pair of CUDA events around them; smaller workloads flush L2 before
each step and time each step with its own events.  ``isolated_call`` adds the
decode call timed alone with L2 flushed.  ``e2e`` is the same metric
through the public API with per-step inputs (q, new K/V, slots, tables,
lengths) copied from pinned host memory and the output copied back inside the
timed region; the KV cache itself stays resident, as it does in serving.

Multi-GPU: decode shards by sequence with no exchange, so each rank runs its
own batch (seed + rank); ``value`` sums all ranks' bytes over the slowest
rank's time (weak scaling).  ``--impl reference`` times the float64 CPU oracle
on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attn achieved HBM GB/s & % of GB300 peak; decode tokens/s per layer"
WORKLOAD_DESC = {
    "l3-70b": "Llama-3-70B-shaped serving batch: 256 seqs, 64 q / 8 kv heads (GQA 8), head_dim 128, "
              "block_size 16, seq_lens lognormal(median 600, sigma 1) clipped to [16, 8192] + 1 appended "
              "token each, shuffled pool (needed + 10%)",
    "l3-8b": "Llama-3-8B-shaped decode layer: 64 seqs, 32 q / 8 kv heads, head_dim 128, block_size 16, "
             "seq_lens U[512, 2048]",
    "long": "Long-context split-K: 8 seqs, 32 q / 8 kv heads, head_dim 128, block_size 16, seq_lens U[32768, 131072]",
    "tiny": "Tiny: 4 seqs, 8 q / 8 kv heads, head_dim 64, block_size 16, seq_lens U[1, 128] + 1",
    "prefix-b8": "Prefix sharing + CoW, block_size 8",
    "prefix-b16": "Prefix sharing + CoW, block_size 16",
    "prefix-b32": "Prefix sharing + CoW, block_size 32",
}
# Steps per chunk of the end-to-end loop (one cross-stream wait per chunk).
E2E_CHUNK = 4
# Kernel source files whose change invalidates the recorded ncu traffic.
DOMINANT_SOURCES = ["paged_kv_cache_122_gb300/csrc/decode_tc.cu", "paged_kv_cache_122_gb300/csrc/sm100.cuh",
                    "paged_kv_cache_122_gb300/csrc/decode.cuh", "paged_kv_cache_122_gb300/csrc/decode_api.cu",
                    "paged_kv_cache_122_gb300/csrc/block_scan.cuh"]
# DRAM bytes per launch of the dominant kernel from one ncu capture, and the
# hash of its sources at that time (profiles/ holds the summary).
RECORDED_TRAFFIC = {"sources_sha1": "66e29afac64e0ca3c432b97dec24cb0ccb78e151", "bytes_per_launch": 1125091840, "workload": "l3-70b"}


def sources_sha1() -> str:
    h = hashlib.sha1()
    for rel in DOMINANT_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# Clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3][1:]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm)
# ---------------------------------------------------------------------------

CPU_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
try:
    os.sched_setaffinity(0, {{sorted(os.sched_getaffinity(0))[0]}})
except Exception:
    pass
import oracle
from paged_kv_cache_122_gb300 import workloads as W, metrics as M
w = W.get({workload!r}, {seed})
sel = list(range(min({nseq}, w.num_seqs)))
wc = W.custom({seed}, w.seq_lens[sel], w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
t = W.make_tensors(wc, "cpu")
q, kc, vc = (W.bits(t[k]) for k in ("q", "k_cache", "v_cache"))
nbytes = M.useful_bytes(wc)["attention"]
times = []
t_end = time.perf_counter() + {budget}
while True:
    t0 = time.perf_counter()
    oracle.paged_decode_attention(q, kc, vc, wc.block_tables, wc.seq_lens, wc.scale, wc.block_size)
    times.append(time.perf_counter() - t0)
    if time.perf_counter() > t_end or len(times) >= {max_reps}:
        break
print(json.dumps({{"times": times, "bytes": nbytes, "seqs": len(sel), "tokens": int(wc.seq_lens.sum())}}))
"""


BM_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
try:
    os.sched_setaffinity(0, {{sorted(os.sched_getaffinity(0))[0]}})
except Exception:
    pass
from paged_kv_cache_122_gb300 import BlockManager, workloads as W
w = W.get({workload!r}, {seed})
N, B, K = w.num_seqs, w.block_size, {steps}
lens = [int(x) for x in w.seq_lens]
MB = -(-(max(lens) + K) // B)
ids = np.arange(N, dtype=np.int64)
# Every sequence gets private blocks here (no prefix sharing): size the pool for that.
POOL = sum(-(-(L + K) // B) for L in lens) + N
def native():
    bm = BlockManager(POOL, B)
    for s in range(N):
        bm.add_sequence(s)
        bm.append_slots(np.full(lens[s], s, dtype=np.int64))
    tables = np.empty((N, MB), dtype=np.int32); sl = np.empty(N, dtype=np.int32)
    ts = []
    for _ in range(K):
        t0 = time.perf_counter()
        bm.append_slots(ids); bm.take_copies(); bm.export(ids, MB, tables, sl)
        ts.append(time.perf_counter() - t0)
    return ts
def reference():
    import oracle
    bm = oracle.CowBlockManager(POOL, B)
    for s in range(N):
        bm.new_sequence(str(s))
        for _ in range(lens[s]):
            bm.append_slot(str(s))
    ts = []
    for _ in range(K):
        t0 = time.perf_counter()
        slots = [bm.append_slot(str(s)) for s in range(N)]
        pairs = bm.take_copies()
        tables = np.full((N, MB), -1, dtype=np.int32)
        for s in range(N):
            tb = bm.tables[str(s)]
            tables[s, :len(tb)] = tb
        sl = np.array([bm.lengths[str(s)] for s in range(N)], dtype=np.int32)
        ts.append(time.perf_counter() - t0)
    return ts
out = {{"native": native()}}
if {with_oracle}:
    out["oracle"] = reference()
print(json.dumps(out))
"""


# All host cores: the same oracle over the same sample, one sequence per work
# item, in a pool of single-threaded worker processes started with spawn (the
# subprocess that owns the pool never touches the GPU).  The sample's arrays are
# written once to a temporary folder and memory-mapped by every worker.
POOL_SNIPPET = r"""
import json, os, sys, time, tempfile, shutil
sys.path.insert(0, {root!r})
import numpy as np
import multiprocessing as mp
import bench
from paged_kv_cache_122_gb300 import workloads as W, metrics as M
w = W.get({workload!r}, {seed})
sel = list(range(min({nseq}, w.num_seqs)))
wc = W.custom({seed}, w.seq_lens[sel], w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
t = W.make_tensors(wc, "cpu")
folder = tempfile.mkdtemp(prefix="pk_oracle_pool_")
try:
    for name, arr in (("q", W.bits(t["q"])), ("k", W.bits(t["k_cache"])), ("v", W.bits(t["v_cache"])),
                      ("bt", np.asarray(wc.block_tables)), ("lens", np.asarray(wc.seq_lens))):
        np.save(os.path.join(folder, name + ".npy"), arr)
    del t
    cores = len(os.sched_getaffinity(0))
    order = sorted(range(len(sel)), key=lambda s: -int(wc.seq_lens[s]))     # longest first
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=bench._pool_init,
                  initargs=(folder, float(wc.scale), int(wc.block_size))) as pool:
        list(pool.imap_unordered(bench._pool_task, order))                   # warm-up pass
        times = []
        t_end = time.perf_counter() + {budget}
        while True:
            t0 = time.perf_counter()
            list(pool.imap_unordered(bench._pool_task, order))
            times.append(time.perf_counter() - t0)
            if time.perf_counter() > t_end or len(times) >= 1000:
                break
finally:
    shutil.rmtree(folder, ignore_errors=True)
print(json.dumps({{"times": times, "bytes": M.useful_bytes(wc)["attention"], "seqs": len(sel),
                  "tokens": int(wc.seq_lens.sum()), "cores": cores}}))
"""

_POOL = None


def _pool_init(folder, scale, block_size):
    """Worker start-up of the all-cores oracle pass: map the sample's arrays."""
    global _POOL
    import numpy as np

    def ld(name, mode=None):
        return np.load(os.path.join(folder, name + ".npy"), mmap_mode=mode)
    _POOL = (ld("q"), ld("k", "r"), ld("v", "r"), ld("bt"), ld("lens"), scale, block_size)


def _pool_task(s):
    """One work item of the all-cores oracle pass: sequence ``s``."""
    import oracle
    q, kc, vc, bt, lens, scale, block_size = _POOL
    oracle.paged_decode_attention(q[s:s + 1], kc, vc, bt[s:s + 1], lens[s:s + 1], scale, block_size)
    return s


def run_cpu_oracle_pool(workload: str, seed: int, nseq: int, budget_s: float, timeout_s: float = 240.0):
    """The oracle over the sample on every host core (one process per core)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = POOL_SNIPPET.format(root=ROOT, workload=workload, seed=seed, nseq=nseq, budget=budget_s)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=timeout_s)
    if res.returncode != 0:
        raise RuntimeError(f"all-cores oracle run failed:\n{res.stderr[-2000:]}")
    return json.loads(res.stdout.strip().splitlines()[-1])


def run_block_manager(workload: str, seed: int, steps: int, with_oracle: bool):
    """Host block-manager time of one decode step (append every sequence, take
    the copy pairs, export tables and lengths), on one pinned host core."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    code = BM_SNIPPET.format(root=ROOT, workload=workload, seed=seed, steps=steps, with_oracle=with_oracle)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if res.returncode != 0:
        raise RuntimeError(f"block-manager timing failed:\n{res.stderr[-2000:]}")
    return json.loads(res.stdout.strip().splitlines()[-1])


def run_cpu_oracle(workload: str, seed: int, nseq: int, budget_s: float, max_reps: int = 1000):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = CPU_SNIPPET.format(root=ROOT, workload=workload, seed=seed, nseq=nseq, budget=budget_s,
                              max_reps=max_reps)
    cmd = [sys.executable, "-c", code]
    res = subprocess.run(cmd, capture_output=True, text=True, env=env)
    if res.returncode != 0:
        raise RuntimeError(f"CPU oracle run failed:\n{res.stderr[-2000:]}")
    return json.loads(res.stdout.strip().splitlines()[-1])


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return ws, rank, local


def aggregate_over_ranks(device_ms: float, e2e_ms: float, step_bytes: float, device):
    """Whole-job figures over the ranks: the slowest rank's times and the sum
    of every rank's bytes (each rank runs its own batch)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([device_ms, e2e_ms], dtype=torch.float64, device=device)
    b = torch.tensor([step_bytes], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t[0]), float(t[1]), float(b[0])


def contiguous_tables(w):
    """Block tables of the same lengths with every sequence's blocks back to
    back (bt[s, i] = base_s + i): the paging-overhead control layout.  None
    when the pool is too small for it (a workload whose sequences share
    blocks holds fewer blocks than its sequences' lengths add up to)."""
    import numpy as np
    bt = np.full_like(w.block_tables, -1)
    base = 0
    for s in range(w.num_seqs):
        nb = -(-int(w.seq_lens[s]) // w.block_size)
        if base + nb > w.num_blocks:
            return None
        bt[s, :nb] = np.arange(base, base + nb, dtype=np.int32)
        base += nb
    return bt


class L2Flush:
    """Leaves L2 cold and clean before a timed call: a 256 MiB write (twice
    the 129 MB L2) evicts whatever the call could reuse, then a read of
    another 256 MiB buffer evicts the dirty lines that write left, so that
    their write-back to HBM happens here, outside the timed region, and not
    inside the next timed call."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.view(-1, 64).amax(dim=0)      # a plain read of the second buffer


def time_decode(fn, steps, flush, stream):
    """Mean device time (ms) of fn() over `steps` calls, L2 flushed before each."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def workload_report(name, seed, dev, steps, flush, peak):
    """Decode-only GB/s of another workload (context for the bench line)."""
    import torch
    import paged_kv_cache_122_gb300 as pk
    from paged_kv_cache_122_gb300 import metrics as M, workloads as W
    w = W.get(name, seed)
    t = W.make_tensors(w, dev)
    ub = M.useful_bytes(w)
    ws = pk.new_workspace((pk.pk_decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                        w.max_seq_len)), dev)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
    if w.copy_pairs.shape[0]:
        pk.copy_blocks(t["k_cache"], t["v_cache"], t["copy_pairs"])
    if w.num_new_tokens:
        pk.reshape_and_cache(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])

    def fn():
        pk.pk_paged_attention_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                     w.scale, w.block_size, w.max_seq_len, ws)
    for _ in range(3):
        fn()
    stream = torch.cuda.current_stream(dev)
    ms = time_decode(fn, steps, flush, stream)
    gbs = ub["attention"] / (ms * 1e-3) / 1e9
    rep = {"decode_ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
           "tokens_per_s_per_layer": round(w.num_seqs / (ms * 1e-3), 1),
           "timing": "one call at a time, L2 flushed before each"}
    if ub["kv_unique"] >= torch.cuda.get_device_properties(dev).L2_cache_size:
        # Back to back, alternating between two copies of the cache (as the
        # bench line's steps run): each call's K/V is larger than L2, and the
        # call before it read the other copy, so nothing it reads is left in
        # L2 from its previous use.
        kc2, vc2 = t["k_cache"].clone(), t["v_cache"].clone()
        pairs = [(t["k_cache"], t["v_cache"]), (kc2, vc2)]

        def fn2(i):
            pk.pk_paged_attention_decode(out, t["q"], pairs[i & 1][0], pairs[i & 1][1], t["block_tables"],
                                         t["seq_lens"], w.scale, w.block_size, w.max_seq_len, ws)
        for i in range(4):
            fn2(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n2 = max(steps, 100)
        a.record(stream)
        for i in range(n2):
            fn2(i)
        b.record(stream)
        torch.cuda.synchronize()
        ms2 = a.elapsed_time(b) / n2
        gbs2 = ub["attention"] / (ms2 * 1e-3) / 1e9
        rep["back_to_back"] = {"decode_ms": round(ms2, 4), "gbs": round(gbs2, 1), "frac": round(gbs2 / peak, 4),
                               "tokens_per_s_per_layer": round(w.num_seqs / (ms2 * 1e-3), 1),
                               "timing": f"{n2} calls back to back alternating between two copies of the cache"}
        del kc2, vc2, pairs
    # The cache writes alone (each call repeats the same copies and writes, so
    # it is idempotent); GB/s of bytes read plus written.
    if w.copy_pairs.shape[0]:
        cms = time_decode(lambda: pk.copy_blocks(t["k_cache"], t["v_cache"], t["copy_pairs"]), steps, flush, stream)
        rep["copy_blocks_us"] = round(cms * 1e3, 2)
        rep["copy_blocks_gbs"] = round(ub["copies"] / (cms * 1e-3) / 1e9, 1)
    if w.num_new_tokens:
        ams = time_decode(lambda: pk.reshape_and_cache(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"],
                                                       t["slot_mapping"]), steps, flush, stream)
        rep["reshape_and_cache_us"] = round(ams * 1e3, 2)
        rep["reshape_and_cache_gbs"] = round(ub["append"] / (ams * 1e-3) / 1e9, 1)
    if ub["kv_unique"] != ub["kv"]:
        uniq = (ub["attention"] - ub["kv"] + ub["kv_unique"]) / (ms * 1e-3) / 1e9
        rep["gbs_unique_bytes"] = round(uniq, 1)
    del t, ws, out
    torch.cuda.empty_cache()
    return rep


def swap_report(w, t, dev, nblocks=1024, reps=5):
    """Swap `nblocks` random blocks of the pool out to a pinned host pool and
    back in: one pk_swap_blocks launch per direction, against one
    cudaMemcpyAsync per block and tensor (what "many small transfers" means)."""
    import torch
    import paged_kv_cache_122_gb300 as pk
    import numpy as np
    rng = np.random.default_rng(7)
    src = rng.choice(w.num_blocks, size=nblocks, replace=False)
    pairs_out = torch.from_numpy(np.stack([src, np.arange(nblocks)], 1).astype(np.int64)).to(dev)
    pairs_in = torch.from_numpy(np.stack([np.arange(nblocks), src], 1).astype(np.int64)).to(dev)
    shape = (nblocks,) + tuple(t["k_cache"].shape[1:])
    hk = torch.empty(shape, dtype=torch.bfloat16, pin_memory=True)
    hv = torch.empty(shape, dtype=torch.bfloat16, pin_memory=True)
    stream = torch.cuda.current_stream(dev)
    nbytes = 2 * nblocks * hk[0].numel() * 2

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream); fn(); b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    kc, vc = t["k_cache"], t["v_cache"]
    out_ms = timed(lambda: pk.swap_blocks(hk, hv, kc, vc, pairs_out))
    in_ms = timed(lambda: pk.swap_blocks(kc, vc, hk, hv, pairs_in))
    src_l = src.tolist()

    def per_block_out():
        for i, b in enumerate(src_l):
            hk[i].copy_(kc[b], non_blocking=True)
            hv[i].copy_(vc[b], non_blocking=True)

    def per_block_in():
        for i, b in enumerate(src_l):
            kc[b].copy_(hk[i], non_blocking=True)
            vc[b].copy_(hv[i], non_blocking=True)
    pb_out = timed(per_block_out)
    pb_in = timed(per_block_in)
    assert pk.pk_get_device_error(dev) == 0
    gb = lambda ms: round(nbytes / (ms * 1e-3) / 1e9, 1)
    return {"blocks": nblocks, "bytes": nbytes,
            "out_one_launch_gbs": gb(out_ms), "in_one_launch_gbs": gb(in_ms),
            "out_per_block_copies_gbs": gb(pb_out), "in_per_block_copies_gbs": gb(pb_in),
            "what": f"{nblocks} random blocks (K+V, {hk[0].numel() * 4} B each) device pool <-> pinned "
                    "host pool; one pk_swap_blocks launch per direction vs one cudaMemcpyAsync per block "
                    "and tensor (median of 5)"}


def multi_query_report(w, t, dev, flush, peak, q_per_seq=2, steps=20):
    """Speculative-verification shape: q_per_seq newest tokens of every
    sequence of the batch as causal queries over the paged cache (one MMA
    column per query token and query head: G * q <= 16)."""
    import torch
    import paged_kv_cache_122_gb300 as pk
    from paged_kv_cache_122_gb300 import metrics as M
    N = w.num_seqs
    cu = torch.arange(N + 1, dtype=torch.int32, device=dev) * q_per_seq
    g = torch.Generator(device=dev).manual_seed(99)
    q = torch.randn(N * q_per_seq, w.num_heads, w.head_dim, generator=g, device=dev, dtype=torch.bfloat16)
    out = torch.empty_like(q)

    def fn():
        pk.paged_attention_multi_query(q, cu, q_per_seq, t["k_cache"], t["v_cache"], t["block_tables"],
                                       t["seq_lens"], w.scale, out=out, max_seq_len=w.max_seq_len)
    for _ in range(3):
        fn()
    ms = time_decode(fn, steps, flush, torch.cuda.current_stream(dev))
    assert pk.pk_get_device_error(dev) == 0
    ub = M.useful_bytes(w)
    nbytes = ub["kv"] + q_per_seq * ub["q_o"]
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"q_per_seq": q_per_seq, "ms": round(ms, 4), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
            "query_tokens_per_s_per_layer": round(N * q_per_seq / (ms * 1e-3), 1),
            "what": f"{N} sequences x {q_per_seq} newest tokens as causal queries (G={w.group}), "
                    "paged_attention_multi_query, L2 flushed between calls"}


def prefill_report(dev, flush, steps=10, N=16, prior=4096, chunk=512):
    """Chunked prefill: `chunk` new prompt tokens per sequence (causal among
    themselves) over `prior` earlier tokens, Llama-3-70B heads (64 q / 8 kv,
    d 128, block 16); FLOPs count only the visible (query, key) pairs."""
    import torch
    import paged_kv_cache_122_gb300 as pk
    from paged_kv_cache_122_gb300 import workloads as W
    L = prior + chunk
    w = W.custom(3, [L] * N, 64, 8, 128, 16)
    t = W.make_tensors(w, dev)
    cu = torch.arange(N + 1, dtype=torch.int32, device=dev) * chunk
    g = torch.Generator(device=dev).manual_seed(5)
    q = torch.randn(N * chunk, 64, 128, generator=g, device=dev, dtype=torch.bfloat16)
    out = torch.empty_like(q)

    def fn():
        pk.paged_attention_multi_query(q, cu, chunk, t["k_cache"], t["v_cache"], t["block_tables"], t["seq_lens"],
                                       w.scale, out=out, max_seq_len=w.max_seq_len)
    for _ in range(3):
        fn()
    ms = time_decode(fn, steps, flush, torch.cuda.current_stream(dev))
    assert pk.pk_get_device_error(dev) == 0
    visible = N * sum(prior + r + 1 for r in range(chunk))          # (query token, key) pairs
    flops = 4.0 * 128 * 64 * visible                                 # QK^T and PV, every query head
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    peak = float(peaks.get("bf16_tflops") or 0) or None
    tf = flops / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 4), "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / peak, 4) if peak else None,
            "prompt_tokens_per_s_per_layer": round(N * chunk / (ms * 1e-3), 1),
            "what": f"{N} sequences x {chunk}-token prompt chunk over {prior} earlier tokens, 64 q / 8 kv heads, "
                    "d 128, block 16; paged_attention_multi_query (two 128-row query tiles per CTA); causal FLOPs"}


def multi_layer_report(w, t, dev, layers, steps, workspace, out, peak):
    """One attention step of a `layers`-layer model (the Llama-3-70B batch has
    80): the copy-on-write copies and the append of every layer in one launch
    each, then one decode per layer over that layer's own caches.  Layer 0 is
    the workload's cache; the others are filled on the GPU (values do not
    matter for timing; parity is in the tests).  The caches (GBs per layer)
    far exceed L2, so no flush is needed."""
    import torch
    import paged_kv_cache_122_gb300 as pk
    from paged_kv_cache_122_gb300 import metrics as M
    gen = torch.Generator(device=dev).manual_seed(4321)
    kcs, vcs = [t["k_cache"]], [t["v_cache"]]
    for _ in range(layers - 1):
        kcs.append(torch.randn(t["k_cache"].shape, generator=gen, device=dev, dtype=torch.bfloat16))
        vcs.append(torch.randn(t["v_cache"].shape, generator=gen, device=dev, dtype=torch.bfloat16))
    lk, lv = pk.LayerPointers(kcs), pk.LayerPointers(vcs)
    lkn, lvn = pk.LayerPointers([t["k_new"]] * layers), pk.LayerPointers([t["v_new"]] * layers)
    stream = torch.cuda.current_stream(dev)

    def prelude():
        if w.copy_pairs.shape[0]:
            pk.pk_copy_blocks_layers(lk, lv, t["copy_pairs"])
        if w.num_new_tokens:
            pk.pk_reshape_and_cache_layers(lkn, lvn, lk, lv, t["slot_mapping"])

    def prelude_per_layer():
        for l in range(layers):
            if w.copy_pairs.shape[0]:
                pk.copy_blocks(kcs[l], vcs[l], t["copy_pairs"])
            if w.num_new_tokens:
                pk.reshape_and_cache(t["k_new"], t["v_new"], kcs[l], vcs[l], t["slot_mapping"])

    def decode_all():
        for l in range(layers):
            pk.pk_paged_attention_decode(out, t["q"], kcs[l], vcs[l], t["block_tables"], t["seq_lens"], w.scale,
                                         w.block_size, w.max_seq_len, workspace)

    prelude(); decode_all(); prelude_per_layer()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in ev:
        e[0].record(stream); prelude(); e[1].record(stream); decode_all(); e[2].record(stream)
    pl = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in pl:
        e[0].record(stream); prelude_per_layer(); e[1].record(stream)
    torch.cuda.synchronize(dev)
    assert pk.pk_get_device_error(dev) == 0
    step = statistics.median(e[0].elapsed_time(e[2]) for e in ev)
    app = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    dec = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    app_pl = statistics.median(e[0].elapsed_time(e[1]) for e in pl)
    ub = M.useful_bytes(w)
    gbs = ub["attention"] * layers / (dec * 1e-3) / 1e9
    rep = {"layers": layers, "step_ms": round(step, 3),
           "what": "copy + append of all layers in one launch each, then one decode per layer (median of "
                   f"{steps} steps; {layers} separate K/V caches of {w.num_blocks} blocks)",
           "decode_ms_per_layer": round(dec / layers, 4), "decode_gbs": round(gbs, 1),
           "decode_frac": round(gbs / peak, 4),
           "append_all_layers_one_launch_us": round(app * 1e3, 2),
           "append_per_layer_launches_us": round(app_pl * 1e3, 2),
           "tokens_per_s_all_layers": round(w.num_seqs / (step * 1e-3), 1)}
    del kcs, vcs, lk, lv
    torch.cuda.empty_cache()
    return rep


def run_ours(args):
    import torch
    import paged_kv_cache_122_gb300 as pk
    from paged_kv_cache_122_gb300 import metrics as M, workloads as W

    ws, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk.load_library()
    pk.pk_set_decode_path(args.decode_path)
    w = W.get(args.workload, args.seed + rank)
    if args.shape:
        # The workload's lengths with other head counts / head dim (kernel
        # comparisons): attention only, no appends or copies.
        H, Hkv, D = (int(x) for x in args.shape.split(":"))
        w = W.custom(args.seed + rank, w.seq_lens, H, Hkv, D, w.block_size)
    t = W.make_tensors(w, dev)
    ub = M.useful_bytes(w)
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
    ws_bytes = pk.pk_decode_workspace_bytes(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.max_seq_len)
    workspace = pk.new_workspace(ws_bytes, dev)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)

    # When a step's K/V is far larger than L2, steps run back to back as in
    # serving, with no flush: consecutive steps use two separate copies of the
    # cache (two layers of the model), so nothing a step reads was left in L2
    # by the step before.  Smaller workloads flush L2 before every step.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    stream_mode = ub["kv_unique"] >= 2 * l2_bytes
    caches = [(t["k_cache"], t["v_cache"])]
    if stream_mode:
        caches.append((t["k_cache"].clone(), t["v_cache"].clone()))

    def attend(o=out, q=t["q"], bt=t["block_tables"], sl=t["seq_lens"], c=0):
        kc, vc = caches[c % len(caches)]
        pk.pk_paged_attention_decode(o, q, kc, vc, bt, sl, w.scale, w.block_size, w.max_seq_len, workspace)

    def prelude(kn=t["k_new"], vn=t["v_new"], sm=t["slot_mapping"], c=0):
        kc, vc = caches[c % len(caches)]
        if w.copy_pairs.shape[0]:
            pk.copy_blocks(kc, vc, t["copy_pairs"])
        if w.num_new_tokens:
            pk.reshape_and_cache(kn, vn, kc, vc, sm)

    # Launches of this library per step: copy, append, then the decode kernel
    # and its merge (the merge runs when a sequence can span several CTAs /
    # partitions: > 128 tokens on tensor cores, > 512 on CUDA cores).
    max_tiles = w.num_seqs * w.num_kv_heads * ((w.max_seq_len + 127) // 128)
    tensor_core = args.decode_path.startswith("tensor_core") or \
        (args.decode_path == "auto" and max_tiles >= torch.cuda.get_device_properties(dev).multi_processor_count)
    merge = w.max_seq_len > (128 if tensor_core else 512)
    launches_per_step = (1 if w.copy_pairs.shape[0] else 0) + (1 if w.num_new_tokens else 0) + 1 + (1 if merge else 0)

    for i in range(args.warmup):
        prelude(c=i)
        attend(c=i)
    torch.cuda.synchronize(dev)
    assert pk.pk_get_device_error(dev) == 0

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    timed_launches = launches_per_step * args.steps
    with ClockSampler(local) as clocks:
        if stream_mode:
            # The K timed steps back to back, one pair of events around them;
            # then the decode call alone the same way (the roofline's launch
            # duration).
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush()
            e0.record(stream)
            for i in range(args.steps):
                prelude(c=i)
                attend(c=i)
            e1.record(stream)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for i in range(args.steps):
                attend(c=i)
            a1.record(stream)
            torch.cuda.synchronize(dev)
            total_ms = e0.elapsed_time(e1)
            attn_avg_ms = a0.elapsed_time(a1) / args.steps
            timed_launches += (1 + (1 if merge else 0)) * args.steps
        else:
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
            for i in range(args.steps):
                flush()                                       # cold, clean L2 between steps (outside the events)
                ev[i][0].record(stream)
                prelude()
                ev[i][1].record(stream)
                attend()
                ev[i][2].record(stream)
            torch.cuda.synchronize(dev)
            total_ms = sum(e[0].elapsed_time(e[2]) for e in ev)
            attn_avg_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
        if ws > 1:
            torch.distributed.barrier()
    assert pk.pk_get_device_error(dev) == 0

    # One call at a time with L2 cold and clean before each (context, and the
    # cache writes' own time).
    iso_steps = max(10, min(args.steps, 200))
    iso = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(iso_steps)]
    for i in range(iso_steps):
        flush()
        iso[i][0].record(stream)
        prelude()
        iso[i][1].record(stream)
        attend()
        iso[i][2].record(stream)
    torch.cuda.synchronize(dev)
    iso_attn_ms = [e[1].elapsed_time(e[2]) for e in iso]
    iso_pre_ms = [e[0].elapsed_time(e[1]) for e in iso]

    # End to end through the public API with host buffers, as a serving loop
    # runs it: every step copies its inputs from pinned host memory and reads
    # its output back, on two copy streams, so that uploads and downloads
    # overlap the kernels of other steps.  The compute stream waits on the copy
    # streams once per chunk of E2E_CHUNK steps (their uploads are issued
    # together before the chunk, their downloads after each step): a wait on
    # another stream's event between two steps costs the next step's launch
    # its overlap with the previous call (≈ 4.6 µs per step on l3-70b).
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens")
    host = {k: t[k].cpu().pin_memory() for k in names}
    nsets = 2 * E2E_CHUNK
    dbufs = [{k: torch.empty_like(t[k]) for k in host} for _ in range(nsets)]
    outs = [out] + [torch.empty_like(out) for _ in range(nsets - 1)]
    out_hosts = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(nsets)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_step = [torch.cuda.Event() for _ in range(nsets)]   # a step's kernels done
    ev_in = [torch.cuda.Event() for _ in range(2)]         # a chunk's uploads done
    ev_done = [torch.cuda.Event() for _ in range(2)]       # a chunk's kernels done
    ev_out = [torch.cuda.Event() for _ in range(2)]        # a chunk's downloads done

    def e2e_chunk(i0, n):
        j, cp = i0 // E2E_CHUNK, (i0 // E2E_CHUNK) & 1
        with torch.cuda.stream(up):
            if j >= 2:
                up.wait_event(ev_done[cp])         # chunk j-2 has consumed these buffer sets
            for i in range(i0, i0 + n):
                for k, v in host.items():
                    dbufs[i % nsets][k].copy_(v, non_blocking=True)
            ev_in[cp].record(up)
        stream.wait_event(ev_in[cp])
        if j >= 2:
            stream.wait_event(ev_out[cp])          # chunk j-2's outputs have been read back
        for i in range(i0, i0 + n):
            b = i % nsets
            prelude(dbufs[b]["k_new"], dbufs[b]["v_new"], dbufs[b]["slot_mapping"], c=i)
            attend(outs[b], dbufs[b]["q"], dbufs[b]["block_tables"], dbufs[b]["seq_lens"], c=i)
            ev_step[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_step[b])
                out_hosts[b].copy_(outs[b], non_blocking=True)
        ev_done[cp].record(stream)
        ev_out[cp].record(down)

    def e2e_run(n):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        up.wait_event(start)
        for i0 in range(0, n, E2E_CHUNK):
            e2e_chunk(i0, min(E2E_CHUNK, n - i0))
        for cp in range(min(2, (n + E2E_CHUNK - 1) // E2E_CHUNK)):
            stream.wait_event(ev_out[cp])
        end.record(stream)
        return start, end

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize(dev)
    e0, e1 = e2e_run(args.steps)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    assert pk.pk_get_device_error(dev) == 0
    assert torch.equal(out_hosts[(args.steps - 1) % nsets], outs[(args.steps - 1) % nsets].cpu())

    # Paging-overhead control: the same kernel and lengths, contiguous tables.
    contig = contiguous_tables(w)
    ctl_steps = max(10, min(args.steps, 100))
    paged_ms = time_decode(lambda: attend(), ctl_steps, flush, stream)
    contig_ms = None
    if contig is not None:
        bt_contig = torch.from_numpy(contig).to(dev)
        contig_ms = time_decode(lambda: attend(bt=bt_contig), ctl_steps, flush, stream)
    assert pk.pk_get_device_error(dev) == 0

    others = {}
    swap = swap_report(w, t, dev) if args.report_workloads and rank == 0 else None
    mqr = None
    if args.report_workloads and rank == 0 and w.group * 2 <= 16:
        mqr = multi_query_report(w, t, dev, flush, load_peaks()[0])
    pfr = prefill_report(dev, flush) if args.report_workloads and rank == 0 else None
    if args.report_workloads and rank == 0:
        peak0, _ = load_peaks()
        for name in ("l3-8b", "long", "prefix-b8", "prefix-b16", "prefix-b32", "tiny"):
            if name != args.workload:
                others[name] = workload_report(name, args.seed, dev, 20, flush, peak0)

    multi = None
    if args.layers > 1 and rank == 0:
        peak0, _ = load_peaks()
        multi = multi_layer_report(w, t, dev, args.layers, 5, workspace, out, peak0)

    if ws > 1:
        total_ms, e2e_ms, all_bytes = aggregate_over_ranks(total_ms, e2e_ms, float(ub["step"]), dev)
    else:
        all_bytes = float(ub["step"])

    if rank != 0:
        return None
    peak, peak_kind = load_peaks()
    ms_per_step = total_ms / args.steps
    value = all_bytes * args.steps / (total_ms * 1e-3) / 1e9
    attn_gbs = ub["attention"] / (attn_avg_ms * 1e-3) / 1e9
    iso_ms = statistics.median(iso_attn_ms)
    if stream_mode:
        l2_note = (f"inputs larger than L2: each step reads {ub['kv_unique'] / 1e9:.2f} GB of K/V "
                   f"({ub['kv_unique'] / l2_bytes:.1f}x the {l2_bytes / 1e6:.0f} MB L2) from one of two separate "
                   "caches used alternately (two layers), so nothing a step reads was left in L2 by the step "
                   "before; the K steps run back to back with no flush, one pair of CUDA events around them "
                   "(L2 flushed once before the first); the roofline's launch duration comes from K decode "
                   "calls timed the same way")
    else:
        l2_note = ("flushed between timed steps outside the events (256 MiB write, then a 256 MiB read so that "
                   "the write's dirty lines are written back before the step)")
    traffic = None
    if (RECORDED_TRAFFIC["sources_sha1"] == sources_sha1() and RECORDED_TRAFFIC["workload"] == args.workload
            and not args.shape):
        traffic = RECORDED_TRAFFIC["bytes_per_launch"]
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: {WORKLOAD_DESC[args.workload]}" + (
                f"; its lengths with {w.num_heads} q / {w.num_kv_heads} kv heads, head_dim {w.head_dim}, "
                "attention only" if args.shape else ""),
            "num_seqs": w.num_seqs, "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size, "num_blocks": w.num_blocks,
            "tokens_attended": ub["tokens"], "new_tokens": w.num_new_tokens,
            "copy_pairs": int(w.copy_pairs.shape[0]), "seed": args.seed,
            "useful_bytes_per_step": ub["step"], "attention_bytes": ub["attention"],
            "unique_kv_bytes": ub["kv_unique"],
            "l2": l2_note,
            "parallelism": f"replicas x{ws} (independent batches, no collective)",
            "decode_path": args.decode_path,
        },
        "pct_of_peak": round(100.0 * value / peak, 2),
        "tokens_per_s_per_layer": round(w.num_seqs * ws / (ms_per_step * 1e-3), 1),
        "roofline": {
            "kernel": "paged_attention_decode",
            "bound": "hbm",
            "achieved": round(attn_gbs, 2),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s",
            "frac": round(attn_gbs / peak, 4),
            "traffic": traffic,
            "avg_launch_ms": round(attn_avg_ms, 5),
            "algorithmic_bytes_per_launch": ub["attention"],
        },
        "e2e": {
            "value": round(all_bytes * args.steps / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms / args.steps, 5),
            "pipelining": f"inputs uploaded and outputs read back every step from/to pinned host memory on two "
                          f"copy streams overlapping other steps' kernels; {2 * E2E_CHUNK} buffer sets, the "
                          f"compute stream waiting on the copy streams once per {E2E_CHUNK} steps",
        },
        "paging_overhead": {
            "paged_decode_ms": round(paged_ms, 5),
            "contiguous_decode_ms": round(contig_ms, 5) if contig_ms else None,
            "overhead": round(paged_ms / contig_ms - 1.0, 4) if contig_ms else None,
            "skipped": None if contig_ms else "the sequences share blocks: laid out back to back they would need "
                                             "more blocks than the pool holds",
            "note": "same kernel and lengths with bt[s, i] = base_s + i; the pages quote a 20-26% kernel "
                    "slowdown vs a contiguous kernel for the 2023 paged kernel (context, not a target)",
        },
        "isolated_call": {
            "decode_ms": round(iso_ms, 5),
            "gbs": round(ub["attention"] / (iso_ms * 1e-3) / 1e9, 1),
            "frac": round(ub["attention"] / (iso_ms * 1e-3) / 1e9 / peak, 4),
            "what": f"one decode call at a time, L2 cold and clean before each (256 MiB write + read), CUDA "
                    f"events around the call, median of {iso_steps} (no overlap with a neighbouring launch)",
        },
        "gpu_launches": timed_launches,
        "clocks": clocks.summary(),
    }
    pre_bytes = ub["append"] + ub["copies"]
    pre_ms = statistics.median(iso_pre_ms)
    if pre_bytes > 0 and pre_ms > 0:
        res["cache_ops"] = {
            "what": "copy_blocks (the copy-on-write pairs, if any) then reshape_and_cache of a step, between "
                    "their own events (L2 cold before each step, median of the isolated steps); bytes read "
                    "plus written",
            "us_per_step": round(pre_ms * 1e3, 2),
            "bytes_per_step": pre_bytes,
            "gbs": round(pre_bytes / (pre_ms * 1e-3) / 1e9, 1),
        }
    if others:
        res["other_workloads"] = others
    if multi:
        res["multi_layer"] = multi
    if swap:
        res["block_swap"] = swap
    if mqr:
        res["multi_query"] = mqr
    if pfr:
        res["chunked_prefill"] = pfr
    if rank == 0:
        r = run_block_manager(args.workload, args.seed, 50, not args.no_cpu_baseline)
        nat = statistics.median(r["native"]) * 1e6
        bmr = {"what": f"host block manager, one decode step of {w.num_seqs} sequences: append a slot to "
                       "each, take the copy pairs, export tables and lengths (one pinned core, median of 50)",
               "native_us_per_step": round(nat, 2),
               "appends_per_s": round(w.num_seqs / (nat * 1e-6), 1)}
        if "oracle" in r:
            ref_us = statistics.median(r["oracle"]) * 1e6
            bmr["cpu_baseline"] = {"kind": "oracle", "us_per_step": round(ref_us, 2), "cores": 1}
        res["block_manager"] = bmr
    if not args.no_cpu_baseline:
        r = run_cpu_oracle(args.workload, args.seed, args.cpu_seqs, args.cpu_budget)
        tot = sum(r["times"])
        res["cpu_baseline"] = {
            "value": round(r["bytes"] * len(r["times"]) / tot / 1e9, 4),
            "unit": "GB/s",
            "cores": 1,
            "kind": "oracle",
            "sample": f"float64 oracle decode attention over the first {r['seqs']} sequences "
                      f"({r['tokens']} tokens) of the same workload, {len(r['times'])} passes, "
                      f"{tot:.1f} s on one pinned host core",
        }
        if args.cpu_all_cores_budget > 0:
            try:
                rp = run_cpu_oracle_pool(args.workload, args.seed, args.cpu_seqs, args.cpu_all_cores_budget)
                totp = sum(rp["times"])
                res["cpu_baseline"]["all_cores"] = {
                    "value": round(rp["bytes"] * len(rp["times"]) / totp / 1e9, 4),
                    "unit": "GB/s",
                    "cores": rp["cores"],
                    "sample": f"the same {rp['seqs']} sequences, one sequence per work item on a pool of "
                              f"{rp['cores']} single-threaded processes, {len(rp['times'])} passes, {totp:.1f} s",
                }
            except Exception as e:                      # context only: never costs the bench line
                res["cpu_baseline"]["all_cores"] = {"error": str(e)[-300:]}
    return res


def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    # Each step: the oracle over a bounded sample of the workload (its first
    # --ref-seqs sequences; by default as many as keep the whole run near a
    # minute: 32 at 20 steps, one at 640 steps or more); warm-up passes are
    # discarded.
    nseq = args.ref_seqs if args.ref_seqs > 0 else max(1, min(32, 640 // (args.steps + args.warmup)))
    r = run_cpu_oracle(args.workload, args.seed, nseq, budget_s=1e9, max_reps=args.steps + args.warmup)
    times = r["times"][args.warmup:] or r["times"]
    tot = sum(times)
    value = r["bytes"] * len(times) / tot / 1e9
    sample = (f"float64 oracle decode attention over the first {r['seqs']} sequences ({r['tokens']} tokens) "
              f"of the workload per step, one pinned host core")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": len(times),
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot / len(times), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOAD_DESC[args.workload]}", "seed": args.seed},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="l3-70b", choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--report-workloads", action="store_true",
                    help="also time decode alone on the other workloads (extra context in the line)")
    ap.add_argument("--layers", type=int, default=1,
                    help="also time one attention step of a model with this many layers (separate caches; "
                         "multi-layer copy/append launches), e.g. 80 for Llama-3-70B")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the chunked-prefill workload (16 x 512-token chunks over 4096 earlier tokens) "
                         "and print its report; a small case for profiling the prefill kernel")
    ap.add_argument("--multi-query-only", action="store_true",
                    help="time only the speculative-verification workload (the workload's sequences, 2 newest "
                         "tokens each as causal queries) and print its report; a case for profiling")
    ap.add_argument("--shape", default="",
                    help="H:Hkv:D -- the workload's sequence lengths with these head counts and head dim "
                         "(attention only; for kernel comparisons such as small groups or head dim 64)")
    ap.add_argument("--cpu-seqs", type=int, default=256)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--cpu-all-cores-budget", type=float, default=6.0,
                    help="seconds of timed passes of the oracle on all host cores (0: skip)")
    ap.add_argument("--ref-seqs", type=int, default=0,
                    help="sequences per step of the reference arm (0: sized from --steps, see run_reference)")
    ap.add_argument("--decode-path", default="auto", choices=["auto", "cuda_core", "tensor_core"],
                    help="kernel family of paged_attention_decode (auto: tensor cores)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)          # at least 3 untimed warm-up steps
    if args.prefill_only:
        import torch
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps({"prefill": prefill_report(dev, L2Flush(dev), steps=args.steps)}), flush=True)
        return
    if args.multi_query_only:
        import torch
        from paged_kv_cache_122_gb300 import workloads as W
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        w = W.get(args.workload, args.seed)
        t = W.make_tensors(w, dev)
        rep = multi_query_report(w, t, dev, L2Flush(dev), load_peaks()[0], steps=args.steps)
        print(json.dumps({"multi_query": rep}), flush=True)
        return
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
