"""Torch-facing binding of the C ABI: checks tensors, passes pointers.

Every function here only marshals arguments (shapes, dtypes, device pointers,
the current CUDA stream) into one C call; all work runs in the library's CUDA
kernels.  Names follow the C entry points (``pk_*``); the unprefixed names are
the pages' spelling of the same calls.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence, Tuple

import torch

from . import _native
from ._native import check, load

_WORKSPACES = {}


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _stream(device: torch.device, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def pk_decode_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                              max_seq_len: int) -> int:
    return int(load().pk_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A decode workspace of ``nbytes`` (at least one byte; its contents on
    entry do not matter to the C call)."""
    return torch.empty(max(1, nbytes), dtype=torch.uint8, device=device)


def workspace_for(device: torch.device, nbytes: int, stream=None) -> Optional[torch.Tensor]:
    """A cached scratch buffer of at least ``nbytes`` for ``device`` and stream."""
    if nbytes == 0:
        return None
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device, s.cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = new_workspace(nbytes, device)
        _WORKSPACES[key] = ws
    return ws


def pk_paged_attention_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                              v_cache: torch.Tensor, block_tables: torch.Tensor,
                              seq_lens: torch.Tensor, scale: float, block_size: Optional[int] = None,
                              max_seq_len: Optional[int] = None,
                              workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention into ``out`` ([N, H, D], bf16 or fp32).  See the C header."""
    dev = q.device
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bf16 or fp32")
    _need(out, "out", out.dtype, 3, dev)
    N, H, D = q.shape
    P, B, Hkv, Dk = k_cache.shape
    if block_size is not None and block_size != B:
        raise ValueError(f"block_size {block_size} does not match the cache's {B}")
    if tuple(v_cache.shape) != tuple(k_cache.shape) or Dk != D:
        raise ValueError("k_cache / v_cache / q shapes disagree")
    if tuple(out.shape) != (N, H, D) or block_tables.shape[0] != N or seq_lens.shape[0] != N:
        raise ValueError("out / block_tables / seq_lens do not match q's batch")
    MB = block_tables.shape[1]
    if max_seq_len is None:
        max_seq_len = MB * B
    ws_bytes = pk_decode_workspace_bytes(N, H, Hkv, D, max_seq_len)
    if workspace is None:
        workspace = workspace_for(dev, ws_bytes, stream)
    elif workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError("workspace too small")
    with torch.cuda.device(dev):
        st = load().pk_paged_attention_decode(
            _ptr(out), _native.PK_FP32 if out.dtype == torch.float32 else _native.PK_BF16, _ptr(q),
            _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), MB, _ptr(seq_lens), int(max_seq_len),
            N, H, Hkv, D, P, B, float(scale), _ptr(workspace),
            0 if workspace is None else workspace.numel() * workspace.element_size(),
            _stream(dev, stream))
    check("pk_paged_attention_decode", st)
    return out


def pk_selftest_decode_wait_timeout(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                    v_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                    scale: float, max_seq_len: int, workspace: torch.Tensor, stall_tile: int,
                                    wait_limit_us: int, stream=None) -> int:
    """Self-test of the bounded waits (see the C header): a decode call on the
    tensor-core kernel whose CTA 0 stops issuing copies at ``stall_tile``, so
    its waits give up after ``wait_limit_us``.  Returns the call's status."""
    dev = q.device
    N, H, D = q.shape
    P, B, Hkv, _ = k_cache.shape
    with torch.cuda.device(dev):
        return int(load().pk_selftest_decode_wait_timeout(
            _ptr(out), _native.PK_FP32 if out.dtype == torch.float32 else _native.PK_BF16, _ptr(q),
            _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
            int(max_seq_len), N, H, Hkv, D, P, B, float(scale), _ptr(workspace),
            workspace.numel() * workspace.element_size(), int(stall_tile), int(wait_limit_us),
            _stream(dev, stream)))


def pk_selftest_decode_stale_lengths(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                     v_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                     scale: float, max_seq_len: int, stale_seq_lens: torch.Tensor,
                                     workspace: torch.Tensor, stream=None) -> int:
    """Self-test of the length check after the programmatic wait (see the C
    header): a decode call on the tensor-core kernel that plans first from
    ``stale_seq_lens`` and must plan again from ``seq_lens``.  Returns the
    call's status."""
    dev = q.device
    N, H, D = q.shape
    P, B, Hkv, _ = k_cache.shape
    with torch.cuda.device(dev):
        return int(load().pk_selftest_decode_stale_lengths(
            _ptr(out), _native.PK_FP32 if out.dtype == torch.float32 else _native.PK_BF16, _ptr(q),
            _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
            int(max_seq_len), N, H, Hkv, D, P, B, float(scale), _ptr(stale_seq_lens), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(dev, stream)))


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                           block_size: Optional[int] = None, *, out_dtype=torch.bfloat16,
                           max_seq_len: Optional[int] = None, out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """``paged_attention_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, block_size)``."""
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    return pk_paged_attention_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                                     block_size, max_seq_len, workspace, stream)


def paged_attention_multi_query(q: torch.Tensor, cu_q_lens: torch.Tensor, max_q_len: int,
                                k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                                seq_lens: torch.Tensor, scale: float, *, out_dtype=torch.bfloat16,
                                max_seq_len: Optional[int] = None, out: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal attention of several new tokens per sequence (rows cu_q_lens[s] ..
    cu_q_lens[s+1]-1 of q, the sequence's newest tokens) over the paged cache;
    returns [total_q, H, D].  See the C header."""
    dev = q.device
    _need(q, "q", torch.bfloat16, 3)
    _need(cu_q_lens, "cu_q_lens", torch.int32, 1, dev)
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    Tq, H, D = q.shape
    P, B, Hkv, Dk = k_cache.shape
    N, MB = block_tables.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or Dk != D:
        raise ValueError("k_cache / v_cache / q shapes disagree")
    if seq_lens.shape[0] != N or cu_q_lens.shape[0] != N + 1:
        raise ValueError("seq_lens / cu_q_lens do not match the block tables' batch")
    if out is None:
        out = torch.empty((Tq, H, D), dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, 3, dev)
    if tuple(out.shape) != (Tq, H, D) or out.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out must be bf16 or fp32 [total_q, H, D]")
    if max_seq_len is None:
        max_seq_len = MB * B
    ws_bytes = pk_decode_workspace_bytes(N, H, Hkv, D, max_seq_len)
    if workspace is None:
        workspace = workspace_for(dev, ws_bytes, stream)
    with torch.cuda.device(dev):
        st = load().pk_paged_attention_multi_query(
            _ptr(out), _native.PK_FP32 if out.dtype == torch.float32 else _native.PK_BF16, _ptr(q), Tq,
            _ptr(cu_q_lens), int(max_q_len), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), MB,
            _ptr(seq_lens), int(max_seq_len), N, H, Hkv, D, P, B, float(scale), _ptr(workspace),
            0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(dev, stream))
    check("pk_paged_attention_multi_query", st)
    return out


pk_paged_attention_multi_query = paged_attention_multi_query


def pk_reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         slot_mapping: torch.Tensor, stream=None) -> None:
    """Write new tokens' K/V ([T, Hkv, D] bf16) to their int64 slots.  See the C header."""
    dev = k_cache.device
    _need(k, "k", torch.bfloat16, 3, dev)
    _need(v, "v", torch.bfloat16, 3, dev)
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    T, Hkv, D = k.shape
    P, B, Hc, Dc = k_cache.shape
    if tuple(v.shape) != (T, Hkv, D) or (Hc, Dc) != (Hkv, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k / v / cache shapes disagree")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    with torch.cuda.device(dev):
        st = load().pk_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                         T, Hkv, D, P, B, _stream(dev, stream))
    check("pk_reshape_and_cache", st)


reshape_and_cache = pk_reshape_and_cache


def pk_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs: torch.Tensor,
                   stream=None) -> None:
    """Copy whole blocks for every (src, dst) row of an int64 [n, 2] tensor.  See the C header."""
    dev = k_cache.device
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(src_dst_pairs, "src_dst_pairs", torch.int64, 2, dev)
    if src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [n, 2]")
    P, B, Hkv, D = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache shapes disagree")
    with torch.cuda.device(dev):
        st = load().pk_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src_dst_pairs),
                                   src_dst_pairs.shape[0], Hkv, D, P, B, _stream(dev, stream))
    check("pk_copy_blocks", st)


copy_blocks = pk_copy_blocks


def pk_swap_blocks(dst_k: torch.Tensor, dst_v: torch.Tensor, src_k: torch.Tensor, src_v: torch.Tensor,
                   pairs: torch.Tensor, stream=None) -> None:
    """Copy whole blocks from one pool to another (e.g. device <-> pinned host)
    for every (src, dst) row of an int64 [n, 2] device tensor.  A pool may be a
    CUDA tensor or a pinned CPU tensor.  See the C header."""
    dev = pairs.device
    if not pairs.is_cuda:
        raise ValueError("pairs must be a CUDA tensor")
    for name, t in (("dst_k", dst_k), ("dst_v", dst_v), ("src_k", src_k), ("src_v", src_v)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 [P, B, Hkv, D] tensor")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    _need(pairs, "pairs", torch.int64, 2, dev)
    if pairs.shape[1] != 2:
        raise ValueError("pairs must be [n, 2]")
    if src_k.shape != src_v.shape or dst_k.shape != dst_v.shape or src_k.shape[1:] != dst_k.shape[1:]:
        raise ValueError("pool shapes disagree")
    P_src, B, Hkv, D = src_k.shape
    with torch.cuda.device(dev):
        st = load().pk_swap_blocks(_ptr(dst_k), _ptr(dst_v), _ptr(src_k), _ptr(src_v), _ptr(pairs),
                                   pairs.shape[0], Hkv, D, B, P_src, dst_k.shape[0], _stream(dev, stream))
    check("pk_swap_blocks", st)


swap_blocks = pk_swap_blocks


class LayerPointers:
    """A device array of the data pointers of per-layer tensors (what the
    ``*_layers`` calls take).  Build it once per set of layers: it holds a
    reference to the tensors so that their memory stays alive."""

    def __init__(self, tensors: Sequence[torch.Tensor]):
        tensors = list(tensors)
        if not tensors:
            raise ValueError("need at least one layer")
        dev = tensors[0].device
        shape = tuple(tensors[0].shape)
        for i, t in enumerate(tensors):
            _need(t, f"layer {i}", torch.bfloat16, len(shape), dev)
            if tuple(t.shape) != shape:
                raise ValueError("every layer must have the same shape")
        self.tensors = tensors
        self.shape = shape
        self.device = dev
        self.ptrs = torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=dev)

    def __len__(self):
        return len(self.tensors)


def _layers(x) -> LayerPointers:
    return x if isinstance(x, LayerPointers) else LayerPointers(x)


def pk_reshape_and_cache_layers(k_layers, v_layers, k_cache_layers, v_cache_layers,
                                slot_mapping: torch.Tensor, stream=None) -> None:
    """The append of every layer in one launch: layer l's new rows go to layer
    l's caches at the shared slots.  Arguments are lists of per-layer tensors
    or prebuilt ``LayerPointers``.  See the C header."""
    k, v, kc, vc = (_layers(x) for x in (k_layers, v_layers, k_cache_layers, v_cache_layers))
    n = len(k)
    if not (len(v) == len(kc) == len(vc) == n):
        raise ValueError("every argument needs the same number of layers")
    dev = kc.device
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    if len(k.shape) != 3 or len(kc.shape) != 4 or v.shape != k.shape or vc.shape != kc.shape:
        raise ValueError("layers must be [T, Hkv, D] rows and [P, B, Hkv, D] caches")
    T, Hkv, D = k.shape
    P, B, Hc, Dc = kc.shape
    if (Hc, Dc) != (Hkv, D) or slot_mapping.shape[0] != T:
        raise ValueError("k / cache / slot_mapping shapes disagree")
    with torch.cuda.device(dev):
        st = load().pk_reshape_and_cache_layers(_ptr(k.ptrs), _ptr(v.ptrs), _ptr(kc.ptrs), _ptr(vc.ptrs),
                                                _ptr(slot_mapping), T, n, Hkv, D, P, B, _stream(dev, stream))
    check("pk_reshape_and_cache_layers", st)


def pk_copy_blocks_layers(k_cache_layers, v_cache_layers, src_dst_pairs: torch.Tensor, stream=None) -> None:
    """The copy-on-write block copies of every layer in one launch.  See the C header."""
    kc, vc = _layers(k_cache_layers), _layers(v_cache_layers)
    if len(kc) != len(vc) or kc.shape != vc.shape or len(kc.shape) != 4:
        raise ValueError("k / v cache layers disagree")
    dev = kc.device
    _need(src_dst_pairs, "src_dst_pairs", torch.int64, 2, dev)
    if src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [n, 2]")
    P, B, Hkv, D = kc.shape
    with torch.cuda.device(dev):
        st = load().pk_copy_blocks_layers(_ptr(kc.ptrs), _ptr(vc.ptrs), _ptr(src_dst_pairs), src_dst_pairs.shape[0],
                                          len(kc), Hkv, D, P, B, _stream(dev, stream))
    check("pk_copy_blocks_layers", st)


def pk_gather_kv(k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                 seq_lens: torch.Tensor, seq_lens_host, max_seq_len: Optional[int] = None,
                 stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Contiguous [sum L, Hkv, D] K and V gathered through the tables, and row offsets."""
    dev = k_cache.device
    _need(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _need(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(seq_lens, "seq_lens", torch.int32, 1, dev)
    P, B, Hkv, D = k_cache.shape
    N, MB = block_tables.shape
    lens = [int(x) for x in seq_lens_host]
    cu = [0]
    for L in lens[:-1]:
        cu.append(cu[-1] + L)
    total = sum(lens)
    cu_t = torch.tensor(cu, dtype=torch.int64, device=dev)
    out_k = torch.empty((max(total, 1), Hkv, D), dtype=torch.bfloat16, device=dev)
    out_v = torch.empty_like(out_k)
    if max_seq_len is None:
        max_seq_len = max(lens) if lens else 0
    with torch.cuda.device(dev):
        st = load().pk_gather_kv(_ptr(out_k), _ptr(out_v), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), MB,
                                 _ptr(seq_lens), _ptr(cu_t), int(max_seq_len), N, Hkv, D, P, B,
                                 _stream(dev, stream))
    check("pk_gather_kv", st)
    return out_k[:total], out_v[:total], cu_t


def pk_set_decode_path(path) -> int:
    """Choose the decode kernel: "auto", "cuda_core" or "tensor_core" (or
    0/1/2).

    Returns the previous setting as an int.
    """
    names = {"auto": _native.PATH_AUTO, "cuda_core": _native.PATH_CUDA_CORE,
             "tensor_core": _native.PATH_TENSOR_CORE}
    code = names[path] if isinstance(path, str) else int(path)
    prev = load().pk_set_decode_path(code)
    if prev < 0:
        check("pk_set_decode_path", prev)
    return prev


def pk_get_device_error(device=None, stream=None) -> int:
    """Read and clear the device error word (synchronises the stream)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    code = ctypes.c_uint(0)
    with torch.cuda.device(dev):
        st = load().pk_get_device_error(ctypes.byref(code), _stream(dev, stream))
    check("pk_get_device_error", st)
    return int(code.value)
