"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU.  CPU only: no call here
launches a kernel (every call either fails validation or, with no device,
returns PK_ERR_NO_DEVICE)."""
import ctypes
import os
import re

import pytest
import torch

from conftest import ROOT
from paged_kv_cache_122_gb300 import _native, build

HEADER = os.path.join(ROOT, "include", "pagedkv.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))
NULL = None


@pytest.fixture(scope="module")
def lib():
    if not build.up_to_date():
        build.build()
    return _native.load()


def _declared_functions(headers=None):
    names = set()
    for h in headers or HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(pk_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_three_step_calls():
    names = _declared_functions([HEADER])
    for n in ("pk_paged_attention_decode", "pk_reshape_and_cache", "pk_copy_blocks",
              "pk_decode_workspace_bytes", "pk_gather_kv", "pk_get_device_error", "pk_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n
        assert n in _native.SIGNATURES, f"binding lacks {n}"


def test_status_strings_and_version(lib):
    assert lib.pk_version() >> 16 == 1
    for code in _native.STATUS_NAMES:
        assert lib.pk_status_string(code)
    assert lib.pk_status_string(12345) == b"unknown status"
    assert lib.pk_set_decode_path(7) == -3
    assert lib.pk_set_decode_path(3) == -3            # the removed head-batched family
    assert lib.pk_set_decode_path(1) == 0 and lib.pk_set_decode_path(0) == 1


def test_workspace_bound(lib):
    f = lib.pk_decode_workspace_bytes
    slots = 2 * 1024 * 8384                             # tensor-core kernel: 2 slots per CTA
    assert f(4, 8, 8, 64, 16) == 0                      # every sequence fits one tile: nothing is split
    assert f(4, 8, 2, 64, 128) == 0
    assert f(4, 8, 2, 64, 129) == slots                 # 2 KV heads: per-head tiles of 128 tokens
    assert f(4, 8, 8, 64, 129) == slots                 # 8 KV heads: head pairs, the same slots
    assert f(8, 32, 8, 128, 131072) == max(8 * 32 * 512 * 130 * 4, slots)
    assert f(1, 6, 4, 128, 4096) == 0                   # 6 % 4 != 0
    assert f(1, 8, 8, 96, 4096) == 0                    # head_dim unsupported
    assert f(-1, 8, 8, 64, 10) == 0


def _fake(n=1):
    # Host addresses, never dereferenced: validation fails first, or there is
    # no device and the call returns before any launch.
    buf = (ctypes.c_uint8 * (64 * n))()
    base = (ctypes.addressof(buf) + 15) & ~15
    _fake.keep = buf
    return ctypes.c_void_p(base)


def _decode(lib, **kw):
    a = dict(out=_fake(), dt=0, q=_fake(), kc=_fake(), vc=_fake(), bt=_fake(), mb=4, sl=_fake(), msl=64,
             n=2, h=8, hkv=2, d=128, nb=16, b=16, scale=0.088, ws=_fake(), wsb=1 << 30, st=None)
    a.update(kw)
    return lib.pk_paged_attention_decode(a["out"], a["dt"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"],
                                         a["msl"], a["n"], a["h"], a["hkv"], a["d"], a["nb"], a["b"], a["scale"],
                                         a["ws"], a["wsb"], a["st"])


def test_decode_host_validation(lib):
    assert _decode(lib, h=6, hkv=4) == -2                   # heads not a multiple of kv heads
    assert _decode(lib, d=96) == -3                          # head_dim
    assert _decode(lib, b=64) == -3                          # block size
    assert _decode(lib, h=24, hkv=8) == -3                   # group of 3
    assert _decode(lib, dt=7) == -3                          # out dtype
    assert _decode(lib, msl=65) == -2                        # longer than the table can hold
    assert _decode(lib, n=-1) == -2
    assert _decode(lib, scale=float("nan")) == -2
    assert _decode(lib, n=0) == 0                            # empty batch is a no-op
    assert _decode(lib, out=NULL) == -1
    assert _decode(lib, kc=NULL) == -1
    assert _decode(lib, q=ctypes.c_void_p(_fake().value + 2)) == -6
    if not torch.cuda.is_available():
        assert _decode(lib) == -7                            # valid, but no device here
        assert _decode(lib, mb=64, msl=1024, ws=NULL) == -4  # needs split-K scratch


def test_selftest_host_validation(lib):
    f = lib.pk_selftest_decode_wait_timeout

    def call(stall=1, limit_us=5000, **kw):
        a = dict(out=_fake(), dt=0, q=_fake(), kc=_fake(), vc=_fake(), bt=_fake(), mb=4, sl=_fake(), msl=64,
                 n=2, h=8, hkv=2, d=128, nb=16, b=16, scale=0.088, ws=_fake(), wsb=1 << 30)
        a.update(kw)
        return f(a["out"], a["dt"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"], a["msl"], a["n"], a["h"],
                 a["hkv"], a["d"], a["nb"], a["b"], a["scale"], a["ws"], a["wsb"], stall, limit_us, None)
    assert call(stall=0) == -2 and call(stall=-3) == -2       # a stall must name a tile >= 1
    assert call(limit_us=50) == -2 and call(limit_us=2000000) == -2
    assert call(d=96) == -3                                   # then the decode call's own checks
    assert call(n=0) == 0
    if not torch.cuda.is_available():
        assert call() == -7


def test_stale_lengths_selftest_host_validation(lib):
    f = lib.pk_selftest_decode_stale_lengths

    def call(**kw):
        a = dict(out=_fake(), dt=0, q=_fake(), kc=_fake(), vc=_fake(), bt=_fake(), mb=4, sl=_fake(), msl=64,
                 n=2, h=8, hkv=2, d=128, nb=16, b=16, scale=0.088, stale=_fake(), ws=_fake(), wsb=1 << 30)
        a.update(kw)
        return f(a["out"], a["dt"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"], a["msl"], a["n"], a["h"],
                 a["hkv"], a["d"], a["nb"], a["b"], a["scale"], a["stale"], a["ws"], a["wsb"], None)
    assert call(stale=NULL) == -1                             # the stale lengths are required
    assert call(d=96) == -3                                   # then the decode call's own checks
    assert call(n=0) == 0
    if not torch.cuda.is_available():
        assert call() == -7


def test_cache_ops_host_validation(lib):
    f = lib.pk_reshape_and_cache
    assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 4, 8, 100, 16, 16, None) == -3
    assert f(_fake(), _fake(), _fake(), _fake(), _fake(), -1, 8, 128, 16, 16, None) == -2
    assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 0, 8, 128, 16, 16, None) == 0
    assert f(NULL, _fake(), _fake(), _fake(), _fake(), 4, 8, 128, 16, 16, None) == -1
    g = lib.pk_copy_blocks
    assert g(_fake(), _fake(), _fake(), 3, 8, 128, 16, 12, None) == -3
    assert g(_fake(), _fake(), _fake(), 0, 8, 128, 16, 16, None) == 0
    assert g(_fake(), NULL, _fake(), 2, 8, 128, 16, 16, None) == -1
    h = lib.pk_gather_kv
    assert h(_fake(), _fake(), _fake(), _fake(), _fake(), 2, _fake(), _fake(), 64, 1, 8, 128, 4, 16, None) == -2
    if not torch.cuda.is_available():
        assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 4, 8, 128, 16, 16, None) == -7
        assert g(_fake(), _fake(), _fake(), 2, 8, 128, 16, 16, None) == -7
        code = ctypes.c_uint(99)
        assert lib.pk_get_device_error(ctypes.byref(code), None) == -7 and code.value == 0


def test_multi_layer_cache_ops_host_validation(lib):
    f = lib.pk_reshape_and_cache_layers
    #   k_layers   v_layers   kc_layers  vc_layers  slots     T  L   Hkv D    P   B
    assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 4, 80, 8, 100, 16, 16, None) == -3
    assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 4, -1, 8, 128, 16, 16, None) == -2
    assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 4, 65536, 8, 128, 16, 16, None) == -2
    assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 4, 0, 8, 128, 16, 16, None) == 0
    assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 0, 80, 8, 128, 16, 16, None) == 0
    assert f(_fake(), _fake(), NULL, _fake(), _fake(), 4, 80, 8, 128, 16, 16, None) == -1
    assert f(ctypes.c_void_p(_fake().value + 4), _fake(), _fake(), _fake(), _fake(), 4, 80, 8, 128, 16, 16, None) == -6
    g = lib.pk_copy_blocks_layers
    #   kc_layers  vc_layers  pairs    n  L   Hkv D    P   B
    assert g(_fake(), _fake(), _fake(), 3, 80, 8, 128, 16, 12, None) == -3
    assert g(_fake(), _fake(), _fake(), 3, 32768, 8, 128, 16, 16, None) == -2
    assert g(_fake(), _fake(), _fake(), 0, 80, 8, 128, 16, 16, None) == 0
    assert g(_fake(), NULL, _fake(), 2, 80, 8, 128, 16, 16, None) == -1
    if not torch.cuda.is_available():
        assert f(_fake(), _fake(), _fake(), _fake(), _fake(), 4, 80, 8, 128, 16, 16, None) == -7
        assert g(_fake(), _fake(), _fake(), 2, 80, 8, 128, 16, 16, None) == -7


def test_multi_query_host_validation(lib):
    f = lib.pk_paged_attention_multi_query
    def call(tq=8, cu="fake", mq=2, h=16, hkv=2, d=128, msl=64, nseq=4):
        return f(_fake(), 0, _fake(), tq, _fake() if cu == "fake" else cu, mq, _fake(), _fake(), _fake(), 4,
                 _fake(), msl, nseq, h, hkv, d, 16, 16, 0.1, _fake(), 1 << 30, None)
    assert call(d=64, hkv=3) == -2            # 16 heads do not split into 3 KV heads
    assert call(d=96) == -3
    assert call(tq=0) == 0 and call(nseq=0) == 0
    assert call(cu=NULL) == -1
    assert call(tq=-1) == -2
    if not torch.cuda.is_available():
        assert call() == -7



def test_swap_blocks_host_validation(lib):
    f = lib.pk_swap_blocks

    def call(dk="fake", n=2, hkv=8, d=128, b=16, src_nb=32, dst_nb=16, dst_k_off=0):
        dk = ctypes.c_void_p(_fake().value + dst_k_off) if dk == "fake" else dk
        return f(dk, _fake(), _fake(), _fake(), _fake(), n, hkv, d, b, src_nb, dst_nb, None)
    assert call(n=-1) == -2
    assert call(src_nb=-1) == -2 and call(dst_nb=-1) == -2
    assert call(hkv=0) == -2 and call(b=0) == -2
    assert call(d=96) == -3                                   # head_dim
    assert call(b=12) == -3                                   # block size
    assert call(n=0) == 0                                     # no pairs: a no-op
    assert call(dk=NULL) == -1
    assert call(dst_k_off=8) == -6                            # not 16-byte aligned
    if not torch.cuda.is_available():
        assert call() == -7                                   # valid, but no device here


def test_decode_noalloc_host_validation(lib):
    f = lib.pk_paged_attention_decode_noalloc

    def call(out="fake", dt=0, n=2, h=8, hkv=2, d=128, b=16, mb=4, msl=64, scale=0.088, q_off=0):
        out = _fake() if out == "fake" else out
        return f(out, dt, ctypes.c_void_p(_fake().value + q_off), _fake(), _fake(), _fake(), mb, _fake(), msl,
                 n, h, hkv, d, 16, b, scale, None)
    assert call(h=6, hkv=4) == -2                             # heads not a multiple of kv heads
    assert call(msl=65) == -2                                 # longer than the table can hold
    assert call(n=-1) == -2 and call(n=65536) == -2
    assert call(h=40000, hkv=40000) == -2                     # the regular call's KV-head bound
    assert call(scale=float("inf")) == -2
    assert call(dt=7) == -3 and call(d=96) == -3 and call(b=64) == -3
    assert call(h=24, hkv=8) == -3                            # group of 3
    assert call(n=0) == 0                                     # empty batch: a no-op
    assert call(out=NULL) == -1
    assert call(q_off=2) == -6                                # not 16-byte aligned
    if not torch.cuda.is_available():
        assert call() == -7                                   # valid, but no device here


def test_binding_refuses_cpu_tensors():
    import paged_kv_cache_122_gb300 as pk
    q = torch.zeros(1, 8, 64, dtype=torch.bfloat16)
    kc = torch.zeros(4, 16, 8, 64, dtype=torch.bfloat16)
    bt = torch.zeros(1, 1, dtype=torch.int32)
    sl = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        pk.paged_attention_decode(q, kc, kc, bt, sl, 0.125, 16)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError, match="no CPU fallback"):
        _native.load(str(tmp_path / "absent.so"))
