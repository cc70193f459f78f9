"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
function include/kda.h declares, and rejects bad arguments on the host before
any launch (all checks are on metadata; the pointers below are never
dereferenced).  Fail-closed behaviour: "vllm-ascend KDA state copy" page,
"Startup preparation" and "Numeric contract" (S = 0 launches nothing)."""
import ctypes
import os
import re

import pytest

import kimi_delta_attention_varlen_gb300 as kda
from kimi_delta_attention_varlen_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

OK, NULL, DTYPE, LAYOUT, SHAPE, RANGE, WORKSPACE, CUDA, UNSUPPORTED, ALIGN = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9
A = 0x10000  # a 256-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def L():
    build.build()
    return _abi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert names == sorted(_abi.EXPORTED)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in (OK, NULL, DTYPE, LAYOUT, SHAPE, RANGE, WORKSPACE, CUDA, UNSUPPORTED, ALIGN):
        assert L.kda_status_string(code)
    assert b"unknown" in L.kda_status_string(12345)


def cache(data=A, dtype=0, n=8, h=2, v=32, k=32, stride=None, reserved=0):
    return _abi.KdaCache(data, dtype, reserved, n, h, v, k, h * v * k if stride is None else stride)


def gather(L, c, idx=A, it=0, sel=4, flags=None, packed=A):
    return L.kda_state_gather(ctypes.byref(c) if c is not None else None, idx, it, sel, flags, packed, None)


def test_gather_rejections(L):
    assert gather(L, None) == NULL
    assert gather(L, cache(data=0)) == NULL
    assert gather(L, cache(dtype=7)) == DTYPE
    assert gather(L, cache(n=0)) == LAYOUT
    assert gather(L, cache(h=0)) == LAYOUT
    assert gather(L, cache(stride=2 * 32 * 32 - 1)) == LAYOUT  # overlapping pages
    assert gather(L, cache(reserved=1)) == LAYOUT
    assert gather(L, cache(), it=5) == DTYPE
    assert gather(L, cache(), sel=-1) == SHAPE
    assert gather(L, cache(), idx=None) == NULL
    assert gather(L, cache(), packed=None) == NULL
    assert gather(L, cache(), idx=A + 2) == ALIGN
    assert gather(L, cache(data=A + 2)) == ALIGN
    assert gather(L, cache(n=1 << 40, stride=1 << 30)) == RANGE


def test_empty_selection_is_a_no_op(L):
    # S = 0 validates metadata and returns without touching the GPU
    assert gather(L, cache(), idx=None, sel=0, packed=None) == OK
    c = cache()
    assert L.kda_state_scatter(ctypes.byref(c), None, 0, 0, None, 0, None) == OK
    assert gather(L, cache(n=0), sel=0) == LAYOUT  # metadata is still checked


def test_scatter_rejections(L):
    c = cache()
    assert L.kda_state_scatter(ctypes.byref(c), A, 0, 4, A, 9, None) == DTYPE
    assert L.kda_state_scatter(ctypes.byref(c), A, 3, 4, A, 0, None) == DTYPE
    assert L.kda_state_scatter(ctypes.byref(c), A, 0, -2, A, 0, None) == SHAPE
    assert L.kda_state_scatter(ctypes.byref(c), A, 0, 4, None, 0, None) == NULL
    assert L.kda_state_scatter(ctypes.byref(c), A + 1, 0, 4, A, 0, None) == ALIGN
    assert L.kda_state_scatter(ctypes.byref(c), A, 0, 4, A + 2, 0, None) == ALIGN


def test_workspace_size(L):
    assert L.kda_prefill_workspace_size(1000, 3, 4, 128, 128) > 0
    assert L.kda_prefill_workspace_size(1000, 3, 4, 128, 64) == 0  # dk != dv not built
    assert L.kda_prefill_workspace_size(1000, 3, 4, 96, 96) == 0
    assert L.kda_prefill_workspace_size(1000, 0, 4, 128, 128) == 0
    small = L.kda_prefill_workspace_size(640, 1, 4, 128, 128)
    big = L.kda_prefill_workspace_size(6400, 1, 4, 128, 128)
    assert big > small
    # more sequences never shrink it (each may add a partial chunk)
    assert L.kda_prefill_workspace_size(640, 10, 4, 128, 128) > small
    # zero tokens still needs the header and chunk table
    assert L.kda_prefill_workspace_size(0, 2, 4, 64, 64) > 0


def prefill(L, **kw):
    a = dict(q=A, k=A, v=A, io=1, g=A, beta=A, cu=A, B=2, T=100, h=4, dk=128, dv=128, scale=0.1, l2=1,
             init=None, init_dtype=0, final=A, out=A, ws=A, ws_bytes=1 << 40, stream=None)
    a.update(kw)
    return L.kda_prefill_varlen(a["q"], a["k"], a["v"], a["io"], a["g"], a["beta"], a["cu"], a["B"], a["T"],
                                a["h"], a["dk"], a["dv"], a["scale"], a["l2"], a["init"], a["init_dtype"],
                                a["final"], a["out"], a["ws"], a["ws_bytes"], a["stream"])


def test_prefill_rejections(L):
    assert prefill(L, io=4) == DTYPE
    assert prefill(L, init=A, init_dtype=3) == DTYPE
    assert prefill(L, B=0) == SHAPE
    assert prefill(L, T=-1) == SHAPE
    assert prefill(L, h=0) == SHAPE
    assert prefill(L, dk=128, dv=64) == UNSUPPORTED
    assert prefill(L, dk=48, dv=48) == UNSUPPORTED
    assert prefill(L, T=1 << 31) == RANGE
    assert prefill(L, T=1 << 30, h=128) == RANGE  # chunk-preparation grid: 2^24 chunks x 128 heads
    assert prefill(L, B=1 << 25, h=8) == RANGE  # state-pass grid: 2^28 pairs x up to 8 value slices
    assert prefill(L, cu=None) == NULL
    assert prefill(L, ws=None) == NULL
    assert prefill(L, q=None) == NULL
    assert prefill(L, out=None) == NULL
    assert prefill(L, q=A + 8) == ALIGN
    assert prefill(L, g=A + 4) == ALIGN
    assert prefill(L, final=A + 8) == ALIGN
    assert prefill(L, ws=A + 16) == WORKSPACE
    need = L.kda_prefill_workspace_size(100, 2, 4, 128, 128)
    assert prefill(L, io=0, ws_bytes=need - 1) == WORKSPACE  # fp32: the records must fit
    compact = L.kda_prefill_workspace_size_compact(100, 2, 4, 128, 128, 1)
    assert prefill(L, ws_bytes=compact - 1) == WORKSPACE     # bf16, head size 128: the compact form


def test_compact_workspace_size(L):
    full = L.kda_prefill_workspace_size(73364, 16, 32, 128, 128)
    compact = L.kda_prefill_workspace_size_compact(73364, 16, 32, 128, 128, 1)
    # bf16 at head size 128: the header and chunk table only, no per-chunk records
    assert 0 < compact < 64 << 10 and full > 2_700_000_000
    assert L.kda_prefill_workspace_size_compact(73364, 16, 32, 128, 128, 0) == full  # fp32: records
    assert L.kda_prefill_workspace_size_compact(640, 2, 4, 64, 64, 1) == L.kda_prefill_workspace_size(640, 2, 4, 64, 64)
    assert L.kda_prefill_workspace_size_compact(640, 2, 4, 128, 128, 7) == 0  # unknown dtype
    assert L.kda_prefill_workspace_size_compact(640, 2, 4, 48, 48, 1) == 0    # head size not built


def cached(L, c, **kw):
    a = dict(q=A, k=A, v=A, io=1, g=A, beta=A, cu=A, B=2, T=100, h=2, dk=32, dv=32, scale=0.1, l2=1, idx_in=A,
             flags=None, idx_out=None, it=0, final=None, ckpt=None, ckpt_dtype=0, every=0, slots=0, out=A, ws=A,
             ws_bytes=1 << 40)
    a.update(kw)
    return L.kda_prefill_varlen_cached(a["q"], a["k"], a["v"], a["io"], a["g"], a["beta"], a["cu"], a["B"], a["T"],
                                       a["h"], a["dk"], a["dv"], a["scale"], a["l2"],
                                       ctypes.byref(c) if c is not None else None, a["idx_in"], a["flags"],
                                       a["idx_out"], a["it"], a["final"], a["ckpt"], a["ckpt_dtype"], a["every"],
                                       a["slots"], a["out"], a["ws"], a["ws_bytes"], None)


def test_cached_prefill_rejections(L):
    c = cache()
    assert cached(L, None) == NULL
    assert cached(L, cache(data=0)) == NULL
    assert cached(L, cache(h=3)) == SHAPE           # cache heads != h
    assert cached(L, c, dk=64, dv=64) == SHAPE
    assert cached(L, c, it=5) == DTYPE
    assert cached(L, c, idx_in=None) == NULL
    assert cached(L, c, idx_in=A + 2) == ALIGN
    assert cached(L, c, idx_out=A + 4, it=1) == ALIGN
    assert cached(L, cache(data=A + 4)) == ALIGN    # rows must be 16-byte aligned
    assert cached(L, cache(stride=2 * 32 * 32 + 2)) == ALIGN
    assert cached(L, c, ckpt=A, every=100) == SHAPE  # not a multiple of 64
    assert cached(L, c, ckpt=A, every=0) == SHAPE
    assert cached(L, c, ckpt=A, every=64, slots=-1) == SHAPE
    assert cached(L, c, ckpt=A, every=64, ckpt_dtype=5) == DTYPE
    assert cached(L, c, ckpt=A + 8, every=64, slots=4) == ALIGN
    assert cached(L, c, io=4) == DTYPE
    assert cached(L, c, final=A + 8) == ALIGN
    need = L.kda_prefill_workspace_size(100, 2, 2, 32, 32)
    assert cached(L, c, ws_bytes=need - 1) == WORKSPACE


def test_checkpoint_count(L):
    def count(offsets, every):
        arr = (ctypes.c_int32 * len(offsets))(*offsets)
        return L.kda_prefill_checkpoint_count(arr, len(offsets) - 1, every)
    assert count([0, 130, 130, 384], 64) == 2 + 0 + 3
    assert count([0, 130, 130, 384], 128) == 1 + 0 + 1
    assert count([0, 63], 64) == 0
    assert count([0, 10, 5], 64) == -1   # decreasing
    assert count([0, 64], 100) == -1     # not a multiple of 64
    assert L.kda_prefill_checkpoint_count(None, 1, 64) == -1
    assert kda.kda_prefill_checkpoint_count([0, 256, 320], 64) == 5


def test_int8_checkpoint_rejections(L):
    c = cache(dtype=1)
    st = L.kda_ckpt_store_int8
    ld = L.kda_ckpt_load_int8
    assert st(None, A, A, 0, 4, A, A, 4, None) == NULL
    assert st(ctypes.byref(c), A, A, 3, 4, A, A, 4, None) == DTYPE
    assert st(ctypes.byref(c), A, A, 0, -1, A, A, 4, None) == SHAPE
    assert st(ctypes.byref(c), A, A, 0, 4, A, A, -1, None) == SHAPE
    assert st(ctypes.byref(cache(v=16, k=32)), A, A, 0, 4, A, A, 4, None) == UNSUPPORTED
    assert st(ctypes.byref(c), None, None, 0, 0, None, None, 4, None) == OK  # empty: nothing launched
    assert st(ctypes.byref(c), None, A, 0, 4, A, A, 4, None) == NULL
    assert st(ctypes.byref(c), A, A, 0, 4, None, A, 4, None) == NULL
    assert st(ctypes.byref(c), A, A, 0, 4, A + 8, A, 4, None) == ALIGN
    assert st(ctypes.byref(c), A, A, 0, 4, A, A + 4, 4, None) == ALIGN
    assert st(ctypes.byref(cache(dtype=1, stride=2 * 32 * 32 + 4)), A, A, 0, 4, A, A, 4, None) == ALIGN
    assert ld(A, A, 4, A, A, 0, 4, None, None) == NULL
    assert ld(A, A, 4, A + 2, A, 0, 4, ctypes.byref(c), None) == ALIGN
    assert ld(None, A, 4, A, A, 0, 4, ctypes.byref(c), None) == NULL
    assert ld(A, A, 4, A, A, 0, 0, ctypes.byref(c), None) == OK


def test_target_verify_rejections(L):
    c = cache(dtype=1)
    V = L.kda_target_verify

    def call(cc=c, pool=c, **kw):
        a = dict(q=A, k=A, v=A, io=1, g=A, beta=A, R=4, Lt=3, h=2, dk=32, dv=32, idx=A, inter=A, it=0, out=A)
        a.update(kw)
        return V(a["q"], a["k"], a["v"], a["io"], a["g"], a["beta"], a["R"], a["Lt"], a["h"], a["dk"], a["dv"], 0.1,
                 1, ctypes.byref(cc) if cc is not None else None, a["idx"],
                 ctypes.byref(pool) if pool is not None else None, a["inter"], a["it"], a["out"], None)
    assert call(cc=None) == NULL
    assert call(pool=None) == NULL
    assert call(io=3) == DTYPE
    assert call(Lt=0) == SHAPE
    assert call(R=-1) == SHAPE
    assert call(h=3) == SHAPE
    assert call(pool=cache(dtype=0, h=2, v=64, k=64)) == SHAPE
    assert call(dk=48, dv=48) == UNSUPPORTED
    assert call(R=0, q=None) == OK
    assert call(inter=None) == NULL
    assert call(q=None) == NULL
    assert call(g=A + 4) == ALIGN
    assert call(pool=cache(dtype=1, stride=2 * 32 * 32 + 4)) == ALIGN


def decode(L, c, **kw):
    a = dict(q=A, k=A, v=A, io=1, g=A, beta=A, R=8, h=2, dk=32, dv=32, scale=0.1, l2=1, idx=A, it=0, out=A)
    a.update(kw)
    return L.kda_decode_step(a["q"], a["k"], a["v"], a["io"], a["g"], a["beta"], a["R"], a["h"], a["dk"],
                             a["dv"], a["scale"], a["l2"], ctypes.byref(c) if c is not None else None,
                             a["idx"], a["it"], a["out"], None)


def test_decode_rejections(L):
    c = cache(dtype=1)
    assert decode(L, None) == NULL
    assert decode(L, c, io=2) == DTYPE
    assert decode(L, c, it=2) == DTYPE
    assert decode(L, c, R=-1) == SHAPE
    assert decode(L, c, h=3) == SHAPE  # cache holds 2 heads
    assert decode(L, c, dk=64, dv=64) == SHAPE
    assert decode(L, c, dk=32, dv=16) == UNSUPPORTED
    assert decode(L, c, R=0, q=None) == OK  # empty batch: nothing launched
    assert decode(L, c, idx=None) == NULL
    assert decode(L, c, out=None) == NULL
    assert decode(L, c, q=A + 4) == ALIGN
    assert decode(L, cache(dtype=1, stride=2 * 32 * 32 + 3)) == ALIGN


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        kda.kda_status_string(0)


def test_selftest_bounded_wait_rejections(L):
    assert L.kda_selftest_bounded_wait(None, 1000, 0, None) == NULL
    assert L.kda_selftest_bounded_wait(ctypes.c_void_p(A), 0, 0, None) == RANGE


def conv(L, **kw):
    a = dict(x=A, io=1, cu=A, B=2, T=100, C=64, W=4, w=A, b=None, act=1, init=None, fin=None, sd=1, y=A)
    a.update(kw)
    return L.kda_conv1d_varlen(a["x"], a["io"], a["cu"], a["B"], a["T"], a["C"], a["W"], a["w"], a["b"], a["act"],
                               a["init"], a["fin"], a["sd"], a["y"], None)


def test_conv1d_rejections(L):
    assert conv(L, W=5) == UNSUPPORTED
    assert conv(L, W=1) == UNSUPPORTED
    assert conv(L, C=12) == SHAPE
    assert conv(L, act=2) == SHAPE
    assert conv(L, io=4) == DTYPE
    assert conv(L, C=65536 * 1024) == RANGE  # channel blocks beyond the grid's y dimension
    assert conv(L, T=1 << 30, C=1 << 20) == RANGE  # (token block, channel block) pairs beyond 2^31 - 1
    assert conv(L, B=0) == SHAPE
    assert conv(L, w=None) == NULL
    assert conv(L, x=A + 8) == ALIGN
