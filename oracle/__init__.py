"""Plain fp64 CPU oracle for the KDA serving hot path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
baseline leg of the benchmark may import this package.  The CUDA library never
imports, links or calls it, and it shares no code with the CUDA library.

``kda_oracle.c`` holds the definitions (literal masked gather/scatter,
token-by-token recurrence, decode step); this module compiles it with gcc and
wraps it with ctypes.  ``chunked.py`` restates the chunkwise (UT/WY) form used
by the "Support Kimi-K3 on NPU" report's extend listing, as an independent
formulation the tests pin the sequential recurrence against.

All functions take and return numpy arrays.  Floating inputs are float64
(callers upcast bf16/fp32 device tensors exactly before calling).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

F32 = 0
BF16 = 1
EPS = 1e-6  # L2-normalisation epsilon: x / sqrt(sum(x^2) + EPS)

_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_VP = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into a shared library (gcc, -O2, no host-specific flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_f32_to_bf16.argtypes = [_VP, _VP, ctypes.c_int64]
            lib.oracle_f32_to_bf16.restype = None
            lib.oracle_gather.argtypes = [_VP, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, _I64, _VP, ctypes.c_int64, _VP]
            lib.oracle_gather.restype = ctypes.c_int
            lib.oracle_scatter.argtypes = [_VP, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, _I64, ctypes.c_int64, _VP, ctypes.c_int]
            lib.oracle_scatter.restype = ctypes.c_int
            lib.oracle_prefill.argtypes = [_D, _D, _D, _D, _D, _I64, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _D,
                                           ctypes.c_double, ctypes.c_int, ctypes.c_double, _D, _D,
                                           ctypes.c_int]
            lib.oracle_prefill.restype = ctypes.c_int
            lib.oracle_prefill_ckpt.argtypes = lib.oracle_prefill.argtypes[:16] + [ctypes.c_int64, _D,
                                                                                 ctypes.c_int]
            lib.oracle_prefill_ckpt.restype = ctypes.c_int
            lib.oracle_ckpt_store_int8.argtypes = [_VP, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _I64, _I64,
                                                   ctypes.c_int64, _VP, _VP, ctypes.c_int64]
            lib.oracle_ckpt_store_int8.restype = ctypes.c_int
            lib.oracle_ckpt_load_int8.argtypes = [_VP, _VP, ctypes.c_int64, _I64, _I64, ctypes.c_int64, _VP,
                                                  ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int64]
            lib.oracle_ckpt_load_int8.restype = ctypes.c_int
            lib.oracle_conv1d_varlen.argtypes = [_D, _I64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _D,
                                                 _D, ctypes.c_int, _D, _D, _D]
            lib.oracle_conv1d_varlen.restype = ctypes.c_int
            lib.oracle_conv1d_update.argtypes = [_D, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _D, _D,
                                                 ctypes.c_int, _VP, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                 _I64, _D]
            lib.oracle_conv1d_update.restype = ctypes.c_int
            lib.oracle_target_verify.argtypes = [_D, _D, _D, _D, _D, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                                 ctypes.c_int, ctypes.c_double, _VP, ctypes.c_int, ctypes.c_int64,
                                                 ctypes.c_int64, _I64, _VP, ctypes.c_int, ctypes.c_int64,
                                                 ctypes.c_int64, _I64, _D, ctypes.c_int]
            lib.oracle_target_verify.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [_D, _D, _D, _D, _D, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                          ctypes.c_int, ctypes.c_double, _VP, ctypes.c_int,
                                          ctypes.c_int64, ctypes.c_int64, _I64, _D, ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _ptr(a: np.ndarray, ctype=None):
    if ctype is None:
        return ctypes.c_void_p(a.ctypes.data)
    return a.ctypes.data_as(ctype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def f32_to_bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f32_to_bf16(_ptr(x), _ptr(y), x.size)
    return y


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype in (np.uint16, np.int16):
        return BF16
    raise TypeError(f"cache/packed arrays must be float32 or bf16 bit patterns (uint16), got {arr.dtype}")


def gather(cache_flat: np.ndarray, n_rows: int, payload: int, row_stride: int, idx, flags=None):
    """Literal masked gather.  cache_flat: float32 or uint16 (bf16 bits), n_rows*row_stride
    elements.  Returns packed [selected, payload] in the cache's element type."""
    cache_flat = np.ascontiguousarray(cache_flat)
    dt = _dtype_code(cache_flat)
    idx = _i64(idx).reshape(-1)
    sel = idx.size
    packed = np.empty((sel, payload), dtype=cache_flat.dtype)
    fl = None
    if flags is not None:
        fl = np.ascontiguousarray(flags, dtype=np.uint8).reshape(-1)
        assert fl.size == sel
    rc = _load().oracle_gather(_ptr(cache_flat), dt, n_rows, payload, row_stride, _ptr(idx, _I64),
                               None if fl is None else _ptr(fl), sel, _ptr(packed))
    if rc != 0:
        raise ValueError(f"oracle_gather rejected its arguments ({rc})")
    return packed


def scatter(cache_flat: np.ndarray, n_rows: int, payload: int, row_stride: int, idx, packed):
    """Literal scatter, in place on ``cache_flat`` (float32 or uint16 bf16 bits).
    packed: [selected, payload], float32 or uint16 bf16 bits."""
    assert cache_flat.flags.c_contiguous
    dt = _dtype_code(cache_flat)
    packed = np.ascontiguousarray(packed)
    pdt = _dtype_code(packed)
    idx = _i64(idx).reshape(-1)
    assert packed.shape[0] == idx.size
    rc = _load().oracle_scatter(_ptr(cache_flat), dt, n_rows, payload, row_stride, _ptr(idx, _I64),
                                idx.size, _ptr(packed), pdt)
    if rc != 0:
        raise ValueError(f"oracle_scatter rejected its arguments ({rc})")
    return cache_flat


def prefill(q, k, v, g, beta, cu_seqlens, init=None, scale=1.0, l2norm=True, eps=EPS,
            nthreads=None):
    """Token-by-token fp64 recurrence over a varlen batch.

    q, k, g: [T, H, K]; v: [T, H, V]; beta: [T, H]; cu_seqlens: [B + 1];
    init: [B, H, V, K] or None.  Returns (out [T, H, V], final [B, H, V, K])."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    cu = _i64(cu_seqlens).reshape(-1)
    T, H, K = q.shape
    V = v.shape[2]
    B = cu.size - 1
    assert k.shape == (T, H, K) and g.shape == (T, H, K) and v.shape == (T, H, V)
    assert beta.shape == (T, H)
    assert cu[0] == 0 and cu[-1] == T
    ini = None
    if init is not None:
        ini = _f64(init)
        assert ini.shape == (B, H, V, K)
    out = np.zeros((T, H, V), dtype=np.float64)
    final = np.zeros((B, H, V, K), dtype=np.float64)
    rc = _load().oracle_prefill(_ptr(q, _D), _ptr(k, _D), _ptr(v, _D), _ptr(g, _D),
                                _ptr(beta, _D), _ptr(cu, _I64), B, H, K, V,
                                None if ini is None else _ptr(ini, _D), float(scale),
                                1 if l2norm else 0, float(eps), _ptr(out, _D), _ptr(final, _D),
                                nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_prefill failed ({rc})")
    return out, final


def prefill_ckpt(q, k, v, g, beta, cu_seqlens, every, init=None, scale=1.0, l2norm=True, eps=EPS,
                 nthreads=None):
    """prefill plus checkpoints: returns (out, final, ckpt [slots, H, V, K]) where slot
    first_b + m - 1 holds the state of sequence b after its first m * every tokens
    (m = 1 .. len_b // every) and first_b = sum of len_b' // every over b' < b."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    cu = _i64(cu_seqlens).reshape(-1)
    T, H, K = q.shape
    V = v.shape[2]
    B = cu.size - 1
    assert cu[0] == 0 and cu[-1] == T and every > 0
    ini = None
    if init is not None:
        ini = _f64(init)
        assert ini.shape == (B, H, V, K)
    slots = int(sum((cu[b + 1] - cu[b]) // every for b in range(B)))
    out = np.zeros((T, H, V), dtype=np.float64)
    final = np.zeros((B, H, V, K), dtype=np.float64)
    ckpt = np.zeros((max(slots, 1), H, V, K), dtype=np.float64)
    rc = _load().oracle_prefill_ckpt(_ptr(q, _D), _ptr(k, _D), _ptr(v, _D), _ptr(g, _D),
                                     _ptr(beta, _D), _ptr(cu, _I64), B, H, K, V,
                                     None if ini is None else _ptr(ini, _D), float(scale),
                                     1 if l2norm else 0, float(eps), _ptr(out, _D), _ptr(final, _D),
                                     int(every), _ptr(ckpt, _D), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_prefill_ckpt failed ({rc})")
    return out, final, ckpt[:slots]


def ckpt_store_int8(active_flat: np.ndarray, n_rows: int, row_stride: int, H: int, V: int, K: int,
                    src, dst, qdata: np.ndarray, scale: np.ndarray) -> None:
    """Quantise active rows (float32, or bf16 as uint16 bits; rows of row_stride elements
    holding [H, V, K]) into qdata [slots, H, V, K] int8 and scale [slots, H, K] float32, in
    place, for pairs (src[s], dst[s]) with valid indices."""
    assert active_flat.flags.c_contiguous and qdata.flags.c_contiguous and scale.flags.c_contiguous
    assert qdata.dtype == np.int8 and scale.dtype == np.float32
    src, dst = _i64(src).reshape(-1), _i64(dst).reshape(-1)
    assert src.size == dst.size
    rc = _load().oracle_ckpt_store_int8(active_flat.ctypes.data, _dtype_code(active_flat), n_rows, row_stride,
                                        H, V, K, _ptr(src, _I64), _ptr(dst, _I64), src.size,
                                        qdata.ctypes.data, scale.ctypes.data, qdata.shape[0])
    if rc != 0:
        raise ValueError(f"oracle_ckpt_store_int8 failed ({rc})")


def ckpt_load_int8(qdata: np.ndarray, scale: np.ndarray, src, dst, active_flat: np.ndarray, n_rows: int,
                   row_stride: int, H: int, V: int, K: int) -> None:
    """Dequantise checkpoint slots src[s] into active rows dst[s] (in place)."""
    assert active_flat.flags.c_contiguous and qdata.flags.c_contiguous and scale.flags.c_contiguous
    src, dst = _i64(src).reshape(-1), _i64(dst).reshape(-1)
    assert src.size == dst.size
    rc = _load().oracle_ckpt_load_int8(qdata.ctypes.data, scale.ctypes.data, qdata.shape[0], _ptr(src, _I64),
                                       _ptr(dst, _I64), src.size, active_flat.ctypes.data,
                                       _dtype_code(active_flat), n_rows, row_stride, H, V, K)
    if rc != 0:
        raise ValueError(f"oracle_ckpt_load_int8 failed ({rc})")


ACT = {"none": 0, "silu": 1}


def conv1d_varlen(x, cu_seqlens, weight, bias=None, activation="none", init=None):
    """Depthwise causal convolution over a varlen batch.  x: [T, C]; weight: [C, W];
    bias: [C] or None; init: [B, W-1, C] or None.  Returns (y [T, C], final [B, W-1, C])."""
    x, w = _f64(x), _f64(weight)
    cu = _i64(cu_seqlens).reshape(-1)
    T, C = x.shape
    W = w.shape[1]
    B = cu.size - 1
    assert w.shape == (C, W) and cu[0] == 0 and cu[-1] == T
    b = None if bias is None else _f64(bias)
    ini = None if init is None else _f64(init)
    if ini is not None:
        assert ini.shape == (B, W - 1, C)
    y = np.zeros((T, C), dtype=np.float64)
    final = np.zeros((B, max(W - 1, 0), C), dtype=np.float64)
    rc = _load().oracle_conv1d_varlen(_ptr(x, _D), _ptr(cu, _I64), B, C, W, _ptr(w, _D),
                                      None if b is None else _ptr(b, _D), ACT[activation],
                                      None if ini is None else _ptr(ini, _D), _ptr(y, _D), _ptr(final, _D))
    if rc != 0:
        raise ValueError(f"oracle_conv1d_varlen failed ({rc})")
    return y, final


def conv1d_update(x, weight, cache_flat: np.ndarray, n_rows: int, row_stride: int, idx, bias=None,
                  activation="none"):
    """One token per request on conv-state cache rows ([W-1, C] each, float32 or bf16 bits),
    in place.  Returns y [R, C]."""
    x, w = _f64(x), _f64(weight)
    R, C = x.shape
    W = w.shape[1]
    assert cache_flat.flags.c_contiguous
    idx = _i64(idx).reshape(-1)
    assert idx.size == R
    b = None if bias is None else _f64(bias)
    y = np.zeros((R, C), dtype=np.float64)
    rc = _load().oracle_conv1d_update(_ptr(x, _D), R, C, W, _ptr(w, _D), None if b is None else _ptr(b, _D),
                                      ACT[activation], cache_flat.ctypes.data, _dtype_code(cache_flat), n_rows,
                                      row_stride, _ptr(idx, _I64), _ptr(y, _D))
    if rc != 0:
        raise ValueError(f"oracle_conv1d_update failed ({rc})")
    return y


def target_verify(q, k, v, g, beta, cache_flat: np.ndarray, n_rows: int, row_stride: int, idx,
                  pool_flat: np.ndarray, pool_rows: int, pool_stride: int, inter_idx, scale=1.0, l2norm=True,
                  eps=EPS, nthreads=None):
    """L draft tokens per request from cache row idx[r] (read only); the state after token t
    of request r goes to pool row inter_idx[r, t] (float32 or bf16 bits; rows of pool_stride
    elements holding [H, V, K]), in place.  q, k, g: [R, L, H, K]; v: [R, L, H, V];
    beta: [R, L, H].  Returns out [R, L, H, V]."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    R, L, H, K = q.shape
    V = v.shape[3]
    assert cache_flat.flags.c_contiguous and pool_flat.flags.c_contiguous
    idx = _i64(idx).reshape(-1)
    ii = _i64(inter_idx).reshape(-1)
    assert idx.size == R and ii.size == R * L
    out = np.zeros((R, L, H, V), dtype=np.float64)
    rc = _load().oracle_target_verify(_ptr(q, _D), _ptr(k, _D), _ptr(v, _D), _ptr(g, _D), _ptr(beta, _D), R, L,
                                      H, K, V, float(scale), 1 if l2norm else 0, float(eps), cache_flat.ctypes.data,
                                      _dtype_code(cache_flat), n_rows, row_stride, _ptr(idx, _I64),
                                      pool_flat.ctypes.data, _dtype_code(pool_flat), pool_rows, pool_stride,
                                      _ptr(ii, _I64), _ptr(out, _D), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_target_verify failed ({rc})")
    return out


def decode(q, k, v, g, beta, cache_flat: np.ndarray, n_rows: int, row_stride: int, idx,
           scale=1.0, l2norm=True, eps=EPS, nthreads=None):
    """One recurrent token per request, in place on ``cache_flat`` (float32 or uint16
    bf16 bits; rows of row_stride elements holding [H, V, K]).  Returns out [R, H, V]."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    R, H, K = q.shape
    V = v.shape[2]
    assert cache_flat.flags.c_contiguous
    dt = _dtype_code(cache_flat)
    idx = _i64(idx).reshape(-1)
    assert idx.size == R
    out = np.zeros((R, H, V), dtype=np.float64)
    rc = _load().oracle_decode(_ptr(q, _D), _ptr(k, _D), _ptr(v, _D), _ptr(g, _D),
                               _ptr(beta, _D), R, H, K, V, float(scale), 1 if l2norm else 0,
                               float(eps), _ptr(cache_flat), dt, n_rows, row_stride,
                               _ptr(idx, _I64), _ptr(out, _D), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_decode failed ({rc})")
    return out
