"""ctypes binding of libkda.so (the C ABI declared in include/kda.h).

Argument marshalling only: every function here turns torch tensors into the
pointers and sizes the C ABI takes, calls it, and raises KdaError on a
non-zero status.  All computation runs in the CUDA kernels of libkda.so;
there is no fallback of any kind.  If the library has not been built, the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libkda.so")

KDA_F32 = 0
KDA_BF16 = 1
KDA_I32 = 0
KDA_I64 = 1
KDA_NOALLOC_SCRATCH_BYTES = 128 << 20  # include/kda.h

# Every symbol include/kda.h declares.
EXPORTED = (
    "kda_state_gather",
    "kda_state_scatter",
    "kda_prefill_workspace_size",
    "kda_prefill_workspace_size_compact",
    "kda_prefill_varlen",
    "kda_prefill_varlen_timed",
    "kda_prefill_varlen_noalloc",
    "kda_prefill_noalloc_status",
    "kda_prefill_varlen_cached",
    "kda_prefill_checkpoint_count",
    "kda_target_verify",
    "kda_conv1d_varlen",
    "kda_conv1d_update",
    "kda_ckpt_store_int8",
    "kda_ckpt_load_int8",
    "kda_decode_step",
    "kda_status_string",
    "kda_last_cuda_error_string",
    "kda_prefill_workspace_status",
    "kda_selftest_bounded_wait",
)


class KdaCache(ctypes.Structure):
    """Mirror of the C struct kda_cache."""
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("n_rows", ctypes.c_int64),
        ("h", ctypes.c_int64),
        ("v", ctypes.c_int64),
        ("k", ctypes.c_int64),
        ("row_stride", ctypes.c_int64),
    ]


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().kda_status_string(status).decode()
        if status == -7:
            msg += f" ({lib().kda_last_cuda_error_string().decode()})"
        super().__init__(f"{what}: {msg}")


_lock = threading.Lock()
_lib = None


def lib():
    """Load libkda.so once and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libkda.so is not built ({LIB_PATH} missing): run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        cache_p = ctypes.POINTER(KdaCache)
        L.kda_state_gather.argtypes = [cache_p, vp, i32, i64, vp, vp, vp]
        L.kda_state_gather.restype = ctypes.c_int
        L.kda_state_scatter.argtypes = [cache_p, vp, i32, i64, vp, i32, vp]
        L.kda_state_scatter.restype = ctypes.c_int
        L.kda_prefill_workspace_size.argtypes = [i64, i64, i32, i32, i32]
        L.kda_prefill_workspace_size.restype = sz
        L.kda_prefill_workspace_size_compact.argtypes = [i64, i64, i32, i32, i32, i32]
        L.kda_prefill_workspace_size_compact.restype = sz
        L.kda_prefill_varlen.argtypes = [vp, vp, vp, i32, vp, vp, vp, i64, i64, i32, i32, i32, f32, i32,
                                         vp, i32, vp, vp, vp, sz, vp]
        L.kda_prefill_varlen.restype = ctypes.c_int
        L.kda_prefill_varlen_timed.argtypes = L.kda_prefill_varlen.argtypes + [ctypes.POINTER(ctypes.c_void_p)]
        L.kda_prefill_varlen_timed.restype = ctypes.c_int
        L.kda_prefill_varlen_noalloc.argtypes = L.kda_prefill_varlen.argtypes[:18] + [vp]
        L.kda_prefill_varlen_noalloc.restype = ctypes.c_int
        L.kda_prefill_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
        L.kda_prefill_noalloc_status.restype = ctypes.c_int
        L.kda_prefill_varlen_cached.argtypes = [vp, vp, vp, i32, vp, vp, vp, i64, i64, i32, i32, i32, f32, i32,
                                                cache_p, vp, vp, vp, i32, vp, vp, i32, i32, i64, vp, vp, sz, vp]
        L.kda_prefill_varlen_cached.restype = ctypes.c_int
        L.kda_prefill_checkpoint_count.argtypes = [ctypes.POINTER(ctypes.c_int32), i64, i32]
        L.kda_prefill_checkpoint_count.restype = i64
        L.kda_target_verify.argtypes = [vp, vp, vp, i32, vp, vp, i64, i32, i32, i32, i32, f32, i32, cache_p, vp,
                                        cache_p, vp, i32, vp, vp]
        L.kda_target_verify.restype = ctypes.c_int
        L.kda_conv1d_varlen.argtypes = [vp, i32, vp, i64, i64, i64, i32, vp, vp, i32, vp, vp, i32, vp, vp]
        L.kda_conv1d_varlen.restype = ctypes.c_int
        L.kda_conv1d_update.argtypes = [vp, i32, i64, i64, i32, vp, vp, i32, cache_p, vp, i32, vp, vp]
        L.kda_conv1d_update.restype = ctypes.c_int
        L.kda_ckpt_store_int8.argtypes = [cache_p, vp, vp, i32, i64, vp, vp, i64, vp]
        L.kda_ckpt_store_int8.restype = ctypes.c_int
        L.kda_ckpt_load_int8.argtypes = [vp, vp, i64, vp, vp, i32, i64, cache_p, vp]
        L.kda_ckpt_load_int8.restype = ctypes.c_int
        L.kda_decode_step.argtypes = [vp, vp, vp, i32, vp, vp, i64, i32, i32, i32, f32, i32, cache_p, vp, i32,
                                      vp, vp]
        L.kda_decode_step.restype = ctypes.c_int
        L.kda_status_string.argtypes = [i32]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_last_cuda_error_string.argtypes = []
        L.kda_last_cuda_error_string.restype = ctypes.c_char_p
        L.kda_prefill_workspace_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
        L.kda_prefill_workspace_status.restype = ctypes.c_int
        L.kda_selftest_bounded_wait.argtypes = [vp, ctypes.c_uint32, ctypes.c_int32, vp]
        L.kda_selftest_bounded_wait.restype = ctypes.c_int
        _lib = L
        return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise KdaError(rc, what)
