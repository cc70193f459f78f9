"""Kimi Delta Attention (KDA) serving hot path on GB300 (sm_103a).

Thin Python binding of the C ABI in include/kda.h (libkda.so).  The functions
keep the C names; they take torch tensors (device memory) and only marshal
arguments - every step of the computation runs in the library's CUDA kernels.

    kda_state_gather(cache, idx, packed, flags=None)
    kda_state_scatter(cache, idx, packed)
    kda_prefill_workspace_size(total_tokens, num_seqs, h, dk, dv)
    kda_prefill_varlen(q, k, v, g, beta, cu_seqlens, out, workspace, ...)
    kda_decode_step(q, k, v, g, beta, cache, idx, out, ...)

`cache` is a 4-D tensor view [N, H, V, K] whose inner [H, V, K] block is dense
and whose stride(0) >= H*V*K (page gaps allowed); its data_ptr() already
includes any storage offset.
"""
from __future__ import annotations

import ctypes

import torch

from ._abi import (EXPORTED, KDA_BF16, KDA_F32, KDA_I32, KDA_I64, LIB_PATH, KdaCache, KdaError,
                   _check, lib)

__all__ = [
    "kda_state_gather", "kda_state_scatter", "kda_prefill_workspace_size", "kda_prefill_workspace_size_compact",
    "kda_prefill_varlen",
    "kda_prefill_varlen_cached", "kda_prefill_checkpoint_count", "kda_prefill_varlen_noalloc",
    "kda_prefill_noalloc_status", "kda_decode_step",
    "kda_ckpt_store_int8", "kda_ckpt_load_int8", "kda_conv1d_varlen", "kda_conv1d_update", "kda_target_verify",
    "kda_status_string", "kda_prefill_workspace_status", "kda_selftest_bounded_wait", "cache_descriptor",
    "KdaError", "EXPORTED", "LIB_PATH",
]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KDA_F32
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"expected float32 or bfloat16, got {t.dtype}")


def _itype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.int32:
        return KDA_I32
    if t.dtype == torch.int64:
        return KDA_I64
    raise TypeError(f"indices must be int32 or int64, got {t.dtype}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _ptr(t):
    return None if t is None else t.data_ptr()


def cache_descriptor(cache: torch.Tensor) -> KdaCache:
    """kda_cache for a [N, H, V, K] view with a dense inner block."""
    _need(cache.dim() == 4, "cache must be a 4-D view [N, H, V, K]")
    N, H, V, K = cache.shape
    for d, want in ((1, V * K), (2, K), (3, 1)):
        _need(cache.size(d) == 1 or cache.stride(d) == want,
              "cache rows must hold a dense [H, V, K] block")
    return KdaCache(cache.data_ptr(), _dtype_code(cache), 0, N, H, V, K, cache.stride(0))


def _index_vector(idx: torch.Tensor) -> None:
    _need(idx.dim() == 1 and idx.is_contiguous(), "indices must be a contiguous 1-D tensor")


def kda_state_gather(cache: torch.Tensor, idx: torch.Tensor, packed: torch.Tensor,
                     flags: torch.Tensor | None = None, stream=None) -> None:
    """packed[s] = cache[idx[s]] for valid indices with a true flag, else zeros."""
    d = cache_descriptor(cache)
    _index_vector(idx)
    S = idx.numel()
    _need(packed.is_contiguous() and packed.dtype == cache.dtype and
          tuple(packed.shape) == (S, *cache.shape[1:]), "packed must be contiguous [S, H, V, K], cache dtype")
    if flags is not None:
        _need(flags.dtype in (torch.bool, torch.uint8) and flags.is_contiguous() and flags.numel() == S,
              "flags must be a contiguous bool tensor of length S")
    rc = lib().kda_state_gather(ctypes.byref(d), _ptr(idx), _itype_code(idx), S, _ptr(flags), _ptr(packed),
                                _stream(stream))
    _check(rc, "kda_state_gather")


def kda_state_scatter(cache: torch.Tensor, idx: torch.Tensor, packed: torch.Tensor, stream=None) -> None:
    """cache[idx[s]] = packed[s] converted to the cache dtype, for valid indices."""
    d = cache_descriptor(cache)
    _index_vector(idx)
    S = idx.numel()
    _need(packed.is_contiguous() and tuple(packed.shape) == (S, *cache.shape[1:]),
          "packed must be contiguous [S, H, V, K]")
    rc = lib().kda_state_scatter(ctypes.byref(d), _ptr(idx), _itype_code(idx), S, _ptr(packed),
                                 _dtype_code(packed), _stream(stream))
    _check(rc, "kda_state_scatter")


def kda_prefill_workspace_size(total_tokens: int, num_seqs: int, h: int, dk: int, dv: int) -> int:
    return int(lib().kda_prefill_workspace_size(total_tokens, num_seqs, h, dk, dv))



def kda_prefill_workspace_size_compact(total_tokens: int, num_seqs: int, h: int, dk: int, dv: int,
                                       dtype=torch.bfloat16) -> int:
    """Smallest workspace the prefill accepts for inputs of `dtype`: for bf16 at head size
    128 the chunk table only (the call then runs the fused kernel, with no per-chunk records
    in memory); otherwise kda_prefill_workspace_size."""
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib().kda_prefill_workspace_size_compact(total_tokens, num_seqs, h, dk, dv, code))

def kda_prefill_varlen(q, k, v, g, beta, cu_seqlens, out, workspace, *, scale: float | None = None,
                       qk_l2norm: bool = True, init_state=None, final_state=None, stream=None,
                       events=None) -> None:
    """Chunkwise gated delta-rule prefill over a cu_seqlens varlen batch.

    q, k: [T, H, K]; v, out: [T, H, V] (bf16 or fp32, one dtype); g: [T, H, K] fp32;
    beta: [T, H] fp32; cu_seqlens: [B + 1] int32; init_state: [B, H, V, K] fp32/bf16 or
    None; final_state: [B, H, V, K] fp32 or None; workspace: uint8 device tensor of at
    least kda_prefill_workspace_size(T, B, H, K, V) bytes.  events: optional list of four
    torch.cuda.Event (timing enabled) recorded at the boundaries of the three kernels
    (kda_prefill_varlen_timed); a None entry leaves that boundary unrecorded."""
    T, H, K = q.shape
    V = v.shape[2]
    B = cu_seqlens.numel() - 1
    for name, t, shape in (("q", q, (T, H, K)), ("k", k, (T, H, K)), ("v", v, (T, H, V)),
                           ("out", out, (T, H, V)), ("g", g, (T, H, K)), ("beta", beta, (T, H))):
        _need(tuple(t.shape) == shape and t.is_contiguous(), f"{name} must be contiguous {shape}")
    _need(k.dtype == q.dtype and v.dtype == q.dtype and out.dtype == q.dtype, "q, k, v, out share a dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g and beta must be float32")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous() and B >= 1,
          "cu_seqlens must be a contiguous int32 tensor of B + 1 >= 2 offsets")
    init_code = 0
    if init_state is not None:
        _need(tuple(init_state.shape) == (B, H, V, K) and init_state.is_contiguous(),
              "init_state must be contiguous [B, H, V, K]")
        init_code = _dtype_code(init_state)
    if final_state is not None:
        _need(tuple(final_state.shape) == (B, H, V, K) and final_state.is_contiguous() and
              final_state.dtype == torch.float32, "final_state must be contiguous float32 [B, H, V, K]")
    _need(workspace.dtype == torch.uint8 and workspace.is_contiguous(), "workspace must be a uint8 tensor")
    if scale is None:
        scale = K ** -0.5
    args = (_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(g), _ptr(beta), _ptr(cu_seqlens), B, T, H, K, V,
            float(scale), 1 if qk_l2norm else 0, _ptr(init_state), init_code, _ptr(final_state), _ptr(out),
            _ptr(workspace), workspace.numel(), _stream(stream))
    if events is None:
        _check(lib().kda_prefill_varlen(*args), "kda_prefill_varlen")
        return
    _need(len(events) == 4, "events: four torch.cuda.Event (None leaves that boundary unrecorded)")
    handles = []
    for ev in events:
        if ev is None:
            handles.append(None)
            continue
        if not ev.cuda_event:  # torch creates the event lazily at its first record
            ev.record()
        handles.append(ev.cuda_event)
    arr = (ctypes.c_void_p * 4)(*handles)
    _check(lib().kda_prefill_varlen_timed(*args, arr), "kda_prefill_varlen_timed")


def kda_prefill_checkpoint_count(cu_seqlens, ckpt_every: int) -> int:
    """Checkpoint slots kda_prefill_varlen_cached writes: sum of len_b // ckpt_every over
    the sequences of cu_seqlens (a host int32 tensor or a list of offsets)."""
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu().contiguous()
    n = lib().kda_prefill_checkpoint_count(ctypes.cast(cu.data_ptr(), ctypes.POINTER(ctypes.c_int32)),
                                           cu.numel() - 1, int(ckpt_every))
    _need(n >= 0, "cu_seqlens must be non-decreasing and ckpt_every a positive multiple of 64")
    return int(n)


def kda_prefill_varlen_cached(q, k, v, g, beta, cu_seqlens, out, workspace, cache, idx_in, *,
                              flags=None, idx_out=None, final_state=None, checkpoints=None,
                              ckpt_every: int = 0, scale: float | None = None, qk_l2norm: bool = True,
                              stream=None) -> None:
    """kda_prefill_varlen with initial states read from cache rows idx_in (with flags, the
    gather rule) and final states written to cache rows idx_out (the scatter rule, cast
    to the cache dtype), in one pass; optional checkpoints [slots, H, V, K] (fp32 or bf16)
    hold the state after every ckpt_every tokens of each sequence (sequence-major; see
    kda_prefill_checkpoint_count)."""
    T, H, K = q.shape
    V = v.shape[2]
    B = cu_seqlens.numel() - 1
    for name, t, shape in (("q", q, (T, H, K)), ("k", k, (T, H, K)), ("v", v, (T, H, V)),
                           ("out", out, (T, H, V)), ("g", g, (T, H, K)), ("beta", beta, (T, H))):
        _need(tuple(t.shape) == shape and t.is_contiguous(), f"{name} must be contiguous {shape}")
    _need(k.dtype == q.dtype and v.dtype == q.dtype and out.dtype == q.dtype, "q, k, v, out share a dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g and beta must be float32")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous() and B >= 1,
          "cu_seqlens must be a contiguous int32 tensor of B + 1 >= 2 offsets")
    d = cache_descriptor(cache)
    _index_vector(idx_in)
    _need(idx_in.numel() == B, "idx_in must hold one index per sequence")
    if idx_out is not None:
        _index_vector(idx_out)
        _need(idx_out.numel() == B and idx_out.dtype == idx_in.dtype,
              "idx_out: one index per sequence, idx_in's dtype")
    if flags is not None:
        _need(flags.dtype in (torch.bool, torch.uint8) and flags.is_contiguous() and flags.numel() == B,
              "flags must be a contiguous bool tensor of length B")
    if final_state is not None:
        _need(tuple(final_state.shape) == (B, H, V, K) and final_state.is_contiguous() and
              final_state.dtype == torch.float32, "final_state must be contiguous float32 [B, H, V, K]")
    slots, ck_code = 0, 0
    if checkpoints is not None:
        _need(checkpoints.dim() == 4 and tuple(checkpoints.shape[1:]) == (H, V, K) and checkpoints.is_contiguous(),
              "checkpoints must be contiguous [slots, H, V, K]")
        slots, ck_code = checkpoints.shape[0], _dtype_code(checkpoints)
    _need(workspace.dtype == torch.uint8 and workspace.is_contiguous(), "workspace must be a uint8 tensor")
    if scale is None:
        scale = K ** -0.5
    rc = lib().kda_prefill_varlen_cached(
        _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(g), _ptr(beta), _ptr(cu_seqlens), B, T, H, K, V,
        float(scale), 1 if qk_l2norm else 0, ctypes.byref(d), _ptr(idx_in), _ptr(flags), _ptr(idx_out),
        _itype_code(idx_in), _ptr(final_state), _ptr(checkpoints), ck_code, int(ckpt_every), slots, _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "kda_prefill_varlen_cached")


def kda_target_verify(q, k, v, g, beta, cache, idx, pool, inter_idx, out, *, scale: float | None = None,
                      qk_l2norm: bool = True, stream=None) -> None:
    """L draft tokens per request from cache rows idx[r] (read only); outputs to out and the
    state after token t of request r to pool row inter_idx[r, t].  q, k, g: [R, L, H, K];
    v, out: [R, L, H, V]; beta: [R, L, H]; cache, pool: [N, H, V, K] views."""
    R, L, H, K = q.shape
    V = v.shape[3]
    for name, t, shape in (("q", q, (R, L, H, K)), ("k", k, (R, L, H, K)), ("v", v, (R, L, H, V)),
                           ("out", out, (R, L, H, V)), ("g", g, (R, L, H, K)), ("beta", beta, (R, L, H))):
        _need(tuple(t.shape) == shape and t.is_contiguous(), f"{name} must be contiguous {shape}")
    _need(k.dtype == q.dtype and v.dtype == q.dtype and out.dtype == q.dtype, "q, k, v, out share a dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g and beta must be float32")
    _index_vector(idx)
    _need(idx.numel() == R, "idx must hold one index per request")
    _need(inter_idx.is_contiguous() and tuple(inter_idx.shape) == (R, L) and inter_idx.dtype == idx.dtype,
          "inter_idx must be a contiguous [R, L] tensor of idx's dtype")
    dc, dp = cache_descriptor(cache), cache_descriptor(pool)
    if scale is None:
        scale = K ** -0.5
    rc = lib().kda_target_verify(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(g), _ptr(beta), R, L, H, K, V,
                                 float(scale), 1 if qk_l2norm else 0, ctypes.byref(dc), _ptr(idx), ctypes.byref(dp),
                                 _ptr(inter_idx), _itype_code(idx), _ptr(out), _stream(stream))
    _check(rc, "kda_target_verify")


_ACT = {"none": 0, "silu": 1}


def _conv_weights(weight, bias, C):
    _need(weight.dtype == torch.float32 and weight.dim() == 2 and weight.shape[0] == C and weight.is_contiguous(),
          "weight must be a contiguous float32 [C, W] tensor")
    if bias is not None:
        _need(bias.dtype == torch.float32 and tuple(bias.shape) == (C,) and bias.is_contiguous(),
              "bias must be a contiguous float32 [C] tensor")
    return weight.shape[1]


def kda_conv1d_varlen(x, cu_seqlens, weight, y, *, bias=None, activation: str = "none", init_state=None,
                      final_state=None, stream=None) -> None:
    """Depthwise causal convolution over a varlen batch: x, y [T, C] (bf16 / fp32);
    weight [C, W] fp32; bias [C] fp32 or None; init/final states [B, W-1, C] (fp32 / bf16,
    one dtype) or None."""
    T, C = x.shape
    B = cu_seqlens.numel() - 1
    W = _conv_weights(weight, bias, C)
    _need(tuple(y.shape) == (T, C) and y.dtype == x.dtype and x.is_contiguous() and y.is_contiguous(),
          "x and y must be contiguous [T, C] tensors of one dtype")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous() and B >= 1,
          "cu_seqlens must be a contiguous int32 tensor of B + 1 >= 2 offsets")
    st_code = 0
    for name, t in (("init_state", init_state), ("final_state", final_state)):
        if t is not None:
            _need(tuple(t.shape) == (B, W - 1, C) and t.is_contiguous(), f"{name} must be contiguous [B, W-1, C]")
            st_code = _dtype_code(t)
    if init_state is not None and final_state is not None:
        _need(init_state.dtype == final_state.dtype, "init_state and final_state share a dtype")
    rc = lib().kda_conv1d_varlen(_ptr(x), _dtype_code(x), _ptr(cu_seqlens), B, T, C, W, _ptr(weight), _ptr(bias),
                                 _ACT[activation], _ptr(init_state), _ptr(final_state), st_code, _ptr(y),
                                 _stream(stream))
    _check(rc, "kda_conv1d_varlen")


def kda_conv1d_update(x, weight, conv_cache, idx, y, *, bias=None, activation: str = "none", stream=None) -> None:
    """One token per request on conv-state cache rows in place: x, y [R, C]; conv_cache a
    [N, 1, W-1, C] view (rows of W-1 states, oldest first); idx [R] int32/int64."""
    R, C = x.shape
    W = _conv_weights(weight, bias, C)
    _need(tuple(y.shape) == (R, C) and y.dtype == x.dtype and x.is_contiguous() and y.is_contiguous(),
          "x and y must be contiguous [R, C] tensors of one dtype")
    _index_vector(idx)
    _need(idx.numel() == R, "idx must hold one index per request")
    d = cache_descriptor(conv_cache)
    rc = lib().kda_conv1d_update(_ptr(x), _dtype_code(x), R, C, W, _ptr(weight), _ptr(bias), _ACT[activation],
                                 ctypes.byref(d), _ptr(idx), _itype_code(idx), _ptr(y), _stream(stream))
    _check(rc, "kda_conv1d_update")


def _ckpt_pools(cache, qdata, scale):
    _, H, V, K = cache.shape
    _need(qdata.dtype == torch.int8 and qdata.dim() == 4 and tuple(qdata.shape[1:]) == (H, V, K) and
          qdata.is_contiguous(), "qdata must be a contiguous int8 [slots, H, V, K] tensor")
    _need(scale.dtype == torch.float32 and tuple(scale.shape) == (qdata.shape[0], H, K) and scale.is_contiguous(),
          "scale must be a contiguous float32 [slots, H, K] tensor")


def kda_ckpt_store_int8(cache, src_rows, dst_slots, qdata, scale, stream=None) -> None:
    """Quantise active cache rows src_rows[s] into int8 checkpoint slots dst_slots[s]:
    per (slot, head, k) scale = max_v |x| / 127, codes round(x / scale) in [-127, 127]."""
    d = cache_descriptor(cache)
    _index_vector(src_rows)
    _index_vector(dst_slots)
    _need(src_rows.numel() == dst_slots.numel() and src_rows.dtype == dst_slots.dtype,
          "src_rows and dst_slots: same length and dtype")
    _ckpt_pools(cache, qdata, scale)
    rc = lib().kda_ckpt_store_int8(ctypes.byref(d), _ptr(src_rows), _ptr(dst_slots), _itype_code(src_rows),
                                   src_rows.numel(), _ptr(qdata), _ptr(scale), qdata.shape[0], _stream(stream))
    _check(rc, "kda_ckpt_store_int8")


def kda_ckpt_load_int8(qdata, scale, src_slots, cache, dst_rows, stream=None) -> None:
    """Dequantise int8 checkpoint slots src_slots[s] into active cache rows dst_rows[s]."""
    d = cache_descriptor(cache)
    _index_vector(src_slots)
    _index_vector(dst_rows)
    _need(src_slots.numel() == dst_rows.numel() and src_slots.dtype == dst_rows.dtype,
          "src_slots and dst_rows: same length and dtype")
    _ckpt_pools(cache, qdata, scale)
    rc = lib().kda_ckpt_load_int8(_ptr(qdata), _ptr(scale), qdata.shape[0], _ptr(src_slots), _ptr(dst_rows),
                                  _itype_code(src_slots), src_slots.numel(), ctypes.byref(d), _stream(stream))
    _check(rc, "kda_ckpt_load_int8")


def kda_decode_step(q, k, v, g, beta, cache, idx, out, *, scale: float | None = None,
                    qk_l2norm: bool = True, stream=None) -> None:
    """One recurrent token per request on cache rows, in place.

    q, k: [R, H, K]; v, out: [R, H, V] (bf16 or fp32); g: [R, H, K] fp32; beta: [R, H] fp32;
    cache: [N, H, V, K] view; idx: [R] int32/int64."""
    R, H, K = q.shape
    V = v.shape[2]
    for name, t, shape in (("q", q, (R, H, K)), ("k", k, (R, H, K)), ("v", v, (R, H, V)),
                           ("out", out, (R, H, V)), ("g", g, (R, H, K)), ("beta", beta, (R, H))):
        _need(tuple(t.shape) == shape and t.is_contiguous(), f"{name} must be contiguous {shape}")
    _need(k.dtype == q.dtype and v.dtype == q.dtype and out.dtype == q.dtype, "q, k, v, out share a dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g and beta must be float32")
    _index_vector(idx)
    _need(idx.numel() == R, "idx must hold one index per request")
    d = cache_descriptor(cache)
    if scale is None:
        scale = K ** -0.5
    rc = lib().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(g), _ptr(beta), R, H, K, V,
                               float(scale), 1 if qk_l2norm else 0, ctypes.byref(d), _ptr(idx),
                               _itype_code(idx), _ptr(out), _stream(stream))
    _check(rc, "kda_decode_step")


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(status).decode()


def kda_prefill_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Device status word of the last prefill on this workspace (0 = all waits completed).
    Synchronises the stream."""
    out = ctypes.c_int32(-1)
    _check(lib().kda_prefill_workspace_status(_ptr(workspace), ctypes.byref(out), _stream(stream)),
           "kda_prefill_workspace_status")
    return int(out.value)


def kda_selftest_bounded_wait(status: torch.Tensor, polls: int, arrive: bool, stream=None) -> None:
    """One CTA waits, with the kernels' bounded mbarrier wait (at most `polls` polls), on a
    barrier that gets its arrival (`arrive`) or never does; writes 0 (completed) or 1
    (expired) to the device int32 tensor `status`.  Asynchronous."""
    if status.dtype != torch.int32 or status.numel() < 1:
        raise ValueError("status must be a device int32 tensor")
    _check(lib().kda_selftest_bounded_wait(_ptr(status), int(polls), 1 if arrive else 0, _stream(stream)),
           "kda_selftest_bounded_wait")


def kda_prefill_varlen_noalloc(q, k, v, g, beta, cu_seqlens, out, *, scale: float | None = None,
                               qk_l2norm: bool = True, init_state=None, final_state=None, stream=None) -> None:
    """kda_prefill_varlen without a workspace argument, for callers that cannot
    allocate device memory (a host program with no device allocator, or a runtime
    whose device memory is fixed at start-up and allows no allocation while
    serving).  The kernels use a fixed scratch array of the library
    (KDA_NOALLOC_SCRATCH_BYTES); batches that need more raise KdaError
    (KDA_ERR_WORKSPACE).  The first call on a device looks up the scratch address
    (make it before any stream capture); calls that overlap on the GPU race."""
    T, H, K = q.shape
    V = v.shape[2]
    B = cu_seqlens.numel() - 1
    for name, t, shape in (("q", q, (T, H, K)), ("k", k, (T, H, K)), ("v", v, (T, H, V)),
                           ("out", out, (T, H, V)), ("g", g, (T, H, K)), ("beta", beta, (T, H))):
        _need(tuple(t.shape) == shape and t.is_contiguous(), f"{name} must be contiguous {shape}")
    _need(k.dtype == q.dtype and v.dtype == q.dtype and out.dtype == q.dtype, "q, k, v, out share a dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32, "g and beta must be float32")
    _need(cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous() and B >= 1,
          "cu_seqlens must be a contiguous int32 tensor of B + 1 >= 2 offsets")
    init_code = 0
    if init_state is not None:
        _need(tuple(init_state.shape) == (B, H, V, K) and init_state.is_contiguous(),
              "init_state must be contiguous [B, H, V, K]")
        init_code = _dtype_code(init_state)
    if final_state is not None:
        _need(tuple(final_state.shape) == (B, H, V, K) and final_state.is_contiguous() and
              final_state.dtype == torch.float32, "final_state must be contiguous float32 [B, H, V, K]")
    if scale is None:
        scale = K ** -0.5
    rc = lib().kda_prefill_varlen_noalloc(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(g), _ptr(beta),
                                          _ptr(cu_seqlens), B, T, H, K, V, float(scale), 1 if qk_l2norm else 0,
                                          _ptr(init_state), init_code, _ptr(final_state), _ptr(out),
                                          _stream(stream))
    _check(rc, "kda_prefill_varlen_noalloc")


def kda_prefill_noalloc_status(stream=None) -> int:
    """Device status word of the last kda_prefill_varlen_noalloc call on the current
    device (0 = every internal wait completed; the codes of kda_prefill_workspace_status).
    The caller never sees the library's fixed scratch array, so this is the only way to
    read it.  Synchronises the stream."""
    out = ctypes.c_int32(-1)
    _check(lib().kda_prefill_noalloc_status(ctypes.byref(out), _stream(stream)), "kda_prefill_noalloc_status")
    return int(out.value)
