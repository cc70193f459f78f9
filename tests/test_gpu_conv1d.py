"""GPU parity of the short causal convolution (prefill over a varlen batch and the
per-request decode update) against the fp64 oracle.

Outputs: |d| <= 1e-5 * S (+ half a bf16 step of |y| for bf16 outputs), S = |bias| +
sum |w x| the magnitude of the terms (fp32 accumulation of at most five terms, the
SiLU's slope is below 1.1, and its fast exponential and division add a few ulps of
|y|, far below 1e-5 S; for bf16 outputs the sigmoid comes from one hardware tanh,
relative error about 2^-11, i.e. |y| 2^-12, inside the half bf16 step allowed).
States hold inputs: bit for bit (bf16 states of fp32
inputs round to nearest even, as the oracle's cast)."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import (kda_conv1d_update, kda_conv1d_varlen, kda_state_gather,
                                               kda_state_scatter)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import f64, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


def magnitude(x, cu, w, bias, init):
    """S_t[c] = |bias| + sum_i |w[c][i] x_{t-(W-1)+i}[c]| with the same window as the convolution."""
    absx = np.abs(x)
    ini = None if init is None else np.abs(init)
    s, _ = oracle.conv1d_varlen(absx, cu, np.abs(w), None if bias is None else np.abs(bias), "none", ini)
    return s


def check_out(got, ref, S, bf16):
    tol = 1e-5 * S + 1e-30
    if bf16:
        tol = tol + np.abs(ref) * 2.0 ** -8
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} outputs off, worst {float((err - tol).max()):.3e}"


def state_bits(vals64, dtype):
    if dtype == torch.float32:
        return vals64.astype(np.float32).view(np.uint32)
    return oracle.f32_to_bf16_bits(vals64.astype(np.float32))


def dev_bits(t):
    r = raw(t)
    return r.view(np.uint32) if t.dtype == torch.float32 else r


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("act", ["none", "silu"])
@pytest.mark.parametrize("state_dtype", [None, torch.float32, torch.bfloat16])
def test_conv1d_varlen_against_oracle(W, io, act, state_dtype):
    lengths = [0, 1, 2, 15, 16, 17, 0, 0, 100, 7, 0]
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    T, B, C = cu[-1], len(lengths), 1040  # two channel blocks, the second partial
    g = wl.generator(W * 10 + (io == torch.float32), "cpu")
    x = torch.randn(T, C, generator=g).to(io)
    w = torch.randn(C, W, generator=g)
    bias = torch.randn(C, generator=g)
    init = None
    if state_dtype is not None:
        init = torch.randn(B, W - 1, C, generator=g).to(state_dtype)
    xd, wd, bd = x.to(DEV), w.to(DEV), bias.to(DEV)
    y = torch.full((T, C), float("nan"), dtype=io, device=DEV)
    fin = None if state_dtype is None else torch.full((B, W - 1, C), float("nan"), dtype=state_dtype, device=DEV)
    kda_conv1d_varlen(xd, torch.tensor(cu, dtype=torch.int32, device=DEV), wd, y, bias=bd, activation=act,
                      init_state=None if init is None else init.to(DEV), final_state=fin)
    torch.cuda.synchronize()
    ini64 = None if init is None else f64(init)
    y_ref, f_ref = oracle.conv1d_varlen(f64(x), cu, f64(w), f64(bias), act, ini64)
    check_out(f64(y), y_ref, magnitude(f64(x), cu, f64(w), f64(bias), ini64), io == torch.bfloat16)
    if fin is not None:
        np.testing.assert_array_equal(dev_bits(fin), state_bits(f_ref, state_dtype))


def test_conv_states_move_with_the_state_copy_calls():
    """A conv-state cache row [W-1, C] is a kda_cache with h = 1: gather -> conv ->
    scatter updates the rows exactly as the oracle's states."""
    W, C, N = 4, 256, 6
    lengths = [5, 40, 0]
    cu = [0, 5, 45, 45]
    B, T = 3, 45
    pc = wl.paged_cache(N, 1, W - 1, C, torch.bfloat16, (W - 1) * C + 64, seed=3, device=DEV)
    gidx = torch.tensor([4, -1, 1], dtype=torch.int32, device=DEV)
    packed = torch.empty(B, 1, W - 1, C, dtype=torch.bfloat16, device=DEV)
    kda_state_gather(pc.view, gidx, packed)
    g = wl.generator(5, "cpu")
    x = torch.randn(T, C, generator=g).to(torch.bfloat16).to(DEV)
    w = torch.randn(C, W, generator=g).to(DEV)
    y = torch.empty_like(x)
    fin = torch.empty(B, 1, W - 1, C, dtype=torch.bfloat16, device=DEV)
    kda_conv1d_varlen(x, torch.tensor(cu, dtype=torch.int32, device=DEV), w, y, activation="silu",
                      init_state=packed.view(B, W - 1, C), final_state=fin.view(B, W - 1, C))
    kda_state_scatter(pc.view, gidx, fin)
    torch.cuda.synchronize()
    ini = f64(packed.view(B, W - 1, C))
    y_ref, f_ref = oracle.conv1d_varlen(f64(x), cu, f64(w), None, "silu", ini)
    check_out(f64(y), y_ref, magnitude(f64(x), cu, f64(w), None, ini), True)
    for b, r in ((0, 4), (2, 1)):
        np.testing.assert_array_equal(raw(pc.view[r, 0]), state_bits(f_ref[b], torch.bfloat16))


@pytest.mark.parametrize("W", [2, 4])
@pytest.mark.parametrize("cache_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("itype", [torch.int32, torch.int64])
def test_conv1d_update_against_oracle(W, cache_dtype, io, itype):
    R, C, N = 7, 2056, 9
    pc = wl.paged_cache(N, 1, W - 1, C, cache_dtype, (W - 1) * C + 32, seed=W, device=DEV)
    idx = torch.tensor([3, -1, 8, 0, N + 4, 5, 2], dtype=itype)
    g = wl.generator(17, "cpu")
    x = torch.randn(R, C, generator=g).to(io)
    w = torch.randn(C, W, generator=g)
    bias = torch.randn(C, generator=g)
    host = raw(pc.backing)
    body = np.ascontiguousarray(host[pc.front:pc.front + N * pc.row_stride])
    # the oracle's window before the token, for the magnitude bound
    states = np.zeros((R, W - 1, C))
    for r, row in enumerate(idx.tolist()):
        if 0 <= row < N:
            states[r] = f64(pc.view[row, 0])
    y = torch.empty(R, C, dtype=io, device=DEV)
    kda_conv1d_update(x.to(DEV), w.to(DEV), pc.view, idx.to(DEV), y, bias=bias.to(DEV), activation="silu")
    torch.cuda.synchronize()
    y_ref = oracle.conv1d_update(f64(x), f64(w), body, N, pc.row_stride, idx.numpy(), bias=f64(bias),
                                 activation="silu")
    S = magnitude(f64(x), list(range(R + 1)), f64(w), f64(bias), states)
    check_out(f64(y), y_ref, S, io == torch.bfloat16)
    want = host.copy()
    want[pc.front:pc.front + N * pc.row_stride] = body
    np.testing.assert_array_equal(raw(pc.backing), want)  # updated rows bit for bit, everything else untouched
