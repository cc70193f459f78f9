"""GPU parity of the next rows at the sizes and launch configurations bench.py times,
on sampled outputs the oracle evaluates one by one:

- target verification of the decode workload (R = 512, L = 4, bf16 cache
  [2048, 32, 128, 128], bf16 pool): sampled requests' outputs and every pool slot
  they write (outputs max|d| <= 2e-2 max|ref|, states ||dS|| <= 1e-2 ||S_ref||);
- the short convolution over the varlen batch's tokens (x [T, 3 H D] bf16, width 4,
  SiLU, bf16 states): sampled channel groups over all tokens (the conv tests'
  magnitude tolerance) and their final states bit for bit;
- INT8 checkpoints of 256 fp32 states of the [1024, 32, 128, 128] cache: sampled
  pairs' codes and scales bit for bit, and the rows loaded back."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import (kda_ckpt_load_int8, kda_ckpt_store_int8, kda_conv1d_varlen,
                                               kda_target_verify)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_state_close, f64, raw
from tests.test_gpu_conv1d import check_out, magnitude, state_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_target_verify_full_workload_sampled():
    w = wl.decode()
    R, L, H, D, N = w.R, 4, w.H, w.K, w.cache_rows
    P = H * D * D
    t = wl.token_inputs(R * L, H, D, D, w.io_dtype, seed=41, device=DEV)
    inp = {n: x.view(R, L, *x.shape[1:]) for n, x in t.items()}
    pc = wl.paged_cache(N, H, D, D, w.cache_dtype, None, seed=5, device=DEV)
    idx = w.idx.clone()
    pool = torch.empty(R * L, H, D, D, dtype=w.cache_dtype, device=DEV)
    inter = torch.arange(R * L, dtype=torch.int32, device=DEV).view(R, L)
    out = torch.empty(R, L, H, D, dtype=w.io_dtype, device=DEV)
    kda_target_verify(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pc.view, idx.to(DEV), pool, inter, out)
    torch.cuda.synchronize()
    invalid = [r for r in range(R) if int(idx[r]) < 0]
    sample = sorted({0, 1, 255, 511, *(invalid[:1])})
    rows = [int(idx[r]) for r in sample]
    host = raw(pc.backing)
    mini = np.zeros(len(sample) * P, dtype=host.dtype)
    for j, x in enumerate(rows):
        if x >= 0:
            s0 = pc.front + x * pc.row_stride
            mini[j * P:(j + 1) * P] = host[s0:s0 + P]
    mini_idx = np.array([j if x >= 0 else -1 for j, x in enumerate(rows)], dtype=np.int64)
    mini_pool = np.zeros(len(sample) * L * P, dtype=host.dtype)
    mini_inter = np.arange(len(sample) * L, dtype=np.int64).reshape(len(sample), L)
    pick = torch.tensor(sample, dtype=torch.long, device=DEV)
    o_ref = oracle.target_verify(f64(inp["q"][pick]), f64(inp["k"][pick]), f64(inp["v"][pick]), f64(inp["g"][pick]),
                                 f64(inp["beta"][pick]), mini, len(sample), P, mini_idx, mini_pool, len(sample) * L,
                                 P, mini_inter, scale=D ** -0.5)
    assert_out_close(f64(out[pick]), o_ref)
    got_pool = raw(pool).reshape(-1)
    for j, r in enumerate(sample):
        for tt in range(L):
            s = r * L + tt
            got = got_pool[s * P:(s + 1) * P]
            want = mini_pool[(j * L + tt) * P:(j * L + tt + 1) * P]
            assert_state_close(bf16_bits_to_f64(got), bf16_bits_to_f64(want), what=f"request {r} token {tt}")
    del pool, pc
    torch.cuda.empty_cache()


def test_conv1d_full_batch_sampled_channels():
    w16 = wl.varlen(0)
    cu = [0]
    for n in w16.lengths:
        cu.append(cu[-1] + n)
    T, B, C, W = cu[-1], len(w16.lengths), 3 * w16.H * w16.K, 4
    g = torch.Generator(device=DEV).manual_seed(0)
    x = torch.randn(T, C, generator=g, device=DEV).to(torch.bfloat16)
    wt = torch.randn(C, W, generator=g, device=DEV)
    init = torch.randn(B, W - 1, C, generator=g, device=DEV).to(torch.bfloat16)
    y = torch.empty_like(x)
    fin = torch.empty_like(init)
    kda_conv1d_varlen(x, torch.tensor(cu, dtype=torch.int32, device=DEV), wt, y, activation="silu",
                      init_state=init, final_state=fin)
    torch.cuda.synchronize()
    for c0 in (0, 4096 + 8, C - 8):  # channel groups of one thread each (8 channels)
        cs = slice(c0, c0 + 8)
        xs, ws_, ini = f64(x[:, cs]), f64(wt[cs]), f64(init[:, :, cs])
        y_ref, f_ref = oracle.conv1d_varlen(xs, cu, ws_, None, "silu", ini)
        check_out(f64(y[:, cs]), y_ref, magnitude(xs, cu, ws_, None, ini), True)
        np.testing.assert_array_equal(raw(fin[:, :, cs].contiguous()), state_bits(f_ref, torch.bfloat16))
    del x, y
    torch.cuda.empty_cache()


def test_int8_checkpoints_full_size_sampled():
    N, H, D, pairs = 1024, 32, 128, 256
    P = H * D * D
    pc = wl.paged_cache(N, H, D, D, torch.float32, None, seed=7, device=DEV)
    rows = torch.randperm(N, generator=torch.Generator().manual_seed(21))[:pairs].to(torch.int32)
    slots = torch.arange(pairs, dtype=torch.int32)
    q = torch.empty(pairs, H, D, D, dtype=torch.int8, device=DEV)
    sc = torch.empty(pairs, H, D, dtype=torch.float32, device=DEV)
    kda_ckpt_store_int8(pc.view, rows.to(DEV), slots.to(DEV), q, sc)
    # load every slot back into a second cache, at shifted rows
    back = wl.paged_cache(N, H, D, D, torch.float32, None, seed=0, device=DEV, fill=False)
    dst = (rows + 1) % N
    kda_ckpt_load_int8(q, sc, slots.to(DEV), back.view, dst.to(DEV))
    torch.cuda.synchronize()
    sample = [0, 1, 100, 255]
    host = raw(pc.backing)
    mini = np.zeros(len(sample) * P, dtype=np.float32)
    for j, s in enumerate(sample):
        s0 = pc.front + int(rows[s]) * pc.row_stride
        mini[j * P:(j + 1) * P] = host[s0:s0 + P]
    n = len(sample)
    q_ref = np.zeros((n, H, D, D), dtype=np.int8)
    sc_ref = np.zeros((n, H, D), dtype=np.float32)
    oracle.ckpt_store_int8(mini, n, P, H, D, D, np.arange(n), np.arange(n), q_ref, sc_ref)
    pick = torch.tensor(sample, dtype=torch.long, device=DEV)
    np.testing.assert_array_equal(q[pick].cpu().numpy(), q_ref)
    np.testing.assert_array_equal(sc[pick].cpu().numpy().view(np.uint32), sc_ref.view(np.uint32))
    loaded = np.zeros(n * P, dtype=np.float32)
    oracle.ckpt_load_int8(q_ref, sc_ref, np.arange(n), np.arange(n), loaded, n, P, H, D, D)
    host_back = raw(back.backing)
    for j, s in enumerate(sample):
        s0 = back.front + int(dst[s]) * back.row_stride
        np.testing.assert_array_equal(host_back[s0:s0 + P].view(np.uint32), loaded[j * P:(j + 1) * P].view(np.uint32))
    del pc, back, q
    torch.cuda.empty_cache()
