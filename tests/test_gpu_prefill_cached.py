"""GPU parity of kda_prefill_varlen_cached: initial states read from cache rows by
index (gather rule), final states written back to cache rows (scatter rule) and
chunk-boundary checkpoints.

Checks: bit-identical with the unfused gather -> prefill -> scatter composition
on the GPU (same kernels, only the state addressing differs); the in-place
slot-reuse case against the oracle's gather -> prefill -> scatter; checkpoints
against the oracle's prefix states (state tolerance; fp32 checkpoints of a
sequence whose length is a multiple of the interval equal its final state bit
for bit); slots past the given capacity stay untouched."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import (kda_prefill_checkpoint_count, kda_prefill_varlen,
                                               kda_prefill_varlen_cached, kda_prefill_workspace_size,
                                               kda_prefill_workspace_status, kda_state_gather,
                                               kda_state_scatter)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_state_close, bytes_of, f64, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


def cu_of(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return cu


def workspace(T, B, H, D):
    return torch.empty(kda_prefill_workspace_size(T, B, H, D, D), dtype=torch.uint8, device=DEV)


def make_case(lengths, H, D, io, cache_dtype, itype, seed, n_rows=24, gap=64):
    cu = cu_of(lengths)
    B = len(lengths)
    inp = wl.token_inputs(cu[-1], H, D, D, io, seed=seed, device=DEV, decay_scale=0.3)
    pc = wl.paged_cache(n_rows, H, D, D, cache_dtype, H * D * D + gap, seed=seed + 1, device=DEV)
    idx_in = wl.gather_indices(B, n_rows, 0.25, seed + 2, itype)
    flags = wl.bernoulli_flags(B, 0.75, seed + 3)
    idx_out = wl.scatter_indices(B, n_rows, 0.25, seed + 4, itype)
    return cu, inp, pc, idx_in, flags, idx_out


@pytest.mark.parametrize("D,H,io", [(128, 40, torch.bfloat16), (128, 2, torch.bfloat16), (128, 2, torch.float32),
                                    (64, 3, torch.bfloat16), (32, 2, torch.float32)])
@pytest.mark.parametrize("cache_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("itype", [torch.int32, torch.int64])
def test_cached_equals_unfused_bit_for_bit(D, H, io, cache_dtype, itype):
    """D = 128, bf16: 40 heads x 4 sequences run the tensor-memory state pass with one CTA per
    (sequence, head), 2 heads its value-split form; fp32 with 2 heads the warp-pair register
    pass; the others the register pass with value splits."""
    lengths = [130, 0, 64, 257]
    cu, inp, pc, idx_in, flags, idx_out = make_case(lengths, H, D, io, cache_dtype, itype, seed=D + H)
    B, T = len(lengths), cu[-1]
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    idx_in_d, flags_d, idx_out_d = idx_in.to(DEV), flags.to(DEV), idx_out.to(DEV)
    # unfused: gather -> prefill -> scatter on a copy of the cache
    backing_a = pc.backing.clone()
    view_a = backing_a.as_strided(pc.view.shape, pc.view.stride(), pc.front)
    packed = torch.empty(B, H, D, D, dtype=cache_dtype, device=DEV)
    kda_state_gather(view_a, idx_in_d, packed, flags_d)
    out_a = torch.empty(T, H, D, dtype=io, device=DEV)
    fin_a = torch.empty(B, H, D, D, dtype=torch.float32, device=DEV)
    ws = workspace(T, B, H, D)
    kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out_a, ws,
                       init_state=packed, final_state=fin_a)
    kda_state_scatter(view_a, idx_out_d, fin_a)
    # fused
    out_b = torch.empty_like(out_a)
    fin_b = torch.full_like(fin_a, float("nan"))
    kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out_b, ws, pc.view,
                              idx_in_d, flags=flags_d, idx_out=idx_out_d, final_state=fin_b)
    torch.cuda.synchronize()
    assert kda_prefill_workspace_status(ws) == 0
    assert torch.equal(out_a.view(torch.uint8), out_b.view(torch.uint8))
    assert torch.equal(fin_a.view(torch.uint8), fin_b.view(torch.uint8))
    assert np.array_equal(bytes_of(backing_a), bytes_of(pc.backing))  # rows, gaps and guards


def test_cached_in_place_slot_reuse_against_oracle():
    """idx_out == idx_in (the serving slot-reuse case): each row is read as the initial
    state and overwritten with the final state; compared with the oracle's gather ->
    prefill -> scatter (cast to the bf16 cache)."""
    lengths, H, D = [100, 65, 1], 2, 64
    cu, inp, pc, _, _, _ = make_case(lengths, H, D, torch.bfloat16, torch.bfloat16, torch.int32, seed=7)
    B, T, N = len(lengths), cu[-1], pc.view.shape[0]
    idx = torch.tensor([3, 9, -1], dtype=torch.int32)
    flags = torch.tensor([True, False, True])
    before = raw(pc.backing)
    body = before[pc.front:pc.front + N * pc.row_stride].copy()
    P = H * D * D
    init_bits = oracle.gather(body, N, P, pc.row_stride, idx.numpy(), flags.numpy())  # bf16 bits [B, P]
    init = init_bits.astype(np.uint32) << 16
    init = init.view(np.float32).astype(np.float64).reshape(B, H, D, D)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out = torch.empty(T, H, D, dtype=torch.bfloat16, device=DEV)
    ws = workspace(T, B, H, D)
    kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws, pc.view,
                              idx.to(DEV), flags=flags.to(DEV), idx_out=idx.to(DEV))
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]), f64(inp["beta"]),
                                  cu, init=init, scale=D ** -0.5)
    assert_out_close(f64(out), o_ref)
    for b, r in enumerate(idx.tolist()):
        if 0 <= r < N:
            assert_state_close(f64(pc.view[r]), f_ref[b])
    after = raw(pc.backing)
    touched = np.zeros(after.size, dtype=bool)
    for r in idx.tolist():
        if 0 <= r < N:
            touched[pc.front + r * pc.row_stride:pc.front + r * pc.row_stride + P] = True
    assert np.array_equal(after[~touched], before[~touched])  # every other byte untouched


# tensor-memory (one CTA per pair, value-split), warp-pair and one-warp register passes
@pytest.mark.parametrize("D,H,io", [(128, 40, torch.bfloat16), (128, 2, torch.bfloat16), (128, 2, torch.float32),
                                    (64, 3, torch.bfloat16)])
@pytest.mark.parametrize("ckpt_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("every", [64, 128, 192])
def test_checkpoints_match_oracle(D, H, io, ckpt_dtype, every):
    lengths = [130, 0, 384, 63, 192]
    cu, inp, pc, idx_in, flags, _ = make_case(lengths, H, D, io, torch.float32, torch.int32, seed=every + D)
    B, T, N = len(lengths), cu[-1], pc.view.shape[0]
    n = kda_prefill_checkpoint_count(cu, every)
    assert n == sum(L // every for L in lengths)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out = torch.empty(T, H, D, dtype=io, device=DEV)
    fin = torch.empty(B, H, D, D, dtype=torch.float32, device=DEV)
    ck = torch.full((max(n, 1), H, D, D), float("nan"), dtype=ckpt_dtype, device=DEV)
    ws = workspace(T, B, H, D)
    kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws, pc.view,
                              idx_in.to(DEV), flags=flags.to(DEV), final_state=fin, checkpoints=ck[:n],
                              ckpt_every=every)
    torch.cuda.synchronize()
    assert kda_prefill_workspace_status(ws) == 0
    packed = torch.empty(B, H, D, D, dtype=torch.float32, device=DEV)
    kda_state_gather(pc.view, idx_in.to(DEV), packed, flags.to(DEV))
    heads = [0, H - 1]
    _, _, ck_ref = oracle.prefill_ckpt(f64(inp["q"][:, heads]), f64(inp["k"][:, heads]), f64(inp["v"][:, heads]),
                                       f64(inp["g"][:, heads]), f64(inp["beta"][:, heads]), cu, every,
                                       init=f64(packed[:, heads]), scale=D ** -0.5)
    assert ck_ref.shape[0] == n
    for s in range(n):
        assert_state_close(f64(ck[s, heads]), ck_ref[s], what=f"checkpoint {s}")
    # a sequence whose length is a multiple of `every` ends on a checkpoint: its final state
    slot = -1
    for b, L in enumerate(lengths):
        slot += L // every
        if L > 0 and L % every == 0:
            want = fin[b].to(ckpt_dtype)
            assert torch.equal(ck[slot].view(torch.uint8), want.view(torch.uint8))


def test_checkpoint_slots_past_capacity_are_not_written():
    lengths, H, D, every = [256, 128], 2, 64, 64
    cu, inp, pc, idx_in, flags, _ = make_case(lengths, H, D, torch.bfloat16, torch.float32, torch.int32, seed=5)
    n = kda_prefill_checkpoint_count(cu, every)  # 4 + 2
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out = torch.empty(cu[-1], H, D, dtype=torch.bfloat16, device=DEV)
    ck = torch.full((n, H, D, D), float("nan"), dtype=torch.float32, device=DEV)
    ws = workspace(cu[-1], 2, H, D)
    kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws, pc.view,
                              idx_in.to(DEV), flags=flags.to(DEV), checkpoints=ck[:n - 2], ckpt_every=every)
    torch.cuda.synchronize()
    assert not torch.isnan(ck[:n - 2]).any()
    assert torch.isnan(ck[n - 2:]).all()


def test_full_varlen_workload_fused_equals_unfused():
    """At the benchmark's size (16 sequences U[512, 8192], H = 32, D = 128, fp32 cache
    [1024, 32, 128, 128]): the fused call is bit-identical with gather -> prefill ->
    scatter, outputs and every cache byte."""
    w = wl.varlen()
    H, D = w.H, w.K
    cu = cu_of(w.lengths)
    T, B = cu[-1], w.B
    pc = wl.paged_cache(w.cache_rows, H, D, D, w.cache_dtype, w.cache_stride, seed=w.seed, device=DEV)
    inp = wl.token_inputs(T, H, D, D, w.io_dtype, seed=w.seed, device=DEV)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    gidx, gflags, sidx = w.gather_idx.to(DEV), w.gather_flags.to(DEV), w.scatter_idx.to(DEV)
    backing_a = pc.backing.clone()
    view_a = backing_a.as_strided(pc.view.shape, pc.view.stride(), pc.front)
    packed = torch.empty(B, H, D, D, dtype=pc.view.dtype, device=DEV)
    kda_state_gather(view_a, gidx, packed, gflags)
    out_a = torch.empty(T, H, D, dtype=w.io_dtype, device=DEV)
    fin = torch.empty(B, H, D, D, dtype=torch.float32, device=DEV)
    ws = workspace(T, B, H, D)
    kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out_a, ws, init_state=packed,
                       final_state=fin)
    kda_state_scatter(view_a, sidx, fin)
    out_b = torch.empty_like(out_a)
    kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out_b, ws, pc.view, gidx,
                              flags=gflags, idx_out=sidx)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.uint8), out_b.view(torch.uint8))
    assert torch.equal(backing_a.view(torch.uint8), pc.backing.view(torch.uint8))
    del backing_a, view_a
    torch.cuda.empty_cache()


def test_next_rows_capture_into_a_cuda_graph():
    """The fused prefill, INT8 store, conv1d and verify calls allocate nothing and take the
    stream per call: captured once, a replay on new input values gives the eager results."""
    from kimi_delta_attention_varlen_gb300 import (kda_ckpt_store_int8, kda_conv1d_varlen, kda_target_verify)
    lengths, H, D = [130, 64, 7], 2, 64
    cu = cu_of(lengths)
    T, B = cu[-1], len(lengths)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    pc = wl.paged_cache(8, H, D, D, torch.float32, None, seed=1, device=DEV)
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=2, device=DEV)
    idx = torch.tensor([3, 5, -1], dtype=torch.int32, device=DEV)
    x = torch.randn(T, 3 * H * D, device=DEV).to(torch.bfloat16)
    wt = torch.randn(3 * H * D, 4, device=DEV)
    R, L = 2, 3
    vin = {n: a.view(R, L, *a.shape[1:]) for n, a in wl.token_inputs(R * L, H, D, D, torch.bfloat16, seed=4,
                                                                     device=DEV).items()}
    ridx = torch.tensor([1, 6], dtype=torch.int32, device=DEV)
    inter = torch.arange(R * L, dtype=torch.int32, device=DEV).view(R, L)

    def make_outputs():
        return dict(out=torch.empty(T, H, D, dtype=torch.bfloat16, device=DEV),
                    q8=torch.empty(2, H, D, D, dtype=torch.int8, device=DEV),
                    sc=torch.empty(2, H, D, dtype=torch.float32, device=DEV),
                    y=torch.empty_like(x),
                    pool=torch.empty(R * L, H, D, D, dtype=torch.float32, device=DEV),
                    vout=torch.empty(R, L, H, D, dtype=torch.bfloat16, device=DEV))

    ws = workspace(T, B, H, D)

    def calls(o, cache):
        kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, o["out"], ws, cache,
                                  idx, idx_out=idx)
        kda_ckpt_store_int8(cache, idx[:2].contiguous(), torch.arange(2, dtype=torch.int32, device=DEV), o["q8"],
                            o["sc"])
        kda_conv1d_varlen(x, cu_t, wt, o["y"], activation="silu")
        kda_target_verify(vin["q"], vin["k"], vin["v"], vin["g"], vin["beta"], cache, ridx, o["pool"], inter,
                          o["vout"])

    g_out = make_outputs()
    start = pc.backing.clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        calls(g_out, pc.view)
    # new values in the captured input buffers, the cache restored, then replay
    for t in (inp["q"], inp["v"], x):
        t.copy_(torch.randn(t.shape, device=DEV).to(t.dtype))
    pc.backing.copy_(start)
    graph.replay()
    torch.cuda.synchronize()
    replayed_cache = pc.backing.clone()
    pc.backing.copy_(start)
    e_out = make_outputs()
    calls(e_out, pc.view)
    torch.cuda.synchronize()
    for k in e_out:
        assert torch.equal(g_out[k].view(torch.uint8), e_out[k].view(torch.uint8)), k
    assert torch.equal(replayed_cache.view(torch.uint8), pc.backing.view(torch.uint8))
