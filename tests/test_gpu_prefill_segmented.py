"""GPU parity of the segmented prefill: one sequence at head size 128, bf16, with few
heads and at least two segments of 256 chunks runs its chunk preparation and its
value-split state pass segment by segment, the pass of one segment overlapping the
preparation of the next on a second stream, with the state handed between segments
through the workspace.

Checked against the token-by-token fp64 oracle at the method's tolerances (outputs
max|d| <= 2e-2 max|ref|, states ||dS||_F <= 1e-2 ||S_ref||_F), and bit for bit against
the same sequence run unsegmented (a batch of it and an empty sequence, which takes the
same kernels in one launch each): outputs, final states, checkpoints on and off the
segment boundaries, and the cache row written by the cache-indexed entry point; and
captured into a CUDA graph, whose replay matches the eager call."""
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import (kda_prefill_checkpoint_count, kda_prefill_varlen,
                                               kda_prefill_varlen_cached, kda_prefill_workspace_size,
                                               kda_prefill_workspace_status)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_state_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128
SEG = 256 * 64  # tokens per segment


def workspace(cu, H):
    return torch.empty(kda_prefill_workspace_size(cu[-1], len(cu) - 1, H, D, D), dtype=torch.uint8, device=DEV)


def prefill(inp, cu, H, init, every=0, n_slots=0):
    T, B = cu[-1], len(cu) - 1
    out = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    fin = torch.full((B, H, D, D), float("nan"), device=DEV)
    ws = workspace(cu, H)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    if every:
        rows = wl.paged_cache(B + 2, H, D, D, torch.float32, H * D * D + 64, seed=5, device=DEV)
        rows.view[:B].copy_(init[:B])
        idx_in = torch.arange(B, dtype=torch.int32)
        idx_out = torch.arange(B, dtype=torch.int32) + 2
        ck = torch.full((max(n_slots, 1), H, D, D), float("nan"), device=DEV)
        kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws, rows.view,
                                  idx_in.to(DEV), idx_out=idx_out.to(DEV), final_state=fin, checkpoints=ck[:n_slots],
                                  ckpt_every=every)
        torch.cuda.synchronize()
        assert kda_prefill_workspace_status(ws) == 0
        return out, fin, ck[:n_slots], rows.view[2:2 + B].clone()
    kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws, init_state=init,
                       final_state=fin)
    torch.cuda.synchronize()
    assert kda_prefill_workspace_status(ws) == 0
    return out, fin, None, None


@pytest.mark.parametrize("T,H", [(2 * SEG, 4), (2 * SEG + 37, 8), (3 * SEG - 64 * 3 + 5, 2)])
def test_segmented_equals_unsegmented_and_oracle(T, H):
    """Two segments exactly, two and a 1-chunk tail of 37 tokens, and three segments whose last
    is short: bit-identical with the unsegmented run, and within tolerance of the oracle."""
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=T % 997 + H, device=DEV, decay_scale=0.3)
    init = torch.randn(2, H, D, D, generator=wl.generator(T % 89, DEV), device=DEV) * 0.5
    out_s, fin_s, _, _ = prefill(inp, [0, T], H, init[:1])
    out_u, fin_u, _, _ = prefill(inp, [0, T, T], H, init)
    assert torch.equal(out_s.view(torch.uint8), out_u.view(torch.uint8))
    assert torch.equal(fin_s[0], fin_u[0])
    heads = [0, H - 1]
    o_ref, f_ref = oracle.prefill(f64(inp["q"][:, heads]), f64(inp["k"][:, heads]), f64(inp["v"][:, heads]),
                                  f64(inp["g"][:, heads]), f64(inp["beta"][:, heads]), [0, T],
                                  init=f64(init[:1, heads]), scale=D ** -0.5)
    assert_out_close(f64(out_s[:, heads]), o_ref)
    assert_state_close(f64(fin_s[:, heads]), f_ref)


@pytest.mark.parametrize("every", [4096, SEG])
def test_segmented_checkpoints_and_cache_rows(every):
    """Checkpoints every 4,096 tokens (inside segments and at their ends) or every segment, the
    initial state from a cache row and the final one to another: bit-identical with the
    unsegmented run, the checkpoints within tolerance of the oracle's chunk-boundary states."""
    T, H = 2 * SEG + 1000, 4
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=every % 1000, device=DEV, decay_scale=0.3)
    init = torch.randn(2, H, D, D, generator=wl.generator(every % 97, DEV), device=DEV) * 0.5
    n = kda_prefill_checkpoint_count([0, T], every)
    out_s, fin_s, ck_s, row_s = prefill(inp, [0, T], H, init[:1], every, n)
    out_u, fin_u, ck_u, row_u = prefill(inp, [0, T, T], H, init, every, kda_prefill_checkpoint_count([0, T, T], every))
    assert torch.equal(out_s.view(torch.uint8), out_u.view(torch.uint8))
    assert torch.equal(fin_s[0], fin_u[0])
    assert torch.equal(ck_s, ck_u[:n])
    assert torch.equal(row_s[0], row_u[0]) and torch.equal(row_s[0], fin_s[0])
    heads = [1, 3]
    _, _, ck_ref = oracle.prefill_ckpt(f64(inp["q"][:, heads]), f64(inp["k"][:, heads]), f64(inp["v"][:, heads]),
                                       f64(inp["g"][:, heads]), f64(inp["beta"][:, heads]), [0, T], every,
                                       init=f64(init[:1, heads]), scale=D ** -0.5)
    assert ck_ref.shape[0] == n
    for s in range(n):
        assert_state_close(f64(ck_s[s, heads]), ck_ref[s], what=f"checkpoint {s}")


def test_segmented_capture_into_a_cuda_graph():
    """The segmented prefill forks onto the library's stream and joins back by events, which
    stream capture follows: captured once (after a first call outside capture), a replay on new
    input values gives the eager results bit for bit."""
    T, H = 2 * SEG + 37, 2
    cu = [0, T]
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=3, device=DEV, decay_scale=0.3)
    init = torch.randn(1, H, D, D, generator=wl.generator(4, DEV), device=DEV) * 0.5
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    ws = workspace(cu, H)

    def call(out, fin):
        kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws, init_state=init,
                           final_state=fin)

    outs = [(torch.empty(T, H, D, dtype=torch.bfloat16, device=DEV), torch.empty(1, H, D, D, device=DEV))
            for _ in range(2)]
    call(*outs[0])  # outside capture: the library's stream exists from here on
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call(*outs[1])
    for t in (inp["q"], inp["v"]):
        t.copy_(torch.randn(t.shape, device=DEV).to(t.dtype))
    graph.replay()
    torch.cuda.synchronize()
    call(*outs[0])
    torch.cuda.synchronize()
    assert kda_prefill_workspace_status(ws) == 0
    assert torch.equal(outs[1][0].view(torch.uint8), outs[0][0].view(torch.uint8))
    assert torch.equal(outs[1][1], outs[0][1])


@pytest.mark.parametrize("gate", ["g_minus_50", "mixed_channels"])
def test_segmented_strong_decay(gate):
    """Decays beyond the block split's range (every chunk takes the exact fix-up, whose list is
    cleared between segments): g = -50 everywhere, and channels alternating -0.1 and -40."""
    T, H = 2 * SEG + 100, 2
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=len(gate), device=DEV)
    if gate == "g_minus_50":
        inp["g"].fill_(-50.0)
    else:
        inp["g"].copy_(torch.where(torch.arange(D, device=DEV) % 2 == 0, -0.1, -40.0).expand_as(inp["g"]))
    init = torch.randn(2, H, D, D, generator=wl.generator(6, DEV), device=DEV) * 0.5
    out_s, fin_s, _, _ = prefill(inp, [0, T], H, init[:1])
    out_u, fin_u, _, _ = prefill(inp, [0, T, T], H, init)
    assert torch.equal(out_s.view(torch.uint8), out_u.view(torch.uint8))
    assert torch.equal(fin_s[0], fin_u[0])
    o_ref, f_ref = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]), f64(inp["beta"]),
                                  [0, T], init=f64(init[:1]), scale=D ** -0.5)
    assert_out_close(f64(out_s), o_ref)
    assert_state_close(f64(fin_s), f_ref)


def test_segmented_timed_events():
    """kda_prefill_varlen_timed on the segmented form: all four events recorded in order
    (the state passes overlap the preparation, so events[2] follows the last segment's
    preparation and events[3] the last pass) and the results those of the untimed call."""
    T, H = 2 * SEG + 64, 2
    cu = [0, T]
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=8, device=DEV, decay_scale=0.3)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    ws = workspace(cu, H)
    outs = []
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for events in (None, ev):
        out = torch.empty(T, H, D, dtype=torch.bfloat16, device=DEV)
        kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws, events=events)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.uint8), outs[1].view(torch.uint8))
    for a, b in zip(ev[:-1], ev[1:]):
        assert a.elapsed_time(b) >= 0.0
    assert ev[0].elapsed_time(ev[3]) > 0.0
