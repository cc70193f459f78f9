"""GPU parity of the prefill's compact form: bf16 inputs at head size 128 with a
workspace too small for the per-chunk records (kda_prefill_workspace_size_compact
bytes), which runs the fused kernel (chunk preparation and state pass in one
persistent CTA per SM, every per-chunk quantity kept on chip).

Checked against the token-by-token fp64 oracle at the method's tolerances
(outputs max|d| <= 2e-2 max|ref|, states ||dS||_F <= 1e-2 ||S_ref||_F) on ragged
batches (empty and single-token sequences, tails), every gate regime (the scaled
path, chunks whose gate span takes the exact path, g = -50 where the state
reduces to beta k v^T), without l2norm, with bf16 initial states, through the
cache-indexed entry point with checkpoints, and at the benchmark's full size on
whole sequences; against the two-kernel form on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import (kda_prefill_checkpoint_count, kda_prefill_varlen,
                                               kda_prefill_varlen_cached, kda_prefill_workspace_size,
                                               kda_prefill_workspace_size_compact, kda_prefill_workspace_status,
                                               kda_state_gather)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_state_close, f64, oracle_prefill_from_device

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


def cu_of(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return cu


def compact_ws(T, B, H):
    n = kda_prefill_workspace_size_compact(T, B, H, D, D)
    assert 0 < n < kda_prefill_workspace_size(T, B, H, D, D)
    return torch.empty(n, dtype=torch.uint8, device=DEV)


def run(inp, cu, H, ws, init=None, scale=None, l2norm=True, final=True):
    T, B = cu[-1], len(cu) - 1
    out = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    fin = torch.full((B, H, D, D), float("nan"), device=DEV) if final else None
    kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], torch.tensor(cu, dtype=torch.int32,
                       device=DEV), out, ws, scale=scale, init_state=init, final_state=fin, qk_l2norm=l2norm)
    torch.cuda.synchronize()
    assert kda_prefill_workspace_status(ws) == 0
    return out, fin


def check(inp, cu, H, init, out, fin, scale, l2norm=True, heads=None, seqs=None):
    o_ref, f_ref, toks = oracle_prefill_from_device(inp, cu, init, scale, l2norm, heads, seqs)
    hs = slice(None) if heads is None else list(heads)
    sq = list(range(len(cu) - 1)) if seqs is None else list(seqs)
    if toks:
        assert_out_close(f64(out[torch.tensor(toks, dtype=torch.long, device=DEV)][:, hs]), o_ref)
    if fin is not None:
        assert_state_close(f64(fin[sq][:, hs]), f_ref)


@pytest.mark.parametrize("lengths,H", [([1, 63, 64, 65, 0, 200, 333], 3), ([700, 1, 130, 64], 32), ([0, 0], 4),
                                       ([5], 1)])
@pytest.mark.parametrize("decay", [1.0, 0.01])
def test_compact_ragged_varlen(lengths, H, decay):
    cu = cu_of(lengths)
    inp = wl.token_inputs(cu[-1], H, D, D, torch.bfloat16, seed=len(lengths) + H, device=DEV, decay_scale=decay)
    init = torch.randn(len(lengths), H, D, D, generator=wl.generator(3, DEV), device=DEV) * 0.5
    out, fin = run(inp, cu, H, compact_ws(cu[-1], len(lengths), H), init=init)
    check(inp, cu, H, init, out, fin, D ** -0.5, heads=None if H <= 4 else [0, 13, 31])


@pytest.mark.parametrize("gate", ["span_edge", "span_beyond", "g_minus_50", "mixed_channels", "spikes"])
def test_compact_gate_regimes(gate):
    """span_edge: 64 tokens of g = -1.25 span 115 (log2 units): the scaled path near its
    limit of 120; span_beyond: g = -1.5 spans 138: the exact path, like the rest."""
    lengths, H = [150, 37, 64], 4
    cu = cu_of(lengths)
    inp = wl.token_inputs(cu[-1], H, D, D, torch.bfloat16, seed=len(gate), device=DEV)
    g = inp["g"]
    if gate == "span_edge":
        g.fill_(-1.25)
    elif gate == "span_beyond":
        g.fill_(-1.5)
    elif gate == "g_minus_50":
        g.fill_(-50.0)
    elif gate == "mixed_channels":
        g.copy_(torch.where(torch.arange(D, device=DEV) % 2 == 0, -0.1, -40.0).expand_as(g))
    else:
        spikes = torch.rand(g.shape, generator=wl.generator(78, DEV), device=DEV) < 0.002
        g.copy_(torch.where(spikes, torch.full_like(g, -200.0), g))
    init = torch.randn(len(lengths), H, D, D, generator=wl.generator(34, DEV), device=DEV) * 0.5
    out, fin = run(inp, cu, H, compact_ws(cu[-1], len(lengths), H), init=init)
    check(inp, cu, H, init, out, fin, D ** -0.5)


def test_compact_without_l2norm_bf16_init_and_no_final():
    lengths, H = [129, 64, 3], 2
    cu = cu_of(lengths)
    inp = wl.token_inputs(cu[-1], H, D, D, torch.bfloat16, seed=11, device=DEV, decay_scale=0.3)
    init = (torch.randn(len(lengths), H, D, D, generator=wl.generator(12, DEV), device=DEV) * 0.5).to(torch.bfloat16)
    out, _ = run(inp, cu, H, compact_ws(cu[-1], len(lengths), H), init=init, scale=1.0, l2norm=False, final=False)
    check(inp, cu, H, init.float(), out, None, 1.0, l2norm=False)


def test_compact_matches_two_kernel_form():
    lengths, H = [300, 1, 64, 129], 8
    cu = cu_of(lengths)
    T, B = cu[-1], len(lengths)
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=21, device=DEV)
    init = torch.randn(B, H, D, D, generator=wl.generator(22, DEV), device=DEV) * 0.5
    full = torch.empty(kda_prefill_workspace_size(T, B, H, D, D), dtype=torch.uint8, device=DEV)
    out_a, fin_a = run(inp, cu, H, full, init=init)
    out_b, fin_b = run(inp, cu, H, compact_ws(T, B, H), init=init)
    assert_out_close(f64(out_b), f64(out_a))
    assert_state_close(f64(fin_b), f64(fin_a))


@pytest.mark.parametrize("every", [64, 192])
def test_compact_cached_with_checkpoints(every):
    """Initial states by index from an fp32 cache (flags), final states to other rows,
    checkpoints every `every` tokens: against the oracle's gather -> prefill -> scatter."""
    lengths, H, N = [130, 0, 384, 63, 192], 3, 24
    cu = cu_of(lengths)
    T, B = cu[-1], len(lengths)
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=every, device=DEV, decay_scale=0.3)
    pc = wl.paged_cache(N, H, D, D, torch.float32, H * D * D + 64, seed=every + 1, device=DEV)
    idx_in = wl.gather_indices(B, N, 0.25, every + 2)
    flags = wl.bernoulli_flags(B, 0.75, every + 3)
    idx_out = wl.scatter_indices(B, N, 0.25, every + 4)
    packed = torch.empty(B, H, D, D, device=DEV)
    kda_state_gather(pc.view, idx_in.to(DEV), packed, flags.to(DEV))
    n = kda_prefill_checkpoint_count(cu, every)
    ck = torch.full((max(n, 1), H, D, D), float("nan"), device=DEV)
    out = torch.empty(T, H, D, dtype=torch.bfloat16, device=DEV)
    fin = torch.empty(B, H, D, D, device=DEV)
    ws = compact_ws(T, B, H)
    kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              torch.tensor(cu, dtype=torch.int32, device=DEV), out, ws, pc.view, idx_in.to(DEV),
                              flags=flags.to(DEV), idx_out=idx_out.to(DEV), final_state=fin, checkpoints=ck[:n],
                              ckpt_every=every)
    torch.cuda.synchronize()
    assert kda_prefill_workspace_status(ws) == 0
    o_ref, f_ref, ck_ref = oracle.prefill_ckpt(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]),
                                               f64(inp["beta"]), cu, every, init=f64(packed), scale=D ** -0.5)
    assert_out_close(f64(out), o_ref)
    assert_state_close(f64(fin), f_ref)
    for s in range(n):
        assert_state_close(f64(ck[s]), ck_ref[s], what=f"checkpoint {s}")
    for b, r in enumerate(idx_out.tolist()):
        if 0 <= r < N:  # the row holds the final state, as written to final_state
            assert torch.equal(pc.view[r], fin[b])


def test_compact_full_varlen_workload():
    """The benchmark's batch (16 sequences U[512, 8192], H = 32): every head of the
    longest and the shortest sequence against the oracle."""
    w = wl.varlen()
    H = w.H
    cu = cu_of(w.lengths)
    T, B = cu[-1], w.B
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=w.seed, device=DEV)
    init = torch.randn(B, H, D, D, generator=wl.generator(5, DEV), device=DEV) * 0.5
    out, fin = run(inp, cu, H, compact_ws(T, B, H), init=init)
    order = sorted(range(B), key=lambda b: w.lengths[b])
    for b in (order[0], order[-1]):
        check(inp, cu, H, init, out, fin, D ** -0.5, seqs=[b])
    torch.cuda.empty_cache()
