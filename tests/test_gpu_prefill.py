"""GPU parity of kda_prefill_varlen (and the gather -> prefill -> scatter
composition) against the token-by-token fp64 oracle.

Tolerances (the method's target): outputs max|d| <= 2e-2 max|ref|, final
states ||dS||_F <= 1e-2 ||S_ref||_F; state copies bit-exact.  Cases span
several chunks with ragged tails, empty and single-token sequences, every
built head size, both io dtypes, mild decay (long-range state propagation)
and the degenerate gates; the full-size workloads are checked on sampled
(sequence, head) pairs the oracle evaluates one by one."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import (kda_prefill_varlen, kda_prefill_workspace_size,
                                               kda_prefill_workspace_status, kda_state_gather,
                                               kda_state_scatter)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import (assert_out_close, assert_state_close, bytes_of, f64, oracle_prefill_from_device,
                           raw)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_prefill(inp, cu, H, D, init=None, scale=None, final=True, l2norm=True):
    T = inp["q"].shape[0]
    B = len(cu) - 1
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out = torch.full((T, H, D), float("nan"), dtype=inp["q"].dtype, device=DEV)
    fin = torch.full((B, H, D, D), float("nan"), dtype=torch.float32, device=DEV) if final else None
    ws = torch.empty(kda_prefill_workspace_size(T, B, H, D, D), dtype=torch.uint8, device=DEV)
    kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws,
                       scale=scale, init_state=init, final_state=fin, qk_l2norm=l2norm)
    torch.cuda.synchronize()
    assert kda_prefill_workspace_status(ws) == 0
    return out, fin


def check_against_oracle(inp, cu, H, D, init, out, fin, scale, l2norm=True, heads=None, seqs=None):
    o_ref, f_ref, toks = oracle_prefill_from_device(inp, cu, init, scale, l2norm, heads, seqs)
    hs = slice(None) if heads is None else list(heads)
    sq = list(range(len(cu) - 1)) if seqs is None else list(seqs)
    got_o = f64(out[torch.tensor(toks, dtype=torch.long, device=DEV)][:, hs]) if toks else np.zeros((0,))
    if toks:
        assert_out_close(got_o, o_ref)
    if fin is not None:
        assert_state_close(f64(fin[sq][:, hs]), f_ref)


@pytest.mark.parametrize("D,io", [(128, torch.bfloat16), (64, torch.bfloat16), (32, torch.float32),
                                  (128, torch.float32)])
@pytest.mark.parametrize("decay", [1.0, 0.01])
def test_prefill_ragged_varlen(D, io, decay):
    lengths = [1, 63, 64, 65, 0, 200, 333]
    H = 3
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    inp = wl.token_inputs(cu[-1], H, D, D, io, seed=D + int(decay * 10), device=DEV, decay_scale=decay)
    init = torch.randn(len(lengths), H, D, D, generator=wl.generator(3, DEV), device=DEV) * 0.5
    scale = D ** -0.5
    out, fin = run_prefill(inp, cu, H, D, init=init, scale=scale)
    check_against_oracle(inp, cu, H, D, init, out, fin, scale)
    assert torch.equal(fin[4], init[4])  # the empty sequence keeps its state bit for bit


@pytest.mark.parametrize("H", [64, 4])
@pytest.mark.parametrize("init_kind", ["fp32", "bf16", "none"])
def test_prefill_many_heads(init_kind, H):
    """64 heads: enough (sequence, head) pairs for one CTA per pair (the tensor-memory
    state pass at head size 128, bf16); 4 heads: its value-split form.  Ragged lengths,
    an empty sequence, every init kind."""
    lengths, D = [1, 63, 64, 65, 0, 130], 128
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    inp = wl.token_inputs(cu[-1], H, D, D, torch.bfloat16, seed=40, device=DEV, decay_scale=0.3)
    init = None
    if init_kind != "none":
        init = torch.randn(len(lengths), H, D, D, generator=wl.generator(41, DEV), device=DEV)
        if init_kind == "bf16":
            init = init.to(torch.bfloat16)
    out, fin = run_prefill(inp, cu, H, D, init=init, scale=D ** -0.5)
    ref_init = None if init is None else init.float()
    check_against_oracle(inp, cu, H, D, ref_init, out, fin, D ** -0.5, heads=[0, 17, 63] if H == 64 else None)
    if init is not None:
        assert torch.equal(fin[4], init[4].float())  # the empty sequence keeps its state
    else:
        assert not torch.any(fin[4] != 0)


def test_prefill_bf16_init_and_no_final():
    lengths, H, D = [130, 7], 2, 128
    cu = [0, 130, 137]
    inp = wl.token_inputs(137, H, D, D, torch.bfloat16, seed=5, device=DEV)
    init = torch.randn(2, H, D, D, generator=wl.generator(6, DEV), device=DEV).to(torch.bfloat16)
    out, _ = run_prefill(inp, cu, H, D, init=init, scale=0.1, final=False)
    check_against_oracle(inp, cu, H, D, init.float(), out, None, 0.1)


def test_prefill_zero_tokens_keeps_init():
    H, D = 2, 64
    inp = wl.token_inputs(0, H, D, D, torch.bfloat16, seed=1, device=DEV)
    init = torch.randn(3, H, D, D, generator=wl.generator(2, DEV), device=DEV)
    out, fin = run_prefill(inp, [0, 0, 0, 0], H, D, init=init)
    assert torch.equal(fin, init)


def test_prefill_without_l2norm_and_unit_scale():
    lengths, H, D = [100, 29], 2, 64
    cu = [0, 100, 129]
    inp = wl.token_inputs(129, H, D, D, torch.bfloat16, seed=8, device=DEV)
    out, fin = run_prefill(inp, cu, H, D, scale=1.0, l2norm=False)
    check_against_oracle(inp, cu, H, D, None, out, fin, 1.0, l2norm=False)


def test_degenerate_beta0_g0_keeps_state():
    H, D, T = 2, 128, 150
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=9, device=DEV)
    inp["g"].zero_()
    inp["beta"].zero_()
    init = torch.randn(1, H, D, D, generator=wl.generator(10, DEV), device=DEV)
    out, fin = run_prefill(inp, [0, T], H, D, init=init, scale=D ** -0.5)
    assert_state_close(f64(fin), f64(init))
    check_against_oracle(inp, [0, T], H, D, init, out, fin, D ** -0.5)


def test_degenerate_strong_decay():
    """g = -8 per token (inside the documented gate range): the state keeps almost
    nothing beyond the last token; outputs follow beta_t (k.q) v_t."""
    H, D, T = 2, 128, 140
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=11, device=DEV)
    inp["g"].fill_(-8.0)
    init = torch.randn(1, H, D, D, generator=wl.generator(12, DEV), device=DEV)
    out, fin = run_prefill(inp, [0, T], H, D, init=init, scale=D ** -0.5)
    check_against_oracle(inp, [0, T], H, D, init, out, fin, D ** -0.5)


def test_tiny_workload_gather_prefill_scatter():
    """The tiny workload end to end: gather initial states by index and flag,
    prefill, scatter final states - each step against its oracle."""
    w = wl.tiny()
    H, D = w.H, w.K
    cu = [0]
    for n in w.lengths:
        cu.append(cu[-1] + n)
    pc = wl.paged_cache(w.cache_rows, H, D, D, w.cache_dtype, w.cache_stride, seed=w.seed, device=DEV)
    inp = wl.token_inputs(w.T, H, D, D, w.io_dtype, seed=w.seed, device=DEV)
    packed = torch.empty(w.B, H, D, D, dtype=pc.view.dtype, device=DEV)
    kda_state_gather(pc.view, w.gather_idx.to(DEV), packed, w.gather_flags.to(DEV))
    out, fin = run_prefill(inp, cu, H, D, init=packed, scale=D ** -0.5)
    host_before = raw(pc.backing)
    kda_state_scatter(pc.view, w.scatter_idx.to(DEV), fin)
    torch.cuda.synchronize()
    # gather: bit-exact
    N, P = w.cache_rows, H * D * D
    body = host_before[pc.front:pc.front + N * pc.row_stride]
    want_packed = oracle.gather(body, N, P, pc.row_stride, w.gather_idx.numpy(), w.gather_flags.numpy())
    assert np.array_equal(raw(packed).reshape(w.B, -1), want_packed)
    assert not torch.any(packed[1] != 0) and not torch.any(packed[2] != 0)  # idx -1, flag false
    # prefill: tolerance
    check_against_oracle(inp, cu, H, D, packed, out, fin, D ** -0.5)
    # scatter: bit-exact given the GPU's final states
    oracle.scatter(body, N, P, pc.row_stride, w.scatter_idx.numpy(), raw(fin).reshape(w.B, -1))
    host_before[pc.front:pc.front + N * pc.row_stride] = body
    assert np.array_equal(bytes_of(pc.backing), host_before.view(np.uint8))


def _full_workload(w, sample_pairs, whole_seqs=()):
    H, D = w.H, w.K
    cu = [0]
    for n in w.lengths:
        cu.append(cu[-1] + n)
    pc = wl.paged_cache(w.cache_rows, H, D, D, w.cache_dtype, w.cache_stride, seed=w.seed, device=DEV)
    inp = wl.token_inputs(w.T, H, D, D, w.io_dtype, seed=w.seed, device=DEV)
    packed = torch.empty(w.B, H, D, D, dtype=pc.view.dtype, device=DEV)
    kda_state_gather(pc.view, w.gather_idx.to(DEV), packed, w.gather_flags.to(DEV))
    out, fin = run_prefill(inp, cu, H, D, init=packed, scale=D ** -0.5)
    kda_state_scatter(pc.view, w.scatter_idx.to(DEV), fin)
    torch.cuda.synchronize()
    for b, h in sample_pairs:  # h: one head, or a list of heads the oracle runs in parallel
        hs = list(h) if isinstance(h, (list, tuple)) else [h]
        check_against_oracle(inp, cu, H, D, packed, out, fin, D ** -0.5, heads=hs, seqs=[b])
        r = int(w.scatter_idx[b])
        if 0 <= r < w.cache_rows:  # the scattered row holds exactly the GPU's final state
            assert torch.equal(pc.view[r, hs], fin[b, hs].to(pc.view.dtype))
    for b in whole_seqs:  # every head of these sequences, the oracle's heads run in parallel
        check_against_oracle(inp, cu, H, D, packed, out, fin, D ** -0.5, seqs=[b])
        r = int(w.scatter_idx[b])
        if 0 <= r < w.cache_rows:
            assert torch.equal(pc.view[r], fin[b].to(pc.view.dtype))
    return pc, inp, out, fin


def test_full_varlen_workload_sampled():
    """The 16-sequence batch in the benchmark's launch configuration: all 32 heads of the
    longest and the shortest sequence, plus single heads of others."""
    w = wl.varlen()
    order = sorted(range(w.B), key=lambda b: -w.lengths[b])
    pairs = [(order[1], 0), (order[1], 31), (order[-2], 7), (order[w.B // 2], 19), (order[w.B // 2 + 1], 3)]
    _full_workload(w, pairs, whole_seqs=(order[0], order[-1]))
    torch.cuda.empty_cache()


def test_full_long_sequence_sampled():
    """The 131,072-token sequence (2,048 chunks per head): four heads against the oracle."""
    w = wl.long_seq()
    _full_workload(w, [(0, [0, 5, 18, 31])])
    torch.cuda.empty_cache()


# bf16 at head size 128: 16 or 64 (sequence, head) pairs take the value-split tensor-memory
# pass (two CTAs per pair, one wave), 96 pairs one CTA per pair; fp32 inputs take the
# register passes (warp pairs for 16 pairs, one warp per value group for 64).
@pytest.mark.parametrize("lengths,H,io", [([327, 100, 1, 0], 4, torch.bfloat16), ([150, 71], 32, torch.bfloat16),
                                          ([200, 65, 131], 32, torch.bfloat16), ([327, 100, 1, 0], 4, torch.float32),
                                          ([150, 71], 32, torch.float32)])
def test_prefill_state_pass_dispatch(lengths, H, io):
    """Every state-pass form at head size 128 against the oracle."""
    D = 128
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    inp = wl.token_inputs(cu[-1], H, D, D, io, seed=len(lengths) + H, device=DEV, decay_scale=0.1)
    init = torch.randn(len(lengths), H, D, D, generator=wl.generator(9, DEV), device=DEV) * 0.5
    scale = D ** -0.5
    out, fin = run_prefill(inp, cu, H, D, init=init, scale=scale)
    heads = None if H <= 4 else [0, 13, 31]
    check_against_oracle(inp, cu, H, D, init, out, fin, scale, heads=heads)


def test_timed_prefill_with_unrecorded_boundaries():
    """events=[None, a, b, None] records only the chunk-preparation interval; the outputs
    are those of the untimed call, bit for bit."""
    lengths, H, D = [300, 64, 5], 2, 128
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    T, B = cu[-1], len(lengths)
    inp = wl.token_inputs(T, H, D, D, torch.bfloat16, seed=17, device=DEV)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    ws = torch.empty(kda_prefill_workspace_size(T, B, H, D, D), dtype=torch.uint8, device=DEV)
    outs = []
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for ev in (None, [None, a, b, None]):
        out = torch.empty(T, H, D, dtype=torch.bfloat16, device=DEV)
        kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_t, out, ws, events=ev)
        outs.append(out)
    torch.cuda.synchronize()
    assert a.elapsed_time(b) > 0.0
    assert torch.equal(outs[0].view(torch.uint8), outs[1].view(torch.uint8))


@pytest.mark.parametrize("D,io", [(128, torch.bfloat16), (32, torch.float32)])
@pytest.mark.parametrize("gate", ["mixed_sign", "slow_growth", "range_limit"])
def test_gates_across_the_documented_range(D, io, gate):
    """Gates inside the documented range: signs mixed with a net decay (about a quarter
    of the g > 0), a slow steady growth, and a decay of 79.2 nats over any 8 consecutive
    tokens (beyond the block split's range: the chunks take the exact Gram).  States that grow fast (zero-mean gates of
    spread 0.5) amplify the bf16 operand rounding beyond the tolerance on every path."""
    H, lengths = 2, [150, 37, 64]
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    inp = wl.token_inputs(cu[-1], H, D, D, io, seed=D + len(gate), device=DEV)
    if gate == "mixed_sign":
        inp["g"].copy_(torch.randn(inp["g"].shape, generator=wl.generator(31, DEV), device=DEV) * 0.5 - 0.3)
    elif gate == "slow_growth":
        inp["g"].fill_(0.05)
    else:
        inp["g"].fill_(-9.9)
    init = torch.randn(len(lengths), H, D, D, generator=wl.generator(32, DEV), device=DEV) * 0.5
    out, fin = run_prefill(inp, cu, H, D, init=init, scale=D ** -0.5)
    check_against_oracle(inp, cu, H, D, init, out, fin, D ** -0.5)


# State-pass forms by shape (the launcher's dispatch): the tensor-memory passes (head size 128,
# bf16: one CTA per pair for 96 (sequence, head) pairs, two value-split CTAs per pair for 64
# and 16), the one-warp and warp-pair register passes (fp32, 64 and 16 pairs), and the register
# pass at head sizes 64 and 32.
STRONG_DECAY_FORMS = {
    "tcgen05": (128, torch.bfloat16, [200, 65, 131], 32, [0, 13, 31]),
    "tcgen05_split": (128, torch.bfloat16, [150, 71], 32, [0, 21]),
    "tcgen05_split_few": (128, torch.bfloat16, [327, 100, 1, 0], 4, None),
    "one_warp": (128, torch.float32, [150, 71], 32, [0, 21]),
    "warp_pair": (128, torch.float32, [327, 100, 1, 0], 4, None),
    "d64": (64, torch.bfloat16, [130, 64, 9], 3, None),
    "d32_fp32": (32, torch.float32, [100, 37, 64], 2, None),
}


@pytest.mark.parametrize("form", list(STRONG_DECAY_FORMS))
@pytest.mark.parametrize("gate", ["g_minus_50", "g_minus_1000", "mixed_channels", "spikes"])
def test_strong_decay_gates(form, gate):
    """Decays far beyond the block split's range (e^{g} underflows to 0 within a token or
    a few) against the oracle on every state-pass form: g = -50 and g = -1000 everywhere
    (the state reduces to beta k v^T, the pin of the token-by-token recurrence), channels
    alternating -0.1 and -40, and the configs' gates with isolated -200 spikes."""
    D, io, lengths, H, heads = STRONG_DECAY_FORMS[form]
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    inp = wl.token_inputs(cu[-1], H, D, D, io, seed=D + H + len(gate), device=DEV)
    g = inp["g"]
    if gate == "g_minus_50":
        g.fill_(-50.0)
    elif gate == "g_minus_1000":
        g.fill_(-1000.0)
    elif gate == "mixed_channels":
        g.copy_(torch.where(torch.arange(D, device=DEV) % 2 == 0, -0.1, -40.0).expand_as(g))
    else:
        gen = wl.generator(77, DEV)
        spikes = torch.rand(g.shape, generator=gen, device=DEV) < 0.002
        g.copy_(torch.where(spikes, torch.full_like(g, -200.0), g))
    init = torch.randn(len(lengths), H, D, D, generator=wl.generator(33, DEV), device=DEV) * 0.5
    out, fin = run_prefill(inp, cu, H, D, init=init, scale=D ** -0.5)
    check_against_oracle(inp, cu, H, D, init, out, fin, D ** -0.5, heads=heads)
