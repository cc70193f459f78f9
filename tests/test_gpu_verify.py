"""GPU parity of the speculative target verification against the oracle: outputs
(max|d| <= 2e-2 max|ref|), every intermediate state (||dS||_F <= 1e-2 ||S_ref||_F),
the cache untouched bit for bit, pool slots that are not addressed untouched; and
the commit of an accepted prefix through the state-copy calls."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import (kda_decode_step, kda_state_gather, kda_state_scatter,
                                               kda_target_verify)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_state_close, bytes_of, f64, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


def draft_inputs(R, L, H, D, io, seed):
    t = wl.token_inputs(R * L, H, D, D, io, seed=seed, device=DEV, decay_scale=0.3)
    return {n: x.view(R, L, *x.shape[1:]) for n, x in t.items()}


@pytest.mark.parametrize("D,H", [(128, 3), (64, 2), (32, 4)])
@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("cache_dtype,pool_dtype", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32),
                                                    (torch.bfloat16, torch.float32)])
def test_target_verify_against_oracle(D, H, io, cache_dtype, pool_dtype):
    R, L, N, P = 5, 4, 7, 24
    inp = draft_inputs(R, L, H, D, io, seed=D + H)
    pc = wl.paged_cache(N, H, D, D, cache_dtype, H * D * D + 64, seed=1, device=DEV)
    pool = wl.paged_cache(P, H, D, D, pool_dtype, None, seed=0, device=DEV, fill=False)
    idx = torch.tensor([3, -1, 6, 0, N + 2], dtype=torch.int32)
    inter = torch.arange(R * L, dtype=torch.int32).view(R, L).clone()
    inter[1, 1] = -1
    inter[3, 3] = P + 5
    cache_before, pool_before = raw(pc.backing), raw(pool.backing)
    out = torch.empty(R, L, H, D, dtype=io, device=DEV)
    kda_target_verify(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pc.view, idx.to(DEV), pool.view,
                      inter.to(DEV), out)
    torch.cuda.synchronize()
    assert np.array_equal(raw(pc.backing), cache_before)  # the cache is only read
    body = np.ascontiguousarray(cache_before[pc.front:pc.front + N * pc.row_stride])
    pbody = np.zeros(P * H * D * D, dtype=pool_before.dtype)
    o_ref = oracle.target_verify(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]), f64(inp["beta"]),
                                 body, N, pc.row_stride, idx.numpy(), pbody, P, H * D * D, inter.numpy(),
                                 scale=D ** -0.5)
    assert_out_close(f64(out), o_ref)
    pref = pbody.reshape(P, H, D, D)
    if pool_dtype == torch.bfloat16:
        pref = (pref.astype(np.uint32) << 16).view(np.float32)
    written = set()
    for r in range(R):
        for t in range(L):
            s = int(inter[r, t])
            if 0 <= s < P:
                written.add(s)
                assert_state_close(f64(pool.view[s]), pref[s].astype(np.float64), what=f"state ({r}, {t})")
    after = raw(pool.backing)
    for s in range(P):
        if s not in written:
            lo = pool.front + s * pool.row_stride
            assert np.array_equal(after[lo:lo + H * D * D], pool_before[lo:lo + H * D * D])


def test_commit_accepted_prefix_matches_decode_steps():
    """Verify 4 tokens, accept 3: copying slot inter[r, 2] into the cache row gives the
    state of three decode steps (fp32 cache and pool: both keep fp32 states)."""
    R, L, H, D, N = 3, 4, 2, 128, 5
    inp = draft_inputs(R, L, H, D, torch.bfloat16, seed=9)
    pc = wl.paged_cache(N, H, D, D, torch.float32, None, seed=2, device=DEV)
    ref = pc.backing.clone()
    ref_view = ref.as_strided(pc.view.shape, pc.view.stride(), pc.front)
    pool = wl.paged_cache(R * L, H, D, D, torch.float32, None, seed=0, device=DEV, fill=False)
    idx = torch.tensor([4, 1, 2], dtype=torch.int32, device=DEV)
    inter = torch.arange(R * L, dtype=torch.int32, device=DEV).view(R, L)
    out = torch.empty(R, L, H, D, dtype=torch.bfloat16, device=DEV)
    kda_target_verify(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pc.view, idx, pool.view, inter, out)
    accepted = inter[:, 2].contiguous()
    packed = torch.empty(R, H, D, D, dtype=torch.float32, device=DEV)
    kda_state_gather(pool.view, accepted, packed)
    kda_state_scatter(pc.view, idx, packed)
    dout = torch.empty(R, H, D, dtype=torch.bfloat16, device=DEV)
    for t in range(3):
        kda_decode_step(inp["q"][:, t].contiguous(), inp["k"][:, t].contiguous(), inp["v"][:, t].contiguous(),
                        inp["g"][:, t].contiguous(), inp["beta"][:, t].contiguous(), ref_view, idx, dout)
        assert_out_close(f64(out[:, t]), f64(dout))
    torch.cuda.synchronize()
    for r in idx.tolist():
        assert_state_close(f64(pc.view[r]), f64(ref_view[r]))
    untouched = [r for r in range(N) if r not in idx.tolist()]
    for r in untouched:
        assert np.array_equal(bytes_of(pc.view[r]), bytes_of(ref_view[r]))
