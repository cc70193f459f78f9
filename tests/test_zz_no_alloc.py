"""kda_prefill_varlen_noalloc: the prefill entry point for callers that cannot
allocate device memory (a host program linking only this library, with no
device allocator; a runtime whose device memory is fixed at start-up and that
allows no allocation on the request path).  The same kernels run on the same
inputs, only with the workspace in the library's fixed scratch array, so its
results must be bit-identical to kda_prefill_varlen with a caller workspace -
checked here through the C ABI on two calls in a row, since every call reuses
the one array - and the first batch is also checked against the oracle.  The
status word of the fixed array (kda_prefill_noalloc_status) must read 0 after
each call.  Batches whose records do not fit the array run the compact form
(bf16, head size 128) or are rejected; one long sequence whose records fit runs the
segmented form.  The file is named to be collected last."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_varlen_gb300 as kda
from kimi_delta_attention_varlen_gb300 import _abi
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_state_close, f64, oracle_prefill_from_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _batch(lengths, seed, H=32, D=128):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    inp = wl.token_inputs(cu[-1], H, D, D, torch.bfloat16, seed=seed, device=DEV)
    init = torch.randn(len(lengths), H, D, D, generator=wl.generator(seed + 100, DEV), device=DEV)
    return inp, torch.tensor(cu, dtype=torch.int32, device=DEV), init


def _with_workspace(inp, cu, init):
    T, H, D = inp["q"].shape
    B = cu.numel() - 1
    out = torch.empty(T, H, D, dtype=inp["q"].dtype, device=DEV)
    fin = torch.empty(B, H, D, D, device=DEV)
    ws = torch.empty(kda.kda_prefill_workspace_size(T, B, H, D, D), dtype=torch.uint8, device=DEV)
    kda.kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu, out, ws,
                           init_state=init, final_state=fin)
    return out, fin


def _noalloc(inp, cu, init):
    T, H, D = inp["q"].shape
    B = cu.numel() - 1
    out = torch.full((T, H, D), float("nan"), dtype=inp["q"].dtype, device=DEV)
    fin = torch.full((B, H, D, D), float("nan"), device=DEV)
    kda.kda_prefill_varlen_noalloc(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu, out,
                                   init_state=init, final_state=fin)
    return out, fin


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # two different batches back to back: the second call reuses the scratch the first one left
    for n, (lengths, seed) in enumerate((([700, 1, 130, 64], 1), ([65, 1000, 300], 2))):
        inp, cu, init = _batch(lengths, seed)
        want_out, want_fin = _with_workspace(inp, cu, init)
        got_out, got_fin = _noalloc(inp, cu, init)
        assert kda.kda_prefill_noalloc_status() == 0  # synchronises: every bounded wait completed
        # same kernels, same inputs: bit for bit the workspace entry point's results
        assert torch.equal(got_out, want_out)
        assert torch.equal(got_fin, want_fin)
        if n == 0:  # and the oracle's, on two heads of every sequence
            cu_host = cu.tolist()
            heads = [0, 31]
            o_ref, f_ref, toks = oracle_prefill_from_device(inp, cu_host, init, 128 ** -0.5, heads=heads)
            assert_out_close(f64(got_out[toks][:, heads]), o_ref)
            assert_state_close(f64(got_fin[:, heads]), f_ref)


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    H, D = 32, 128
    T = 64 * 64  # fp32: 64 chunks of 32 heads need more records than the fixed scratch holds
    assert kda.kda_prefill_workspace_size(T, 1, H, D, D) > _abi.KDA_NOALLOC_SCRATCH_BYTES
    cu = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    inp = wl.token_inputs(T, H, D, D, torch.float32, seed=3, device=DEV)
    out = torch.zeros(T, H, D, dtype=torch.float32, device=DEV)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_varlen_noalloc(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu, out)
    assert e.value.status == -6  # KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not torch.any(out != 0)  # nothing was launched


def test_noalloc_runs_a_large_bf16_batch_in_the_compact_form():
    # bf16 at head size 128: a batch beyond the records the scratch holds runs the fused
    # kernel, whose workspace is only the chunk table
    lengths = [4100, 30, 2000]
    H, D = 32, 128
    T = sum(lengths)
    assert kda.kda_prefill_workspace_size(T, len(lengths), H, D, D) > _abi.KDA_NOALLOC_SCRATCH_BYTES
    inp, cu, init = _batch(lengths, 4)
    out, fin = _noalloc(inp, cu, init)
    assert kda.kda_prefill_noalloc_status() == 0
    heads = [0, 31]
    o_ref, f_ref, toks = oracle_prefill_from_device(inp, cu.tolist(), init, 128 ** -0.5, heads=heads)
    assert_out_close(f64(out[toks][:, heads]), o_ref)
    assert_state_close(f64(fin[:, heads]), f_ref)


def test_noalloc_segmented_long_sequence():
    # one sequence of 544 chunks at 2 heads: its records fit the scratch, so it runs the
    # segmented form (the library's second stream) - bit for bit the workspace call's results
    T, H = 544 * 64 - 17, 2
    assert kda.kda_prefill_workspace_size(T, 1, H, 128, 128) <= _abi.KDA_NOALLOC_SCRATCH_BYTES
    inp, cu, init = _batch([T], 5, H=H)
    want_out, want_fin = _with_workspace(inp, cu, init)
    got_out, got_fin = _noalloc(inp, cu, init)
    assert kda.kda_prefill_noalloc_status() == 0
    assert torch.equal(got_out, want_out)
    assert torch.equal(got_fin, want_fin)
