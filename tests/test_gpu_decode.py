"""GPU parity of kda_decode_step against the oracle's one-token step on cache
rows (in place; invalid index -> zero state, output computed, nothing
written).  Written-back rows are compared after the oracle's state is cast to
the cache dtype, with the state tolerance; untouched rows bit-exactly."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import kda_decode_step
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_state_close, bytes_of, f64, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _decode_vs_oracle(R, H, D, io, cache_dtype, N, itype, stride_extra=0, decay=1.0, sample=None):
    inp = wl.token_inputs(R, H, D, D, io, seed=R + D, device=DEV, decay_scale=decay)
    base = torch.randperm(N, generator=wl.generator(3))[:R]
    bad = torch.rand(R, generator=wl.generator(4)) < 0.1
    idx = torch.where(bad, torch.full_like(base, -1), base).to(itype)
    idx[0] = -1
    if R > 1:
        idx[1] = N + 5
    pc = wl.paged_cache(N, H, D, D, cache_dtype, H * D * D + stride_extra, seed=5, device=DEV)
    before = bytes_of(pc.backing)
    out = torch.full((R, H, D), float("nan"), dtype=io, device=DEV)
    kda_decode_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pc.view, idx.to(DEV), out)
    torch.cuda.synchronize()
    rs = list(range(R)) if sample is None else sample
    P = H * D * D
    # oracle on a mini cache holding the sampled requests' rows (pre-step values)
    rows = [int(idx[r]) for r in rs]
    valid = [0 <= x < N for x in rows]
    es = pc.backing.element_size()
    host_before = before.view(np.float32 if es == 4 else np.uint16)
    mini = np.zeros(len(rs) * P, dtype=host_before.dtype)
    for j, (x, ok) in enumerate(zip(rows, valid)):
        if ok:
            s0 = pc.front + x * pc.row_stride
            mini[j * P:(j + 1) * P] = host_before[s0:s0 + P]
    mini_idx = [j if ok else -1 for j, ok in enumerate(valid)]
    pick = torch.tensor(rs, dtype=torch.long, device=DEV)
    o_ref = oracle.decode(f64(inp["q"][pick]), f64(inp["k"][pick]), f64(inp["v"][pick]), f64(inp["g"][pick]),
                          f64(inp["beta"][pick]), mini, len(rs), P, mini_idx, scale=D ** -0.5)
    assert_out_close(f64(out[pick]), o_ref)
    host_after = raw(pc.backing)
    for j, (x, ok) in enumerate(zip(rows, valid)):
        if ok:
            s0 = pc.front + x * pc.row_stride
            got = host_after[s0:s0 + P]
            want = mini[j * P:(j + 1) * P]
            to64 = (lambda a: a.astype(np.float64)) if es == 4 else \
                (lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
            assert_state_close(to64(got), to64(want), what=f"row {x}")
    # rows no request touched, page gaps and guards: unchanged bytes
    touched = np.zeros(host_after.size, dtype=bool)
    for x in idx.tolist():
        if 0 <= x < N:
            touched[pc.front + x * pc.row_stride: pc.front + x * pc.row_stride + P] = True
    assert np.array_equal(host_after[~touched].view(np.uint8), host_before[~touched].view(np.uint8))


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("io,cache_dtype", [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float32),
                                            (torch.float32, torch.float32)])
@pytest.mark.parametrize("itype", [torch.int32, torch.int64])
def test_decode_small(D, io, cache_dtype, itype):
    _decode_vs_oracle(R=37, H=3, D=D, io=io, cache_dtype=cache_dtype, N=64, itype=itype, stride_extra=64)


def test_decode_mild_decay():
    _decode_vs_oracle(R=16, H=4, D=128, io=torch.bfloat16, cache_dtype=torch.float32, N=32,
                      itype=torch.int32, decay=0.01)


def test_decode_full_workload_sampled():
    w = wl.decode()
    _decode_vs_oracle(R=w.R, H=w.H, D=w.K, io=w.io_dtype, cache_dtype=w.cache_dtype, N=w.cache_rows,
                      itype=torch.int32, sample=[0, 1, 2, 3, 100, 257, 400, 511])
    torch.cuda.empty_cache()


def test_decode_steps_equal_prefill():
    """L decode steps on an fp32 cache row reproduce the prefill of those L tokens."""
    from kimi_delta_attention_varlen_gb300 import kda_prefill_varlen, kda_prefill_workspace_size
    H, D, L = 2, 128, 70
    inp = wl.token_inputs(L, H, D, D, torch.bfloat16, seed=13, device=DEV)
    pc = wl.paged_cache(4, H, D, D, torch.float32, None, seed=14, device=DEV)
    init = pc.view[2:3].clone()
    out_p = torch.empty(L, H, D, dtype=torch.bfloat16, device=DEV)
    fin = torch.empty(1, H, D, D, device=DEV)
    ws = torch.empty(kda_prefill_workspace_size(L, 1, H, D, D), dtype=torch.uint8, device=DEV)
    kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                       torch.tensor([0, L], dtype=torch.int32, device=DEV), out_p, ws, init_state=init,
                       final_state=fin)
    idx = torch.tensor([2], dtype=torch.int32, device=DEV)
    out_d = torch.empty(L, H, D, dtype=torch.bfloat16, device=DEV)
    for t in range(L):
        kda_decode_step(inp["q"][t:t + 1], inp["k"][t:t + 1], inp["v"][t:t + 1], inp["g"][t:t + 1],
                        inp["beta"][t:t + 1], pc.view, idx, out_d[t:t + 1])
    torch.cuda.synchronize()
    assert_out_close(f64(out_d), f64(out_p))
    assert_state_close(f64(pc.view[2]), f64(fin[0]))
