"""GPU parity of kda_state_gather / kda_state_scatter against the oracle.

Bit-exact comparisons of the whole backing buffer (payloads, page gaps, guard
bytes) on small layouts, and of sampled rows on the full-size copy workload
(fp32 cache [4096,32,128,128] with 64 KiB page gaps: 8.25 GiB, so rows lie
beyond 4 GiB).  Contract: "vllm-ascend KDA state copy" page, "Numeric
contract"."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_varlen_gb300 import (KdaError, kda_state_gather, kda_state_scatter)
from kimi_delta_attention_varlen_gb300 import workloads as wl
from tests.helpers import bytes_of, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _oracle_gather(pc: wl.PagedCache, idx, flags):
    N, H, V, K = pc.view.shape
    host = raw(pc.backing)[pc.front:pc.front + N * pc.row_stride]
    return oracle.gather(host, N, H * V * K, pc.row_stride, idx.cpu().numpy(),
                         None if flags is None else flags.cpu().numpy())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("itype", [torch.int32, torch.int64])
@pytest.mark.parametrize("gap", [0, 37, 64])  # 37 elements: misaligned rows -> element-wise kernels
def test_gather_small_bitexact(dtype, itype, gap):
    N, H, V, K, S = 23, 3, 16, 32, 70
    P = H * V * K
    pc = wl.paged_cache(N, H, V, K, dtype, P + gap, seed=1, device=DEV)
    idx = wl.gather_indices(S, N, 0.15, seed=2, dtype=itype)
    flags = wl.bernoulli_flags(S, 0.8, seed=3)
    before = bytes_of(pc.backing)
    packed = torch.full((S, H, V, K), 7.0, dtype=dtype, device=DEV)
    kda_state_gather(pc.view, idx.to(DEV), packed, flags.to(DEV))
    torch.cuda.synchronize()
    want = _oracle_gather(pc, idx, flags)
    assert np.array_equal(raw(packed).reshape(S, -1), want)
    assert np.array_equal(bytes_of(pc.backing), before)  # the cache is only read
    # without flags every valid row comes back, duplicates included
    kda_state_gather(pc.view, idx.to(DEV), packed, None)
    torch.cuda.synchronize()
    assert np.array_equal(raw(packed).reshape(S, -1), _oracle_gather(pc, idx, None))


@pytest.mark.parametrize("cache_dtype,packed_dtype", [(torch.float32, torch.float32),
                                                      (torch.bfloat16, torch.bfloat16),
                                                      (torch.bfloat16, torch.float32),
                                                      (torch.float32, torch.bfloat16)])
@pytest.mark.parametrize("itype", [torch.int32, torch.int64])
@pytest.mark.parametrize("gap", [0, 37, 64])
def test_scatter_small_bitexact(cache_dtype, packed_dtype, itype, gap):
    N, H, V, K, S = 29, 2, 32, 32, 20
    P = H * V * K
    pc = wl.paged_cache(N, H, V, K, cache_dtype, P + gap, seed=4, device=DEV)
    idx = wl.scatter_indices(S, N, 0.2, seed=5, dtype=itype)
    packed = torch.randn(S, H, V, K, generator=wl.generator(6, DEV), device=DEV).to(packed_dtype)
    host = raw(pc.backing)
    kda_state_scatter(pc.view, idx.to(DEV), packed)
    torch.cuda.synchronize()
    body = host[pc.front:pc.front + N * pc.row_stride]
    oracle.scatter(body, N, P, pc.row_stride, idx.numpy(), raw(packed).reshape(S, -1))
    host[pc.front:pc.front + N * pc.row_stride] = body
    got = raw(pc.backing)
    assert np.array_equal(got.view(np.uint8), host.view(np.uint8))  # payloads, gaps and guards


def test_empty_selection_launches_nothing():
    pc = wl.paged_cache(4, 2, 8, 8, torch.float32, None, seed=7, device=DEV)
    before = bytes_of(pc.backing)
    idx = torch.empty(0, dtype=torch.int32, device=DEV)
    packed = torch.empty(0, 2, 8, 8, device=DEV)
    kda_state_gather(pc.view, idx, packed)
    kda_state_scatter(pc.view, idx, packed)
    torch.cuda.synchronize()
    assert np.array_equal(bytes_of(pc.backing), before)


def test_bad_layout_is_rejected_before_launch():
    pc = wl.paged_cache(4, 2, 8, 8, torch.float32, None, seed=8, device=DEV)
    overlapping = pc.backing.as_strided((4, 2, 8, 8), (100, 64, 8, 1), pc.front)  # stride < payload
    idx = torch.zeros(2, dtype=torch.int32, device=DEV)
    packed = torch.zeros(2, 2, 8, 8, device=DEV)
    with pytest.raises(KdaError):
        kda_state_gather(overlapping, idx, packed)
    roomy = torch.zeros(4096, device=DEV)
    inner_strided = roomy.as_strided((4, 2, 8, 8), (256, 128, 8, 1), 0)  # heads 128 apart, not 64
    with pytest.raises(ValueError):
        kda_state_gather(inner_strided, idx, packed)


def test_graph_replay_with_swapped_indices_and_flags():
    """Calls capture into a CUDA graph; new index / flag VALUES take effect on replay."""
    N, H, V, K, S = 16, 2, 16, 16, 12
    pc = wl.paged_cache(N, H, V, K, torch.float32, H * V * K + 16, seed=9, device=DEV)
    idx = wl.gather_indices(S, N, 0.2, seed=10).to(DEV)
    flags = wl.bernoulli_flags(S, 0.7, seed=11).to(DEV)
    packed = torch.zeros(S, H, V, K, device=DEV)
    stream = torch.cuda.Stream()
    kda_state_gather(pc.view, idx, packed, flags, stream=stream)  # warm-up outside capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kda_state_gather(pc.view, idx, packed, flags, stream=torch.cuda.current_stream())
    for trial in range(3):
        idx.copy_(wl.gather_indices(S, N, 0.2, seed=20 + trial).to(DEV))
        flags.copy_(wl.bernoulli_flags(S, 0.6, seed=30 + trial).to(DEV))
        packed.fill_(3.0)
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(raw(packed).reshape(S, -1), _oracle_gather(pc, idx.cpu(), flags.cpu()))


@pytest.mark.parametrize("which", ["fp32", "bf16"])
def test_full_size_copy_beyond_4gib(which):
    """Full copy workload: sampled rows checked bit-exactly, including rows whose
    byte offset exceeds 4 GiB, with both int32 and int64 indices."""
    w = wl.copy_fp32() if which == "fp32" else wl.copy_bf16()
    pc = wl.paged_cache(w.N, w.H, w.V, w.K, w.dtype, w.row_stride, seed=w.seed, device=DEV)
    es = pc.backing.element_size()
    assert (w.N - 1) * w.row_stride * es > (1 << 32)
    P = pc.payload
    gidx = wl.gather_indices(w.S, w.N, w.p_invalid, seed=w.seed + 1)
    gidx[:4] = torch.tensor([w.N - 1, w.N - 2, w.N // 2 + 7, 0], dtype=torch.int32)  # far rows
    flags = wl.bernoulli_flags(w.S, w.p_flag, seed=w.seed + 2)
    flags[:4] = True
    packed = torch.empty(w.S, w.H, w.V, w.K, dtype=w.dtype, device=DEV)
    sample = [0, 1, 2, 3] + [int(s) for s in torch.randperm(w.S, generator=wl.generator(5))[:12]]
    for itype in (torch.int32, torch.int64):
        packed.fill_(1.0)
        kda_state_gather(pc.view, gidx.to(itype).to(DEV), packed, flags.to(DEV))
        torch.cuda.synchronize()
        for s in sample:
            r = int(gidx[s])
            valid = 0 <= r < w.N and bool(flags[s])
            row = raw(pc.view[r].reshape(-1)) if valid else None
            mini = np.zeros(P, dtype=raw(packed[s].reshape(-1)).dtype) if row is None else row
            want = oracle.gather(mini, 1, P, P, [0 if valid else -1], None)[0]
            assert np.array_equal(raw(packed[s].reshape(-1)), want), f"row s={s} idx={r}"
    # scatter into unique rows (fp32 packed -> cache dtype)
    sidx = wl.scatter_indices(w.S, w.N, w.p_invalid, seed=w.seed + 3)
    sidx[0] = w.N - 1
    src = torch.randn(w.S, w.H, w.V, w.K, generator=wl.generator(12, DEV), device=DEV)
    probe_rows = sorted({w.N - 1, w.N - 2, 0, 1, 3000} | {int(r) for r in sidx[:6] if 0 <= int(r) < w.N})
    stride = pc.row_stride
    before = {r: raw(pc.backing[pc.front + r * stride: pc.front + (r + 1) * stride]) for r in probe_rows}
    kda_state_scatter(pc.view, sidx.to(torch.int64).to(DEV), src)
    torch.cuda.synchronize()
    sidx_np = sidx.numpy()
    for r in probe_rows:
        host = before[r].copy()
        hits = np.nonzero(sidx_np == r)[0]
        sub_idx = [0] if hits.size else [-1]
        sub_src = raw(src[int(hits[0])].reshape(1, -1)) if hits.size else np.zeros((1, P), np.float32)
        oracle.scatter(host, 1, P, stride, sub_idx, sub_src)
        got = raw(pc.backing[pc.front + r * stride: pc.front + (r + 1) * stride])
        assert np.array_equal(got.view(np.uint8), host.view(np.uint8)), f"row {r}"
    del pc, packed, src
    torch.cuda.empty_cache()
