"""Seeded synthetic inputs shaped like the workloads the pages describe.

This module holds none of the method's arithmetic.  It draws random numbers
(q, k, v ~ N(0,1) with q and k scaled to unit length per (token, head),
g = -softplus(N(0,1)), beta = sigmoid(N(0,1))), builds cu_seqlens and index
vectors, and lays out paged caches whose page gaps and guard bytes hold the
sentinel byte 0xA5.  Both the CUDA path (tests, benchmark) and the CPU oracle
consume what it produces; neither side's results feed back into it.

The five named workloads follow the benchmark configurations:
  tiny      3 sequences (64, 100, 37), H=2, K=V=32, fp32, cache [8,2,32,32]
            with stride(0) = 1.25 x payload, gather [5,-1,5] flags [T,T,F],
            scatter [2,-1,7]
  copy      fp32 cache [4096,32,128,128], stride(0) = payload + 64 KiB,
            256 rows, 10% invalid, flags p=0.8 (also a bf16 cache)
  varlen    16 sequences, lengths U[512, 8192], H=32, K=V=128, bf16,
            initial states from an fp32 cache [1024,...], 20% flags false
  long      one 131072-token sequence, zero initial state, final state to
            one row of an fp32 cache [64,...]
  decode    512 requests x 1 token, bf16 cache [2048,...], unique int32
            indices, 5% invalid
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SENTINEL = 0xA5
GUARD_BYTES = 256


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def cu_seqlens_of(lengths, device="cpu") -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def uniform_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=generator(seed))]


def token_inputs(T: int, H: int, K: int, V: int, io_dtype, seed: int, device="cpu",
                 decay_scale: float = 1.0, unit_qk: bool = True) -> dict:
    """q, k, v (io_dtype), g, beta (fp32) for T tokens, drawn on `device`."""
    gen = generator(seed, device)
    q = torch.randn(T, H, K, generator=gen, device=device)
    k = torch.randn(T, H, K, generator=gen, device=device)
    v = torch.randn(T, H, V, generator=gen, device=device)
    g = -torch.nn.functional.softplus(torch.randn(T, H, K, generator=gen, device=device)) * decay_scale
    beta = torch.sigmoid(torch.randn(T, H, generator=gen, device=device))
    if unit_qk:
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    return {"q": q.to(io_dtype).contiguous(), "k": k.to(io_dtype).contiguous(),
            "v": v.to(io_dtype).contiguous(), "g": g.contiguous(), "beta": beta.contiguous()}


@dataclass
class PagedCache:
    backing: torch.Tensor     # flat storage: guard | rows (payload + gap) | guard
    view: torch.Tensor        # [N, H, V, K] strided view into `backing`
    row_stride: int           # elements
    front: int                # storage offset of row 0, elements

    @property
    def payload(self) -> int:
        _, H, V, K = self.view.shape
        return H * V * K


def paged_cache(n_rows: int, H: int, V: int, K: int, dtype, row_stride: int | None, seed: int,
                device="cpu", fill: bool = True) -> PagedCache:
    """Cache [n_rows, H, V, K] with the given row stride (elements; None = dense).
    Every byte outside the row payloads is the sentinel; payloads are N(0,1)."""
    es = torch.empty((), dtype=dtype).element_size()
    P = H * V * K
    stride = P if row_stride is None else int(row_stride)
    assert stride >= P
    front = GUARD_BYTES // es
    total = front + n_rows * stride + GUARD_BYTES // es
    backing = torch.empty(total, dtype=dtype, device=device)
    backing.view(torch.uint8).fill_(SENTINEL)
    view = backing.as_strided((n_rows, H, V, K), (stride, V * K, K, 1), front)
    if fill:
        gen = generator(seed, device)
        chunk = max(1, (1 << 28) // P)  # fill in slabs of rows to bound temporaries
        for r0 in range(0, n_rows, chunk):
            r1 = min(n_rows, r0 + chunk)
            view[r0:r1].copy_(torch.randn(r1 - r0, H, V, K, generator=gen, device=device).to(dtype))
    return PagedCache(backing, view, stride, front)


def indices_with_invalid(base: torch.Tensor, N: int, p_invalid: float, seed: int, dtype) -> torch.Tensor:
    """Replace a p_invalid fraction of `base` by -1 or by N + r (both invalid)."""
    gen = generator(seed)
    S = base.numel()
    bad = torch.rand(S, generator=gen) < p_invalid
    neg = torch.rand(S, generator=gen) < 0.5
    big = N + torch.randint(0, 1000, (S,), generator=gen)
    out = torch.where(bad, torch.where(neg, torch.full_like(base, -1), big), base)
    return out.to(dtype)


def gather_indices(S: int, N: int, p_invalid: float, seed: int, dtype=torch.int32) -> torch.Tensor:
    base = torch.randint(0, N, (S,), generator=generator(seed))  # duplicates allowed
    return indices_with_invalid(base, N, p_invalid, seed + 1, dtype)


def scatter_indices(S: int, N: int, p_invalid: float, seed: int, dtype=torch.int32) -> torch.Tensor:
    base = torch.randperm(N, generator=generator(seed))[:S]  # unique targets
    return indices_with_invalid(base, N, p_invalid, seed + 1, dtype)


def bernoulli_flags(S: int, p_true: float, seed: int) -> torch.Tensor:
    return torch.rand(S, generator=generator(seed)) < p_true


# ------------------------------------------------------------- workloads --

@dataclass
class PrefillWorkload:
    name: str
    lengths: list
    H: int
    K: int
    V: int
    io_dtype: torch.dtype
    cache_rows: int
    cache_dtype: torch.dtype
    cache_stride: int | None
    gather_idx: torch.Tensor
    gather_flags: torch.Tensor
    scatter_idx: torch.Tensor
    seed: int = 0
    decay_scale: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    @property
    def B(self) -> int:
        return len(self.lengths)


def tiny(seed: int = 0) -> PrefillWorkload:
    P = 2 * 32 * 32
    return PrefillWorkload("tiny: lengths 64,100,37 H=2 K=V=32 fp32", [64, 100, 37], 2, 32, 32, torch.float32,
                           8, torch.float32, P + P // 4,
                           torch.tensor([5, -1, 5], dtype=torch.int32), torch.tensor([True, True, False]),
                           torch.tensor([2, -1, 7], dtype=torch.int32), seed)


def varlen(seed: int = 0, B: int = 16, lo: int = 512, hi: int = 8192) -> PrefillWorkload:
    lengths = uniform_lengths(B, lo, hi, seed)
    rows = torch.randperm(1024, generator=generator(seed + 11))[:B].to(torch.int32)
    flags = torch.rand(B, generator=generator(seed + 12)) >= 0.2
    return PrefillWorkload(f"varlen: B={B} lengths U[{lo},{hi}] H=32 K=V=128 bf16", lengths, 32, 128, 128,
                           torch.bfloat16, 1024, torch.float32, None, rows, flags, rows.clone(), seed)


def long_seq(seed: int = 0, T: int = 131072) -> PrefillWorkload:
    row = torch.randint(0, 64, (1,), generator=generator(seed + 13)).to(torch.int32)
    return PrefillWorkload(f"long: T={T} B=1 H=32 K=V=128 bf16", [T], 32, 128, 128, torch.bfloat16, 64,
                           torch.float32, None, row, torch.tensor([False]), row.clone(), seed)


@dataclass
class CopyWorkload:
    name: str
    N: int
    H: int
    V: int
    K: int
    dtype: torch.dtype
    row_stride: int
    S: int
    p_invalid: float
    p_flag: float
    seed: int = 0


def copy_fp32(seed: int = 0, N: int = 4096, S: int = 256) -> CopyWorkload:
    P = 32 * 128 * 128
    return CopyWorkload(f"copy: fp32 cache [{N},32,128,128] stride payload+64KiB, S={S}", N, 32, 128, 128,
                        torch.float32, P + (64 << 10) // 4, S, 0.1, 0.8, seed)


def copy_bf16(seed: int = 0, N: int = 4096, S: int = 256) -> CopyWorkload:
    P = 32 * 128 * 128
    return CopyWorkload(f"copy: bf16 cache [{N},32,128,128] stride payload+64KiB, S={S}", N, 32, 128, 128,
                        torch.bfloat16, P + (64 << 10) // 2, S, 0.1, 0.8, seed)


@dataclass
class DecodeWorkload:
    name: str
    R: int
    H: int
    K: int
    V: int
    io_dtype: torch.dtype
    cache_rows: int
    cache_dtype: torch.dtype
    idx: torch.Tensor
    seed: int = 0


def decode(seed: int = 0, R: int = 512, N: int = 2048) -> DecodeWorkload:
    base = torch.randperm(N, generator=generator(seed + 21))[:R]
    bad = torch.rand(R, generator=generator(seed + 22)) < 0.05
    idx = torch.where(bad, torch.full_like(base, -1), base).to(torch.int32)
    return DecodeWorkload(f"decode: R={R} H=32 K=V=128 bf16, bf16 cache [{N},32,128,128]", R, 32, 128, 128,
                          torch.bfloat16, N, torch.bfloat16, idx, seed)
