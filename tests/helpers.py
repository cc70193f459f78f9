"""Helpers shared by the tests: host copies, tolerance checks, oracle calls on
device-resident workloads.  Tolerances are the ones the method's target fixes:
outputs max|d| <= 2e-2 * max|ref|; states ||dS||_F <= 1e-2 * ||S_ref||_F;
state copies bit-exact."""
from __future__ import annotations

import numpy as np
import torch

import oracle

OUT_TOL = 2e-2
STATE_TOL = 1e-2


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def raw(t: torch.Tensor) -> np.ndarray:
    """Host copy with the oracle's element types: float32, or bf16 as uint16 bits."""
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    raise TypeError(t.dtype)


def bytes_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.uint8).numpy().copy()


def assert_out_close(got: np.ndarray, ref: np.ndarray, what: str = "out") -> float:
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err <= OUT_TOL * scale, f"{what}: max|d| = {err:.3e} > {OUT_TOL} * {scale:.3e}"
    return err / scale


def assert_state_close(got: np.ndarray, ref: np.ndarray, what: str = "state") -> float:
    nref = float(np.linalg.norm(ref))
    err = float(np.linalg.norm(got - ref))
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    if nref == 0.0:
        assert err == 0.0, f"{what}: expected zeros"
        return 0.0
    assert err <= STATE_TOL * nref, f"{what}: ||d||/||ref|| = {err / nref:.3e} > {STATE_TOL}"
    return err / nref


def oracle_prefill_from_device(inp: dict, cu: list, init, scale: float, l2norm: bool = True,
                               heads=None, seqs=None):
    """Run the oracle on (a sample of) a device-resident prefill batch.
    heads / seqs: lists of head / sequence indices to evaluate (None = all).
    Returns (out [T_sel, H_sel, V], final [B_sel, H_sel, V, K], token index list)."""
    B = len(cu) - 1
    seqs = list(range(B)) if seqs is None else list(seqs)
    hsel = slice(None) if heads is None else list(heads)
    toks, cu_sel = [], [0]
    for b in seqs:
        toks.extend(range(cu[b], cu[b + 1]))
        cu_sel.append(cu_sel[-1] + cu[b + 1] - cu[b])
    tix = torch.tensor(toks, dtype=torch.long, device=inp["q"].device)

    def pick(t):
        return f64(t.index_select(0, tix)[:, hsel])

    ini = None
    if init is not None:
        ini = f64(init[seqs][:, hsel])
    out, fin = oracle.prefill(pick(inp["q"]), pick(inp["k"]), pick(inp["v"]), pick(inp["g"]),
                              pick(inp["beta"]), cu_sel, init=ini, scale=scale, l2norm=l2norm)
    return out, fin, toks
