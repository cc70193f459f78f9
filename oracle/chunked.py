"""Chunkwise (UT / WY) form of the KDA recurrence, fp64 numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

This restates, in plain numpy and for any chunk size C, the steps the
"Support Kimi-K3 on NPU" report's ``_AscendKDAExtendKernel.extend`` listing
performs in order:

  1. L2-normalise q and k per (token, head);
  2. split each sequence of the cu_seqlens batch into chunks of C tokens,
     restarting at every sequence start (the last chunk may be partial);
  3. G = cumulative sum of the log-decay g inside each chunk, per channel
     (the listing scales it by log2(e) to use exp2; that is the same function);
  4. gated K K^T and Q K^T products:
        A_kk[i, j] = beta_i * sum_c k_ic k_jc exp(G_ic - G_jc)   for i > j
        A_qk[i, j] =          sum_c q_ic k_jc exp(G_ic - G_jc)   for i >= j
  5. T = (I + A_kk)^-1 (unit lower triangular solve);
  6. W = T diag(beta) (K * exp(G)),  U = T diag(beta) V;
  7. state pass over chunks in order:
        V_new = U - W S
        O     = scale * ((Q * exp(G)) S + A_qk V_new)
        S     = diag(exp(G_last)) S + (K * exp(G_last - G))^T V_new
     starting from the initial state.

The tests use it as an independent formulation: it must agree with the
token-by-token recurrence of ``kda_oracle.c`` (the affine-composition
property of the "KDA's challenges for AI infra" page, section 1.3, is what
makes the two equal).  Exponentials are taken element by element, exactly.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

from . import EPS


def l2normalise(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def chunk_table(cu_seqlens, C: int):
    """(sequence, first token, last token + 1) for every chunk, sequences in order."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    table = []
    for b in range(cu.size - 1):
        for t0 in range(int(cu[b]), int(cu[b + 1]), C):
            table.append((b, t0, min(t0 + C, int(cu[b + 1]))))
    return table


def chunk_quantities(q, k, v, g, beta, scale=1.0):
    """Steps 3-6 for ONE chunk of one head (q, k already normalised).

    q, k, g: [n, K]; v: [n, V]; beta: [n].  Returns dict with G, A_kk, A_qk, T, W, U."""
    n = q.shape[0]
    G = np.cumsum(g, axis=0)
    lower = np.tril(np.ones((n, n), dtype=bool))
    diff = np.where(lower[:, :, None], G[:, None, :] - G[None, :, :], -np.inf)
    decay = np.exp(diff)  # exp(G_i - G_j) on i >= j, zero above the diagonal
    a_kk = beta[:, None] * np.einsum("ic,jc,ijc->ij", k, k, decay)
    a_kk = np.tril(a_kk, k=-1)
    a_qk = np.einsum("ic,jc,ijc->ij", q, k, decay)
    eye = np.eye(n)
    T = solve_triangular(eye + a_kk, eye, lower=True, unit_diagonal=True)
    W = T @ (beta[:, None] * k * np.exp(G))
    U = T @ (beta[:, None] * v)
    return {"G": G, "A_kk": a_kk, "A_qk": a_qk * scale, "T": T, "W": W, "U": U}


def prefill(q, k, v, g, beta, cu_seqlens, C=64, init=None, scale=1.0, l2norm=True, eps=EPS):
    """Chunked prefill.  Same arguments and results as ``oracle.prefill``."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, H, K = q.shape
    V = v.shape[2]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    B = cu.size - 1
    if l2norm:
        q = l2normalise(q, eps)
        k = l2normalise(k, eps)
    out = np.zeros((T, H, V))
    final = np.zeros((B, H, V, K))
    chunks = chunk_table(cu, C)
    for h in range(H):
        states = {}
        for b in range(B):
            states[b] = init[b, h].T.copy() if init is not None else np.zeros((K, V))
        for b, t0, t1 in chunks:
            S = states[b]
            cq = chunk_quantities(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h],
                                  beta[t0:t1, h], scale)
            G = cq["G"]
            v_new = cq["U"] - cq["W"] @ S
            out[t0:t1, h] = scale * ((q[t0:t1, h] * np.exp(G)) @ S) + cq["A_qk"] @ v_new
            k_tilde = k[t0:t1, h] * np.exp(G[-1][None, :] - G)
            states[b] = np.exp(G[-1])[:, None] * S + k_tilde.T @ v_new
        for b in range(B):
            final[b, h] = states[b].T
    return out, final
