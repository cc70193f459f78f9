"""Pins for the CPU oracle: each test ties the oracle to something other than
itself (a hand-derived worked example, a closed form, an invariant of the
method, a library routine, or an independent formulation), so that a dropped
term, a wrong sign or index or a transposed operand fails at least one test.

Sources of the facts pinned here:
  - "vllm-ascend KDA state copy" page, section "Numeric contract"
    (gather zeros / skips / gaps / casts);
  - "KDA's challenges for AI infra" page, section 1.1 (the recurrence),
    section 1.3 (affine composition of segments), section 9.1 (the unrolled
    sum S_n = M_n..M_1 S_0 + sum_i M_n..M_{i+1} b_i);
  - "Support Kimi-K3 on NPU" report, extend listing (chunked UT form, chunk
    restart at each sequence start, L2 normalisation of q and k).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softplus(x):
    return np.log1p(np.exp(x))


def rand_tokens(seed, lengths, H, K, V, decay=1.0):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    g = -_softplus(rng.standard_normal((T, H, K))) * decay
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, g, beta, cu


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

def test_bf16_golden_table():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rne.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                a, b = line.split()
                rows.append((int(a, 16), int(b, 16)))
    x = np.array([r[0] for r in rows], dtype=np.uint32).view(np.float32)
    got = oracle.f32_to_bf16_bits(x)
    assert [int(v) for v in got] == [r[1] for r in rows]


def test_bf16_matches_torch_rounding():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000).astype(np.float32) * np.float32(1000)
    # force a block of exact ties with both parities of the kept part
    bits = x.view(np.uint32).copy()
    bits[:5000] = (bits[:5000] & 0xFFFF0000) | 0x8000
    x = bits.view(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f32_to_bf16_bits(x), ref)


# --------------------------------------------------------------------------
# state copy contract
# --------------------------------------------------------------------------

SENT = np.uint32(0xA5A5A5A5)


def _golden_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line or ":" not in line:
                continue
            key, val = line.split(":", 1)
            out[key.strip()] = val.split()
    return out


def _small_cache():
    N, P, stride = 3, 2, 3
    cache = np.full(N * stride, SENT, dtype=np.uint32).view(np.float32)
    for r in range(N):
        cache[r * stride:r * stride + P] = [2 * r + 1, 2 * r + 2]
    return cache, N, P, stride


def test_gather_golden():
    gd = _golden_kv("state_copy_small.txt")
    cache, N, P, stride = _small_cache()
    before = cache.copy()
    idx = [int(x) for x in gd["gather_idx"]]
    flags = [int(x) for x in gd["gather_flags"]]
    got = oracle.gather(cache, N, P, stride, idx, flags)
    assert np.array_equal(got.reshape(-1), np.array(gd["gather_out_flags"], dtype=np.float32))
    got = oracle.gather(cache, N, P, stride, idx, None)
    assert np.array_equal(got.reshape(-1), np.array(gd["gather_out_noflags"], dtype=np.float32))
    assert np.array_equal(cache.view(np.uint32), before.view(np.uint32))  # read only


def test_scatter_golden():
    gd = _golden_kv("state_copy_small.txt")
    N, P, stride = 3, 2, 3
    cache = np.full(N * stride, SENT, dtype=np.uint32).view(np.float32)
    for r in range(N):
        cache[r * stride:r * stride + P] = 9.0
    idx = [int(x) for x in gd["scatter_idx"]]
    packed = np.array(gd["scatter_packed"], dtype=np.float32).reshape(3, P)
    oracle.scatter(cache, N, P, stride, idx, packed)
    rows = cache.reshape(N, stride)
    assert np.array_equal(rows[:, :P].reshape(-1), np.array(gd["scatter_rows_after"], dtype=np.float32))
    assert np.all(rows[:, P:].view(np.uint32) == SENT)


def test_scatter_cast_golden():
    gd = _golden_kv("state_copy_small.txt")
    vals = np.array(gd["cast_packed"], dtype=np.float32)
    n = vals.size
    cache = np.full(n + 2, 0xA5A5, dtype=np.uint16)  # one row, payload n, 2 gap elements
    oracle.scatter(cache, 1, n, n + 2, [0], vals.reshape(1, n))
    assert [int(x) for x in cache[:n]] == [int(b, 16) for b in gd["cast_bits"]]
    assert np.all(cache[n:] == 0xA5A5)


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_gather_scatter_contract_random(dtype):
    rng = np.random.default_rng(7)
    N, P, stride, S = 9, 24, 31, 40
    if dtype == np.float32:
        cache = np.full(N * stride, SENT, dtype=np.uint32).view(np.float32)
        payload = rng.standard_normal((N, P)).astype(np.float32)
    else:
        cache = np.full(N * stride, 0xA5A5, dtype=np.uint16)
        payload = rng.integers(0, 0x7F00, size=(N, P), dtype=np.uint16)
    cache.reshape(N, stride)[:, :P] = payload
    gap_before = cache.reshape(N, stride)[:, P:].copy()
    idx = rng.integers(-3, N + 3, size=S)
    flags = rng.integers(0, 2, size=S)
    got = oracle.gather(cache, N, P, stride, idx, flags)
    for s in range(S):
        valid = 0 <= idx[s] < N and flags[s]
        want = payload[idx[s]] if valid else np.zeros(P, dtype=dtype)
        assert np.array_equal(got[s].view(np.uint8), want.view(np.uint8))
    # empty selection: nothing read, nothing produced
    assert oracle.gather(cache, N, P, stride, [], None).shape == (0, P)
    # scatter with unique valid targets; invalid ones skipped; flags play no part
    targets = np.array([4, -1, 0, N, 7, -9], dtype=np.int64)
    src = got[: targets.size]
    oracle.scatter(cache, N, P, stride, targets, src)
    rows = cache.reshape(N, stride)
    for r in range(N):
        hits = [s for s, t in enumerate(targets) if t == r]
        want = src[hits[0]] if hits else payload[r]
        assert np.array_equal(rows[r, :P].view(np.uint8), want.view(np.uint8))
    assert np.array_equal(rows[:, P:].view(np.uint8), gap_before.view(np.uint8))


def test_scatter_bf16_to_f32_is_exact_upcast():
    bits = np.array([[0x3F80, 0xC049, 0x0000, 0x7F7F]], dtype=np.uint16)
    cache = np.zeros(4, dtype=np.float32)
    oracle.scatter(cache, 1, 4, 4, [0], bits)
    want = (bits.astype(np.uint32) << 16).view(np.float32).reshape(-1)
    assert np.array_equal(cache, want)


# --------------------------------------------------------------------------
# recurrence: worked example and closed forms
# --------------------------------------------------------------------------

def _golden_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "kda_two_token.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            if line == "end":
                cases.append(cur)
                cur = None
                continue
            key, val = line.split(":", 1)
            if key == "case":
                cur = {"name": val.strip()}
            else:
                cur[key] = [float(x) for x in val.split()]
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_worked_example(case):
    T = len(case["beta"])
    q = np.array(case["q"]).reshape(T, 1, 2)
    k = np.array(case["k"]).reshape(T, 1, 2)
    v = np.array(case["v"]).reshape(T, 1, 2)
    g = np.array(case["g"]).reshape(T, 1, 2)
    beta = np.array(case["beta"]).reshape(T, 1)
    init = np.array(case["init_vk"]).reshape(1, 1, 2, 2)
    out, final = oracle.prefill(q, k, v, g, beta, [0, T], init=init, scale=case["scale"][0],
                                l2norm=bool(case["l2norm"][0]))
    tol = case["tol"][0]
    np.testing.assert_allclose(out.reshape(-1), case["out"], rtol=0, atol=tol * 10)
    np.testing.assert_allclose(final.reshape(-1), case["final_vk"], rtol=0, atol=tol * 10)
    # the chunked form reproduces the same example
    out_c, final_c = chunked.prefill(q, k, v, g, beta, [0, T], C=2, init=init,
                                     scale=case["scale"][0], l2norm=bool(case["l2norm"][0]))
    np.testing.assert_allclose(out_c.reshape(-1), case["out"], rtol=0, atol=tol * 10)
    np.testing.assert_allclose(final_c.reshape(-1), case["final_vk"], rtol=0, atol=tol * 10)


def test_beta0_g0_leaves_state_unchanged():
    q, k, v, g, beta, cu = rand_tokens(2, [13], 2, 8, 6)
    g[:] = 0.0
    beta[:] = 0.0
    rng = np.random.default_rng(3)
    init = rng.standard_normal((1, 2, 6, 8))
    out, final = oracle.prefill(q, k, v, g, beta, cu, init=init, scale=0.7)
    np.testing.assert_allclose(final, init, rtol=0, atol=1e-14)
    qn = chunked.l2normalise(q)
    want = 0.7 * np.einsum("thk,hvk->thv", qn, init[0])  # o = scale * S0^T q
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-13)


def test_strong_decay_resets_state():
    # exp(-50) ~ 2e-22: the old state is wiped at every token
    q, k, v, g, beta, cu = rand_tokens(4, [9], 3, 8, 5)
    g[:] = -50.0
    init = np.random.default_rng(5).standard_normal((1, 3, 5, 8))
    out, final = oracle.prefill(q, k, v, g, beta, cu, init=init, scale=1.3)
    qn, kn = chunked.l2normalise(q), chunked.l2normalise(k)
    last = 8
    want_final = beta[last][:, None, None] * v[last][:, :, None] * kn[last][:, None, :]
    np.testing.assert_allclose(final[0], want_final, rtol=0, atol=1e-12)
    want_out = 1.3 * beta[:, :, None] * np.sum(kn * qn, axis=-1)[:, :, None] * v
    np.testing.assert_allclose(out, want_out, rtol=0, atol=1e-12)


def test_orthonormal_keys_closed_form():
    K, V, T = 8, 4, 6
    perm = np.random.default_rng(6).permutation(K)[:T]
    q, _, v, g, beta, cu = rand_tokens(7, [T], 1, K, V)
    k = np.zeros((T, 1, K))
    k[np.arange(T), 0, perm] = 1.0
    g[:] = 0.0
    out, final = oracle.prefill(q, k, v, g, beta, cu, l2norm=False)
    S = np.zeros((K, V))
    for t in range(T):
        S[perm[t]] = beta[t, 0] * v[t, 0]  # row pi(t) holds beta_t v_t^T
    np.testing.assert_allclose(final[0, 0], S.T, rtol=0, atol=1e-14)


def test_repeated_key_is_moving_average():
    K, V, T = 6, 3, 11
    rng = np.random.default_rng(8)
    kvec = unit(rng.standard_normal(K))
    q, _, v, g, beta, cu = rand_tokens(9, [T], 1, K, V)
    k = np.tile(kvec, (T, 1, 1))
    g[:] = 0.0
    S0 = rng.standard_normal((K, V))
    _, final = oracle.prefill(q, k, v, g, beta, cu, init=S0.T[None, None], l2norm=False)
    S = final[0, 0].T
    s = kvec @ S0
    for t in range(T):
        s = (1 - beta[t, 0]) * s + beta[t, 0] * v[t, 0]
    np.testing.assert_allclose(kvec @ S, s, rtol=0, atol=1e-12)
    proj = np.eye(K) - np.outer(kvec, kvec)  # the orthogonal complement is untouched
    np.testing.assert_allclose(proj @ S, proj @ S0, rtol=0, atol=1e-12)


def test_delta_rule_read_back():
    """After a write with beta = 1, reading with the same key returns v exactly,
    whatever the decay and the prior state; with beta < 1 the read is the
    beta-blend of v and the decayed prior read (decay acts before the erase)."""
    K, V, T = 8, 5, 7
    q, k, v, g, beta, cu = rand_tokens(10, [T], 2, K, V, decay=0.6)
    init = np.random.default_rng(11).standard_normal((1, 2, V, K))
    kn = unit(k)  # exactly unit keys, normalisation off: k^T k = 1 to rounding
    beta1 = beta.copy()
    beta1[-1] = 1.0
    _, fin = oracle.prefill(q, kn, v, g, beta1, cu, init=init, l2norm=False)
    np.testing.assert_allclose(np.einsum("hk,hvk->hv", kn[-1], fin[0]), v[-1], rtol=0, atol=1e-12)
    _, prev = oracle.prefill(q[:-1], kn[:-1], v[:-1], g[:-1], beta[:-1], [0, T - 1], init=init,
                             l2norm=False)
    _, cur = oracle.prefill(q, kn, v, g, beta, cu, init=init, l2norm=False)
    decayed_read = np.einsum("hk,hvk->hv", kn[-1] * np.exp(g[-1]), prev[0])
    want = (1 - beta[-1])[:, None] * decayed_read + beta[-1][:, None] * v[-1]
    np.testing.assert_allclose(np.einsum("hk,hvk->hv", kn[-1], cur[0]), want, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# recurrence: affine structure (sections 1.3 and 9.1 of the infra page)
# --------------------------------------------------------------------------

def _affine_map(q, k, v, g, beta, K, V):
    """Probe the oracle's segment map F(S0) = M S0 + b (one head): returns (M, b)
    with M: K x K and b: K x V, from K + 1 runs."""
    T = q.shape[0]

    def run(S0):
        _, fin = oracle.prefill(q, k, v, g, beta, [0, T], init=S0.T[None, None])
        return fin[0, 0].T

    b = run(np.zeros((K, V)))
    M = np.zeros((K, K))
    for i in range(K):
        E = np.zeros((K, V))
        E[i, 0] = 1.0
        M[:, i] = (run(E) - b)[:, 0]
    return M, b


def test_single_token_map_is_the_stated_matrix():
    K, V = 5, 3
    q, k, v, g, beta, _ = rand_tokens(12, [1], 1, K, V)
    M, b = _affine_map(q, k, v, g, beta, K, V)
    kn = chunked.l2normalise(k)[0, 0]
    want_M = (np.eye(K) - beta[0, 0] * np.outer(kn, kn)) @ np.diag(np.exp(g[0, 0]))
    want_b = beta[0, 0] * np.outer(kn, v[0, 0])
    np.testing.assert_allclose(M, want_M, rtol=0, atol=1e-13)
    np.testing.assert_allclose(b, want_b, rtol=0, atol=1e-13)


def test_map_acts_on_all_value_columns_alike():
    K, V, T = 5, 4, 6
    q, k, v, g, beta, _ = rand_tokens(13, [T], 1, K, V)
    M, b = _affine_map(q, k, v, g, beta, K, V)
    S0 = np.random.default_rng(14).standard_normal((K, V))
    _, fin = oracle.prefill(q, k, v, g, beta, [0, T], init=S0.T[None, None])
    np.testing.assert_allclose(fin[0, 0].T, M @ S0 + b, rtol=0, atol=1e-12)


def test_affine_composition_and_unrolled_sum():
    K, V, T1, T2 = 4, 3, 5, 4
    q, k, v, g, beta, _ = rand_tokens(15, [T1 + T2], 1, K, V, decay=0.1)
    seg1 = tuple(a[:T1] for a in (q, k, v, g, beta))
    seg2 = tuple(a[T1:] for a in (q, k, v, g, beta))
    M1, b1 = _affine_map(*seg1, K, V)
    M2, b2 = _affine_map(*seg2, K, V)
    M12, b12 = _affine_map(q, k, v, g, beta, K, V)
    # F_C2(F_C1(S)) = M_C2 M_C1 S + M_C2 b_C1 + b_C2
    np.testing.assert_allclose(M12, M2 @ M1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(b12, M2 @ b1 + b2, rtol=0, atol=1e-12)
    # not commutative: the other order gives a different map
    assert np.linalg.norm(M1 @ M2 - M2 @ M1) > 1e-2 * np.linalg.norm(M2 @ M1)
    # S_n = M_n..M_1 S_0 + sum_i M_n..M_{i+1} b_i, from per-token maps
    n = T1 + T2
    maps = [_affine_map(*(a[t:t + 1] for a in (q, k, v, g, beta)), K, V) for t in range(n)]
    S0 = np.random.default_rng(16).standard_normal((K, V))
    prod = np.eye(K)
    for t in range(n):
        prod = maps[t][0] @ prod
    unrolled = prod @ S0
    for i in range(n):
        tail = np.eye(K)
        for t in range(i + 1, n):
            tail = maps[t][0] @ tail
        unrolled += tail @ maps[i][1]
    _, fin = oracle.prefill(q, k, v, g, beta, [0, n], init=S0.T[None, None])
    np.testing.assert_allclose(fin[0, 0].T, unrolled, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# chunked form == sequential recurrence; varlen; decode; edge cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("C", [1, 7, 16, 64])
@pytest.mark.parametrize("decay", [1.0, 0.01])
def test_chunked_equals_sequential(C, decay):
    lengths = [64, 100, 37, 1]
    q, k, v, g, beta, cu = rand_tokens(20 + C, lengths, 2, 16, 12, decay=decay)
    init = np.random.default_rng(21).standard_normal((len(lengths), 2, 12, 16))
    o_s, f_s = oracle.prefill(q, k, v, g, beta, cu, init=init, scale=0.25)
    o_c, f_c = chunked.prefill(q, k, v, g, beta, cu, C=C, init=init, scale=0.25)
    assert np.abs(o_c - o_s).max() <= 1e-10 * max(1.0, np.abs(o_s).max())
    assert np.linalg.norm(f_c - f_s) <= 1e-10 * np.linalg.norm(f_s)


def test_chunk_solve_is_the_inverse():
    q, k, v, g, beta, _ = rand_tokens(22, [64], 1, 32, 32)
    qn, kn = chunked.l2normalise(q[:, 0]), chunked.l2normalise(k[:, 0])
    cq = chunked.chunk_quantities(qn, kn, v[:, 0], g[:, 0], beta[:, 0])
    A = cq["A_kk"]
    assert np.all(np.triu(A) == 0)  # strictly lower
    want = np.linalg.inv(np.eye(64) + A)  # Gaussian elimination
    np.testing.assert_allclose(cq["T"], want, rtol=0, atol=1e-12)
    # brute force of one entry of the gated Gram matrix
    i, j = 40, 17
    brute = beta[i, 0] * sum(kn[i, c] * kn[j, c] * np.exp(np.sum(g[j + 1:i + 1, 0, c]))
                             for c in range(32))
    assert abs(A[i, j] - brute) < 1e-13


def test_varlen_batch_equals_separate_runs():
    lengths = [5, 0, 70, 33]
    q, k, v, g, beta, cu = rand_tokens(23, lengths, 2, 8, 8)
    init = np.random.default_rng(24).standard_normal((4, 2, 8, 8))
    out, final = oracle.prefill(q, k, v, g, beta, cu, init=init)
    for b in range(4):
        t0, t1 = cu[b], cu[b + 1]
        o_b, f_b = oracle.prefill(q[t0:t1], k[t0:t1], v[t0:t1], g[t0:t1], beta[t0:t1],
                                  [0, t1 - t0], init=init[b:b + 1])
        np.testing.assert_array_equal(out[t0:t1], o_b)
        np.testing.assert_array_equal(final[b], f_b[0])
    np.testing.assert_array_equal(final[1], init[1])  # empty sequence keeps its state


def test_empty_batch_and_zero_init():
    q, k, v, g, beta, _ = rand_tokens(25, [0, 0], 1, 4, 4)
    out, final = oracle.prefill(q, k, v, g, beta, [0, 0, 0])
    assert out.shape == (0, 1, 4) and np.all(final == 0)


def test_prefill_equals_decode_steps():
    R_len, H, K, V = 9, 2, 8, 6
    q, k, v, g, beta, cu = rand_tokens(26, [R_len], H, K, V)
    init = np.random.default_rng(27).standard_normal((1, H, V, K)).astype(np.float32)
    out_p, final_p = oracle.prefill(q, k, v, g, beta, cu, init=init.astype(np.float64), scale=0.5)
    N, stride = 3, H * V * K + 5
    cache = np.zeros(N * stride, dtype=np.float32)
    cache.reshape(N, stride)[1, :H * V * K] = init.reshape(-1)
    for t in range(R_len):
        o = oracle.decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], cache, N,
                          stride, [1], scale=0.5)
        np.testing.assert_allclose(o[0], out_p[t], rtol=1e-5, atol=1e-6)
    got = cache.reshape(N, stride)[1, :H * V * K].reshape(H, V, K)
    np.testing.assert_allclose(got, final_p[0], rtol=1e-5, atol=1e-6)


def test_decode_invalid_index_uses_zero_state_and_writes_nothing():
    H, K, V = 2, 4, 4
    q, k, v, g, beta, _ = rand_tokens(28, [3], H, K, V)
    N, stride = 2, H * V * K
    cache = np.full(N * stride, 0xA5A5, dtype=np.uint16)
    before = cache.copy()
    out = oracle.decode(q, k, v, g, beta, cache, N, stride, [-1, N, 5], scale=1.0)
    assert np.array_equal(cache, before)
    qn, kn = chunked.l2normalise(q), chunked.l2normalise(k)
    want = beta[:, :, None] * np.sum(qn * kn, axis=-1)[:, :, None] * v  # S0 = 0
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-13)


def test_decode_bf16_writeback_rounds_to_nearest_even():
    H, K, V = 1, 8, 8
    q, k, v, g, beta, _ = rand_tokens(29, [1], H, K, V)
    rng = np.random.default_rng(30)
    S0 = torch.from_numpy(rng.standard_normal((V, K)).astype(np.float32)).to(torch.bfloat16)
    cache = S0.view(torch.int16).numpy().view(np.uint16).reshape(-1).copy()
    init = S0.to(torch.float64).numpy()[None, None]
    _, fin = oracle.prefill(q, k, v, g, beta, [0, 1], init=init)
    oracle.decode(q, k, v, g, beta, cache, 1, V * K, [0])
    want = oracle.f32_to_bf16_bits(fin[0, 0].astype(np.float32)).reshape(-1)
    assert np.array_equal(cache, want)


def test_value_columns_are_independent():
    K, V, T = 6, 5, 20
    q, k, v, g, beta, cu = rand_tokens(31, [T], 1, K, V)
    init = np.random.default_rng(32).standard_normal((1, 1, V, K))
    out, final = oracle.prefill(q, k, v, g, beta, cu, init=init)
    v2, init2 = v.copy(), init.copy()
    v2[:, :, 3] += 5.0
    init2[:, :, 3, :] -= 2.0
    out2, final2 = oracle.prefill(q, k, v2, g, beta, cu, init=init2)
    keep = [0, 1, 2, 4]
    np.testing.assert_array_equal(out2[:, :, keep], out[:, :, keep])
    np.testing.assert_array_equal(final2[:, :, keep], final[:, :, keep])
    assert np.abs(out2[:, :, 3] - out[:, :, 3]).max() > 1e-3


def test_l2norm_ignores_positive_scaling_of_q_and_k():
    q, k, v, g, beta, cu = rand_tokens(33, [17], 2, 8, 8)
    o1, f1 = oracle.prefill(q, k, v, g, beta, cu)
    o2, f2 = oracle.prefill(q * 3.0, k * 0.5, v, g, beta, cu)
    np.testing.assert_allclose(o2, o1, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(f2, f1, rtol=1e-5, atol=1e-6)


# --------------------------------------------------------------------------
# Chunk-boundary checkpoints
# --------------------------------------------------------------------------

def test_checkpoints_are_prefix_final_states():
    """Slot first_b + m - 1 holds sequence b's state after its first m * every tokens,
    i.e. the final state of a run over just those tokens from the same initial state;
    recording checkpoints changes neither the outputs nor the final states."""
    lengths, every = [130, 0, 64, 63, 200], 64
    q, k, v, g, beta, cu = rand_tokens(40, lengths, 2, 6, 5)
    init = np.random.default_rng(41).standard_normal((5, 2, 5, 6))
    out, final, ck = oracle.prefill_ckpt(q, k, v, g, beta, cu, every, init=init, scale=0.7)
    assert ck.shape == (sum(n // every for n in lengths), 2, 5, 6)
    slot = 0
    for b, n in enumerate(lengths):
        for m in range(1, n // every + 1):
            t0, t1 = cu[b], cu[b] + m * every
            _, f = oracle.prefill(q[t0:t1], k[t0:t1], v[t0:t1], g[t0:t1], beta[t0:t1], [0, t1 - t0],
                                  init=init[b:b + 1], scale=0.7)
            np.testing.assert_array_equal(ck[slot], f[0])
            slot += 1
    o2, f2 = oracle.prefill(q, k, v, g, beta, cu, init=init, scale=0.7)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(final, f2)
    np.testing.assert_array_equal(ck[2], final[2])  # length 64 = every: its only checkpoint is its final state


def test_checkpoint_interval_longer_than_every_sequence_records_nothing():
    q, k, v, g, beta, cu = rand_tokens(42, [10, 127], 1, 4, 4)
    _, _, ck = oracle.prefill_ckpt(q, k, v, g, beta, cu, 128)
    assert ck.shape[0] == 0


# --------------------------------------------------------------------------
# INT8 checkpoints
# --------------------------------------------------------------------------

def _golden_int8():
    vals = {}
    for line in open(os.path.join(GOLDEN, "int8_ckpt_small.txt")):
        if line.startswith("#") or ":" not in line:
            continue
        key, rest = line.split(":", 1)
        vals[key.strip()] = [float(x) for x in rest.split()]
    return vals


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_int8_checkpoint_golden(dtype):
    gv = _golden_int8()
    V, K = int(gv["V"][0]), int(gv["K"][0])
    x = np.array(gv["state_v_major"], dtype=np.float32)
    stride = V * K + 3  # a gap after the row
    N = 2
    act = np.full(N * stride, 99.0, dtype=np.float32)
    act[stride:stride + V * K] = x  # row 1
    if dtype == "bf16":
        act = oracle.f32_to_bf16_bits(act)
    q = np.full((3, 1, V, K), 55, dtype=np.int8)
    sc = np.full((3, 1, K), -1.0, dtype=np.float32)
    oracle.ckpt_store_int8(act, N, stride, 1, V, K, [1, -1, 0], [2, 0, 7], q, sc)
    np.testing.assert_array_equal(q[2].reshape(-1), np.array(gv["codes_v_major"], dtype=np.int8))
    np.testing.assert_array_equal(sc[2].reshape(-1), np.array(gv["scale"], dtype=np.float32))
    assert np.all(q[:2] == 55) and np.all(sc[:2] == -1.0)  # invalid src (-1) and dst (7) pairs: skipped
    back = np.full(N * stride, 99.0, dtype=np.float32)
    if dtype == "bf16":
        back = oracle.f32_to_bf16_bits(back)
    oracle.ckpt_load_int8(q, sc, [2, 9], [0, 1], back, N, stride, 1, V, K)
    row0 = back[:V * K]
    if dtype == "bf16":
        row0 = (row0.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(row0, np.array(gv["back_v_major"], dtype=np.float32))
    rest = back[V * K:]
    want = np.full(rest.shape, 99.0, dtype=np.float32)
    if dtype == "bf16":
        want = oracle.f32_to_bf16_bits(want)
    np.testing.assert_array_equal(rest, want)  # gap, row 1 (invalid slot 9): untouched


def test_int8_checkpoint_error_bound_and_extremes():
    """|back - x| <= scale / 2 element-wise (plus fp32 rounding of the product); the
    column's max-abs element maps to +-127; negating the state negates the codes."""
    rng = np.random.default_rng(50)
    H, V, K = 2, 16, 8
    x = (rng.standard_normal((3, H, V, K)) * rng.uniform(0.01, 10, (3, H, 1, K))).astype(np.float32)
    act = x.reshape(-1).copy()
    stride = H * V * K
    q = np.zeros((3, H, V, K), dtype=np.int8)
    sc = np.zeros((3, H, K), dtype=np.float32)
    oracle.ckpt_store_int8(act, 3, stride, H, V, K, [0, 1, 2], [0, 1, 2], q, sc)
    amax = np.abs(x).max(axis=2)
    np.testing.assert_allclose(sc, amax / 127, rtol=1e-6)
    at_max = np.abs(x) == amax[:, :, None, :]
    assert np.all(np.abs(q[at_max]) == 127)
    back = np.zeros_like(act)
    oracle.ckpt_load_int8(q, sc, [0, 1, 2], [0, 1, 2], back, 3, stride, H, V, K)
    err = np.abs(back.reshape(x.shape) - x)
    assert np.all(err <= sc[:, :, None, :] * (0.5 + 1e-5) + 1e-30)
    qn = np.zeros_like(q)
    scn = np.zeros_like(sc)
    oracle.ckpt_store_int8((-x).reshape(-1).copy(), 3, stride, H, V, K, [0, 1, 2], [0, 1, 2], qn, scn)
    np.testing.assert_array_equal(qn, -q)
    np.testing.assert_array_equal(scn, sc)


def test_int8_checkpoint_power_of_two_scaling_keeps_codes():
    """Scaling a state by 2^m is exact in fp32: the scales scale by 2^m, the codes stay."""
    rng = np.random.default_rng(51)
    H, V, K = 1, 8, 4
    x = rng.standard_normal((1, H, V, K)).astype(np.float32)
    q1, s1 = np.zeros((1, H, V, K), np.int8), np.zeros((1, H, K), np.float32)
    q2, s2 = np.zeros_like(q1), np.zeros_like(s1)
    oracle.ckpt_store_int8(x.reshape(-1).copy(), 1, V * K, H, V, K, [0], [0], q1, s1)
    oracle.ckpt_store_int8((x * 8).reshape(-1).copy(), 1, V * K, H, V, K, [0], [0], q2, s2)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s2, s1 * 8)


def test_int8_checkpoint_subnormal_scales_are_zero():
    """A column whose amax / 127 falls below the smallest normal float (every value under
    127 * 2^-126 in magnitude) gets scale 0 and codes 0, whether that scale would be 0 or a
    subnormal; a column just above keeps the ordinary rule (its max maps to +-127)."""
    H, V, K = 1, 4, 4
    tiny = np.float32(np.finfo(np.float32).tiny)  # 2^-126
    x = np.zeros((1, H, V, K), dtype=np.float32)
    x[0, 0, :, 0] = [1e-45, -3e-45, 0.0, 2e-45]           # subnormal inputs: amax / 127 -> 0
    x[0, 0, :, 1] = [100 * tiny, -50 * tiny, 0.0, 1e-40]  # amax / 127 subnormal
    x[0, 0, :, 2] = [127 * tiny * 2, -tiny, 0.0, 3 * tiny]  # amax / 127 = 2^-125: normal
    x[0, 0, :, 3] = [0.5, -1.0, 0.25, 0.0]
    q = np.full((1, H, V, K), 9, dtype=np.int8)
    sc = np.full((1, H, K), -1.0, dtype=np.float32)
    oracle.ckpt_store_int8(x.reshape(-1).copy(), 1, V * K, H, V, K, [0], [0], q, sc)
    assert sc[0, 0, 0] == 0.0 and sc[0, 0, 1] == 0.0
    assert np.all(q[0, 0, :, :2] == 0)
    assert sc[0, 0, 2] == np.float32(2 * tiny)  # 254 * 2^-126 / 127 = 2^-125 exactly
    assert list(q[0, 0, :, 2]) == [127, 0, 0, 2]  # -0.5 -> 0 and 1.5 -> 2: ties to even
    s3 = np.float32(1.0) / np.float32(127.0)      # correctly rounded, as numpy's float32 division
    assert sc[0, 0, 3] == s3
    want = np.rint(x[0, 0, :, 3] / s3).astype(np.int8)  # numpy: IEEE float32 quotient, half-even rint
    assert list(q[0, 0, :, 3]) == list(want) and want[1] == -127
    back = np.full(V * K, 7.0, dtype=np.float32)
    oracle.ckpt_load_int8(q, sc, [0], [0], back, 1, V * K, H, V, K)
    assert np.all(back.reshape(V, K)[:, :2] == 0.0)


# --------------------------------------------------------------------------
# Short causal convolution
# --------------------------------------------------------------------------

def test_conv1d_single_channel_is_numpy_convolve():
    """Zero state, no bias, identity: channel c of y is the first T terms of the full
    convolution of x with the reversed kernel (numpy's textbook routine)."""
    rng = np.random.default_rng(60)
    T, C, W = 37, 3, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    y, _ = oracle.conv1d_varlen(x, [0, T], w)
    for c in range(C):
        np.testing.assert_allclose(y[:, c], np.convolve(x[:, c], w[c, ::-1])[:T], rtol=1e-12, atol=1e-12)


def test_conv1d_impulse_response_and_bias():
    T, C, W = 10, 2, 3
    w = np.array([[1.0, 2.0, 3.0], [-1.0, 0.5, 4.0]])
    x = np.zeros((T, C))
    x[4] = 1.0
    y, final = oracle.conv1d_varlen(x, [0, T], w, bias=np.array([0.25, -1.0]))
    want = np.tile(np.array([0.25, -1.0]), (T, 1))
    want[4] += w[:, 2]  # current-token tap first, then the older ones
    want[5] += w[:, 1]
    want[6] += w[:, 0]
    np.testing.assert_array_equal(y, want)
    np.testing.assert_array_equal(final[0], x[T - 2:])  # the last W-1 inputs, oldest first


def test_conv1d_split_sequence_continues_through_its_state():
    """Running a sequence in two parts, the first part's final state as the second's
    initial state, gives the outputs and final state of one run (the state is exactly
    the window the convolution needs)."""
    rng = np.random.default_rng(61)
    T, C, W = 23, 5, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    b = rng.standard_normal(C)
    init = rng.standard_normal((1, W - 1, C))
    y, f = oracle.conv1d_varlen(x, [0, T], w, bias=b, activation="silu", init=init)
    for cut in (0, 1, 2, 9, T):
        y1, f1 = oracle.conv1d_varlen(x[:cut], [0, cut], w, bias=b, activation="silu", init=init)
        y2, f2 = oracle.conv1d_varlen(x[cut:], [0, T - cut], w, bias=b, activation="silu", init=f1)
        np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-14, atol=1e-14)
        np.testing.assert_array_equal(f2, f)


def test_conv1d_short_and_empty_sequences_keep_older_state_rows():
    W, C = 4, 2
    init = np.arange(2 * 3 * C, dtype=np.float64).reshape(2, 3, C)
    x = np.array([[100.0, 200.0]])
    _, f = oracle.conv1d_varlen(x, [0, 1, 1], np.ones((C, W)), init=init)
    np.testing.assert_array_equal(f[0], np.concatenate([init[0, 1:], x]))  # one token shifts in
    np.testing.assert_array_equal(f[1], init[1])                          # empty: unchanged


def test_conv1d_silu_closed_form():
    x = np.array([[0.0], [1.0], [-2.0], [30.0]])
    y, _ = oracle.conv1d_varlen(x, [0, 4], np.array([[0.0, 1.0]]), activation="silu")
    want = x[:, 0] / (1.0 + np.exp(-x[:, 0]))
    np.testing.assert_allclose(y[:, 0], want, rtol=1e-15)
    assert y[0, 0] == 0.0 and abs(y[3, 0] - 30.0) < 1e-11


def test_conv1d_update_equals_one_token_prefill():
    rng = np.random.default_rng(62)
    R, C, W = 3, 6, 4
    w = rng.standard_normal((C, W))
    b = rng.standard_normal(C)
    x = rng.standard_normal((R, C)).astype(np.float32).astype(np.float64)
    N, stride = 4, (W - 1) * C + 2
    cache = np.zeros(N * stride, dtype=np.float32)
    st = rng.standard_normal((N, W - 1, C)).astype(np.float32)
    for r in range(N):
        cache[r * stride:r * stride + (W - 1) * C] = st[r].reshape(-1)
    idx = [2, -1, 0]
    before = cache.copy()
    y = oracle.conv1d_update(x, w, cache, N, stride, idx, bias=b, activation="silu")
    init = np.stack([st[2], np.zeros((W - 1, C)), st[0]]).astype(np.float64)
    y_ref, f_ref = oracle.conv1d_varlen(x, [0, 1, 2, 3], w, bias=b, activation="silu", init=init)
    np.testing.assert_allclose(y, y_ref, rtol=1e-14, atol=1e-14)
    for r, row in ((0, 2), (2, 0)):
        got = cache[row * stride:row * stride + (W - 1) * C].reshape(W - 1, C)
        np.testing.assert_array_equal(got, f_ref[r].astype(np.float32))
    for row in (1, 3):  # rows not addressed (and the invalid index) are untouched
        np.testing.assert_array_equal(cache[row * stride:(row + 1) * stride], before[row * stride:(row + 1) * stride])
    np.testing.assert_array_equal(cache[(W - 1) * C:stride], before[(W - 1) * C:stride])  # gap


# --------------------------------------------------------------------------
# Speculative target verification
# --------------------------------------------------------------------------

def test_target_verify_is_prefill_with_per_token_states():
    """Verifying L tokens equals prefilling them from the cached state: the same outputs,
    intermediate state t = the checkpoint after t + 1 tokens; the cache is left as it was."""
    rng = np.random.default_rng(70)
    R, L, H, K, V = 3, 5, 2, 6, 4
    q, k, v, g, beta, _ = rand_tokens(71, [R * L], H, K, V)
    N, stride = 4, H * V * K + 3
    cache = rng.standard_normal(N * stride).astype(np.float32)
    before = cache.copy()
    idx = [2, -1, 0]
    P, pstride = 20, H * V * K
    pool = np.full(P * pstride, 7.0, dtype=np.float32)
    inter = np.arange(R * L).reshape(R, L)
    inter[1, 2] = -1      # an invalid slot: not written
    inter[2, 4] = P + 3
    sh = lambda a: a.reshape(R, L, *a.shape[1:])  # noqa: E731
    out = oracle.target_verify(sh(q), sh(k), sh(v), sh(g), sh(beta), cache, N, stride, idx, pool, P, pstride,
                               inter, scale=0.5)
    np.testing.assert_array_equal(cache, before)
    init = np.zeros((R, H, V, K))
    for r, row in enumerate(idx):
        if row >= 0:
            init[r] = cache[row * stride:row * stride + H * V * K].reshape(H, V, K)
    cu = np.arange(0, R * L + 1, L)
    o_ref, _, ck = oracle.prefill_ckpt(q, k, v, g, beta, cu, 1, init=init, scale=0.5)
    np.testing.assert_allclose(out.reshape(R * L, H, V), o_ref, rtol=1e-12, atol=1e-12)
    for r in range(R):
        for t in range(L):
            s = inter[r, t]
            if 0 <= s < P:
                got = pool[s * pstride:(s + 1) * pstride].reshape(H, V, K)
                np.testing.assert_array_equal(got, ck[r * L + t].astype(np.float32))
    np.testing.assert_array_equal(pool[7 * pstride:8 * pstride], np.full(pstride, 7.0, np.float32))  # slot of (1, 2)
