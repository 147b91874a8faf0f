"""Pins for the fp64 CPU oracle: each test checks the oracle against something
other than itself, so that a dropped term, a wrong sign or index, a swapped
forget/predict order or a transposed operand fails at least one of them.

Sources ("page" = the web page, cited by title and section):
  * "Kimi Delta Attention (KDA)" (brain.bigb.es): the delta-rule read-back
    identity, the beta = 1 exact read, the locality of the rank-one write (DeltaNet
    section); the order forget -> predict (Gated DeltaNet section); the DPLR
    transition A_t = D_t (I - beta_t k_t k_t^T) (KDA section); the chunkwise
    schedule with preliminary errors, rho_ij, (I + R_c)^-1, K^end and chi_ij,
    which must give the same states and outputs as the recurrence ("Two
    schedules" section).
  * "K3 架构图解" Ch.08: the worked example 1 + (3 - 1) = 3 (tests/golden).
  * "22580: от GPT-2 до Kimi K3", chunked DeltaNet section: the UT-transform
    forward (T = (I + strict_lower(diag(beta) K K^T))^-1, W = T K_beta,
    U = T V_beta, per-chunk u = U - W S, o = q S + tril(q k^T) u, S += k^T u),
    which is the alpha = 1 case; and the remark that alpha = 0 clears memory
    (Gated DeltaNet section).
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x, axis=-1):
    return x / np.linalg.norm(x, axis=axis, keepdims=True)


def _rand_inputs(rng, T, H, dk, dv, unit_k=True, gate_scale=0.3):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k = _unit(k)
    v = rng.standard_normal((T, H, dv))
    g = -np.log1p(np.exp(rng.standard_normal((T, H, dk)))) * gate_scale
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


def _run(q, k, v, g, beta, S0=None, scale=None, threads=None):
    T, H, _ = q.shape
    cu = np.array([0, T], dtype=np.int64)
    init = None if S0 is None else S0[None]
    out, fin = oracle.kda_fwd(q, k, v, g, beta, cu, init_state=init, scale=scale,
                              threads=threads)
    return out, fin[0]


# --------------------------------------------------------------------------
# Worked example, "K3 架构图解" Ch.08
# --------------------------------------------------------------------------
def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split()
            vals[key] = float(val)
    return vals


def test_worked_example_ch08():
    gv = _read_golden("worked_example_ch08.txt")
    one = lambda x: np.array([[[x]]], dtype=np.float64)  # [T=1, H=1, d=1]
    out, fin = oracle.kda_fwd(one(gv["q"]), one(gv["k"]), one(gv["v"]), one(gv["g"]),
                              np.array([[gv["beta"]]]), np.array([0, 1]),
                              init_state=np.array([[[[gv["state0"]]]]]),
                              scale=gv["scale"])
    assert fin[0, 0, 0, 0] == gv["expected_state"]
    assert out[0, 0, 0] == gv["expected_out"]


# --------------------------------------------------------------------------
# Invariants stated on "Kimi Delta Attention (KDA)"
# --------------------------------------------------------------------------
def test_full_write_reads_back_value_exactly():
    """alpha = 1, beta = 1, unit key: the read with the same key returns v_t."""
    rng = _rng(1)
    T, H, dk, dv = 24, 2, 8, 5
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    g[:] = 0.0
    beta[:] = 1.0
    S0 = rng.standard_normal((H, dk, dv))
    out, _ = _run(k, k, v, g, beta, S0=S0, scale=1.0)  # read with q = k
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)


def _prefix_states(q, k, v, g, beta, S0):
    """State after each prefix [0, t), from the oracle itself (t = 0..T)."""
    T = q.shape[0]
    states = [S0.copy()]
    for t in range(1, T + 1):
        _, fin = _run(q[:t], k[:t], v[:t], g[:t], beta[:t], S0=S0)
        states.append(fin)
    return states


def test_read_back_interpolates():
    """S_t^T k_t = (1 - beta_t) S~_t^T k_t + beta_t v_t for a unit key, where
    S~_t = Diag(alpha_t) S_{t-1} is the state after the forget step."""
    rng = _rng(2)
    T, H, dk, dv = 10, 2, 6, 4
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((H, dk, dv))
    out, _ = _run(k, k, v, g, beta, S0=S0, scale=1.0)
    states = _prefix_states(k, k, v, g, beta, S0)
    for t in range(T):
        for h in range(H):
            S_tilde = np.exp(g[t, h])[:, None] * states[t][h]
            want = (1 - beta[t, h]) * (S_tilde.T @ k[t, h]) + beta[t, h] * v[t, h]
            np.testing.assert_allclose(out[t, h], want, rtol=0, atol=1e-12)


def test_write_is_local_to_the_key_direction():
    """(S_t - S~_t)^T x = 0 for every x orthogonal to k_t, and the write is
    rank one along k_t."""
    rng = _rng(3)
    T, H, dk, dv = 8, 1, 7, 3
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv, unit_k=False)
    S0 = rng.standard_normal((H, dk, dv))
    states = _prefix_states(q, k, v, g, beta, S0)
    for t in range(T):
        kt = k[t, 0]
        delta = states[t + 1][0] - np.exp(g[t, 0])[:, None] * states[t][0]
        for _ in range(4):
            x = rng.standard_normal(dk)
            x -= kt * (kt @ x) / (kt @ kt)
            assert np.abs(delta.T @ x).max() < 1e-12
        assert np.linalg.matrix_rank(delta, tol=1e-10) == 1


def test_zero_write_strength_decays_only():
    """beta = 0: S_T = Diag(prod_t alpha_t) S_0 and o_t reads the decayed S_0;
    with alpha = 1 as well the state is unchanged."""
    rng = _rng(4)
    T, H, dk, dv = 16, 3, 5, 6
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    beta[:] = 0.0
    S0 = rng.standard_normal((H, dk, dv))
    s = 0.37
    out, fin = _run(q, k, v, g, beta, S0=S0, scale=s)
    G = np.cumsum(g, axis=0)  # [T, H, dk]
    for h in range(H):
        np.testing.assert_allclose(fin[h], np.exp(G[-1, h])[:, None] * S0[h],
                                   rtol=1e-12, atol=1e-13)
        for t in range(T):
            want = s * (np.exp(G[t, h])[:, None] * S0[h]).T @ q[t, h]
            np.testing.assert_allclose(out[t, h], want, rtol=1e-11, atol=1e-12)
    g[:] = 0.0
    _, fin = _run(q, k, v, g, beta, S0=S0)
    assert np.array_equal(fin, S0)


def test_zero_retention_clears_memory():
    """alpha_t = 0 (g = -inf) wipes the state before the write, so
    S_t = beta_t k_t v_t^T and o_t = s beta_t (k_t . q_t) v_t."""
    rng = _rng(5)
    T, H, dk, dv = 6, 2, 4, 3
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv, unit_k=False)
    S0 = rng.standard_normal((H, dk, dv))
    g[T - 1] = -np.inf
    out, fin = _run(q, k, v, g, beta, S0=S0, scale=0.5)
    for h in range(H):
        kt, vt, bt, qt = k[-1, h], v[-1, h], beta[-1, h], q[-1, h]
        np.testing.assert_allclose(fin[h], bt * np.outer(kt, vt), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(out[-1, h], 0.5 * bt * (kt @ qt) * vt, rtol=1e-12, atol=1e-14)


def test_forget_comes_before_predict():
    """The error is taken against the decayed state: with a unit key, alpha
    scaling the key channels and beta = 1 the read must still return v_t exactly
    (predict-before-forget would leave (1 - alpha) S k in the read)."""
    rng = _rng(6)
    T, H, dk, dv = 12, 1, 4, 4
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    beta[:] = 1.0
    g[:] = -0.7
    S0 = rng.standard_normal((H, dk, dv)) * 3
    out, _ = _run(k, k, v, g, beta, S0=S0, scale=1.0)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Exact rational brute force over the DPLR transition product
# --------------------------------------------------------------------------
def _fmat(rows, cols, f=Fraction(0)):
    return [[f for _ in range(cols)] for _ in range(rows)]


def _fmul(A, B):
    return [[sum((A[i][p] * B[p][j] for p in range(len(B))), Fraction(0))
             for j in range(len(B[0]))] for i in range(len(A))]


def _fadd(A, B):
    return [[A[i][j] + B[i][j] for j in range(len(A[0]))] for i in range(len(A))]


def _fscale(A, c):
    return [[a * c for a in row] for row in A]


def _eye(n):
    return [[Fraction(int(i == j)) for j in range(n)] for i in range(n)]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_dplr_products_exact(seed):
    """S_t = M_t S_{t-1} + beta_t k_t v_t^T with M_t = (I - beta_t k_t k_t^T) D_t
    (the transpose of the DPLR A_t of the KDA section, for the d_k x d_v layout),
    unrolled as explicit products in exact rational arithmetic:
      S_t = (M_t ... M_1) S_0 + sum_u (M_t ... M_{u+1}) beta_u k_u v_u^T,
      o_t = s S_t^T q_t.
    d_k = 4 (so s = 1/2 exactly) and d_v = 3 (a transposed operand cannot pass)."""
    rng = _rng(100 + seed)
    T, dk, dv = 5, 4, 3
    alphas_pool = [Fraction(1), Fraction(1, 2), Fraction(3, 4), Fraction(2, 3), Fraction(7, 8)]
    small = lambda: Fraction(int(rng.integers(-4, 5)), int(rng.integers(1, 4)))
    q = [[small() for _ in range(dk)] for _ in range(T)]
    k = [[small() for _ in range(dk)] for _ in range(T)]
    v = [[small() for _ in range(dv)] for _ in range(T)]
    a = [[alphas_pool[int(rng.integers(0, 5))] for _ in range(dk)] for _ in range(T)]
    b = [Fraction(int(rng.integers(0, 5)), 4) for _ in range(T)]
    S0 = [[small() for _ in range(dv)] for _ in range(dk)]
    s = Fraction(1, 2)

    M = []
    for t in range(T):
        kk = [[k[t][i] * k[t][j] for j in range(dk)] for i in range(dk)]
        D = [[a[t][i] if i == j else Fraction(0) for j in range(dk)] for i in range(dk)]
        M.append(_fmul(_fadd(_eye(dk), _fscale(kk, -b[t])), D))

    def prod(lo, hi):  # M_hi ... M_{lo}  (1-based inclusive, empty -> I)
        P = _eye(dk)
        for t in range(lo, hi + 1):
            P = _fmul(M[t - 1], P)
        return P

    want_out, want_S = [], None
    for t in range(1, T + 1):
        St = _fmul(prod(1, t), S0)
        for u in range(1, t + 1):
            write = [[b[u - 1] * k[u - 1][i] * v[u - 1][j] for j in range(dv)] for i in range(dk)]
            St = _fadd(St, _fmul(prod(u + 1, t), write))
        want_out.append([s * sum((St[i][j] * q[t - 1][i] for i in range(dk)), Fraction(0))
                         for j in range(dv)])
        want_S = St

    f = lambda X: np.array([[float(x) for x in row] for row in X], dtype=np.float64)
    g = np.log(f(a))
    out, fin = oracle.kda_fwd(f(q)[:, None], f(k)[:, None], f(v)[:, None], g[:, None],
                              f([b]).T, np.array([0, T]), init_state=f(S0)[None, None],
                              scale=0.5)
    np.testing.assert_allclose(out[:, 0], f(want_out), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin[0, 0], f(want_S), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# An independent schedule: the chunkwise algebra of the "Two schedules"
# section, restated here in fp64 (exact pairwise decays, a library solve).
# --------------------------------------------------------------------------
def _chunkwise(q, k, v, g, beta, S0, C, scale):
    """One head, one sequence.  For a chunk with incoming state S (d_k x d_v):
      G_i     = sum of g over chunk rows 0..i (decay from the chunk start through i)
      ebar_i  = beta_i (v_i - S^T (exp(G_i) * k_i))        preliminary errors
      rho_ij  = beta_i k_j^T D_{j+1:i} k_i,  j < i,  D_{j+1:i} = exp(G_i - G_j)
      E       = (I + R)^-1 Ebar                            (rows are errors)
      o_i     = s (S^T (exp(G_i) * q_i) + sum_{j<=i} (k_j^T D_{j+1:i} q_i) e_j)
      S_next  = Diag(exp(G_last)) S + sum_i (exp(G_last - G_i) * k_i) e_i^T
    """
    T, dk = q.shape
    S = S0.copy()
    out = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        Q, K, V, Gt, B = q[sl], k[sl], v[sl], np.cumsum(g[sl], axis=0), beta[sl]
        n = Q.shape[0]
        Ebar = B[:, None] * (V - (np.exp(Gt) * K) @ S)
        R = np.zeros((n, n))
        X = np.zeros((n, n))
        for i in range(n):
            for j in range(i + 1):
                dec = np.exp(Gt[i] - Gt[j])
                if j < i:
                    R[i, j] = B[i] * np.sum(K[j] * dec * K[i])
                X[i, j] = np.sum(K[j] * dec * Q[i])
        E = np.linalg.solve(np.eye(n) + R, Ebar)
        out[sl] = scale * ((np.exp(Gt) * Q) @ S + X @ E)
        S = np.exp(Gt[-1])[:, None] * S + (np.exp(Gt[-1] - Gt) * K).T @ E
    return out, S


@pytest.mark.parametrize("C", [1, 16, 64])
def test_chunkwise_schedule_matches_recurrence(C):
    """Same states and outputs from both schedules (agreement ~1e-9 or better)."""
    rng = _rng(7)
    T, dk, dv = 150, 16, 12  # ragged last chunk for C = 16 and 64
    q, k, v, g, beta = _rand_inputs(rng, T, 1, dk, dv, gate_scale=0.2)
    S0 = rng.standard_normal((1, dk, dv)) * 0.5
    out, fin = _run(q, k, v, g, beta, S0=S0)
    co, cS = _chunkwise(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0], C, dk ** -0.5)
    np.testing.assert_allclose(out[:, 0], co, rtol=0, atol=1e-10)
    np.testing.assert_allclose(fin[0], cS, rtol=0, atol=1e-10)


def _deltanet_ut(q, k, v, beta, C):
    """alpha = 1 (DeltaNet) chunk form with the UT transform, per the chunked
    DeltaNet section: T = (I + strict_lower(diag(beta) K K^T))^-1 built by forward
    substitution, W = T (beta K), U = T (beta V); per chunk u = U - W S,
    o = q S + tril(q k^T) u, S += k^T u.  No output scale on that page."""
    L, d = q.shape
    S = np.zeros((d, v.shape[1]))
    out = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        sl = slice(c0, c0 + C)
        Q, K, V, B = q[sl], k[sl], v[sl], beta[sl]
        A = np.tril((B[:, None] * K) @ K.T, -1)
        Tm = np.eye(C)
        for i in range(C):  # row i of (I + A)^-1 = e_i - sum_{j<i} A_ij row_j
            Tm[i] = np.eye(C)[i] - A[i, :i] @ Tm[:i]
        W, U = Tm @ (B[:, None] * K), Tm @ (B[:, None] * V)
        u = U - W @ S
        out[sl] = Q @ S + np.tril(Q @ K.T) @ u
        S = S + K.T @ u
    return out, S


def test_chunkwise_reduces_to_deltanet_ut_form():
    rng = _rng(8)
    T, d = 128, 8
    q, k, v, g, beta = _rand_inputs(rng, T, 1, d, d)
    g[:] = 0.0
    zero = np.zeros((d, d))
    co, cS = _chunkwise(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], zero, 32, 1.0)
    do, dS = _deltanet_ut(q[:, 0], k[:, 0], v[:, 0], beta[:, 0], 32)
    np.testing.assert_allclose(co, do, rtol=0, atol=1e-11)
    np.testing.assert_allclose(cS, dS, rtol=0, atol=1e-11)
    out, fin = _run(q, k, v, g, beta, S0=zero[None], scale=1.0)
    np.testing.assert_allclose(out[:, 0], do, rtol=0, atol=1e-10)
    np.testing.assert_allclose(fin[0], dS, rtol=0, atol=1e-10)


# --------------------------------------------------------------------------
# Checkpoint semantics, packing, threads
# --------------------------------------------------------------------------
def test_split_prefill_resumes_from_state():
    rng = _rng(9)
    T1, T2, H, dk, dv = 37, 50, 2, 8, 8
    q, k, v, g, beta = _rand_inputs(rng, T1 + T2, H, dk, dv)
    S0 = rng.standard_normal((H, dk, dv))
    out, fin = _run(q, k, v, g, beta, S0=S0)
    o1, s1 = _run(q[:T1], k[:T1], v[:T1], g[:T1], beta[:T1], S0=S0)
    o2, s2 = _run(q[T1:], k[T1:], v[T1:], g[T1:], beta[T1:], S0=s1)
    np.testing.assert_array_equal(np.concatenate([o1, o2]), out)
    np.testing.assert_array_equal(s2, fin)


def test_packed_varlen_equals_separate_runs_and_is_head_equivariant():
    rng = _rng(10)
    lens = [5, 0, 64, 17, 1]
    H, dk, dv = 3, 8, 4
    T = sum(lens)
    q, k, v, g, beta = _rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    out, fin = oracle.kda_fwd(q, k, v, g, beta, cu, init_state=S0, threads=3)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        o, s = oracle.kda_fwd(q[sl], k[sl], v[sl], g[sl], beta[sl], np.array([0, lens[n]]),
                              init_state=S0[n:n + 1])
        np.testing.assert_array_equal(out[sl], o)
        np.testing.assert_array_equal(fin[n], s[0])
    assert np.array_equal(fin[1], S0[1])  # empty sequence keeps its state
    perm = [2, 0, 1]
    po, pf = oracle.kda_fwd(q[:, perm], k[:, perm], v[:, perm], g[:, perm], beta[:, perm], cu,
                            init_state=S0[:, perm])
    np.testing.assert_array_equal(po, out[:, perm])
    np.testing.assert_array_equal(pf, fin[:, perm])


def test_result_independent_of_thread_count():
    rng = _rng(11)
    q, k, v, g, beta = _rand_inputs(rng, 40, 8, 8, 8)
    cu = np.array([0, 10, 40])
    a = oracle.kda_fwd(q, k, v, g, beta, cu, threads=1)
    b = oracle.kda_fwd(q, k, v, g, beta, cu, threads=7)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_decode_steps_match_one_sequence_run():
    rng = _rng(12)
    steps, N, H, d = 9, 3, 2, 6
    q, k, v, g, beta = (x.reshape((steps, N) + x.shape[1:]) if x.ndim == 3 else x.reshape(steps, N, H)
                        for x in _rand_inputs(rng, steps * N, H, d, d))
    S0 = rng.standard_normal((N, H, d, d))
    out, fin = oracle.kda_decode_steps(q, k, v, g, beta, S0)
    for n in range(N):
        o, s = _run(q[:, n], k[:, n], v[:, n], g[:, n], beta[:, n], S0=S0[n])
        np.testing.assert_array_equal(out[:, n], o)
        np.testing.assert_array_equal(fin[n], s)
