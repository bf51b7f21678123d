"""The chunked form of the recurrence, restated in fp64 numpy and checked
against the oracle's per-token loop (CPU only; no CUDA code involved).

Variational Linear Attention, §3.3, eq. 9-11, taken C tokens at a time from
the state A_c, S_c before the chunk (U^, K^ the unit rows u^_t, k^_t):

* eq. 9 over the chunk: with Z' = A_c U^T and Guu = U^ Z', the pivots of the
  LDL^T factorisation of I + Guu are the delta_t, and Z = Z' L^-T holds the
  Sherman-Morrison vectors z_t = A_{t-1} u^_t; the chunk's rank-C downdate
  is A_{c+1} = A_c - Z' (I + Guu)^-1 Z'^T (Woodbury) = A_c - N N^T with
  N = Z D^-1/2, the sum of the tokens' z_t z_t^T / delta_t.
  Gaussian elimination of [I + Guu | Guk] gives L, the pivots and
  X = L^-1 Guk together (Guk = U^ A_c K^T).
* the gate of eq. 10: a_t = A_t k^_t = w_t - sum_{q<=t} (z_q / delta_q) X[q][t]
  with w_t = A_c k^_t.
* eq. 10-11 over the chunk: the residual writes are a unit lower-triangular
  solve e_t = v_t - S_c k^_t - sum_{s<t} (k^_t . alpha^_s) e_s, the readout is
  o_t = (S_c phi_t + sum_{s<=t} e_s (alpha^_s . phi_t)) / den_t, and
  S_{c+1} = S_c + E alpha^T.

These identities are exact, so the restatement must agree with the oracle to
fp64 rounding for every chunk size; C = 1 is the per-token loop itself. The
planted mistakes at the end (a strict triangle where the sum includes its
diagonal and the reverse, a dropped 1/delta, the wrong triangle of the Gram
matrices, D^-1 in place of D^-1/2 in the update) must each move the result
well past that rounding.
"""
import numpy as np
import pytest

import oracle


def unit_rows(x):
    return x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), 1e-12)


def phi(x):
    # ELU + 1 (§3.3, eq. 11)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def eliminate(M, G):
    """Gaussian elimination of the augmented [M | G] without pivoting, M
    symmetric positive definite: returns the unit lower L and the pivots of
    M = L diag(delta) L^T, and L^-1 G (what the G columns end as)."""
    n = M.shape[0]
    aug = np.concatenate([M, G], axis=1).astype(np.float64)
    L = np.eye(n)
    for t in range(n):
        for r in range(t + 1, n):
            L[r, t] = aug[r, t] / aug[t, t]
            aug[r, t:] -= L[r, t] * aug[t, t:]
    return L, np.diag(aug[:, :n]).copy(), aug[:, n:]


def chunked_forward(q, k, v, u, lambda0, eps, chunk, S0=None, A0=None, zk0=None, mistake=None):
    """One head [T, d] in chunks of `chunk` tokens; returns o, S, A, zk."""
    T, d = q.shape
    A = np.eye(d) / lambda0 if A0 is None else A0.copy()
    S = np.zeros((d, d)) if S0 is None else S0.copy()
    zk = np.zeros(d) if zk0 is None else zk0.copy()
    o = np.empty((T, d))
    for c0 in range(0, T, chunk):
        n = min(chunk, T - c0)
        sl = slice(c0, c0 + n)
        Uh, Kh = unit_rows(u[sl]), unit_rows(k[sl])
        # eq. 9 for the whole chunk
        Zp = A @ Uh.T                      # z'_t = A_c u^_t (columns)
        W = A @ Kh.T                       # w_t = A_c k^_t
        Guu, Guk = Uh @ Zp, Uh @ W
        if mistake == "gram_triangle":
            Guu = np.triu(Guu) + np.triu(Guu, 1).T * 0.5
        L, delta, X = eliminate(np.eye(n) + Guu, Guk)
        Z = np.linalg.solve(L, Zp.T).T     # Z = Z' L^-T
        Y = Z if mistake == "no_rdelta" else Z / delta
        N = Z / (delta if mistake == "update_rdelta" else np.sqrt(delta))  # N = Z D^-1/2
        A_next = A - N @ N.T
        # the gate of eq. 10: a_t = w_t - sum_{q<=t} (z_q / delta_q) X[q][t]
        tri = np.triu(X, 1) if mistake == "gate_strict" else np.triu(X)
        Ag = W - Y @ tri
        alpha = Ag / np.maximum(np.linalg.norm(Ag, axis=0), 1e-12)
        # eq. 10-11 for the whole chunk
        Lk = Kh @ alpha                    # Lk[t][s] = k^_t . alpha^_s
        R = v[sl].T - S @ Kh.T             # v_t - S_c k^_t
        Ls = np.tril(Lk) if mistake == "solve_diag" else np.tril(Lk, -1)
        E = np.linalg.solve(np.eye(n) + Ls, R.T).T
        Pq = phi(q[sl])
        zks = zk + np.cumsum(phi(k[sl]), axis=0)
        den = np.maximum(np.sum(Pq * zks, axis=1), eps)
        Lq = Pq @ alpha                    # Lq[t][s] = phi_t . alpha^_s
        o[sl] = ((S @ Pq.T + E @ np.tril(Lq).T) / den).T
        S = S + E @ alpha.T
        A = A_next
        zk = zks[-1]
    return o, S, A, zk


def _inputs(seed, BH, T, d, state=False):
    rng = np.random.default_rng(seed)
    q, k, v, u = (rng.standard_normal((BH, T, d)) for _ in range(4))
    if not state:
        return (q, k, v, u), (None, None, None)
    S0 = rng.standard_normal((BH, d, d)) * 0.3
    # a carried A: the inverse of lambda0 I plus some unit outer products,
    # symmetric positive definite as every A_t of eq. 9 is
    A0 = np.empty((BH, d, d))
    for h in range(BH):
        P = unit_rows(rng.standard_normal((3 * d, d)))
        A0[h] = np.linalg.inv(0.1 * np.eye(d) + P.T @ P)
    zk0 = np.abs(rng.standard_normal((BH, d))) * 5.0
    return (q, k, v, u), (S0, A0, zk0)


def _rel(x, ref):
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("chunk", [1, 7, 16])
@pytest.mark.parametrize("state", [False, True])
def test_chunked_form_matches_per_token_loop(orc, chunk, state):
    BH, T, d = 3, 16 * 3 + 5, 24  # several chunks and a ragged tail
    (q, k, v, u), (S0, A0, zk0) = _inputs(11 + chunk, BH, T, d, state)
    o_r, S_r, A_r, zk_r = orc.forward_f64(q, k, v, u, 0.1, 1e-4, S0, A0, zk0)
    for h in range(BH):
        st = (None, None, None) if not state else (S0[h], A0[h], zk0[h])
        o, S, A, zk = chunked_forward(q[h], k[h], v[h], u[h], 0.1, 1e-4, chunk, *st)
        for name, x, ref in (("o", o, o_r[h]), ("S", S, S_r[h]), ("A", A, A_r[h]), ("zk", zk, zk_r[h])):
            assert _rel(x, ref) < 1e-10, (name, h, _rel(x, ref))


@pytest.mark.parametrize("case", ["u_zero", "one_partial_chunk"])
def test_degenerate_cases(orc, case):
    """u = 0 (the unit guard gives u^ = 0: delta_t = 1, A never moves, the
    fixed-A variant) and a sequence shorter than one chunk."""
    BH, T, d = 2, (40 if case == "u_zero" else 5), 24
    (q, k, v, u), _ = _inputs(31, BH, T, d)
    if case == "u_zero":
        u = np.zeros_like(u)
    o_r, S_r, A_r, zk_r = orc.forward_f64(q, k, v, u, 0.1, 1e-4)
    for h in range(BH):
        o, S, A, zk = chunked_forward(q[h], k[h], v[h], u[h], 0.1, 1e-4, 16)
        for name, x, ref in (("o", o, o_r[h]), ("S", S, S_r[h]), ("A", A, A_r[h]), ("zk", zk, zk_r[h])):
            assert _rel(x, ref) < 1e-10, (case, name, h, _rel(x, ref))
    if case == "u_zero":
        assert np.array_equal(A_r[0], np.eye(d) / 0.1)


def test_ldl_pivots_are_the_sherman_morrison_denominators(orc):
    """The pivots of I + U^ A_c U^T are the delta_t = 1 + u^_t . A_{t-1} u^_t
    of eq. 9 that the per-token loop forms one at a time."""
    T, d = 16, 24
    (q, k, v, u), _ = _inputs(5, 1, T, d)
    ref = orc.forward(q, k, v, u, 0.1, 1e-4, trace=True)
    Uh = unit_rows(u[0])
    A0 = np.eye(d) / 0.1
    _, delta, _ = eliminate(np.eye(T) + Uh @ A0 @ Uh.T, np.zeros((T, 1)))
    # the oracle widens fp32 copies of the inputs; compare on those
    Uh32 = unit_rows(u[0].astype(np.float32).astype(np.float64))
    _, delta32, _ = eliminate(np.eye(T) + Uh32 @ A0 @ Uh32.T, np.zeros((T, 1)))
    assert np.allclose(delta32, ref.delta[0], rtol=1e-12, atol=0)
    assert np.allclose(delta, delta32, rtol=1e-5)


def test_symmetric_update_is_the_woodbury_downdate():
    """N N^T with N = Z' L^-T D^-1/2 is Z' (I + U^ A U^^T)^-1 Z'^T, the rank-C
    Woodbury downdate, and also the product of the chunk's C Sherman-Morrison
    steps of eq. 9 taken one token at a time."""
    rng = np.random.default_rng(31)
    d, n = 24, 16
    B = rng.standard_normal((d, d))
    A = B @ B.T / d + np.eye(d)                      # symmetric positive definite
    Uh = unit_rows(rng.standard_normal((n, d)))
    Zp = A @ Uh.T
    L, delta, _ = eliminate(np.eye(n) + Uh @ Zp, np.zeros((n, 1)))
    N = np.linalg.solve(L, Zp.T).T / np.sqrt(delta)
    woodbury = Zp @ np.linalg.solve(np.eye(n) + Uh @ Zp, Zp.T)
    assert np.max(np.abs(N @ N.T - woodbury)) < 1e-12 * np.max(np.abs(woodbury))
    As = A.copy()
    for t in range(n):                               # eq. 9, token by token
        z = As @ Uh[t]
        As = As - np.outer(z, z) / (1.0 + Uh[t] @ z)
    assert np.max(np.abs((A - N @ N.T) - As)) < 1e-12 * np.max(np.abs(A))


@pytest.mark.parametrize("mistake", ["gate_strict", "solve_diag", "no_rdelta", "gram_triangle", "update_rdelta"])
def test_planted_mistakes_are_caught(orc, mistake):
    BH, T, d = 1, 16 * 2 + 3, 24
    (q, k, v, u), _ = _inputs(23, BH, T, d)
    o_r, S_r, A_r, _ = orc.forward_f64(q, k, v, u, 0.1, 1e-4)
    o, S, A, _ = chunked_forward(q[0], k[0], v[0], u[0], 0.1, 1e-4, 16, mistake=mistake)
    worst = max(_rel(o, o_r[0]), _rel(S, S_r[0]), _rel(A, A_r[0]))
    assert worst > 1e-3, (mistake, worst)
