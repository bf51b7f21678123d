"""The chunked form of the reverse sweep, restated in fp64 numpy and checked
against the oracle's per-token backward (CPU only; no CUDA code involved).

Variational Linear Attention, §3.3, eq. 9-11, differentiated; the oracle's
backward applies the adjoint of each per-token step in reverse order. Taken a
chunk of C tokens at a time, with the states S_c, A_c before the chunk (from
checkpoints) and the adjoints H_S = dL/dS, H_A = dL/dA after it:

* S adjoint. dv_t + sum_{s>t} (k^_s . alpha^_t) dv_s
  = H_S alpha^_t + sum_{s>=t} (phi_s . alpha^_t) gO_s / den_s. This is the
  forward's unit-triangular system transposed, with the same Gram matrices.
  g_alpha_t = H_S^T e_t + sum_{s>=t} phi_s (gO_s . e_t) / den_s
  - sum_{s>t} k^_s (dv_s . e_t). The adjoint before the chunk is
  H_S + sum_s gO_s phi_s^T / den_s - sum_s dv_s k^_s^T.
* A adjoint. g_z_t (the adjoint of z_t = A_{t-1} u^_t) follows a C-step
  recurrence on d-vectors. Its only d x d terms are H_A z_t and H_A^T z_t,
  and the rest are sums over s >= t of the chunk's own vectors. The u^ and k^
  gradients take A_c g_z and A_c g_a, then corrections over the chunk's z_s.
  The adjoint before the chunk is H_A + sum_s g_a_s k^_s^T + sum_s g_z_s u^_s^T.

So a chunk touches d x d matrices only through products with d x C blocks:
H_S alpha^, H_S^T E, S_c^T dV, S_c^T gO, H_A Z, H_A^T Z, A_c g_Z, A_c g_A,
and two rank-2C updates. Everything else is C x C Gram matrices,
triangular solves and a C-step recurrence per chunk. These identities are
exact, so the restatement must match the oracle to fp64 rounding for every
chunk size. Each planted mistake must move a gradient well past that.
"""
import numpy as np
import pytest

import oracle
from test_chunk_algebra import _inputs, eliminate, phi, unit_rows


def dphi(x):
    """Derivative of ELU + 1."""
    return np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))


def unit_grad_rows(x, g):
    """Gradient through x^ = x / max(||x||, 1e-12), row by row."""
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    xg = np.sum(x * g, axis=-1, keepdims=True)
    safe = np.maximum(n, 1e-12)
    out = (g - x / safe * (xg / safe)) / safe
    return np.where(n < 1e-12, g / 1e-12, out)


def forward_chunks(q, k, v, u, lambda0, eps, C, S0=None, A0=None, zk0=None):
    """Chunked forward keeping what the reverse sweep reads: the states at
    chunk starts and the per-token vectors."""
    T, d = q.shape
    A = np.eye(d) / lambda0 if A0 is None else A0.copy()
    S = np.zeros((d, d)) if S0 is None else S0.copy()
    zk = np.zeros(d) if zk0 is None else zk0.copy()
    chunks = []
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        sl = slice(c0, c0 + n)
        Uh, Kh = unit_rows(u[sl]), unit_rows(k[sl])
        Zp, W = A @ Uh.T, A @ Kh.T
        L, delta, X = eliminate(np.eye(n) + Uh @ Zp, Uh @ W)
        Z = np.linalg.solve(L, Zp.T).T
        Y = Z / delta
        N = Z / np.sqrt(delta)             # A_{c+1} = A_c - N N^T
        Ag = W - Y @ np.triu(X)
        an = np.linalg.norm(Ag, axis=0)
        al = Ag / np.maximum(an, 1e-12)
        Lk = Kh @ al
        R = v[sl].T - S @ Kh.T
        E = np.linalg.solve(np.eye(n) + np.tril(Lk, -1), R.T).T
        PQ, PK = phi(q[sl]), phi(k[sl])
        ZK = zk + np.cumsum(PK, axis=0)
        raw = np.sum(PQ * ZK, axis=1)
        den = np.maximum(raw, eps)
        Lq = PQ @ al
        O = ((S @ PQ.T + E @ np.tril(Lq).T) / den).T
        chunks.append(dict(sl=sl, n=n, S=S.copy(), A=A.copy(), Uh=Uh, Kh=Kh, Z=Z.T, delta=delta,
                           a=Ag.T, an=an, al=al.T, E=E.T, PQ=PQ, PK=PK, ZK=ZK, den=den,
                           clamp=raw < eps, O=O))
        S = S + E @ al.T
        A = A - N @ N.T
        zk = ZK[-1]
    return chunks, (S, A, zk)


def chunked_backward(q, k, v, u, lambda0, eps, C, gO, gS, gA, gzk, S0=None, A0=None, zk0=None, mistake=None):
    T, d = q.shape
    chunks, _ = forward_chunks(q, k, v, u, lambda0, eps, C, S0, A0, zk0)
    dq, dk, dv, du = (np.zeros((T, d)) for _ in range(4))
    HS = np.zeros((d, d)) if gS is None else gS.copy()   # dL/dS after the chunk
    HA = np.zeros((d, d)) if gA is None else gA.copy()   # dL/dA after the chunk
    gz = np.zeros(d) if gzk is None else gzk.copy()      # dL/dz^key after the chunk
    for ch in reversed(chunks):
        sl, n = ch["sl"], ch["n"]
        Kh, Uh, Z, dl, al, an, E = ch["Kh"], ch["Uh"], ch["Z"], ch["delta"], ch["al"], ch["an"], ch["E"]
        PQ, PK, ZK, den, O = ch["PQ"], ch["PK"], ch["ZK"], ch["den"], ch["O"]
        Sc, Ac = ch["S"], ch["A"]
        GO = gO[sl]
        GOd = GO / den[:, None]                            # gO_s / den_s
        # ---- S adjoint: dv_t + sum_{s>t} (k^_s . al_t) dv_s = HS al_t + sum_{s>=t} (phq_s . al_t) gO_s/den_s
        Lk = Kh @ al.T                                     # Lk[s][t] = k^_s . al_t
        Lq = PQ @ al.T                                     # Lq[s][t] = phq_s . al_t
        lq = np.tril(Lq, -1) if mistake == "rhs_strict" else np.tril(Lq)
        RHS = (HS @ al.T).T + lq.T @ GOd                   # row t: sum_{s>=t} Lq[s][t] gOd_s
        DV = np.empty((n, d))
        for t in range(n - 1, -1, -1):
            DV[t] = RHS[t] - Lk[t + 1:, t] @ DV[t + 1:]
        # g_alpha_t = G_t^T e_t
        GE = GO @ E.T                                      # GE[s][t] = gO_s . e_t
        DE = DV @ E.T                                      # DE[s][t] = dv_s . e_t
        g_al = (HS.T @ E.T).T
        for t in range(n):
            g_al[t] += (GE[t:, t] / den[t:]) @ PQ[t:] - DE[t + 1:, t] @ Kh[t + 1:]
        # g_k^ from e: -(S_c^T dv_t + sum_{s<t} al_s (e_s . dv_t))
        EDV = E @ DV.T                                     # EDV[s][t] = e_s . dv_t
        g_kh = -(Sc.T @ DV.T).T
        for t in range(n):
            g_kh[t] -= EDV[:t, t] @ al[:t]
        # g_phq = (S_c^T gO_t + sum_{s<=t} al_s (e_s . gO_t)) / den_t, plus g_den zk_t
        EGO = E @ GO.T
        g_pq = (Sc.T @ GO.T).T
        for t in range(n):
            g_pq[t] += EGO[:t + 1, t] @ al[:t + 1]
        g_pq /= den[:, None]
        g_den = np.where(ch["clamp"], 0.0, -np.sum(GO * O, axis=1) / den)
        g_pq += g_den[:, None] * ZK
        # z^key: g_phk_t = gzk_after + sum_{s>=t} g_den_s phq_s
        g_pk = np.empty((n, d))
        for t in range(n - 1, -1, -1):
            gz = gz + g_den[t] * PQ[t]
            g_pk[t] = gz
        HS_prev = HS + GOd.T @ PQ - DV.T @ Kh
        # ---- A adjoint
        a = ch["a"]
        g_a = unit_grad_rows(a, g_al)
        HZ, HtZ = (HA @ Z.T).T, (HA.T @ Z.T).T              # H_A z_t, H_A^T z_t
        GZ = np.zeros((n, d))
        g_uh = np.zeros((n, d))
        for t in range(n - 1, -1, -1):
            zt = Z[t]
            Gz = HZ[t] + (Kh[t:] @ zt) @ g_a[t:] + (Uh[t + 1:] @ zt) @ GZ[t + 1:]
            Gtz = HtZ[t] + (g_a[t:] @ zt) @ Kh[t:] + (GZ[t + 1:] @ zt) @ Uh[t + 1:]
            if mistake == "no_transpose_term":
                Gtz = Gz
            gdel = (zt @ Gz) / dl[t] ** 2
            GZ[t] = -(Gz + Gtz) / dl[t] + (0.0 if mistake == "no_gdelta" else gdel) * Uh[t]
            g_uh[t] = gdel * zt
        # g_u^ += A_{t-1} g_z_t = A_c g_z_t - sum_{s<t} z_s (z_s . g_z_t) / delta_s
        ZGZ = Z @ GZ.T
        g_uh += (Ac @ GZ.T).T
        for t in range(n):
            m = t + 1 if mistake == "a_after" else t
            g_uh[t] -= (ZGZ[:m, t] / dl[:m]) @ Z[:m]
        # g_k^ += A_t g_a_t = A_c g_a_t - sum_{s<=t} z_s (z_s . g_a_t) / delta_s
        ZGA = Z @ g_a.T
        g_kh += (Ac @ g_a.T).T
        for t in range(n):
            g_kh[t] -= (ZGA[:t + 1, t] / dl[:t + 1]) @ Z[:t + 1]
        HA_prev = HA + g_a.T @ Kh + GZ.T @ Uh
        # ---- inputs
        dv[sl] = DV
        du[sl] = unit_grad_rows(u[sl], g_uh)
        dk[sl] = unit_grad_rows(k[sl], g_kh) + g_pk * dphi(k[sl])
        dq[sl] = g_pq * dphi(q[sl])
        HS, HA = HS_prev, HA_prev
    return dict(dq=dq, dk=dk, dv=dv, du=du, dS0=HS, dA0=HA, dzk0=gz)


def _seeds(BH, T, d, seed=9):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((BH, T, d)), rng.standard_normal((BH, d, d)) * 0.1,
            rng.standard_normal((BH, d, d)) * 0.1, rng.standard_normal((BH, d)) * 0.1)


def _worst(out, ref, h):
    return {key: float(np.linalg.norm(out[key] - ref[key][h]) / max(np.linalg.norm(ref[key][h]), 1e-300))
            for key in ("dq", "dk", "dv", "du", "dS0", "dA0", "dzk0")}


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("chunk", [1, 7, 16])
@pytest.mark.parametrize("state", [False, True])
def test_chunked_reverse_sweep_matches_oracle(orc, chunk, state):
    BH, T, d = 2, 16 * 3 + 5, 24  # several chunks and a ragged tail
    (q, k, v, u), (S0, A0, zk0) = _inputs(3, BH, T, d, state)
    gO, gS, gA, gzk = _seeds(BH, T, d)
    ref = orc.backward(q, k, v, u, 0.1, 1e-4, S0, A0, zk0, gO, gS, gA, gzk)
    for h in range(BH):
        st = (None, None, None) if not state else (S0[h], A0[h], zk0[h])
        out = chunked_backward(q[h], k[h], v[h], u[h], 0.1, 1e-4, chunk, gO[h], gS[h], gA[h], gzk[h], *st)
        worst = _worst(out, ref, h)
        assert max(worst.values()) < 1e-10, worst


@pytest.mark.parametrize("mistake", ["rhs_strict", "no_transpose_term", "no_gdelta", "a_after"])
def test_planted_mistakes_are_caught(orc, mistake):
    BH, T, d = 1, 16 * 2 + 3, 24
    (q, k, v, u), _ = _inputs(3, BH, T, d)
    gO, gS, gA, gzk = _seeds(BH, T, d)
    ref = orc.backward(q, k, v, u, 0.1, 1e-4, None, None, None, gO, gS, gA, gzk)
    out = chunked_backward(q[0], k[0], v[0], u[0], 0.1, 1e-4, 16, gO[0], gS[0], gA[0], gzk[0], mistake=mistake)
    worst = _worst(out, ref, 0)
    assert max(worst.values()) > 1e-3, (mistake, worst)
