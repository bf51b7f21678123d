"""The precision of a chunked reverse sweep, emulated on the CPU.

The chunked backward of `test_chunk_backward_algebra` is run here in fp32:
first the forward, then the reverse sweep. Every product that a tensor-core
kernel would form (products of d x d states or adjoints with d x C blocks,
rank-C updates, C x C Grams) goes through the same three emulations as in
`test_tf32_split`: split tf32 operands, plain tf32 operands, and exact fp32.
The comparison is with the fp64 oracle's backward, on one head of the
d_h = 96 workload (T = 4096), with dL/do drawn as the benchmark draws it.

* With split operands the worst per-token gradient error stays inside the
  2e-3 parity tolerance.
* With plain tf32 operands it does not.
"""
import numpy as np
import pytest

import oracle
from sherman_morrison_memory_gb300 import workloads as W
from test_tf32_split import TOL, eliminate, mm_f32, mm_plain, mm_split

f32 = np.float32


def unit_rows(x):
    """x / max(||x||, 1e-12) row by row, fp32."""
    return (x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), f32(1e-12))).astype(f32)
def phi(x):
    """ELU + 1, fp32."""
    return np.where(x > 0, x + f32(1), np.exp(np.minimum(x, f32(0)))).astype(f32)
def dphi(x):
    """Derivative of ELU + 1, fp32."""
    return np.where(x > 0, f32(1), np.exp(np.minimum(x, f32(0)))).astype(f32)
def unit_grad_rows(x, g):
    """Gradient through x^ = x / max(||x||, 1e-12), row by row, fp32."""
    n = np.linalg.norm(x, axis=-1, keepdims=True).astype(f32)
    xg = np.sum(x * g, axis=-1, keepdims=True).astype(f32)
    safe = np.maximum(n, f32(1e-12))
    return ((g - x / safe * (xg / safe)) / safe).astype(f32)

def chunked_backward_fp32(q, k, v, u, lambda0, eps, C, gO, gS, gA, gzk, mm):
    """The chunked forward, then the chunked reverse sweep, in fp32; `mm` forms
    the products a tensor-core kernel would."""
    T, d = q.shape
    q, k, v, u, gO = (x.astype(f32) for x in (q, k, v, u, gO))
    A = (np.eye(d) / lambda0).astype(f32); S = np.zeros((d, d), f32); zk = np.zeros(d, f32)
    chunks = []
    for c0 in range(0, T, C):
        n = min(C, T - c0); sl = slice(c0, c0 + n)
        Uh, Kh = unit_rows(u[sl]), unit_rows(k[sl])
        Zp, Wm = mm(A, Uh.T), mm(A, Kh.T)
        L, delta, X = eliminate(np.eye(n, dtype=f32) + mm(Uh, Zp), mm(Uh, Wm))
        Z = np.linalg.solve(L, Zp.T).T.astype(f32)
        Y = (Z / delta).astype(f32)
        N = (Z * (f32(1) / np.sqrt(delta.astype(f32)))).astype(f32)  # N = Z D^-1/2
        Ag = (Wm - Y @ np.triu(X)).astype(f32)
        an = np.linalg.norm(Ag, axis=0).astype(f32)
        al = (Ag / np.maximum(an, f32(1e-12))).astype(f32)
        Lk = mm(Kh, al)
        R = (v[sl].T - mm(S, Kh.T)).astype(f32)
        E = np.linalg.solve(np.eye(n, dtype=f32) + np.tril(Lk, -1), R.T).T.astype(f32)
        PQ, PK = phi(q[sl]), phi(k[sl])
        ZK = (zk + np.cumsum(PK, axis=0)).astype(f32)
        raw = np.sum(PQ * ZK, axis=1).astype(f32)
        den = np.maximum(raw, f32(eps))
        Lq = mm(PQ, al)
        O = ((mm(S, PQ.T) + E @ np.tril(Lq).T) / den).T.astype(f32)
        chunks.append(dict(sl=sl, n=n, S=S, A=A, Uh=Uh, Kh=Kh, Z=Z.T.copy(), delta=delta, a=Ag.T.copy(),
                           al=al.T.copy(), E=E.T.copy(), PQ=PQ, ZK=ZK, den=den, clamp=raw < eps, O=O))
        S = (S + mm(E, al.T)).astype(f32)
        A = (A - mm(N, N.T)).astype(f32)
        zk = ZK[-1]
    dq, dk, dv, du = (np.zeros((T, d), f32) for _ in range(4))
    HS, HA, gz = gS.astype(f32), gA.astype(f32), gzk.astype(f32)
    for ch in reversed(chunks):
        sl, n = ch["sl"], ch["n"]
        Kh, Uh, Z, dl, al, E = ch["Kh"], ch["Uh"], ch["Z"], ch["delta"], ch["al"], ch["E"]
        PQ, ZK, den, O, Sc, Ac = ch["PQ"], ch["ZK"], ch["den"], ch["O"], ch["S"], ch["A"]
        GO = gO[sl]; GOd = (GO / den[:, None]).astype(f32)
        Lk, Lq = mm(Kh, al.T), mm(PQ, al.T)
        RHS = (mm(HS, al.T).T + np.tril(Lq).T @ GOd).astype(f32)
        DV = np.empty((n, d), f32)
        for t in range(n - 1, -1, -1):
            DV[t] = RHS[t] - Lk[t + 1:, t] @ DV[t + 1:]
        GE, DE = mm(GO, E.T), mm(DV, E.T)
        g_al = mm(HS.T, E.T).T.copy()
        for t in range(n):
            g_al[t] += (GE[t:, t] / den[t:]) @ PQ[t:] - DE[t + 1:, t] @ Kh[t + 1:]
        EDV = mm(E, DV.T)
        g_kh = -mm(Sc.T, DV.T).T
        for t in range(n):
            g_kh[t] -= EDV[:t, t] @ al[:t]
        EGO = mm(E, GO.T)
        g_pq = mm(Sc.T, GO.T).T.copy()
        for t in range(n):
            g_pq[t] += EGO[:t + 1, t] @ al[:t + 1]
        g_pq = (g_pq / den[:, None]).astype(f32)
        g_den = np.where(ch["clamp"], f32(0), -np.sum(GO * O, axis=1) / den).astype(f32)
        g_pq = (g_pq + g_den[:, None] * ZK).astype(f32)
        g_pk = np.empty((n, d), f32)
        for t in range(n - 1, -1, -1):
            gz = (gz + g_den[t] * PQ[t]).astype(f32)
            g_pk[t] = gz
        HS_prev = (HS + mm(GOd.T, PQ) - mm(DV.T, Kh)).astype(f32)
        g_a = unit_grad_rows(ch["a"], g_al)
        HZ, HtZ = mm(HA, Z.T).T, mm(HA.T, Z.T).T
        GZ = np.zeros((n, d), f32); g_uh = np.zeros((n, d), f32)
        for t in range(n - 1, -1, -1):
            zt = Z[t]
            Gz = HZ[t] + (Kh[t:] @ zt) @ g_a[t:] + (Uh[t + 1:] @ zt) @ GZ[t + 1:]
            Gtz = HtZ[t] + (g_a[t:] @ zt) @ Kh[t:] + (GZ[t + 1:] @ zt) @ Uh[t + 1:]
            gdel = (zt @ Gz) / dl[t] ** 2
            GZ[t] = -(Gz + Gtz) / dl[t] + gdel * Uh[t]
            g_uh[t] = gdel * zt
        ZGZ = mm(Z, GZ.T)
        g_uh = (g_uh + mm(Ac, GZ.T).T).astype(f32)
        for t in range(n):
            g_uh[t] -= (ZGZ[:t, t] / dl[:t]) @ Z[:t]
        ZGA = mm(Z, g_a.T)
        g_kh = (g_kh + mm(Ac, g_a.T).T).astype(f32)
        for t in range(n):
            g_kh[t] -= (ZGA[:t + 1, t] / dl[:t + 1]) @ Z[:t + 1]
        HA_prev = (HA + mm(g_a.T, Kh) + mm(GZ.T, Uh)).astype(f32)
        dv[sl] = DV; du[sl] = unit_grad_rows(u[sl], g_uh)
        dk[sl] = unit_grad_rows(k[sl], g_kh) + g_pk * dphi(k[sl]); dq[sl] = g_pq * dphi(q[sl])
        HS, HA = HS_prev, HA_prev
    return dict(dq=dq, dk=dk, dv=dv, du=du, dS0=HS, dA0=HA, dzk0=gz)


@pytest.fixture(scope="module")
def errors():
    w = W.WORKLOADS[3]
    q, k, v, u = (x[0, 0] for x in W.make(w, B=1, H=1))
    gO = W.upstream_grad(w, B=1, H=1)[0, 0]
    d = q.shape[1]
    gS, gA, gzk = np.zeros((d, d)), np.zeros((d, d)), np.zeros(d)
    ref = oracle.load().backward(q, k, v, u, w.lambda0, w.eps, None, None, None, gO, gS, gA, gzk)
    out = {}
    for name, mm in (("split", mm_split), ("plain", mm_plain), ("f32", mm_f32)):
        g = chunked_backward_fp32(q, k, v, u, w.lambda0, w.eps, 16, gO, gS, gA, gzk, mm)
        err = {}
        for key in ("dq", "dk", "dv", "du"):
            r = ref[key]
            err[key] = float(np.max(np.linalg.norm(g[key] - r, axis=1) / np.maximum(np.linalg.norm(r, axis=1), 1e-30)))
        for key in ("dS0", "dA0"):
            err[key] = float(np.linalg.norm(g[key] - ref[key]) / np.linalg.norm(ref[key]))
        out[name] = err
    return out


def test_split_products_stay_inside_the_tolerance(errors):
    assert max(errors["split"].values()) < TOL / 3, errors["split"]


def test_plain_tf32_products_miss_the_tolerance(errors):
    assert max(errors["plain"].values()) > 5 * TOL, errors["plain"]
