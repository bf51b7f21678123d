"""The precision argument of the tensor-core path, emulated on the CPU.

tcgen05 `kind::tf32` reads each fp32 operand with its low 13 mantissa bits
dropped. The chunked kernels therefore split every fp32 operand x into
hi = trunc(x) and lo = trunc(x - hi), and form each tensor-core product as
hi*hi + hi*lo + lo*hi. The state, the scalar steps and the sums stay in fp32
otherwise. Here the chunked recurrence of Variational Linear Attention
(§3.3, eq. 9-11; the same algebra as `test_chunk_algebra`) runs in fp32 with
every product the kernels put on the tensor cores emulated three ways: split,
plain tf32 operands, and exact fp32. Each is compared with the fp64 oracle on
one head of the d_h = 96 workload, all 4096 tokens.

* The split stays well inside the 2e-3 parity tolerance, within a few times
  the error of exact fp32 products.
* Plain tf32 operands miss the tolerance. That is why the split is there.

The rank-C update of A is the symmetric N N^T (N = Z D^-1/2), as in the
kernels. With the earlier form M Z'^T (M = Z D^-1 L^-1) the rounding left an
antisymmetric part in A that the downdates never damp while A shrinks, so
the error grew with T: on this head the split's worst o error was about
8e-5 and plain tf32's above 1e-2; with N N^T they are 2e-6 and 2.9e-3.
"""
import numpy as np
import pytest

import oracle
from sherman_morrison_memory_gb300 import workloads as W

f32 = np.float32
TOL = 2e-3  # normwise relative error per token (o) and per head (S, A)


def trunc_tf32(x):
    """fp32 -> the value a tf32 operand read keeps (low 13 mantissa bits cleared)."""
    b = np.ascontiguousarray(x, dtype=f32).view(np.uint32) & np.uint32(0xFFFFE000)
    return b.view(f32)


def mm_split(X, Y):
    X, Y = X.astype(f32), Y.astype(f32)
    xh, yh = trunc_tf32(X), trunc_tf32(Y)
    xl, yl = trunc_tf32(X - xh), trunc_tf32(Y - yh)
    return (xh @ yh + xh @ yl + xl @ yh).astype(f32)


def mm_plain(X, Y):
    return (trunc_tf32(X) @ trunc_tf32(Y)).astype(f32)


def mm_f32(X, Y):
    return (X.astype(f32) @ Y.astype(f32)).astype(f32)


def unit_rows(x):
    return (x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), f32(1e-12))).astype(f32)


def phi(x):
    return np.where(x > 0, x + f32(1), np.exp(np.minimum(x, f32(0)))).astype(f32)


def eliminate(M, G):
    """fp32 Gaussian elimination of [M | G]: unit lower L, pivots, L^-1 G."""
    n = M.shape[0]
    aug = np.concatenate([M, G], axis=1).astype(f32)
    L = np.eye(n, dtype=f32)
    for t in range(n):
        r = f32(1) / aug[t, t]
        for rr in range(t + 1, n):
            L[rr, t] = aug[rr, t] * r
            aug[rr, t:] -= L[rr, t] * aug[t, t:]
    return L, np.diag(aug[:, :n]).copy(), aug[:, n:]


def chunked_fp32(q, k, v, u, lambda0, eps, mm, C=16):
    """One head in fp32, chunks of C tokens; `mm` forms the products that the
    kernels put on the tensor cores."""
    T, d = q.shape
    A = (np.eye(d) / lambda0).astype(f32)
    S = np.zeros((d, d), f32)
    zk = np.zeros(d, f32)
    o = np.empty((T, d), f32)
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        sl = slice(c0, c0 + n)
        Uh, Kh = unit_rows(u[sl]), unit_rows(k[sl])
        Zp, Wm = mm(A, Uh.T), mm(A, Kh.T)                 # [A u | A k]
        Guu, Guk = mm(Uh, Zp), mm(Uh, Wm)                 # Gram matrices
        L, delta, X = eliminate(np.eye(n, dtype=f32) + Guu, Guk)
        Z = np.linalg.solve(L, Zp.T).T.astype(f32)
        Y = (Z / delta).astype(f32)
        N = (Z * (f32(1) / np.sqrt(delta.astype(f32)))).astype(f32)  # N = Z D^-1/2
        A_next = (A - mm(N, N.T)).astype(f32)            # rank-C update of A: A - N N^T
        Ag = (Wm - Y @ np.triu(X)).astype(f32)            # the gate a_t (fp32 FMA)
        nr = np.maximum(np.linalg.norm(Ag, axis=0), f32(1e-12)).astype(f32)
        Lk = (mm(Kh, Ag) / nr).astype(f32)
        R = (v[sl].T - mm(S, Kh.T)).astype(f32)           # v - S_c k^
        E = np.linalg.solve(np.eye(n, dtype=f32) + np.tril(Lk, -1), R.T).T.astype(f32)
        Pq = phi(q[sl])
        zks = (zk + np.cumsum(phi(k[sl]), axis=0)).astype(f32)
        den = np.maximum(np.sum(Pq * zks, axis=1), f32(eps)).astype(f32)
        Lq = (mm(Pq, Ag) / nr).astype(f32)
        o[sl] = ((mm(S, Pq.T) + E @ np.tril(Lq).T) / den).T
        S = (S + mm((E / nr).astype(f32), Ag.T)).astype(f32)  # rank-C update of S
        A = A_next
        zk = zks[-1]
    return o, S, A


@pytest.fixture(scope="module")
def errors():
    w = W.WORKLOADS[3]
    q, k, v, u = (x[0, 0] for x in W.make(w, B=1, H=1))
    o_r, S_r, A_r, _ = oracle.load().forward_f64(q, k, v, u, w.lambda0, w.eps)
    out = {}
    for name, mm in (("split", mm_split), ("plain", mm_plain), ("f32", mm_f32)):
        o, S, A = chunked_fp32(q, k, v, u, w.lambda0, w.eps, mm)
        out[name] = (
            float(np.max(np.linalg.norm(o - o_r, axis=1) / np.linalg.norm(o_r, axis=1))),
            float(np.linalg.norm(S - S_r) / np.linalg.norm(S_r)),
            float(np.linalg.norm(A - A_r) / np.linalg.norm(A_r)),
        )
    return out


def test_split_products_stay_inside_the_tolerance(errors):
    assert max(errors["split"]) < TOL / 5, errors["split"]
    # within a few times exact fp32 products
    assert max(errors["split"]) < 10 * max(errors["f32"]), errors


def test_plain_tf32_products_miss_the_tolerance(errors):
    assert max(errors["plain"]) > TOL, errors["plain"]
    assert max(errors["plain"]) > 100 * max(errors["split"]), errors
