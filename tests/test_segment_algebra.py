"""The two-segment form of the recurrence, restated in fp64 numpy and checked
against the oracle's per-token loop (CPU only; no CUDA code involved).

Variational Linear Attention, §3.2-3.4. The sequence is cut at token L. The
two halves can run side by side because the state at the cut is reachable
without running the first half:

* A. M_t = lambda0 I + sum_{s<=t} u^_s u^_s^T is a prefix sum (§3.2) and
  A_t = M_t^-1 (eq. 9 is Sherman-Morrison on it). So A at the cut is the
  inverse of the first half's prefix sum added to A_0^-1. z^key at the cut is
  z^key_0 + sum_{s<L} phi(k_s).
* S. Eq. 12 (read with the transposed state, S_t^T = F_t S_{t-1}^T + alpha^_t
  v_t^T, F_t = I - alpha^_t k^_t^T) composes associatively. Written on S:
  S_t = S_{t-1} P_t + v_t alpha^_t^T with P_t = I - k^_t alpha^_t^T, so
  S_t = S_L Pi_t + G_t, where Pi_t = P_{L+1} ... P_t and G_t is the second
  half's recurrence from S = 0. Pi_t is that recurrence from S = I with
  v = 0, and its readout Pi_t phi_t / den_t gives
  o_t = o_t(from S = 0) + S_L (Pi_t phi_t / den_t).
  The gates alpha^_t of the second half depend on A only, so both second-half
  runs see the same gates.

These identities are exact, so the restatement must match the oracle to
fp64 rounding at any cut. Each planted mistake (the cut state's A from the
wrong prefix, a dropped or transposed transition, the key sum not carried)
must move the result well past that rounding.
"""
import numpy as np
import pytest

import oracle
from test_chunk_algebra import _inputs, _rel, phi, unit_rows


def segmented(orc, q, k, v, u, lambda0, eps, cut, S0=None, A0=None, zk0=None, mistake=None):
    """One head [T, d] run as two segments [0, cut) and [cut, T); each segment
    is a per-token oracle run. Returns o, S, A, zk."""
    T, d = q.shape
    one = lambda x: None if x is None else x[None]
    # first half: the plain recurrence from the given state
    o1, G0, _, _ = orc.forward_f64(q[None, :cut], k[None, :cut], v[None, :cut], u[None, :cut], lambda0, eps,
                                   one(S0), one(A0), one(zk0))
    # the state at the cut that the second half needs, without the first half's run
    Uh = unit_rows(u[:cut])
    M0 = np.eye(d) * lambda0 if A0 is None else np.linalg.inv(A0)
    pre = Uh[:-1] if mistake == "prefix_short" else Uh
    A_cut = np.linalg.inv(M0 + pre.T @ pre)
    zk_cut = (np.zeros(d) if zk0 is None else zk0) + (0.0 if mistake == "zk_not_carried" else 1.0) * np.sum(
        phi(k[:cut]), axis=0)
    # second half from S = 0, and the transition from S = I with v = 0
    sl = slice(cut, T)
    o2, G1, A_T, zk_T = orc.forward_f64(q[None, sl], k[None, sl], v[None, sl], u[None, sl], lambda0, eps,
                                        np.zeros((1, d, d)), A_cut[None], zk_cut[None])
    of, F1, _, _ = orc.forward_f64(q[None, sl], k[None, sl], np.zeros((1, T - cut, d)), u[None, sl], lambda0, eps,
                                   np.eye(d)[None], A_cut[None], zk_cut[None])
    S_L = G0[0]
    if mistake == "transition_transposed":
        F1 = np.swapaxes(F1, -1, -2)
    if mistake == "no_transition":
        F1 = np.zeros_like(F1)
        of = np.zeros_like(of)
    o = np.concatenate([o1[0], o2[0] + of[0] @ S_L.T], axis=0)
    S = S_L @ F1[0] + G1[0]
    return o, S, A_T[0], zk_T[0]


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("cut", [1, 16, 29, 52])
@pytest.mark.parametrize("state", [False, True])
def test_two_segments_match_the_per_token_loop(orc, cut, state):
    BH, T, d = 2, 53, 24
    (q, k, v, u), (S0, A0, zk0) = _inputs(41 + cut, BH, T, d, state)
    o_r, S_r, A_r, zk_r = orc.forward_f64(q, k, v, u, 0.1, 1e-4, S0, A0, zk0)
    for h in range(BH):
        st = (None, None, None) if not state else (S0[h], A0[h], zk0[h])
        o, S, A, zk = segmented(orc, q[h], k[h], v[h], u[h], 0.1, 1e-4, cut, *st)
        for name, x, ref in (("o", o, o_r[h]), ("S", S, S_r[h]), ("A", A, A_r[h]), ("zk", zk, zk_r[h])):
            assert _rel(x, ref) < 1e-9, (name, h, cut, _rel(x, ref))


@pytest.mark.parametrize("mistake", ["prefix_short", "zk_not_carried", "transition_transposed", "no_transition"])
def test_planted_mistakes_are_caught(orc, mistake):
    T, d, cut = 53, 24, 29
    (q, k, v, u), _ = _inputs(77, 1, T, d)
    o_r, S_r, A_r, zk_r = orc.forward_f64(q, k, v, u, 0.1, 1e-4)
    o, S, A, zk = segmented(orc, q[0], k[0], v[0], u[0], 0.1, 1e-4, cut, mistake=mistake)
    worst = max(_rel(o, o_r[0]), _rel(S, S_r[0]), _rel(A, A_r[0]), _rel(zk, zk_r[0]))
    assert worst > 1e-3, (mistake, worst)
