"""Pins for the fp64 oracle: checks against what the paper and the mathematics
fix, independent of the oracle's own code.

Every pin is a function ``pin_xxx(orc)`` taking an ``oracle.Oracle`` and raising
AssertionError when the oracle disagrees. ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle
with planted mistakes and asserts that each mistake is caught.

Sources (Pandey & Singh, "Variational Linear Attention", arXiv 2605.11196):
  §3.2       A_0 = lambda0^{-1} I, unit penalty directions u_s, A_t = M_t^{-1}
  §3.3 (9)   Sherman-Morrison update of A; delta_t >= 1
  §3.3 (10)  residual write with unit gate alpha^_t = A_t k^_t / ||A_t k^_t||
  §3.3 (11)  ELU+1 readout with key-sum normaliser and eps floor
  §3.4 (12)  S recurrence as an associative scan over (F, G) pairs
  §3.5       u_t = 0 with A fixed at lambda0^{-1} I (the fixed-A ablation)
  §4.1 (13)  Proposition 1: ||S_t||_F <= ||S_0||_F + sum_s ||e_s||
  §4.2 (14)  Proposition 2: Jacobian I - alpha^ k^^T (spectrum; see below)
  §4.2       Corollary 1: the gradient through the recurrence (backward pass)
"""
from __future__ import annotations

import numpy as np

LAMBDA0 = 0.1
EPS = 1e-4


def _phi(x):
    # ELU(x) + 1 (§3.3 eq. 11): x + 1 for x > 0, exp(x) otherwise
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _unit_rows(x):
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, 1e-12)


def _inputs(rng, T, d, lead=(1,)):
    shape = tuple(lead) + (T, d)
    return tuple(rng.standard_normal(shape).astype(np.float32) for _ in range(4))


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------------------
# A-pass: eq. 9 against the direct inverse of the penalty M_t
# ---------------------------------------------------------------------------

def pin_inverse_penalty(orc):
    """A_T equals (lambda0 I + sum_{s<=T} u^_s u^_s^T)^{-1} (§3.2, §3.3 eq. 9).

    The Sherman-Morrison recursion is exact, so the oracle's A must equal the
    inverse that numpy computes directly from the unit penalty directions.
    """
    rng = np.random.default_rng(11)
    for d in (1, 3, 8):
        for lam in (LAMBDA0, 0.37):
            q, k, v, u = _inputs(rng, 40, d)
            uh = _unit_rows(u[0])
            for Tp in (1, 2, 17, 40):
                r = orc.forward(q[:, :Tp], k[:, :Tp], v[:, :Tp], u[:, :Tp], lambda0=lam, eps=EPS)
                M = lam * np.eye(d) + uh[:Tp].T @ uh[:Tp]
                err = _rel(r.A[0], np.linalg.inv(M))
                assert err < 1e-10, f"A_T vs inv(M_T): d={d} lam={lam} T={Tp} rel err {err:.3e}"


def pin_delta(orc):
    """delta_t = 1 + u^_t^T A_{t-1} u^_t with A_{t-1} = M_{t-1}^{-1}, and delta_t >= 1 (§3.3)."""
    rng = np.random.default_rng(12)
    d, T = 6, 30
    q, k, v, u = _inputs(rng, T, d)
    r = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS, trace=True)
    uh = _unit_rows(u[0])
    M = LAMBDA0 * np.eye(d)
    for t in range(T):
        want = 1.0 + uh[t] @ np.linalg.solve(M, uh[t])
        got = r.delta[0, t]
        assert got >= 1.0, f"delta_{t} = {got} < 1"
        assert abs(got - want) <= 1e-11 * want, f"delta_{t}: {got} vs {want}"
        M = M + np.outer(uh[t], uh[t])


def pin_alpha_direction(orc):
    """alpha^_t is the unit vector along A_t k^_t with the UPDATED A_t (§3.3 eq. 10).

    Also checks that the pre-update alternative A_{t-1} k^_t would have been
    distinguishable on these inputs, so the pin has teeth.
    """
    rng = np.random.default_rng(13)
    d, T = 5, 25
    q, k, v, u = _inputs(rng, T, d)
    r = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS, trace=True)
    uh = _unit_rows(u[0])
    kh = _unit_rows(k[0])
    M = LAMBDA0 * np.eye(d)
    worst_pre = 0.0
    for t in range(T):
        pre = np.linalg.solve(M, kh[t])
        M = M + np.outer(uh[t], uh[t])
        want = np.linalg.solve(M, kh[t])
        want /= np.linalg.norm(want)
        got = r.alpha[0, t]
        assert abs(np.linalg.norm(got) - 1.0) < 1e-13, f"||alpha_{t}|| = {np.linalg.norm(got)}"
        assert np.max(np.abs(got - want)) < 1e-11, f"alpha_{t} direction off by {np.max(np.abs(got - want)):.3e}"
        assert np.max(np.abs(r.khat[0, t] - kh[t])) < 1e-14
        worst_pre = max(worst_pre, float(np.max(np.abs(pre / np.linalg.norm(pre) - want))))
    assert worst_pre > 1e-3, "inputs do not separate A_t from A_{t-1}"


def pin_A_spd(orc):
    """A_t stays symmetric positive definite with spectrum in (0, 1/lambda0] (§3.3)."""
    rng = np.random.default_rng(14)
    d, T = 8, 200
    q, k, v, u = _inputs(rng, T, d, lead=(2,))
    r = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS)
    for h in range(2):
        A = r.A[h]
        assert np.max(np.abs(A - A.T)) <= 1e-12 * np.max(np.abs(A))
        ev = np.linalg.eigvalsh(A)
        assert ev.min() > 0 and ev.max() <= 1.0 / LAMBDA0 * (1 + 1e-12), ev


# ---------------------------------------------------------------------------
# Proposition 2 (§4.2, eq. 14), as it holds for the literal update
# ---------------------------------------------------------------------------

def _sigma_max_closed_form(c):
    # For unit a, b with c = a.b, I - a b^T acts as [[1-c, 0], [-s, 1]] on
    # span{b, a}; its largest squared singular value is (3 - 2c + sqrt(5 - 4c)) / 2.
    return np.sqrt((3.0 - 2.0 * c + np.sqrt(5.0 - 4.0 * c)) / 2.0)


def pin_prop2_spectrum(orc):
    """J_t = I - alpha^_t k^_t^T: eigenvalues 1 (d-1 times) and 1 - c_t with
    c_t = alpha^_t . k^_t in (0, 1], so the spectral radius is exactly 1; the
    spectral norm equals the closed form above (1 only when alpha^ = k^).

    The paper states ||J_t||_2 = 1 for all unit alpha^, k^; that holds for the
    spectral radius, and for the norm only in the fixed-A case checked below.
    """
    rng = np.random.default_rng(15)
    d, T = 6, 30
    q, k, v, u = _inputs(rng, T, d)
    r = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS, trace=True)
    for t in range(T):
        a, b = r.alpha[0, t], r.khat[0, t]
        c = float(a @ b)
        assert 0.0 < c <= 1.0 + 1e-12, f"c_{t} = {c}"
        J = np.eye(d) - np.outer(a, b)
        ev = np.sort(np.abs(np.linalg.eigvals(J)))
        assert np.allclose(ev[1:], 1.0, atol=1e-9) and abs(ev[0] - abs(1.0 - c)) < 1e-9, ev
        smax = np.linalg.svd(J, compute_uv=False)[0]
        assert abs(smax - _sigma_max_closed_form(c)) < 1e-12, (smax, _sigma_max_closed_form(c))
    # fixed-A ablation (u = 0, §3.5): alpha^ = k^ and the norm is exactly 1
    u0 = np.zeros_like(u)
    r = orc.forward(q, k, v, u0, lambda0=LAMBDA0, eps=EPS, trace=True)
    for t in range(T):
        J = np.eye(d) - np.outer(r.alpha[0, t], r.khat[0, t])
        assert abs(np.linalg.svd(J, compute_uv=False)[0] - 1.0) < 1e-12


# ---------------------------------------------------------------------------
# S-pass: eq. 10 via Proposition 1 and the associative scan of §3.4
# ---------------------------------------------------------------------------

def pin_prop1_bound(orc):
    """||S_t||_F <= ||S_0||_F + sum_{s<=t} ||e_s|| at every t (§4.1 eq. 13)."""
    rng = np.random.default_rng(16)
    d, T = 6, 24
    q, k, v, u = _inputs(rng, T, d)
    S0 = rng.standard_normal((1, d, d))
    full = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS, S0=S0, trace=True)
    en = np.linalg.norm(full.e[0], axis=-1)
    base = np.linalg.norm(S0[0])
    for t in range(1, T + 1):
        r = orc.forward(q[:, :t], k[:, :t], v[:, :t], u[:, :t], lambda0=LAMBDA0, eps=EPS, S0=S0)
        assert np.linalg.norm(r.S[0]) <= base + en[:t].sum() + 1e-12


def _scan(pairs, lo, hi, rng):
    # (F, G) over tokens [lo, hi) composed in a random tree order; composition
    # (F_r, G_r) o (F_l, G_l) = (F_r F_l, F_r G_l + G_r) (§3.4 eq. 12).
    if hi - lo == 1:
        return pairs[lo]
    mid = int(rng.integers(lo + 1, hi))
    Fl, Gl = _scan(pairs, lo, mid, rng)
    Fr, Gr = _scan(pairs, mid, hi, rng)
    return Fr @ Fl, Fr @ Gl + Gr


def pin_scan(orc):
    """The sequential S equals a brute-force associative scan over (F, G) pairs.

    Eq. 12 as printed (S_t = F_t S_{t-1} + G_t with G_t = e_t alpha^_t^T) does
    not reproduce eq. 10; the consistent reading is the transposed state
    S_t^T = (I - alpha^_t k^_t^T) S_{t-1}^T + alpha^_t v_t^T, which uses only
    alpha^, k^ and the raw values v (not the residuals e).
    """
    rng = np.random.default_rng(17)
    d, T = 5, 37
    q, k, v, u = _inputs(rng, T, d)
    S0 = rng.standard_normal((1, d, d))
    r = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS, S0=S0, trace=True)
    pairs = [(np.eye(d) - np.outer(r.alpha[0, t], r.khat[0, t]),
              np.outer(r.alpha[0, t], v[0, t].astype(np.float64))) for t in range(T)]
    for trial in range(3):
        F, G = _scan(pairs, 0, T, np.random.default_rng(100 + trial))
        ST = F @ S0[0].T + G
        err = _rel(ST.T, r.S[0])
        assert err < 1e-10, f"scan vs sequential rel err {err:.3e}"


# ---------------------------------------------------------------------------
# Closed forms and special cases
# ---------------------------------------------------------------------------

def pin_scalar_closed_form(orc):
    """d = 1: u^, k^ = +-1, so A_t = 1/(lambda0 + t), alpha^_t = k^_t,
    S_t = v_t k^_t and o_t = v_t k^_t phi(q_t) / max(phi(q_t) sum_{s<=t} phi(k_s), eps)."""
    rng = np.random.default_rng(18)
    T = 30
    q, k, v, u = _inputs(rng, T, 1)
    for lam in (LAMBDA0, 2.5):
        r = orc.forward(q, k, v, u, lambda0=lam, eps=EPS)
        kh = np.sign(k[0, :, 0].astype(np.float64))
        qq = q[0, :, 0].astype(np.float64)
        kk = k[0, :, 0].astype(np.float64)
        vv = v[0, :, 0].astype(np.float64)
        zk = np.cumsum(_phi(kk))
        o = vv * kh * _phi(qq) / np.maximum(_phi(qq) * zk, EPS)
        assert abs(r.A[0, 0, 0] - 1.0 / (lam + T)) < 1e-14
        assert abs(r.S[0, 0, 0] - vv[-1] * kh[-1]) < 1e-13
        assert abs(r.zk[0, 0] - zk[-1]) < 1e-12
        assert _rel(r.o[0, :, 0], o) < 1e-12


def pin_single_token(orc):
    """One token from S_0 = 0, A_0 = I/lambda0: with a = 1/lambda0,
    A_1 = a I - a^2 u^ u^^T / (1 + a), S_1 = v alpha^^T, and
    o = v (alpha^ . phi(q)) / max(phi(q) . phi(k), eps)."""
    rng = np.random.default_rng(19)
    d = 5
    for qshift in (0.0, -60.0):  # -60 drives phi(q) . phi(k) below eps
        q, k, v, u = _inputs(rng, 1, d)
        q = (q + np.float32(qshift)).astype(np.float32)
        r = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS)
        a = 1.0 / LAMBDA0
        uh = _unit_rows(u[0, 0])
        kh = _unit_rows(k[0, 0])
        A1 = a * np.eye(d) - a * a * np.outer(uh, uh) / (1.0 + a)
        al = kh - (a / (1.0 + a)) * (uh @ kh) * uh  # A_1 k^ / a
        al /= np.linalg.norm(al)
        vv = v[0, 0].astype(np.float64)
        pq, pk = _phi(q[0, 0].astype(np.float64)), _phi(k[0, 0].astype(np.float64))
        den = max(pq @ pk, EPS)
        if qshift < 0:
            assert den == EPS
        assert _rel(r.A[0], A1) < 1e-13
        assert _rel(r.S[0], np.outer(vv, al)) < 1e-13
        assert _rel(r.o[0, 0], vv * (al @ pq) / den) < 1e-12


def pin_fixed_A_delta_rule(orc):
    """u_t = 0 keeps A at A_0 = I/lambda0 (§3.5 fixed-A ablation), so alpha^ = k^
    and the write is the unit-step delta rule S <- S (I - k^ k^^T) + v k^^T."""
    rng = np.random.default_rng(20)
    d, T = 7, 33
    q, k, v, _ = _inputs(rng, T, d)
    u = np.zeros_like(q)
    S0 = rng.standard_normal((1, d, d))
    r = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS, S0=S0)
    assert np.array_equal(r.A[0], np.eye(d) / LAMBDA0)
    S = S0[0].copy()
    zk = np.zeros(d)
    for t in range(T):
        kh = _unit_rows(k[0, t])
        S = S @ (np.eye(d) - np.outer(kh, kh)) + np.outer(v[0, t].astype(np.float64), kh)
        zk = zk + _phi(k[0, t].astype(np.float64))
        pq = _phi(q[0, t].astype(np.float64))
        assert _rel(r.o[0, t], S @ pq / max(pq @ zk, EPS)) < 1e-11
    assert _rel(r.S[0], S) < 1e-11


def pin_zero_values(orc):
    """v = 0 with S_0 = 0 keeps S = 0 and o = 0 (eq. 10-11)."""
    rng = np.random.default_rng(21)
    q, k, _, u = _inputs(rng, 20, 4)
    v = np.zeros_like(q)
    r = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS)
    assert np.all(r.S == 0) and np.all(r.o == 0)


def pin_zero_key(orc):
    """k_t = 0: the guarded normalisation gives k^ = 0 and alpha^ = 0, so S is
    unchanged and nothing is NaN; z^key still gains phi(0) = 1 per coordinate."""
    rng = np.random.default_rng(22)
    d, T = 4, 6
    q, k, v, u = _inputs(rng, T, d)
    k[:, 3] = 0.0
    r3 = orc.forward(q[:, :3], k[:, :3], v[:, :3], u[:, :3], lambda0=LAMBDA0, eps=EPS)
    r4 = orc.forward(q[:, :4], k[:, :4], v[:, :4], u[:, :4], lambda0=LAMBDA0, eps=EPS)
    assert np.all(np.isfinite(r4.o)) and np.array_equal(r4.S, r3.S)
    assert np.allclose(r4.zk - r3.zk, 1.0, atol=1e-14)


def pin_u_scale_invariance(orc):
    """u enters only through its direction (§3.2: unit penalty directions), so
    rescaling each u_t by a positive factor changes nothing."""
    rng = np.random.default_rng(23)
    d, T = 6, 20
    q, k, v, u = _inputs(rng, T, d)
    s = np.exp(rng.uniform(-3, 3, size=(1, T, 1))).astype(np.float32)
    r1 = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS)
    r2 = orc.forward(q, k, v, (u * s).astype(np.float32), lambda0=LAMBDA0, eps=EPS)
    # u * s is rounded to float32, so directions agree to ~1e-7
    assert _rel(r2.A, r1.A) < 1e-5 and _rel(r2.o, r1.o) < 1e-5


def pin_chunked_state(orc):
    """Running [0, t1) then [t1, T) with the carried (S, A, z^key) equals one run."""
    rng = np.random.default_rng(24)
    d, T, t1 = 5, 29, 11
    q, k, v, u = _inputs(rng, T, d, lead=(2,))
    full = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS)
    a = orc.forward(q[:, :t1], k[:, :t1], v[:, :t1], u[:, :t1], lambda0=LAMBDA0, eps=EPS)
    b = orc.forward(q[:, t1:], k[:, t1:], v[:, t1:], u[:, t1:], lambda0=LAMBDA0, eps=EPS,
                    S0=a.S, A0=a.A, zk0=a.zk)
    assert np.array_equal(np.concatenate([a.o, b.o], axis=1), full.o)
    assert np.array_equal(b.S, full.S) and np.array_equal(b.A, full.A) and np.array_equal(b.zk, full.zk)


def pin_heads_independent(orc):
    """Each (b, h) head is its own recurrence: running heads together or one at
    a time gives identical results."""
    rng = np.random.default_rng(25)
    q, k, v, u = _inputs(rng, 9, 4, lead=(3,))
    allh = orc.forward(q, k, v, u, lambda0=LAMBDA0, eps=EPS)
    for h in range(3):
        one = orc.forward(q[h:h + 1], k[h:h + 1], v[h:h + 1], u[h:h + 1], lambda0=LAMBDA0, eps=EPS)
        assert np.array_equal(one.o[0], allh.o[h]) and np.array_equal(one.S[0], allh.S[h])


def pin_linear_attention_state(orc):
    """Plain cumulative linear attention S = sum_t v_t phi(k_t)^T (§4.1 comparison)."""
    rng = np.random.default_rng(26)
    q, k, v, u = _inputs(rng, 50, 6, lead=(2,))
    S = orc.linear_attention_state(k, v)
    want = np.einsum("hti,htj->hij", v.astype(np.float64), _phi(k.astype(np.float64)))
    assert _rel(S, want) < 1e-12


def pin_linear_attention_closed_forms(orc):
    """Linear attention with k = 0 gives phi(0) = 1, so every column of S is
    sum_t v_t; and the sum is independent of the token order."""
    rng = np.random.default_rng(27)
    T, d = 23, 5
    _, _, v, _ = _inputs(rng, T, d)
    k0 = np.zeros_like(v)
    S = orc.linear_attention_state(k0, v)[0]
    col = v[0].astype(np.float64).sum(axis=0)
    assert np.allclose(S, np.repeat(col[:, None], d, axis=1), rtol=1e-13, atol=1e-13)
    _, k, v, _ = _inputs(rng, T, d)
    perm = rng.permutation(T)
    S1 = orc.linear_attention_state(k, v)[0]
    S2 = orc.linear_attention_state(k[:, perm], v[:, perm])[0]
    assert _rel(S2, S1) < 1e-13


# ---------------------------------------------------------------------------
# backward pass: the oracle's reverse-mode gradient against central finite
# differences of the oracle's forward (pinned above), and against eq. 14
# ---------------------------------------------------------------------------

def _spd(rng, d, lead=(1,)):
    m = rng.standard_normal(tuple(lead) + (d, d))
    return m @ np.swapaxes(m, -1, -2) / d + 2.0 * np.eye(d)


def pin_backward_finite_differences(orc):
    """dL/dx of L = sum gO.o + <gS, S_T> + <gA, A_T> + gzk.zk_T matches the
    central difference (L(x + h r) - L(x - h r)) / 2h along a random direction r,
    for every input and every piece of the initial state."""
    rng = np.random.default_rng(31)
    for T, d, with_state in ((6, 5, True), (4, 3, False)):
        lead = (2,)
        q, k, v, u = (rng.standard_normal(lead + (T, d)) for _ in range(4))
        state = dict(S0=rng.standard_normal(lead + (d, d)), A0=_spd(rng, d, lead),
                     zk0=rng.uniform(0.5, 1.5, lead + (d,))) if with_state else {}
        seeds = dict(gO=rng.standard_normal(lead + (T, d)), gS=rng.standard_normal(lead + (d, d)),
                     gA=rng.standard_normal(lead + (d, d)), gzk=rng.standard_normal(lead + (d,)))

        def loss(**x):
            o, S, A, zk = orc.forward_f64(x["q"], x["k"], x["v"], x["u"], LAMBDA0, EPS,
                                          x.get("S0"), x.get("A0"), x.get("zk0"))
            return (np.sum(seeds["gO"] * o) + np.sum(seeds["gS"] * S) + np.sum(seeds["gA"] * A)
                    + np.sum(seeds["gzk"] * zk))

        g = orc.backward(q, k, v, u, LAMBDA0, EPS, state.get("S0"), state.get("A0"), state.get("zk0"),
                         **seeds)
        args = dict(q=q, k=k, v=v, u=u, **state)
        for name, x in args.items():
            r = rng.standard_normal(x.shape)
            h = 1e-6
            xp, xm = dict(args), dict(args)
            xp[name], xm[name] = x + h * r, x - h * r
            fd = (loss(**xp) - loss(**xm)) / (2 * h)
            an = float(np.sum(g["d" + name] * r))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def pin_backward_state_jacobian(orc):
    """One token, only dL/dS_1 = G seeded: dL/dS_0 = G (I - alpha^ k^^T), the
    state Jacobian of eq. 14 in the orientation S_t = S_{t-1} (I - k^ alpha^^T)
    + v alpha^^T; its largest singular value is the closed form
    sqrt((3 - 2c + sqrt(5 - 4c)) / 2), c = alpha^ . k^."""
    rng = np.random.default_rng(32)
    d = 6
    q, k, v, u = _inputs(rng, 1, d)
    tr = orc.forward(q, k, v, u, LAMBDA0, EPS, trace=True)
    al, kh = tr.alpha[0, 0], tr.khat[0, 0]
    J = np.eye(d) - np.outer(al, kh)
    G = rng.standard_normal((1, d, d))
    g = orc.backward(q, k, v, u, LAMBDA0, EPS, gS=G)
    assert _rel(g["dS0"][0], G[0] @ J) < 1e-12
    c = float(al @ kh)
    smax = np.sqrt((3 - 2 * c + np.sqrt(5 - 4 * c)) / 2)
    # G = x y^T with y the top left singular vector of J: ||G J|| = smax ||G||
    U, sv, Vt = np.linalg.svd(J)
    G1 = np.outer(np.ones(d), U[:, 0])[None]
    g1 = orc.backward(q, k, v, u, LAMBDA0, EPS, gS=G1)
    assert abs(np.linalg.norm(g1["dS0"]) / np.linalg.norm(G1) - smax) < 1e-10


def pin_backward_fixed_A_nonexpansive(orc):
    """Fixed-A ablation (u = 0, A = lambda0^-1 I so alpha^ = k^): each state
    Jacobian is the projection I - k^ k^^T, so ||dL/dS_0||_F <= ||dL/dS_T||_F
    (Corollary 1 holds exactly there), and the gradient of A_0 through the
    penalty directions get a zero gradient (u = 0 makes z = 0)."""
    rng = np.random.default_rng(33)
    T, d = 30, 8
    q, k, v, _ = _inputs(rng, T, d)
    u = np.zeros_like(q)
    G = rng.standard_normal((1, d, d))
    g = orc.backward(q, k, v, u, LAMBDA0, EPS, gS=G)
    assert np.linalg.norm(g["dS0"]) <= np.linalg.norm(G) * (1 + 1e-12)
    assert np.max(np.abs(g["du"])) == 0.0


ALL_PINS = [
    pin_inverse_penalty,
    pin_delta,
    pin_alpha_direction,
    pin_A_spd,
    pin_prop2_spectrum,
    pin_prop1_bound,
    pin_scan,
    pin_scalar_closed_form,
    pin_single_token,
    pin_fixed_A_delta_rule,
    pin_zero_values,
    pin_zero_key,
    pin_u_scale_invariance,
    pin_chunked_state,
    pin_heads_independent,
    pin_linear_attention_state,
    pin_linear_attention_closed_forms,
    pin_backward_finite_differences,
    pin_backward_state_jacobian,
    pin_backward_fixed_A_nonexpansive,
]
