/*
 * vla_oracle.c -- fp64 CPU oracle for the Variational Linear Attention (VLA)
 * forward recurrence and its reverse-mode gradient (backward pass).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the independent reference that the
 * CUDA path is checked against. Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference arm may build, load or call it; the
 * product path never does. It shares no code, header or constant with the
 * CUDA library.
 *
 * Source: "Variational Linear Attention: Stable Associative Memory for
 * Long-Context Transformers" (Pandey, Singh; arXiv 2605.11196), §3.3:
 *   eq. 9   z_t = A_{t-1} u_t,  delta_t = 1 + u_t^T z_t,
 *           A_t = A_{t-1} - z_t z_t^T / delta_t           (Sherman-Morrison)
 *   eq. 10  e_t = v_t - S_{t-1} k^_t,
 *           alpha^_t = A_t k^_t / ||A_t k^_t||,
 *           S_t = S_{t-1} + e_t alpha^_t^T
 *   eq. 11  o_t = S_t phi(q_t) / max(phi(q_t)^T z^key_t, eps),
 *           z^key_t = sum_{s<=t} phi(k_s),  phi = ELU + 1
 * with A_0 = lambda0^{-1} I (lambda0 = 0.1 gives A_0 = 10 I, §3.2) and the
 * penalty directions u_t and the keys used unit-normalised (§3.2, §3.3).
 *
 * Readings of points the paper leaves open (the design notes list each one):
 *  - u_t and k_t are op inputs and are normalised inside the op:
 *    x^ = x / max(||x||, 1e-12); the same guard is used for alpha^.
 *  - phi is applied to the raw (un-normalised) q_t and k_t.
 *  - alpha^_t uses the updated A_t; e_t uses S_{t-1}; o_t uses S_t and a
 *    key sum that includes token t (eq. 10-11 as written).
 *  - z^key is part of the carried state, with S and A.
 *
 * Arithmetic is fp64 throughout; inputs arrive as float32 (which represents
 * every fp32 and bf16 input value exactly) and are widened per element.
 * Heads (b, h) are independent and are distributed over OpenMP threads; the
 * order of operations inside a head is the plain loop below.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* phi(x) = ELU(x) + 1: x + 1 for x > 0, exp(x) otherwise (§3.3, eq. 11). */
static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* out = x / max(||x||, 1e-12) */
static void unit(const double* x, double* out, int d) {
    double nn = 0.0;
    for (int j = 0; j < d; ++j) nn += x[j] * x[j];
    double n = sqrt(nn);
    if (n < 1e-12) n = 1e-12;
    for (int j = 0; j < d; ++j) out[j] = x[j] / n;
}

/*
 * One head. Inputs q, k, v, u point at this head's [T, d] rows. State
 * pointers S0, A0, zk0 may be NULL (then S_0 = 0, A_0 = I / lambda0,
 * z^key_0 = 0). o is [T, d]; S_out and A_out are [d, d] row-major (S[i][j]
 * maps key coordinate j to output i); zk_out is [d]. Every trace pointer may
 * be NULL; when given it receives, per token, delta_t ([T]), alpha^_t, k^_t,
 * u^_t and e_t ([T, d] each).
 */
static void vla_head(int T, int d,
                     const double* q, const double* k, const double* v, const double* u,
                     double lambda0, double eps,
                     const double* S0, const double* A0, const double* zk0,
                     double* o, double* S_out, double* A_out, double* zk_out,
                     double* tr_delta, double* tr_alpha, double* tr_khat,
                     double* tr_uhat, double* tr_e) {
    double* A = (double*)malloc(sizeof(double) * d * d);
    double* S = (double*)malloc(sizeof(double) * d * d);
    double* zk = (double*)malloc(sizeof(double) * d);
    double* x = (double*)malloc(sizeof(double) * d);
    double* uh = (double*)malloc(sizeof(double) * d);
    double* kh = (double*)malloc(sizeof(double) * d);
    double* z = (double*)malloc(sizeof(double) * d);
    double* a = (double*)malloc(sizeof(double) * d);
    double* alpha = (double*)malloc(sizeof(double) * d);
    double* e = (double*)malloc(sizeof(double) * d);
    double* pq = (double*)malloc(sizeof(double) * d);

    /* initial state */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            A[i * d + j] = A0 ? A0[i * d + j] : (i == j ? 1.0 / lambda0 : 0.0);
            S[i * d + j] = S0 ? S0[i * d + j] : 0.0;
        }
    for (int j = 0; j < d; ++j) zk[j] = zk0 ? zk0[j] : 0.0;

    for (int t = 0; t < T; ++t) {
        const double* qt = q + (size_t)t * d;
        const double* kt = k + (size_t)t * d;
        const double* vt = v + (size_t)t * d;
        const double* ut = u + (size_t)t * d;

        /* unit penalty direction and unit key */
        for (int j = 0; j < d; ++j) x[j] = (double)ut[j];
        unit(x, uh, d);
        for (int j = 0; j < d; ++j) x[j] = (double)kt[j];
        unit(x, kh, d);

        /* eq. 9: z = A_{t-1} u^, delta = 1 + u^T z, A_t = A_{t-1} - z z^T / delta */
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += A[i * d + j] * uh[j];
            z[i] = s;
        }
        double delta = 1.0;
        for (int i = 0; i < d; ++i) delta += uh[i] * z[i];
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) A[i * d + j] -= z[i] * z[j] / delta;

        /* eq. 10: alpha^ = A_t k^ / ||A_t k^|| */
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += A[i * d + j] * kh[j];
            a[i] = s;
        }
        unit(a, alpha, d);

        /* eq. 10: e = v - S_{t-1} k^, S_t = S_{t-1} + e alpha^T */
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += S[i * d + j] * kh[j];
            e[i] = (double)vt[i] - s;
        }
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) S[i * d + j] += e[i] * alpha[j];

        /* eq. 11: z^key_t = z^key_{t-1} + phi(k_t); o = S_t phi(q) / max(phi(q)^T z^key_t, eps) */
        for (int j = 0; j < d; ++j) zk[j] += phi((double)kt[j]);
        double den = 0.0;
        for (int j = 0; j < d; ++j) {
            pq[j] = phi((double)qt[j]);
            den += pq[j] * zk[j];
        }
        if (den < eps) den = eps;
        if (o) {
            for (int i = 0; i < d; ++i) {
                double s = 0.0;
                for (int j = 0; j < d; ++j) s += S[i * d + j] * pq[j];
                o[(size_t)t * d + i] = s / den;
            }
        }

        if (tr_delta) tr_delta[t] = delta;
        for (int j = 0; j < d; ++j) {
            if (tr_alpha) tr_alpha[(size_t)t * d + j] = alpha[j];
            if (tr_khat) tr_khat[(size_t)t * d + j] = kh[j];
            if (tr_uhat) tr_uhat[(size_t)t * d + j] = uh[j];
            if (tr_e) tr_e[(size_t)t * d + j] = e[j];
        }
    }

    if (S_out) memcpy(S_out, S, sizeof(double) * d * d);
    if (A_out) memcpy(A_out, A, sizeof(double) * d * d);
    if (zk_out) memcpy(zk_out, zk, sizeof(double) * d);

    free(A); free(S); free(zk); free(x); free(uh); free(kh);
    free(z); free(a); free(alpha); free(e); free(pq);
}

#define OFF(p, n) ((p) ? (p) + (n) : NULL)

/*
 * All heads. Inputs q, k, v, u: [BH, T, d] float32. Optional state:
 * S0, A0 [BH, d, d], zk0 [BH, d]. Outputs (any may be NULL): o [BH, T, d],
 * S_out, A_out [BH, d, d], zk_out [BH, d]. Optional traces: tr_delta [BH, T],
 * tr_alpha, tr_khat, tr_uhat, tr_e [BH, T, d]. nthreads <= 0 uses the OpenMP
 * default. Returns the number of threads used.
 */
int vla_oracle_forward(int BH, int T, int d,
                       const float* q, const float* k, const float* v, const float* u,
                       double lambda0, double eps,
                       const double* S0, const double* A0, const double* zk0,
                       double* o, double* S_out, double* A_out, double* zk_out,
                       double* tr_delta, double* tr_alpha, double* tr_khat,
                       double* tr_uhat, double* tr_e, int nthreads) {
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    if (nthreads > BH && BH > 0) nthreads = BH;
    used = nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int h = 0; h < BH; ++h) {
        size_t in = (size_t)h * T * d, st = (size_t)h * d * d, vec = (size_t)h * d;
        /* widen this head's inputs (exact: fp32 and bf16 values are doubles) */
        double* x = (double*)malloc(sizeof(double) * 4 * (size_t)T * d + 1);
        for (size_t i = 0; i < (size_t)T * d; ++i) {
            x[i] = (double)q[in + i];
            x[(size_t)T * d + i] = (double)k[in + i];
            x[2 * (size_t)T * d + i] = (double)v[in + i];
            x[3 * (size_t)T * d + i] = (double)u[in + i];
        }
        vla_head(T, d, x, x + (size_t)T * d, x + 2 * (size_t)T * d, x + 3 * (size_t)T * d, lambda0, eps,
                 OFF(S0, st), OFF(A0, st), OFF(zk0, vec),
                 OFF(o, in), OFF(S_out, st), OFF(A_out, st), OFF(zk_out, vec),
                 OFF(tr_delta, (size_t)h * T), OFF(tr_alpha, in), OFF(tr_khat, in),
                 OFF(tr_uhat, in), OFF(tr_e, in));
        free(x);
    }
    return used;
}

/* The same with fp64 inputs [BH, T, d] (finite-difference checks of the backward). */
int vla_oracle_forward_f64(int BH, int T, int d,
                           const double* q, const double* k, const double* v, const double* u,
                           double lambda0, double eps,
                           const double* S0, const double* A0, const double* zk0,
                           double* o, double* S_out, double* A_out, double* zk_out) {
    for (int h = 0; h < BH; ++h) {
        size_t in = (size_t)h * T * d, st = (size_t)h * d * d, vec = (size_t)h * d;
        vla_head(T, d, q + in, k + in, v + in, u + in, lambda0, eps,
                 OFF(S0, st), OFF(A0, st), OFF(zk0, vec),
                 OFF(o, in), OFF(S_out, st), OFF(A_out, st), OFF(zk_out, vec),
                 NULL, NULL, NULL, NULL, NULL);
    }
    return 1;
}

/*
 * Plain cumulative linear attention state (the comparison in §4.1 and the
 * linear-attention recurrence S_t = S_{t-1} + v_t phi(k_t)^T, in the same
 * orientation as the VLA state): S_out [BH, d, d] = sum_t v_t phi(k_t)^T.
 */
int vla_oracle_linear_attention_state(int BH, int T, int d,
                                      const float* k, const float* v,
                                      double* S_out, int nthreads) {
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    if (nthreads > BH && BH > 0) nthreads = BH;
    used = nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int h = 0; h < BH; ++h) {
        double* S = S_out + (size_t)h * d * d;
        for (int i = 0; i < d * d; ++i) S[i] = 0.0;
        for (int t = 0; t < T; ++t) {
            const float* kt = k + ((size_t)h * T + t) * d;
            const float* vt = v + ((size_t)h * T + t) * d;
            for (int i = 0; i < d; ++i)
                for (int j = 0; j < d; ++j) S[i * d + j] += (double)vt[i] * phi((double)kt[j]);
        }
    }
    return used;
}

/*
 * Reverse-mode gradient of one head's forward pass (the backward pass the
 * paper's Corollary 1 refers to; §4.2, eq. 14 is the state Jacobian
 * dS_t/dS_{t-1} = I - alpha^_t k^_t^T used below in transposed orientation).
 *
 * Loss seeds: gO [T, d] = dL/do_t (may be NULL: zero), gST, gAT [d, d] and
 * gzkT [d] = dL/dS_T, dL/dA_T, dL/dz^key_T (each may be NULL: zero).
 * Outputs: dq, dk, dv, du [T, d]; dS0, dA0 [d, d], dzk0 [d] (any may be NULL).
 *
 * The forward pass is rerun storing every state S_t, A_t and the per-token
 * vectors; the sweep then visits t = T-1 .. 0 applying, in reverse order, the
 * adjoint of each step of eq. 9-11:
 *   o_t = S_t phi_q / den       gS += gO_t phi_q^T / den, g_phiq = S_t^T gO_t / den,
 *                               g_den = -(gO_t . o_t) / den  (0 where den = eps)
 *   den = phi_q . zk_t          g_phiq += g_den zk_t, g_zk += g_den phi_q
 *   zk_t = zk_{t-1} + phi(k_t)  g_phik = g_zk
 *   S_t = S_{t-1} + e alpha^T   g_e = gS alpha, g_alpha = gS^T e
 *   e = v_t - S_{t-1} k^        g_v = g_e, gS -= g_e k^^T, g_k^ = -S_{t-1}^T g_e
 *   alpha = a / ||a||           g_a = (g_alpha - alpha (alpha . g_alpha)) / ||a||
 *   a = A_t k^                  gA += g_a k^^T, g_k^ += A_t^T g_a
 *   A_t = A_{t-1} - z z^T/delta g_z = -(gA + gA^T) z / delta, g_delta = z^T gA z / delta^2
 *   delta = 1 + u^ . z          g_u^ = g_delta z, g_z += g_delta u^
 *   z = A_{t-1} u^              gA += g_z u^^T, g_u^ += A_{t-1}^T g_z
 *   x^ = x / max(||x||, 1e-12)  g_x = (g_x^ - x^ (x^ . g_x^)) / ||x||  (g_x^ / 1e-12 below the guard)
 *   phi(x)                      g_x += g_phi * (x > 0 ? 1 : exp(x))
 * and ends with dS0 = gS, dA0 = gA, dzk0 = g_zk.
 */
static void unit_grad(const double* x, const double* g, double* out, int d) {
    double nn = 0.0;
    for (int j = 0; j < d; ++j) nn += x[j] * x[j];
    double n = sqrt(nn);
    if (n < 1e-12) {
        for (int j = 0; j < d; ++j) out[j] = g[j] / 1e-12;
        return;
    }
    double xg = 0.0;
    for (int j = 0; j < d; ++j) xg += x[j] * g[j];
    for (int j = 0; j < d; ++j) out[j] = (g[j] - x[j] / n * (xg / n)) / n;
}

static double dphi(double x) { return x > 0.0 ? 1.0 : exp(x); }

static void vla_head_backward(int T, int d,
                              const double* q, const double* k, const double* v, const double* u,
                              double lambda0, double eps,
                              const double* S0, const double* A0, const double* zk0,
                              const double* gO, const double* gST, const double* gAT, const double* gzkT,
                              double* dq, double* dk, double* dv, double* du,
                              double* dS0, double* dA0, double* dzk0) {
    const size_t dd = (size_t)d * d;
    /* states S_t, A_t for t = 0..T (index 0 = initial) and per-token vectors */
    double* Ss = (double*)malloc(sizeof(double) * dd * (T + 1));
    double* As = (double*)malloc(sizeof(double) * dd * (T + 1));
    double* zks = (double*)malloc(sizeof(double) * (size_t)d * (T + 1));
    double* uh = (double*)malloc(sizeof(double) * (size_t)d * T + 1);
    double* kh = (double*)malloc(sizeof(double) * (size_t)d * T + 1);
    double* zz = (double*)malloc(sizeof(double) * (size_t)d * T + 1);
    double* aa = (double*)malloc(sizeof(double) * (size_t)d * T + 1);
    double* al = (double*)malloc(sizeof(double) * (size_t)d * T + 1);
    double* ee = (double*)malloc(sizeof(double) * (size_t)d * T + 1);
    double* pq = (double*)malloc(sizeof(double) * (size_t)d * T + 1);
    double* dl = (double*)malloc(sizeof(double) * T + 1);
    double* na = (double*)malloc(sizeof(double) * T + 1);
    double* dn = (double*)malloc(sizeof(double) * T + 1);
    int* cl = (int*)malloc(sizeof(int) * T + 1);

    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            As[i * d + j] = A0 ? A0[i * d + j] : (i == j ? 1.0 / lambda0 : 0.0);
            Ss[i * d + j] = S0 ? S0[i * d + j] : 0.0;
        }
    for (int j = 0; j < d; ++j) zks[j] = zk0 ? zk0[j] : 0.0;

    /* forward, the same steps as vla_head, keeping everything */
    for (int t = 0; t < T; ++t) {
        const double *Ap = As + dd * t, *Sp = Ss + dd * t;
        double *A = As + dd * (t + 1), *S = Ss + dd * (t + 1);
        double *ut = uh + (size_t)t * d, *kt = kh + (size_t)t * d, *z = zz + (size_t)t * d;
        double *a = aa + (size_t)t * d, *alpha = al + (size_t)t * d, *e = ee + (size_t)t * d;
        double* pqt = pq + (size_t)t * d;
        unit(u + (size_t)t * d, ut, d);
        unit(k + (size_t)t * d, kt, d);
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += Ap[i * d + j] * ut[j];
            z[i] = s;
        }
        double delta = 1.0;
        for (int i = 0; i < d; ++i) delta += ut[i] * z[i];
        dl[t] = delta;
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) A[i * d + j] = Ap[i * d + j] - z[i] * z[j] / delta;
        double nn = 0.0;
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += A[i * d + j] * kt[j];
            a[i] = s;
            nn += s * s;
        }
        na[t] = sqrt(nn);
        unit(a, alpha, d);
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += Sp[i * d + j] * kt[j];
            e[i] = v[(size_t)t * d + i] - s;
        }
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) S[i * d + j] = Sp[i * d + j] + e[i] * alpha[j];
        double den = 0.0;
        for (int j = 0; j < d; ++j) {
            zks[(size_t)(t + 1) * d + j] = zks[(size_t)t * d + j] + phi(k[(size_t)t * d + j]);
            pqt[j] = phi(q[(size_t)t * d + j]);
            den += pqt[j] * zks[(size_t)(t + 1) * d + j];
        }
        cl[t] = den < eps;
        dn[t] = cl[t] ? eps : den;
    }

    /* reverse sweep */
    double* gS = (double*)calloc(dd, sizeof(double));
    double* gA = (double*)calloc(dd, sizeof(double));
    double* gzk = (double*)calloc(d, sizeof(double));
    double* gpq = (double*)malloc(sizeof(double) * d);
    double* ge = (double*)malloc(sizeof(double) * d);
    double* gal = (double*)malloc(sizeof(double) * d);
    double* ga = (double*)malloc(sizeof(double) * d);
    double* gkh = (double*)malloc(sizeof(double) * d);
    double* guh = (double*)malloc(sizeof(double) * d);
    double* gz = (double*)malloc(sizeof(double) * d);
    double* ot = (double*)malloc(sizeof(double) * d);
    double* tmp = (double*)malloc(sizeof(double) * d);
    if (gST) memcpy(gS, gST, sizeof(double) * dd);
    if (gAT) memcpy(gA, gAT, sizeof(double) * dd);
    if (gzkT) memcpy(gzk, gzkT, sizeof(double) * d);
    for (int t = T - 1; t >= 0; --t) {
        const double *A = As + dd * (t + 1), *Ap = As + dd * t;
        const double *S = Ss + dd * (t + 1), *Sp = Ss + dd * t;
        const double *ut = uh + (size_t)t * d, *kt = kh + (size_t)t * d, *z = zz + (size_t)t * d;
        const double *alpha = al + (size_t)t * d, *e = ee + (size_t)t * d, *pqt = pq + (size_t)t * d;
        const double* zkt = zks + (size_t)(t + 1) * d;
        const double den = dn[t], delta = dl[t];
        /* o_t = S_t phi_q / den */
        double go_o = 0.0;
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += S[i * d + j] * pqt[j];
            ot[i] = s / den;
        }
        for (int j = 0; j < d; ++j) gpq[j] = 0.0;
        if (gO) {
            const double* g = gO + (size_t)t * d;
            for (int i = 0; i < d; ++i) {
                go_o += g[i] * ot[i];
                for (int j = 0; j < d; ++j) gS[i * d + j] += g[i] * pqt[j] / den;
            }
            for (int j = 0; j < d; ++j) {
                double s = 0.0;
                for (int i = 0; i < d; ++i) s += S[i * d + j] * g[i];
                gpq[j] = s / den;
            }
        }
        const double gden = cl[t] ? 0.0 : -go_o / den;
        for (int j = 0; j < d; ++j) {
            gpq[j] += gden * zkt[j];
            gzk[j] += gden * pqt[j];
        }
        /* S_t = S_{t-1} + e alpha^T;  e = v - S_{t-1} k^ */
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int j = 0; j < d; ++j) s += gS[i * d + j] * alpha[j];
            ge[i] = s;
        }
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += gS[i * d + j] * e[i];
            gal[j] = s;
        }
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) gS[i * d + j] -= ge[i] * kt[j];
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += Sp[i * d + j] * ge[i];
            gkh[j] = -s;
        }
        /* alpha = a / ||a||, a = A_t k^ */
        {
            double ag = 0.0;
            for (int j = 0; j < d; ++j) ag += alpha[j] * gal[j];
            const double n = na[t] < 1e-12 ? 1e-12 : na[t];
            for (int j = 0; j < d; ++j) ga[j] = na[t] < 1e-12 ? gal[j] / n : (gal[j] - alpha[j] * ag) / n;
        }
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) gA[i * d + j] += ga[i] * kt[j];
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += A[i * d + j] * ga[i];
            gkh[j] += s;
        }
        /* A_t = A_{t-1} - z z^T / delta;  delta = 1 + u^ . z;  z = A_{t-1} u^ */
        double zgz = 0.0;
        for (int i = 0; i < d; ++i) {
            double s1 = 0.0, s2 = 0.0;
            for (int j = 0; j < d; ++j) {
                s1 += gA[i * d + j] * z[j];
                s2 += gA[j * d + i] * z[j];
            }
            gz[i] = -(s1 + s2) / delta;
            zgz += z[i] * s1;
        }
        const double gdelta = zgz / (delta * delta);
        for (int j = 0; j < d; ++j) {
            guh[j] = gdelta * z[j];
            gz[j] += gdelta * ut[j];
        }
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) gA[i * d + j] += gz[i] * ut[j];
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += Ap[i * d + j] * gz[i];
            guh[j] += s;
        }
        /* normalisations and phi */
        unit_grad(u + (size_t)t * d, guh, tmp, d);
        if (du) memcpy(du + (size_t)t * d, tmp, sizeof(double) * d);
        unit_grad(k + (size_t)t * d, gkh, tmp, d);
        for (int j = 0; j < d; ++j) {
            if (dk) dk[(size_t)t * d + j] = tmp[j] + gzk[j] * dphi(k[(size_t)t * d + j]);
            if (dq) dq[(size_t)t * d + j] = gpq[j] * dphi(q[(size_t)t * d + j]);
            if (dv) dv[(size_t)t * d + j] = ge[j];
        }
    }
    if (dS0) memcpy(dS0, gS, sizeof(double) * dd);
    if (dA0) memcpy(dA0, gA, sizeof(double) * dd);
    if (dzk0) memcpy(dzk0, gzk, sizeof(double) * d);

    free(Ss); free(As); free(zks); free(uh); free(kh); free(zz); free(aa); free(al); free(ee); free(pq);
    free(dl); free(na); free(dn); free(cl);
    free(gS); free(gA); free(gzk); free(gpq); free(ge); free(gal); free(ga); free(gkh); free(guh); free(gz);
    free(ot); free(tmp);
}

/*
 * All heads, fp64 inputs and seeds: q, k, v, u, gO [BH, T, d]; S0, A0, gST,
 * gAT [BH, d, d]; zk0, gzkT [BH, d] (optional ones may be NULL). Outputs dq,
 * dk, dv, du [BH, T, d], dS0, dA0 [BH, d, d], dzk0 [BH, d] (may be NULL).
 */
int vla_oracle_backward(int BH, int T, int d,
                        const double* q, const double* k, const double* v, const double* u,
                        double lambda0, double eps,
                        const double* S0, const double* A0, const double* zk0,
                        const double* gO, const double* gST, const double* gAT, const double* gzkT,
                        double* dq, double* dk, double* dv, double* du,
                        double* dS0, double* dA0, double* dzk0, int nthreads) {
    int used = 1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    if (nthreads > BH && BH > 0) nthreads = BH;
    used = nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int h = 0; h < BH; ++h) {
        size_t in = (size_t)h * T * d, st = (size_t)h * d * d, vec = (size_t)h * d;
        vla_head_backward(T, d, q + in, k + in, v + in, u + in, lambda0, eps,
                          OFF(S0, st), OFF(A0, st), OFF(zk0, vec),
                          OFF(gO, in), OFF(gST, st), OFF(gAT, st), OFF(gzkT, vec),
                          OFF(dq, in), OFF(dk, in), OFF(dv, in), OFF(du, in),
                          OFF(dS0, st), OFF(dA0, st), OFF(dzk0, vec));
    }
    return used;
}
