/*
 * vla_oracle.c -- fp64 CPU oracle for the Variational Linear Attention (VLA)
 * forward recurrence.
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
 * Readings of points the paper leaves open (each is listed in the design doc):
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
                     const float* q, const float* k, const float* v, const float* u,
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
        const float* qt = q + (size_t)t * d;
        const float* kt = k + (size_t)t * d;
        const float* vt = v + (size_t)t * d;
        const float* ut = u + (size_t)t * d;

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
        vla_head(T, d, q + in, k + in, v + in, u + in, lambda0, eps,
                 OFF(S0, st), OFF(A0, st), OFF(zk0, vec),
                 OFF(o, in), OFF(S_out, st), OFF(A_out, st), OFF(zk_out, vec),
                 OFF(tr_delta, (size_t)h * T), OFF(tr_alpha, in), OFF(tr_khat, in),
                 OFF(tr_uhat, in), OFF(tr_e, in));
    }
    return used;
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
