// vla_backward.cuh -- reverse-mode gradient of the VLA forward recurrence
// ("Variational Linear Attention", arXiv 2605.11196, §3.3 eq. 9-11; the state
// Jacobian of §4.2 eq. 14 is the adjoint step of the S recurrence below).
// Included by vla_forward.cu inside namespace vla.
//
// One CTA per (b, h), two phases:
//  1. the forward recurrence, token by token, writing a tape to the workspace:
//     z_t (eq. 9), alpha^_t and ||a_t|| (eq. 10), e_t (eq. 10), delta_t and
//     den_t (eq. 11), and S, A every BW_CK tokens;
//  2. the reverse sweep t = T-1 .. 0 applying the adjoint of each step of
//     eq. 9-11 in reverse order (the same order as the fp64 oracle's). S_{t-1}
//     and A_{t-1} are rebuilt from S_t, A_t by undoing the step's rank-1
//     update (S_{t-1} = S_t - e alpha^^T, A_{t-1} = A_t + z z^T / delta) and
//     reset from the checkpoint every BW_CK tokens.
// S, A and the adjoints dL/dS, dL/dA live in shared memory ([D][D+1] fp32);
// thread i of a 96-thread group owns row (or column) i of a matrix-vector
// product.

namespace bw {

constexpr int CK = 64;  // checkpoint interval (tokens)

template <int D>
struct BLay {
    static constexpr int NG = 6;              // 6 groups of D threads for the matrix-vector rounds
    static constexpr int THREADS = NG * D;    // 576 at d = 96
    static constexpr int LD = D + 1;          // odd row stride: row and column walks are conflict-free
    static constexpr int MAT = D * LD;
    // tape per token: z | alpha | e (D each), then delta, ||a||, den (signed:
    // negative = the eps floor was taken)
    static constexpr int TREC = 3 * D + 4;
    static constexpr int NVEC = 24;           // shared d-vectors
    static constexpr size_t SMEM = ((size_t)4 * MAT + (size_t)NVEC * D + 64) * 4;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// shared vector slots
enum {
    V_UH, V_KH, V_PQ, V_PK, V_ZK, V_Z, V_AL, V_E, V_GO, V_O, V_GPQ, V_GE, V_GAL, V_GA, V_GKH, V_GZ, V_GUH, V_T0,
    V_T1, V_T2, V_T3, V_T4, V_T5, V_T6
};
// shared scalars
enum { X_NU, X_NK, X_DEN, X_DELTA, X_NA, X_R0, X_R1, X_R2, X_R3, X_R4, X_R5, X_R6, X_R7, X_NX };

// block-wide sum of one value per thread (every thread gets the result);
// `red` holds THREADS/32 floats; callers separate uses with __syncthreads
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) v += __shfl_xor_sync(0xffffffffu, v, h);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) s += red[i];
    return s;
}

__device__ __forceinline__ float phi_d(float x) { return x > 0.f ? 1.f : expf(x); }  // d phi / dx

template <int D, typename TIn>
__global__ void __launch_bounds__(BLay<D>::THREADS, 1)
    vla_backward_kernel(const Params p, const float* dO, const float* dST, const float* dAT, const float* dzkT,
                        float* dq, float* dk, float* dv, float* du, float* dS0, float* dA0, float* dzk0,
                        float* tape, float* ckpt) {
    using L = BLay<D>;
    constexpr int NT = L::THREADS, LD = L::LD;
    extern __shared__ __align__(16) float sh[];
    float* S = sh;
    float* A = S + L::MAT;
    float* gS = A + L::MAT;
    float* gA = gS + L::MAT;
    float* vec = gA + L::MAT;
    float* sx = vec + L::NVEC * D;   // scalars
    float* red = sx + 16;            // block reductions (NT / 32 <= 32 floats)
    auto V = [&](int slot) { return vec + slot * D; };

    const int tid = threadIdx.x, grp = tid / D, li = tid - grp * D;
    const int bh = blockIdx.x, T = p.T;
    const size_t hin = (size_t)bh * T * D;
    const TIn* gq = static_cast<const TIn*>(p.q) + hin;
    const TIn* gk = static_cast<const TIn*>(p.k) + hin;
    const TIn* gv = static_cast<const TIn*>(p.v) + hin;
    const TIn* gu = static_cast<const TIn*>(p.u) + hin;
    float* tp = tape + (size_t)bh * T * L::TREC;
    float* cp = ckpt + (size_t)bh * ((T + CK - 1) / CK + 1) * 2 * D * D;
    bool nonfinite = false;

    // ------------------------------------------------------------------
    // phase 1: forward with tape
    // ------------------------------------------------------------------
    for (int e = tid; e < D * D; e += NT) {
        const int i = e / D, j = e - i * D;
        A[i * LD + j] = p.A0 ? p.A0[(size_t)bh * D * D + e] : (i == j ? p.inv_lambda0 : 0.f);
        S[i * LD + j] = p.S0 ? p.S0[(size_t)bh * D * D + e] : 0.f;
    }
    if (tid < D) V(V_ZK)[tid] = p.zk0 ? p.zk0[(size_t)bh * D + tid] : 0.f;
    __syncthreads();
    for (int t = 0; t < T; ++t) {
        if (t % CK == 0) {
            float* c = cp + (size_t)(t / CK) * 2 * D * D;
            for (int e = tid; e < D * D; e += NT) {
                const int i = e / D, j = e - i * D;
                c[e] = S[i * LD + j];
                c[D * D + e] = A[i * LD + j];
            }
        }
        // inputs of the token; norms, phi, key sum and den (eq. 11)
        float nu = 0.f, nk = 0.f, pd = 0.f;
        if (tid < D) {
            const float uv = ld_in<TIn>(gu + (size_t)t * D, tid), kv = ld_in<TIn>(gk + (size_t)t * D, tid);
            const float qv = ld_in<TIn>(gq + (size_t)t * D, tid);
            nu = uv * uv;
            nk = kv * kv;
            const float zk = V(V_ZK)[tid] + phi(kv);
            V(V_ZK)[tid] = zk;
            const float pq = phi(qv);
            V(V_PQ)[tid] = pq;
            pd = pq * zk;
            V(V_T0)[tid] = uv;
            V(V_T1)[tid] = kv;
        }
        nu = block_sum<NT>(nu, red);
        nk = block_sum<NT>(nk, red);
        pd = block_sum<NT>(pd, red);
        const float iu = 1.f / fmaxf(sqrtf(nu), 1e-12f), ik = 1.f / fmaxf(sqrtf(nk), 1e-12f);
        if (tid < D) {
            V(V_UH)[tid] = V(V_T0)[tid] * iu;
            V(V_KH)[tid] = V(V_T1)[tid] * ik;
        }
        __syncthreads();
        // eq. 9: z = A u^ (rows), e = v - S k^ (rows; S_{t-1})
        if (grp == 0) {
            float s = 0.f;
            for (int j = 0; j < D; ++j) s = fmaf(A[li * LD + j], V(V_UH)[j], s);
            V(V_Z)[li] = s;
        } else if (grp == 1) {
            float s = 0.f;
            for (int j = 0; j < D; ++j) s = fmaf(S[li * LD + j], V(V_KH)[j], s);
            V(V_E)[li] = ld_in<TIn>(gv + (size_t)t * D, li) - s;
        }
        __syncthreads();
        const float delta = 1.f + block_sum<NT>(tid < D ? V(V_UH)[tid] * V(V_Z)[tid] : 0.f, red);
        const float rdl = 1.f / delta;
        for (int e = tid; e < D * D; e += NT) {
            const int i = e / D, j = e - i * D;
            A[i * LD + j] = fmaf(-V(V_Z)[i] * rdl, V(V_Z)[j], A[i * LD + j]);
        }
        __syncthreads();
        // eq. 10: a = A_t k^, alpha^ = a / ||a||, S_t = S_{t-1} + e alpha^^T
        if (grp == 0) {
            float s = 0.f;
            for (int j = 0; j < D; ++j) s = fmaf(A[li * LD + j], V(V_KH)[j], s);
            V(V_T2)[li] = s;
        }
        __syncthreads();
        const float na = sqrtf(block_sum<NT>(tid < D ? V(V_T2)[tid] * V(V_T2)[tid] : 0.f, red));
        const float ina = 1.f / fmaxf(na, 1e-12f);
        if (tid < D) V(V_AL)[tid] = V(V_T2)[tid] * ina;
        __syncthreads();
        for (int e = tid; e < D * D; e += NT) {
            const int i = e / D, j = e - i * D;
            S[i * LD + j] = fmaf(V(V_E)[i], V(V_AL)[j], S[i * LD + j]);
        }
        // tape
        float* r = tp + (size_t)t * L::TREC;
        if (tid < D) {
            r[tid] = V(V_Z)[tid];
            r[D + tid] = V(V_AL)[tid];
            r[2 * D + tid] = V(V_E)[tid];
        }
        if (tid == 0) {
            r[3 * D] = delta;
            r[3 * D + 1] = na;
            r[3 * D + 2] = pd < p.eps ? -p.eps : pd;
            if (!isfinite(delta) || !isfinite(na) || !isfinite(pd)) nonfinite = true;
        }
        __syncthreads();
    }

    // ------------------------------------------------------------------
    // phase 2: reverse sweep
    // ------------------------------------------------------------------
    for (int e = tid; e < D * D; e += NT) {
        const int i = e / D, j = e - i * D;
        const size_t g = (size_t)bh * D * D + e;
        gS[i * LD + j] = dST ? dST[g] : 0.f;
        gA[i * LD + j] = dAT ? dAT[g] : 0.f;
    }
    float gzk = 0.f;  // thread tid < D: dL/dz^key_t[tid]
    if (tid < D) gzk = dzkT ? dzkT[(size_t)bh * D + tid] : 0.f;
    __syncthreads();
    for (int t = T - 1; t >= 0; --t) {
        const float* r = tp + (size_t)t * L::TREC;
        float qv = 0.f, kv = 0.f, uv = 0.f;
        if (tid < D) {
            uv = ld_in<TIn>(gu + (size_t)t * D, tid);
            kv = ld_in<TIn>(gk + (size_t)t * D, tid);
            qv = ld_in<TIn>(gq + (size_t)t * D, tid);
            V(V_Z)[tid] = r[tid];
            V(V_AL)[tid] = r[D + tid];
            V(V_E)[tid] = r[2 * D + tid];
            V(V_PQ)[tid] = phi(qv);
            V(V_GO)[tid] = dO ? dO[((size_t)bh * T + t) * D + tid] : 0.f;
            V(V_T0)[tid] = uv;
            V(V_T1)[tid] = kv;
        }
        const float delta = r[3 * D], na = r[3 * D + 1], dsg = r[3 * D + 2];
        const bool clamped = dsg < 0.f;
        const float den = clamped ? -dsg : dsg;
        const float nu = block_sum<NT>(uv * uv, red), nk = block_sum<NT>(kv * kv, red);
        const float iu = 1.f / fmaxf(sqrtf(nu), 1e-12f), ik = 1.f / fmaxf(sqrtf(nk), 1e-12f);
        if (tid < D) {
            V(V_UH)[tid] = uv * iu;
            V(V_KH)[tid] = kv * ik;
        }
        __syncthreads();
        // round 1 (gS, gA are the adjoints of S_t, A_t before this token's terms):
        // o = S_t phi_q / den, S_t^T gO, gS alpha, gS^T e, gA z, gA^T z
        {
            const float* M;
            const float* x;
            bool col;
            int out;
            switch (grp) {
                case 0: M = S; x = V(V_PQ); col = false; out = V_O; break;
                case 1: M = S; x = V(V_GO); col = true; out = V_GPQ; break;
                case 2: M = gS; x = V(V_AL); col = false; out = V_GE; break;
                case 3: M = gS; x = V(V_E); col = true; out = V_GAL; break;
                case 4: M = gA; x = V(V_Z); col = false; out = V_T2; break;
                default: M = gA; x = V(V_Z); col = true; out = V_T3; break;
            }
            float s = 0.f;
            if (col) {
                for (int i = 0; i < D; ++i) s = fmaf(M[i * LD + li], x[i], s);
            } else {
                for (int j = 0; j < D; ++j) s = fmaf(M[li * LD + j], x[j], s);
            }
            V(out)[li] = s;
        }
        __syncthreads();
        // scalars of the adjoint step
        const float go_o = block_sum<NT>(tid < D ? V(V_GO)[tid] * V(V_O)[tid] : 0.f, red) / den;  // gO . o_t
        const float pq_al = block_sum<NT>(tid < D ? V(V_PQ)[tid] * V(V_AL)[tid] : 0.f, red);
        const float go_e = block_sum<NT>(tid < D ? V(V_GO)[tid] * V(V_E)[tid] : 0.f, red);
        const float gden = clamped ? 0.f : -go_o / den;
        if (tid < D) {
            // gS_t = gS + gO phi_q^T / den: its products with alpha and e
            V(V_GE)[tid] = fmaf(V(V_GO)[tid], pq_al / den, V(V_GE)[tid]);                    // g_e = gS_t alpha
            V(V_GAL)[tid] = fmaf(V(V_PQ)[tid], go_e / den, V(V_GAL)[tid]);                   // g_alpha = gS_t^T e
            V(V_GPQ)[tid] = fmaf(gden, V(V_ZK)[tid], V(V_GPQ)[tid] / den);                   // g_phiq
            gzk = fmaf(gden, V(V_PQ)[tid], gzk);
        }
        __syncthreads();
        const float al_gal = block_sum<NT>(tid < D ? V(V_AL)[tid] * V(V_GAL)[tid] : 0.f, red);
        const float e_ge = block_sum<NT>(tid < D ? V(V_E)[tid] * V(V_GE)[tid] : 0.f, red);
        const float ina = na < 1e-12f ? 1e12f : 1.f / na;
        if (tid < D)  // g_a = (g_alpha - alpha (alpha . g_alpha)) / ||a||
            V(V_GA)[tid] = (na < 1e-12f ? V(V_GAL)[tid] : fmaf(-V(V_AL)[tid], al_gal, V(V_GAL)[tid])) * ina;
        __syncthreads();
        // round 2: S_t^T g_e (then S_{t-1}^T g_e = S_t^T g_e - alpha (e . g_e)), A_t^T g_a
        if (grp == 0) {
            float s = 0.f;
            for (int i = 0; i < D; ++i) s = fmaf(S[i * LD + li], V(V_GE)[i], s);
            V(V_T4)[li] = s;
        } else if (grp == 1) {
            float s = 0.f;
            for (int i = 0; i < D; ++i) s = fmaf(A[i * LD + li], V(V_GA)[i], s);
            V(V_T5)[li] = s;
        }
        __syncthreads();
        // g_k^ = -S_{t-1}^T g_e + A_t^T g_a; the A adjoint now includes g_a k^^T:
        // (gA + g_a k^^T) z and its transpose product, z^T gA z
        const float kz = block_sum<NT>(tid < D ? V(V_KH)[tid] * V(V_Z)[tid] : 0.f, red);
        const float az = block_sum<NT>(tid < D ? V(V_GA)[tid] * V(V_Z)[tid] : 0.f, red);
        const float zgz0 = block_sum<NT>(tid < D ? V(V_Z)[tid] * V(V_T2)[tid] : 0.f, red);
        if (tid < D) {
            V(V_GKH)[tid] = -fmaf(-V(V_AL)[tid], e_ge, V(V_T4)[tid]) + V(V_T5)[tid];
            const float gaz = fmaf(V(V_GA)[tid], kz, V(V_T2)[tid]);   // (gA + g_a k^^T) z
            const float gatz = fmaf(V(V_KH)[tid], az, V(V_T3)[tid]);  // (gA + g_a k^^T)^T z
            V(V_GZ)[tid] = -(gaz + gatz) / delta;
        }
        const float zgz = fmaf(az, kz, zgz0);
        const float gdelta = zgz / (delta * delta);
        __syncthreads();
        if (tid < D) V(V_GZ)[tid] = fmaf(gdelta, V(V_UH)[tid], V(V_GZ)[tid]);
        __syncthreads();
        // round 3: A_t^T g_z (A_{t-1}^T g_z = A_t^T g_z + z (z . g_z) / delta)
        if (grp == 0) {
            float s = 0.f;
            for (int i = 0; i < D; ++i) s = fmaf(A[i * LD + li], V(V_GZ)[i], s);
            V(V_T6)[li] = s;
        }
        __syncthreads();
        const float zgzz = block_sum<NT>(tid < D ? V(V_Z)[tid] * V(V_GZ)[tid] : 0.f, red);
        if (tid < D) V(V_GUH)[tid] = fmaf(gdelta, V(V_Z)[tid], fmaf(V(V_Z)[tid], zgzz / delta, V(V_T6)[tid]));
        __syncthreads();
        // gradients of the token's inputs
        const float ugu = block_sum<NT>(tid < D ? V(V_UH)[tid] * V(V_GUH)[tid] : 0.f, red);
        const float kgk = block_sum<NT>(tid < D ? V(V_KH)[tid] * V(V_GKH)[tid] : 0.f, red);
        if (tid < D) {
            const size_t o = ((size_t)bh * T + t) * D + tid;
            const float dut = nu < 1e-24f ? V(V_GUH)[tid] * 1e12f : fmaf(-V(V_UH)[tid], ugu, V(V_GUH)[tid]) * iu;
            const float dkt = nk < 1e-24f ? V(V_GKH)[tid] * 1e12f : fmaf(-V(V_KH)[tid], kgk, V(V_GKH)[tid]) * ik;
            du[o] = dut;
            dk[o] = fmaf(gzk, phi_d(kv), dkt);
            dq[o] = V(V_GPQ)[tid] * phi_d(qv);
            dv[o] = V(V_GE)[tid];
            if (!isfinite(dut) || !isfinite(dk[o]) || !isfinite(dq[o]) || !isfinite(dv[o])) nonfinite = true;
            // z^key_{t-1} = z^key_t - phi(k_t)
            V(V_ZK)[tid] -= phi(kv);
        }
        // adjoints of S_{t-1}, A_{t-1}; states S_{t-1}, A_{t-1}
        //   gS += gO phi_q^T / den - g_e k^^T;  gA += g_a k^^T + g_z u^^T
        //   S_{t-1} = S_t - e alpha^^T;  A_{t-1} = A_t + z z^T / delta
        const bool reload = (t % CK == 0);
        const float rden = 1.f / den, rdl = 1.f / delta;
        const float* c = cp + (size_t)(t / CK) * 2 * D * D;
        for (int e = tid; e < D * D; e += NT) {
            const int i = e / D, j = e - i * D;
            const int x = i * LD + j;
            gS[x] = fmaf(V(V_GO)[i] * rden, V(V_PQ)[j], fmaf(-V(V_GE)[i], V(V_KH)[j], gS[x]));
            gA[x] = fmaf(V(V_GA)[i], V(V_KH)[j], fmaf(V(V_GZ)[i], V(V_UH)[j], gA[x]));
            if (reload) {
                S[x] = c[e];
                A[x] = c[D * D + e];
            } else {
                S[x] = fmaf(-V(V_E)[i], V(V_AL)[j], S[x]);
                A[x] = fmaf(V(V_Z)[i] * rdl, V(V_Z)[j], A[x]);
            }
        }
        __syncthreads();
    }
    for (int e = tid; e < D * D; e += NT) {
        const int i = e / D, j = e - i * D;
        const size_t g = (size_t)bh * D * D + e;
        if (dS0) dS0[g] = gS[i * LD + j];
        if (dA0) dA0[g] = gA[i * LD + j];
    }
    if (tid < D && dzk0) dzk0[(size_t)bh * D + tid] = gzk;
    if (nonfinite) record_failure(p.status, BIT_NONFINITE, ROLE_S, bh, -1);
}

}  // namespace bw
