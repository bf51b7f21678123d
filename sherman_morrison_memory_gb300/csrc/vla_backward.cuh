// vla_backward.cuh -- reverse-mode gradient of the VLA forward recurrence
// ("Variational Linear Attention", arXiv 2605.11196, §3.3 eq. 9-11; the state
// Jacobian of §4.2 eq. 14 is the adjoint step of the S recurrence below).
// Included by vla_forward.cu inside namespace vla.
//
// The forward pass runs first, on the chunked tensor-core kernels in their
// TAPE mode (vla_tc.cuh for d <= 96, vla_tc2.cuh for d = 128): they write a
// tape to the workspace (per token z_t (eq. 9), alpha^_t and ||a_t|| (eq. 10),
// e_t (eq. 10), delta_t, den_t (eq. 11), ||u_t||^2, ||k_t||^2), S, A and
// z^key every CK tokens, and the final state. Then one CTA per (b, h) runs
// the reverse sweep t = T-1 .. 0, applying the adjoint of each step of
// eq. 9-11 in reverse order. S_{t-1} and A_{t-1} are rebuilt from S_t, A_t by
// undoing the step's rank-1 update (S_{t-1} = S_t - e alpha^^T,
// A_{t-1} = A_t + z z^T / delta) and reloaded from the checkpoint every CK
// tokens.
//
// S, A and the adjoints dL/dS, dL/dA stay in registers for the whole kernel:
// warp w owns rows 8w .. 8w+7 and lane l owns columns l, l+32, .. of each.
// A row product M x is a lane-local partial sum reduced across the warp by a
// halving exchange (9 shuffles for 8 rows); a column product M^T x is a
// warp-local partial sum reduced across warps through shared memory. Dot
// products of d-vectors are recomputed by every warp (butterfly shuffles)
// instead of block-wide reductions. Per token the sweep needs two block
// barriers. Token inputs and the tape are prefetched 3 tokens ahead into a
// shared-memory ring with cp.async.
//
// Identities that save a product per reverse step (A is symmetric):
//   A_t u^ = z / delta,  A_t k^ = alpha^ ||a||,  A_{t-1} g = A_t g + z (z.g) / delta,
// so the reverse step has two passes of matrix-vector products, not three.

namespace bw {

constexpr int CK = 64;  // checkpoint interval (tokens)

template <int D, typename TIn>
struct BLay {
    static constexpr int RW = 8;                // rows per warp
    static constexpr int NW = D / RW;           // warps
    static constexpr int THREADS = 32 * NW;     // 384 at d = 96
    static constexpr int CL = D / 32;           // columns per lane: j = lane + 32 c
    // tape per token: z | alpha^ | e (D each), then delta, ||a||, den (signed:
    // negative = the eps floor was taken), ||u||^2, ||k||^2, 3 unused
    static constexpr int TREC = 3 * D + 8;
    static constexpr int CREC = 2 * D * D + D;  // checkpoint: S | A | z^key
    static constexpr int NB2 = 5;               // reverse ring depth (prefetch 3 tokens ahead, 1 slot in use
                                                // by the deferred k/u gradients of the previous token)
    // ring slot (bytes): raw u | k | q (TIn), then dL/do (fp32), then the tape
    // record
    static constexpr int IN_B = D * (int)sizeof(TIn);
    static constexpr int U = 0, K = IN_B, Q = 2 * IN_B, G = 3 * IN_B, TP = 3 * IN_B + 4 * D;
    static constexpr int SLOT_B = TP + 4 * TREC;
    // shared memory (bytes)
    static constexpr int RING = 0;
    static constexpr int P1 = RING + NB2 * SLOT_B;    // pass-1 column partials [NW][3][D]
    static constexpr int C1 = P1 + NW * 3 * D * 4;    // their sums [3][D]
    static constexpr int R1 = C1 + 3 * D * 4;         // pass-1 row products [2 parities][2][D]
    static constexpr int P2 = R1 + 2 * 2 * D * 4;     // pass-2 column partials [NW][D]
    static constexpr int R2 = P2 + NW * D * 4;        // pass-2 row products [2][D]
    static constexpr int DP = R2 + 2 * D * 4;         // per-warp dot partials [4][NW]
    static constexpr int DS = DP + 4 * NW * 4;        // their sums [4]
    static constexpr int RED = DS + 4 * 4;            // [D/32 warps][2] dot partials of the k/u gradients
    static constexpr int SMEM = RED + 8 * 4;
    static_assert(D % 32 == 0 && D <= 96, "register tiles hold 8 rows x d/32 columns of each of four d x d matrices");
    static_assert(SLOT_B % 16 == 0 && IN_B % 16 == 0, "cp.async chunks");
    static_assert(3 * IN_B / 16 + D / 4 + TREC / 4 <= THREADS, "one prefetch chunk per thread");
    static_assert(NW - 3 * CL == CL, "the warps left over by the column sums are d/32");
};

__device__ __forceinline__ float phi_d(float x) { return x > 0.f ? 1.f : expf(x); }  // d phi / dx

__device__ __forceinline__ float rcpa(float x) {  // 1/x, approximate (1 ulp)
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float inv_norm(float n2) { return fminf(rsqrtf(n2), 1e12f); }  // 1 / max(sqrt(n2), 1e-12)

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// element j of a TIn row held in shared memory, as float
template <typename TIn>
__device__ __forceinline__ float lds_in(const unsigned char* base, int j);
template <>
__device__ __forceinline__ float lds_in<float>(const unsigned char* base, int j) {
    return reinterpret_cast<const float*>(base)[j];
}
template <>
__device__ __forceinline__ float lds_in<__nv_bfloat16>(const unsigned char* base, int j) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[j]);
}

// elements r0 .. r0+7 of a row in shared memory (r0 a multiple of 8): one or
// two 16-byte broadcast loads
template <typename TIn>
__device__ __forceinline__ void lds8(const unsigned char* base, int r0, float (&x)[8]);
template <>
__device__ __forceinline__ void lds8<float>(const unsigned char* base, int r0, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(base)[r0 / 4];
    const float4 b = reinterpret_cast<const float4*>(base)[r0 / 4 + 1];
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
template <>
__device__ __forceinline__ void lds8<__nv_bfloat16>(const unsigned char* base, int r0, float (&x)[8]) {
    const uint4 a = reinterpret_cast<const uint4*>(base)[r0 / 8];
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void lds8f(const float* base, int r0, float (&x)[8]) {
    lds8<float>(reinterpret_cast<const unsigned char*>(base), r0, x);
}

// Row sums of a warp's 8 rows: p[r] is this lane's partial sum for row r.
// Returns the full sum of row (lane >> 2); each row ends in 4 lanes.
__device__ __forceinline__ float rowsum8(const float (&p)[8]) {
    const int l = threadIdx.x & 31;
    const bool b4 = l & 16, b3 = l & 8, b2 = l & 4;
    float q[4], r[2];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float send = b4 ? p[m] : p[m + 4];
        const float keep = b4 ? p[m + 4] : p[m];
        q[m] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const float send = b3 ? q[m] : q[m + 2];
        const float keep = b3 ? q[m + 2] : q[m];
        r[m] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? r[0] : r[1];
    float s = (b2 ? r[1] : r[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    return s;
}

// (x, x), and rows r, r+1 of an 8-row register tile, as packed FMA operands
// (the d x d tiles hold rows r0 + 2 rp and r0 + 2 rp + 1 in one float2)
__device__ __forceinline__ float2 dup2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 pair2(const float (&x)[8], int r) { return make_float2(x[r], x[r + 1]); }

// x[c] for the warp-uniform column index c < N, without local memory
template <int N>
__device__ __forceinline__ float pick(const float (&x)[N], int c) {
    float v = x[0];
#pragma unroll
    for (int i = 1; i < N; ++i) v = c == i ? x[i] : v;
    return v;
}

template <int D, typename TIn>
__device__ __forceinline__ void prefetch_rev(unsigned char* slot, const TIn* gu, const TIn* gk, const TIn* gq,
                                             const float* go, const float* tp, int t) {
    using L = BLay<D, TIn>;
    constexpr int NC = L::IN_B / 16, NG = D / 4, NR = L::TREC / 4;
    const int tid = threadIdx.x;
    if (tid < 3 * NC) {
        const int part = tid / NC, off = tid - part * NC;
        const TIn* src = part == 0 ? gu : part == 1 ? gk : gq;
        cp_async16(slot + part * L::IN_B + off * 16,
                   reinterpret_cast<const unsigned char*>(src + (size_t)t * D) + off * 16);
    } else if (tid < 3 * NC + NG) {
        const int off = tid - 3 * NC;
        if (go) cp_async16(slot + L::G + off * 16, go + (size_t)t * D + off * 4);
    } else if (tid < 3 * NC + NG + NR) {
        const int off = tid - 3 * NC - NG;
        cp_async16(slot + L::TP + off * 16, tp + (size_t)t * L::TREC + off * 4);
    }
}

// dL/dk_t and dL/du_t (column j = 32 jw + lane) from the pass-2 products of
// token t (P2, R2) and its scalars; run by the d/32 warps that the column sums
// of the next step leave free. Returns fma(gradients, 0): 0 unless one is NaN
// or Inf (branch-free, like every per-element check of the sweep).
template <int D, typename TIn>
__device__ __forceinline__ float ku_grads(const unsigned char* sl, const float* P2, const float* R2, float* RED,
                                         int jw, float gzk, float e_ge, float kz, float gdl, float zgz, float az,
                                         float nac, float dl, float nu, float nk, float* dk, float* du) {
    using L = BLay<D, TIn>;
    const int l = threadIdx.x & 31, j = 32 * jw + l;
    const float* rec = reinterpret_cast<const float*>(sl + L::TP);
    float st = 0.f;
#pragma unroll
    for (int v = 0; v < L::NW; ++v) st += P2[v * D + j];
    const float aga = R2[j], aw1 = R2[D + j];
    const float zj = rec[j], alj = rec[D + j];
    const float kj = lds_in<TIn>(sl + L::K, j);
    const float iu = inv_norm(nu), ik = inv_norm(nk), rdl = rcpa(dl);
    const float khj = kj * ik, uhj = lds_in<TIn>(sl + L::U, j) * iu;
    const float gkh = aga - fmaf(-alj, e_ge, st);                                          // A_t g_a - S_{t-1}^T g_e
    const float atgz = fmaf(gdl * rdl, zj, -(aw1 + fmaf(aga, kz, alj * nac * az)) * rdl);  // A_t g_z
    const float zgzf = -zgz * (dl + 1.f) * rdl * rdl;                                      // z . g_z
    const float guh = fmaf(zj, fmaf(zgzf, rdl, gdl), atgz);                                // A_{t-1} g_z + g_delta z
    float d2[2] = {uhj * guh, khj * gkh};
    allreduce<2, 16>(d2);
    if (l == 0) {
        RED[2 * jw] = d2[0];
        RED[2 * jw + 1] = d2[1];
    }
    named_bar(1, D);
    float ugu = 0.f, kgk = 0.f;
#pragma unroll
    for (int v = 0; v < L::CL; ++v) {
        ugu += RED[2 * v];
        kgk += RED[2 * v + 1];
    }
    const float dut = nu < 1e-24f ? guh * 1e12f : fmaf(-uhj, ugu, guh) * iu;
    const float dkt = fmaf(gzk, phi_d(kj), nk < 1e-24f ? gkh * 1e12f : fmaf(-khj, kgk, gkh) * ik);
    du[j] = dut;
    dk[j] = dkt;
    return fmaf(dut, 0.f, dkt * 0.f);
}

// The reverse sweep (four d x d matrices in registers: d <= 96). fin: the
// forward's final S [B*H, d, d] | A [B*H, d, d] | z^key [B*H, d], or NULL for
// T = 0 (the sweep then starts and ends at the initial state).
template <int D, typename TIn>
__global__ void __launch_bounds__(BLay<D, TIn>::THREADS, 1)
    vla_backward_kernel(const Params p, const float* dO, const float* dST, const float* dAT, const float* dzkT,
                        float* dq, float* dk, float* dv, float* du, float* dS0, float* dA0, float* dzk0,
                        float* tape, float* ckpt, const float* fin) {
    using L = BLay<D, TIn>;
    constexpr int RW = L::RW, CL = L::CL, NW = L::NW, NB2 = L::NB2;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* ring = smem + L::RING;
    float* P1 = reinterpret_cast<float*>(smem + L::P1);
    float* C1 = reinterpret_cast<float*>(smem + L::C1);
    float* R1 = reinterpret_cast<float*>(smem + L::R1);
    float* P2 = reinterpret_cast<float*>(smem + L::P2);
    float* R2 = reinterpret_cast<float*>(smem + L::R2);
    float* DP = reinterpret_cast<float*>(smem + L::DP);
    float* DS = reinterpret_cast<float*>(smem + L::DS);
    float* RED = reinterpret_cast<float*>(smem + L::RED);

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int r0 = w * RW;           // first row owned by this warp
    const int rr = r0 + (l >> 2);    // the row whose sums rowsum8 leaves in this lane
    const int bh = blockIdx.x, T = p.T;
    const size_t hin = (size_t)bh * T * D, hdd = (size_t)bh * D * D;
    const TIn* gq = static_cast<const TIn*>(p.q) + hin;
    const TIn* gk = static_cast<const TIn*>(p.k) + hin;
    const TIn* gu = static_cast<const TIn*>(p.u) + hin;
    const float* go_h = dO ? dO + hin : nullptr;
    float* tp = tape + (size_t)bh * T * L::TREC;
    float* cp = ckpt + (size_t)bh * ((T + CK - 1) / CK + 1) * L::CREC;
    float gchk = 0.f;  // fma(gradient, 0, .) of every gradient written: 0 unless one is NaN or Inf

    // S, A (and gS, gA below): rows r0 + 2 rp (.x) and r0 + 2 rp + 1 (.y),
    // columns l + 32 c, updated by packed FP32 FMAs (two rows per instruction)
    float2 S2[RW / 2][CL], A2[RW / 2][CL];
    float zk[CL];
    auto a0 = [&](int i, int j) { return p.A0 ? p.A0[hdd + i * D + j] : (i == j ? p.inv_lambda0 : 0.f); };
    auto s0 = [&](int i, int j) { return p.S0 ? p.S0[hdd + i * D + j] : 0.f; };
#pragma unroll
    for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const int i = r0 + 2 * rp, j = l + 32 * c;
            A2[rp][c] = make_float2(a0(i, j), a0(i + 1, j));
            S2[rp][c] = make_float2(s0(i, j), s0(i + 1, j));
        }
#pragma unroll
    for (int c = 0; c < CL; ++c) zk[c] = p.zk0 ? p.zk0[(size_t)bh * D + l + 32 * c] : 0.f;

    // the forward kernel (the chunked tensor-core kernel with its tape) has
    // written the tape, the checkpoints and its final state to `fin`
    if (fin) {
        const size_t BH = gridDim.x;
#pragma unroll
        for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                const size_t e = hdd + (size_t)(r0 + 2 * rp) * D + l + 32 * c;
                S2[rp][c] = make_float2(fin[e], fin[e + D]);
                A2[rp][c] = make_float2(fin[BH * D * D + e], fin[BH * D * D + e + D]);
            }
#pragma unroll
        for (int c = 0; c < CL; ++c) zk[c] = fin[2 * BH * D * D + (size_t)bh * D + l + 32 * c];
    }

    // ------------------------------------------------------------------
    // reverse sweep
    // ------------------------------------------------------------------
    cp_wait<0>();
    __syncthreads();  // ring free, tape visible to the whole CTA
    float2 gS2[RW / 2][CL], gA2[RW / 2][CL];
    float gzk[CL];
#pragma unroll
    for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const size_t e = hdd + (r0 + 2 * rp) * D + l + 32 * c;
            gS2[rp][c] = dST ? make_float2(dST[e], dST[e + D]) : dup2(0.f);
            gA2[rp][c] = dAT ? make_float2(dAT[e], dAT[e + D]) : dup2(0.f);
        }
#pragma unroll
    for (int c = 0; c < CL; ++c) gzk[c] = dzkT ? dzkT[(size_t)bh * D + l + 32 * c] : 0.f;
    if (!dO)
        for (int i = tid; i < NB2 * D; i += L::THREADS)
            reinterpret_cast<float*>(ring + (i / D) * L::SLOT_B + L::G)[i % D] = 0.f;
    for (int s = 0; s < 3; ++s) {
        const int tok = T - 1 - s;
        if (tok >= 0) prefetch_rev<D, TIn>(ring + (tok % NB2) * L::SLOT_B, gu, gk, gq, go_h, tp, tok);
        cp_commit();
    }
    cp_wait<1>();
    __syncthreads();
    const bool ku_warp = w >= NW - CL;  // the warps that compute dL/dk, dL/du
    const int jw = w - (NW - CL);
    // scalars of the token whose k/u gradients are pending
    float j_ege = 0.f, j_kz = 0.f, j_gdl = 0.f, j_zgz = 0.f, j_az = 0.f, j_nac = 1.f, j_dl = 1.f, j_nu = 1.f,
          j_nk = 1.f;
    for (int t = T - 1; t >= 0; --t) {
        const unsigned char* sl = ring + (t % NB2) * L::SLOT_B;
        const float* rec = reinterpret_cast<const float*>(sl + L::TP);
        const float* gov = reinterpret_cast<const float*>(sl + L::G);
        float* r1 = R1 + (t & 1) * 2 * D;
        const float dl = rec[3 * D], na = rec[3 * D + 1], dsg = rec[3 * D + 2];
        const float nu = rec[3 * D + 3], nk = rec[3 * D + 4];
        const bool clamped = dsg < 0.f;
        const float rden = rcpa(clamped ? -dsg : dsg), rdl = rcpa(dl);
        const float iu = inv_norm(nu), ik = inv_norm(nk);
        const bool tiny = na < 1e-12f;
        const float nac = fmaxf(na, 1e-12f), ina = rcpa(nac);
        const size_t orow = ((size_t)bh * T + t) * D;

        // this lane's columns
        float uh[CL], kh[CL], pq[CL], zc[CL], al[CL];
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const int j = l + 32 * c;
            uh[c] = lds_in<TIn>(sl + L::U, j) * iu;
            kh[c] = lds_in<TIn>(sl + L::K, j) * ik;
            pq[c] = phi(lds_in<TIn>(sl + L::Q, j));
            zc[c] = rec[j];
            al[c] = rec[D + j];
        }
        // product pass 1 (gS, gA: adjoints of S_t, A_t before this token's terms)
        //   rows: gS alpha^, gA z;  columns: gS^T e, S_t^T dL/do, gA^T z
        {
            float pg[RW], pz[RW];
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp) {
                float2 ag = dup2(0.f), az2 = dup2(0.f);
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    ag = __ffma2_rn(gS2[rp][c], dup2(al[c]), ag);
                    az2 = __ffma2_rn(gA2[rp][c], dup2(zc[c]), az2);
                }
                pg[2 * rp] = ag.x;
                pg[2 * rp + 1] = ag.y;
                pz[2 * rp] = az2.x;
                pz[2 * rp + 1] = az2.y;
            }
            const float gsal = rowsum8(pg), gaz = rowsum8(pz);
            if ((l & 3) == 0) {
                r1[rr] = gsal;
                r1[D + rr] = gaz;
            }
        }
        // token dots and this warp's share of the dots of the column products:
        // phi_q.alpha^, dL/do.e, k^.z, phi_q.z, alpha^.z | phi_q.S^T gO, alpha^.gS^T e
        // (= e.gS alpha^), z.gS^T e, z.gA^T z
        float d9[9] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        {
            float er[RW], gor[RW], zr[RW], qe[CL], qo[CL], qz[CL];
            lds8f(rec + 2 * D, r0, er);
            lds8f(gov, r0, gor);
            lds8f(rec, r0, zr);
            {
                float2 qe2[CL], qo2[CL], qz2[CL];
#pragma unroll
                for (int c = 0; c < CL; ++c) qe2[c] = qo2[c] = qz2[c] = dup2(0.f);
#pragma unroll
                for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
                    for (int c = 0; c < CL; ++c) {
                        qe2[c] = __ffma2_rn(gS2[rp][c], pair2(er, 2 * rp), qe2[c]);
                        qo2[c] = __ffma2_rn(S2[rp][c], pair2(gor, 2 * rp), qo2[c]);
                        qz2[c] = __ffma2_rn(gA2[rp][c], pair2(zr, 2 * rp), qz2[c]);
                    }
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    qe[c] = qe2[c].x + qe2[c].y;
                    qo[c] = qo2[c].x + qo2[c].y;
                    qz[c] = qz2[c].x + qz2[c].y;
                }
            }
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                const int j = l + 32 * c;
                P1[(w * 3 + 0) * D + j] = qe[c];
                P1[(w * 3 + 1) * D + j] = qo[c];
                P1[(w * 3 + 2) * D + j] = qz[c];
                d9[0] = fmaf(pq[c], al[c], d9[0]);
                d9[1] = fmaf(gov[j], rec[2 * D + j], d9[1]);
                d9[2] = fmaf(kh[c], zc[c], d9[2]);
                d9[3] = fmaf(pq[c], zc[c], d9[3]);
                d9[4] = fmaf(al[c], zc[c], d9[4]);
                d9[5] = fmaf(pq[c], qo[c], d9[5]);
                d9[6] = fmaf(al[c], qe[c], d9[6]);
                d9[7] = fmaf(zc[c], qe[c], d9[7]);
                d9[8] = fmaf(zc[c], qz[c], d9[8]);
            }
        }
        allreduce<5, 16>(d9);             // token dots: every lane needs them
        reduce_scatter<4, 16>(d9 + 5, l);  // this warp's shares: one lane per dot writes it
        {
            const int x = rs_index<4, 16>(l, 0);
            if (x >= 0) DP[x * NW + w] = d9[5];
        }
        cp_wait<1>();
        __syncthreads();  // B1 (also publishes token t-1's slot)
        // the slot of token t+2 is free: prefetch token t-3 into it
        if (t >= 3) prefetch_rev<D, TIn>(ring + ((t - 3) % NB2) * L::SLOT_B, gu, gk, gq, go_h, tp, t - 3);
        cp_commit();
        if (tid < 3 * D) {
            const int x = tid / D, j = tid - x * D;
            float s = 0.f;
#pragma unroll
            for (int v = 0; v < NW; ++v) s += P1[(v * 3 + x) * D + j];
            C1[x * D + j] = s;
        } else {
            if (w == NW - 1 && l < 4) {
                float s = 0.f;
#pragma unroll
                for (int v = 0; v < NW; ++v) s += DP[l * NW + v];
                DS[l] = s;
            }
            if (t + 1 < T) {  // dL/dk, dL/du of token t+1
                gchk += ku_grads<D, TIn>(ring + ((t + 1) % NB2) * L::SLOT_B, P2, R2, RED, jw, pick<CL>(gzk, jw),
                                         j_ege, j_kz, j_gdl, j_zgz, j_az, j_nac, j_dl, j_nu, j_nk,
                                         dk + orow + D, du + orow + D);
            }
        }
        __syncthreads();  // B2

        // scalars of the adjoint step
        const float c1n = d9[0], c2n = d9[1], kz = d9[2];
        const float c1 = c1n * rden, c2 = c2n * rden;
        const float s_o = DS[0], s_ae = DS[1], s_ze = DS[2], s_zz = DS[3];
        const float gden = clamped ? 0.f : -s_o * rden * rden;     // -(dL/do . o) / den
        const float al_gal = fmaf(c2, c1n, s_ae);                   // alpha^ . g_alpha
        const float e_ge = fmaf(c1, c2n, s_ae);                     // e . g_e
        const float galz = fmaf(c2, d9[3], s_ze);                   // g_alpha . z
        const float az = (tiny ? galz : fmaf(-al_gal, d9[4], galz)) * ina;  // g_a . z
        const float zgz = fmaf(az, kz, s_zz);                       // z^T (gA + g_a k^^T) z
        const float gdl = zgz * rdl * rdl;                          // dL/d delta
        // columns: g_a, w1 = (gA + gA^T) z, g_z, dL/dphi_q
        float gac[CL], w1c[CL], gzc[CL];
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const int j = l + 32 * c;
            const float gal = fmaf(pq[c], c2, C1[j]);
            gac[c] = (tiny ? gal : fmaf(-al[c], al_gal, gal)) * ina;
            w1c[c] = r1[D + j] + C1[2 * D + j];
            // g_z = -((gA + g_a k^^T) z + (gA + g_a k^^T)^T z) / delta + g_delta u^
            gzc[c] = fmaf(gdl, uh[c], -(w1c[c] + fmaf(gac[c], kz, kh[c] * az)) * rdl);
            const float gpq = fmaf(gden, zk[c], C1[D + j] * rden);
            gzk[c] = fmaf(gden, pq[c], gzk[c]);
            if (w == 0) {
                const float x = gpq * phi_d(lds_in<TIn>(sl + L::Q, j));
                dq[orow + j] = x;
                gchk = fmaf(x, 0.f, gchk);
            }
        }
        // rows: g_e
        float ger[RW];
        {
            float a8[RW], b8[RW];
            lds8f(r1, r0, a8);   // gS alpha^
            lds8f(gov, r0, b8);  // dL/do
#pragma unroll
            for (int r = 0; r < RW; ++r) ger[r] = fmaf(b8[r], c1, a8[r]);
        }
        if (l < RW) {
            const float x = pick<RW>(ger, l);
            dv[orow + r0 + l] = x;
            gchk = fmaf(x, 0.f, gchk);
        }
        // product pass 2: columns S_t^T g_e; rows A_t g_a, A_t w1
        {
            float pa[RW], pw[RW];
            float2 qg2[CL];
#pragma unroll
            for (int c = 0; c < CL; ++c) qg2[c] = dup2(0.f);
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp) {
                float2 a2 = dup2(0.f), w2 = dup2(0.f);
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    qg2[c] = __ffma2_rn(S2[rp][c], pair2(ger, 2 * rp), qg2[c]);
                    a2 = __ffma2_rn(A2[rp][c], dup2(gac[c]), a2);
                    w2 = __ffma2_rn(A2[rp][c], dup2(w1c[c]), w2);
                }
                pa[2 * rp] = a2.x;
                pa[2 * rp + 1] = a2.y;
                pw[2 * rp] = w2.x;
                pw[2 * rp + 1] = w2.y;
            }
            const float aga = rowsum8(pa), aw1 = rowsum8(pw);
            if ((l & 3) == 0) {
                R2[rr] = aga;
                R2[D + rr] = aw1;
            }
#pragma unroll
            for (int c = 0; c < CL; ++c) P2[w * D + l + 32 * c] = qg2[c].x + qg2[c].y;
        }
        // adjoints of S_{t-1}, A_{t-1}:
        //   gS += dL/do phi_q^T / den - g_e k^^T;  gA += g_a k^^T + g_z u^^T
        {
            float gor[RW];
            lds8f(gov, r0, gor);
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp) {
                const float2 gs = make_float2(gor[2 * rp] * rden, gor[2 * rp + 1] * rden);
                const float2 mg = make_float2(-ger[2 * rp], -ger[2 * rp + 1]);
#pragma unroll
                for (int c = 0; c < CL; ++c)
                    gS2[rp][c] = __ffma2_rn(gs, dup2(pq[c]), __ffma2_rn(mg, dup2(kh[c]), gS2[rp][c]));
            }
        }
        {
            // this warp's rows of g_a and g_z: rows r0 .. r0+7 are columns held by
            // lanes (r0 mod 32) .. +7 in slot r0 / 32
            const int cs = r0 >> 5, lb = r0 & 31;
            const float ga_s = pick<CL>(gac, cs), gz_s = pick<CL>(gzc, cs);
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp) {
                const float2 gar = make_float2(__shfl_sync(FULL, ga_s, lb + 2 * rp), __shfl_sync(FULL, ga_s, lb + 2 * rp + 1));
                const float2 gzr = make_float2(__shfl_sync(FULL, gz_s, lb + 2 * rp), __shfl_sync(FULL, gz_s, lb + 2 * rp + 1));
#pragma unroll
                for (int c = 0; c < CL; ++c)
                    gA2[rp][c] = __ffma2_rn(gar, dup2(kh[c]), __ffma2_rn(gzr, dup2(uh[c]), gA2[rp][c]));
            }
        }
        // states before the token: S_{t-1} = S_t - e alpha^^T, A_{t-1} = A_t + z z^T / delta,
        // z^key_{t-1} = z^key_t - phi(k_t); exact copies at checkpoints
        if (t % CK == 0) {
            const float* c = cp + (size_t)(t / CK) * L::CREC;
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
                for (int cc = 0; cc < CL; ++cc) {
                    const int e = (r0 + 2 * rp) * D + l + 32 * cc;
                    S2[rp][cc] = make_float2(c[e], c[e + D]);
                    A2[rp][cc] = make_float2(c[D * D + e], c[D * D + e + D]);
                }
#pragma unroll
            for (int cc = 0; cc < CL; ++cc) zk[cc] = c[2 * D * D + l + 32 * cc];
        } else {
            float er[RW], zr[RW];
            lds8f(rec + 2 * D, r0, er);
            lds8f(rec, r0, zr);
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp) {
                const float2 zs = make_float2(zr[2 * rp] * rdl, zr[2 * rp + 1] * rdl);
                const float2 me = make_float2(-er[2 * rp], -er[2 * rp + 1]);
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    S2[rp][c] = __ffma2_rn(me, dup2(al[c]), S2[rp][c]);
                    A2[rp][c] = __ffma2_rn(zs, dup2(zc[c]), A2[rp][c]);
                }
            }
#pragma unroll
            for (int c = 0; c < CL; ++c) zk[c] -= phi(lds_in<TIn>(sl + L::K, l + 32 * c));
        }
        j_ege = e_ge, j_kz = kz, j_gdl = gdl, j_zgz = zgz, j_az = az, j_nac = nac, j_dl = dl, j_nu = nu, j_nk = nk;
    }
    __syncthreads();  // pass-2 products of token 0 visible
    if (T > 0 && ku_warp) {
        gchk += ku_grads<D, TIn>(ring, P2, R2, RED, jw, pick<CL>(gzk, jw), j_ege, j_kz, j_gdl, j_zgz, j_az, j_nac,
                                 j_dl, j_nu, j_nk, dk + (size_t)bh * T * D, du + (size_t)bh * T * D);
    }
#pragma unroll
    for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const size_t e = hdd + (r0 + 2 * rp) * D + l + 32 * c;
            if (dS0) {
                dS0[e] = gS2[rp][c].x;
                dS0[e + D] = gS2[rp][c].y;
            }
            if (dA0) {
                dA0[e] = gA2[rp][c].x;
                dA0[e + D] = gA2[rp][c].y;
            }
        }
    if (w == 0 && dzk0)
#pragma unroll
        for (int c = 0; c < CL; ++c) dzk0[(size_t)bh * D + l + 32 * c] = gzk[c];
    if (gchk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_S, bh, -1);
}

}  // namespace bw
