// vla_backward_split.cuh -- the reverse sweep of vla_backward.cuh as two
// kernels, one per state ("Variational Linear Attention", arXiv 2605.11196,
// §3.3 eq. 9-11, reverse mode). Included by vla_forward.cu inside namespace
// vla, after vla_backward.cuh.
//
// The adjoint of the S recurrence (eq. 10 second half, eq. 11) needs nothing
// from the A side: with g_alpha = (gS + dL/do phi_q^T / den)^T e, the gate's
// gradient before its normalisation is
//   g_a = (g_alpha - alpha^ (alpha^ . g_alpha)) / ||a||,
// and every other S-side quantity (g_e, dL/dv, dL/dq, the z^key adjoint, the
// S part of dL/dk^) follows from S, gS and the tape. The A side (eq. 9, eq. 10
// first half) needs g_a and nothing else from the S side. So:
//  * the S side sweeps t = T-1 .. 0 with S and gS in registers, writes
//    dL/dq, dL/dv, the S part of dL/dk (the z^key term and the projected
//    -S_{t-1}^T g_e, both linear in the S side), and g_a over the tape's e_t
//    (no later step reads e_t);
//  * the A side sweeps with A and gA, reads g_a from the tape, writes dL/du
//    and adds the A part of dL/dk (the projected A_t g_a).
// Each side holds two d x d matrices, half of the single-kernel sweep, so
// d = 128 fits (8 rows x 4 columns of each per thread, 512 threads).
//
// vla_backward_pair_kernel runs both sides at once, as a cluster of two CTAs
// per head: CTA 0 the S side, CTA 1 the A side a few tokens behind it. After
// the first block barrier of its step for token t, one otherwise idle S-side
// thread publishes t + 1 (every write of the steps for tokens > t is done:
// g_a of those tokens, the S part of dL/dk of tokens > t + 1) with a release
// store at cluster scope into a counter in the A side's shared memory; 0 and
// -1 follow the last step and the last dL/dk. The A side reads the counter
// with acquire loads before it prefetches a token's tape record, in one
// thread and then a block barrier, with a time limit (VLA_ERR_TIMEOUT; after
// it runs out the A side waits no more and its results are not meaningful).
// The test hook Params::stall_producer makes the S side publish nothing, so
// that the limit runs out. The S side never waits for the A side, and both CTAs meet at a cluster barrier
// before they exit, so neither leaves while the other may still write into
// its shared memory.
//
// The register layout, the row and column products, the checkpoints and the
// identities that save products are those of vla_backward.cuh.

namespace bw {

// ring slot (bytes) and shared memory of the S-side sweep
template <int D, typename TIn>
struct SLay {
    static constexpr int RW = 8, NW = D / RW, THREADS = 32 * NW, CL = D / 32;
    static constexpr int TREC = 3 * D + 8;
    static constexpr int CREC = 2 * D * D + D;
    static constexpr int NB = 5;  // prefetch 3 tokens ahead, 1 slot held by the deferred dL/dk
    static constexpr int IN_B = D * (int)sizeof(TIn);
    static constexpr int K = 0, Q = IN_B, G = 2 * IN_B, TP = 2 * IN_B + 4 * D;
    static constexpr int SLOT_B = TP + 4 * TREC;
    static constexpr int RING = 0;
    static constexpr int P1 = RING + NB * SLOT_B;   // pass-1 column partials [NW][2][D]
    static constexpr int C1 = P1 + NW * 2 * D * 4;  // their sums [2][D]
    static constexpr int R1 = C1 + 2 * D * 4;       // pass-1 row products [2 parities][D]
    static constexpr int P2 = R1 + 2 * D * 4;       // pass-2 column partials [NW][D]
    static constexpr int DP = P2 + NW * D * 4;      // per-warp dot partials [2][NW]
    static constexpr int DS = DP + 2 * NW * 4;      // their sums [2] (+2 unused)
    static constexpr int RED = DS + 4 * 4;          // [CL] dot partials of the deferred dL/dk
    static constexpr int SMEM = RED + 4 * 4;
    static_assert(D % 32 == 0 && D <= 128 && CL <= 4, "8 rows x d/32 columns per thread");
    static_assert(SLOT_B % 16 == 0 && IN_B % 16 == 0 && TREC % 4 == 0, "cp.async chunks");
    static_assert(2 * IN_B / 16 + D / 4 + TREC / 4 <= THREADS, "one prefetch chunk per thread");
    static_assert(NW == 4 * CL, "column sums on 2 CL warps, the dot sums on one more, dL/dk on the last CL");
};

// ring slot (bytes) and shared memory of the A-side sweep
template <int D, typename TIn>
struct ALay {
    static constexpr int RW = 8, NW = D / RW, THREADS = 32 * NW, CL = D / 32;
    static constexpr int TREC = 3 * D + 8;
    static constexpr int CREC = 2 * D * D + D;
    static constexpr int NB = 5;
    static constexpr int IN_B = D * (int)sizeof(TIn);
    static constexpr int U = 0, K = IN_B, TP = 2 * IN_B;
    static constexpr int SLOT_B = TP + 4 * TREC;
    static constexpr int RING = 0;
    static constexpr int P1 = RING + NB * SLOT_B;  // pass-1 column partials [NW][D]
    static constexpr int C1 = P1 + NW * D * 4;     // their sums [D]
    static constexpr int R1 = C1 + D * 4;          // pass-1 row products [2 parities][D]
    static constexpr int R2 = R1 + 2 * D * 4;      // pass-2 row products [2][D]
    static constexpr int DP = R2 + 2 * D * 4;      // per-warp dot partials [NW]
    static constexpr int DS = DP + NW * 4;         // their sum (+3 unused)
    static constexpr int RED = DS + 4 * 4;         // [CL][2] dot partials of the deferred dL/dk, dL/du
    static constexpr int SMEM = RED + 8 * 4;
    static_assert(D % 32 == 0 && D <= 128 && CL <= 4, "8 rows x d/32 columns per thread");
    static_assert(SLOT_B % 16 == 0 && IN_B % 16 == 0 && TREC % 4 == 0, "cp.async chunks");
    static_assert(2 * IN_B / 16 + TREC / 4 <= THREADS, "one prefetch chunk per thread");
    static_assert(NW == 4 * CL, "column sums on CL warps, the dot sum on one more, dL/dk, dL/du on the last CL");
};

// the two-CTA form: the counter sits past both sides' shared memory
template <int D, typename TIn>
struct PairLay {
    static constexpr int FLAG = (std::max(SLay<D, TIn>::SMEM, ALay<D, TIn>::SMEM) + 15) / 16 * 16;
    static constexpr int SMEM = FLAG + 16;
    // the S-side thread that publishes progress: lane 31 of a warp with no
    // work between the step's two block barriers (else of the warp that sums
    // the two dots, whose lanes 0 and 1 work there)
    static constexpr int NW = SLay<D, TIn>::NW, CL = SLay<D, TIn>::CL;
    static constexpr int PUB = 32 * ((2 * CL + 1 < NW - CL) ? 2 * CL + 1 : 2 * CL) + 31;
    static_assert(SLay<D, TIn>::THREADS == ALay<D, TIn>::THREADS, "both sides run on CTAs of one size");
};

__device__ __forceinline__ uint32_t pair_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t pair_peer(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// every thread of both CTAs
__device__ __forceinline__ void pair_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void pair_publish(uint32_t raddr, int v) {
    asm volatile("st.release.cluster.shared::cluster.s32 [%0], %1;" ::"r"(raddr), "r"(v) : "memory");
}
__device__ __forceinline__ int pair_read(const int* f) {
    int v;
    asm volatile("ld.acquire.cluster.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(f)) : "memory");
    return v;
}
// wait until the counter is at most `target`; false once `limit_ns` has passed
__device__ __noinline__ bool pair_wait(const int* f, int target, uint64_t limit_ns) {
    if (pair_read(f) <= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        __nanosleep(32);
        if (pair_read(f) <= target) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

template <int D, typename TIn>
__device__ __forceinline__ void prefetch_s(unsigned char* slot, const TIn* gk, const TIn* gq, const float* go,
                                           const float* tp, int t) {
    using L = SLay<D, TIn>;
    constexpr int NC = L::IN_B / 16, NG = D / 4, NR = L::TREC / 4;
    const int tid = threadIdx.x;
    if (tid < 2 * NC) {
        const int part = tid / NC, off = tid - part * NC;
        const TIn* src = part == 0 ? gk : gq;
        cp_async16(slot + part * L::IN_B + off * 16,
                   reinterpret_cast<const unsigned char*>(src + (size_t)t * D) + off * 16);
    } else if (tid < 2 * NC + NG) {
        const int off = tid - 2 * NC;
        if (go) cp_async16(slot + L::G + off * 16, go + (size_t)t * D + off * 4);
    } else if (tid < 2 * NC + NG + NR) {
        const int off = tid - 2 * NC - NG;
        cp_async16(slot + L::TP + off * 16, tp + (size_t)t * L::TREC + off * 4);
    }
}

template <int D, typename TIn>
__device__ __forceinline__ void prefetch_a(unsigned char* slot, const TIn* gu, const TIn* gk, const float* tp,
                                           int t) {
    using L = ALay<D, TIn>;
    constexpr int NC = L::IN_B / 16, NR = L::TREC / 4;
    const int tid = threadIdx.x;
    if (tid < 2 * NC) {
        const int part = tid / NC, off = tid - part * NC;
        const TIn* src = part == 0 ? gu : gk;
        cp_async16(slot + part * L::IN_B + off * 16,
                   reinterpret_cast<const unsigned char*>(src + (size_t)t * D) + off * 16);
    } else if (tid < 2 * NC + NR) {
        const int off = tid - 2 * NC;
        cp_async16(slot + L::TP + off * 16, tp + (size_t)t * L::TREC + off * 4);
    }
}

// The S part of dL/dk_t (column j = 32 jw + lane) from token t's pass-2
// column partials (S_t^T g_e):
//   gzk phi'(k) - P(S_{t-1}^T g_e) / ||k||,  S_{t-1}^T g_e = S_t^T g_e - alpha^ (e . g_e),
// P the projection off k^. Run by the last d/32 warps. Returns fma(dL/dk, 0): 0
// unless it is NaN or Inf.
template <int D, typename TIn>
__device__ __forceinline__ float k_grad_s(const unsigned char* sl, const float* P2, float* RED, int jw, float gzk,
                                         float e_ge, float nk, float* dk) {
    using L = SLay<D, TIn>;
    const int l = threadIdx.x & 31, j = 32 * jw + l;
    const float* rec = reinterpret_cast<const float*>(sl + L::TP);
    float st = 0.f;
#pragma unroll
    for (int v = 0; v < L::NW; ++v) st += P2[v * D + j];
    const float sk = fmaf(-rec[D + j], e_ge, st);
    const float kj = lds_in<TIn>(sl + L::K, j);
    const float ik = inv_norm(nk), khj = kj * ik;
    float d1 = khj * sk;
    allreduce<1, 16>(&d1);
    if (l == 0) RED[jw] = d1;
    named_bar(1, D);
    float ks = 0.f;
#pragma unroll
    for (int v = 0; v < L::CL; ++v) ks += RED[v];
    const float dkt = fmaf(gzk, phi_d(kj), nk < 1e-24f ? -sk * 1e12f : -fmaf(-khj, ks, sk) * ik);
    dk[j] = dkt;
    return dkt * 0.f;
}

// dL/du_t and the A part of dL/dk_t (column j = 32 jw + lane) from token t's
// pass-2 row products (A_t g_a, A_t w1) and its scalars; the A part
// P(A_t g_a) / ||k|| is added to the S part already in dk. Run by the last
// d/32 warps. Returns fma(gradients, 0): 0 unless one is NaN or Inf.
template <int D, typename TIn>
__device__ __forceinline__ float ku_grad_a(const unsigned char* sl, const float* R2, float* RED, int jw, float kz,
                                          float gdl, float zgz, float az, float nac, float dl, float nu, float nk,
                                          float* dk, float* du) {
    using L = ALay<D, TIn>;
    const int l = threadIdx.x & 31, j = 32 * jw + l;
    const float* rec = reinterpret_cast<const float*>(sl + L::TP);
    const float aga = R2[j], aw1 = R2[D + j];
    const float zj = rec[j], alj = rec[D + j];
    const float kj = lds_in<TIn>(sl + L::K, j);
    const float iu = inv_norm(nu), ik = inv_norm(nk), rdl = rcpa(dl);
    const float khj = kj * ik, uhj = lds_in<TIn>(sl + L::U, j) * iu;
    const float atgz = fmaf(gdl * rdl, zj, -(aw1 + fmaf(aga, kz, alj * nac * az)) * rdl);  // A_t g_z
    const float zgzf = -zgz * (dl + 1.f) * rdl * rdl;                                      // z . g_z
    const float guh = fmaf(zj, fmaf(zgzf, rdl, gdl), atgz);                                // A_{t-1} g_z + g_delta z
    float d2[2] = {uhj * guh, khj * aga};
    allreduce<2, 16>(d2);
    if (l == 0) {
        RED[2 * jw] = d2[0];
        RED[2 * jw + 1] = d2[1];
    }
    named_bar(1, D);
    float ugu = 0.f, kga = 0.f;
#pragma unroll
    for (int v = 0; v < L::CL; ++v) {
        ugu += RED[2 * v];
        kga += RED[2 * v + 1];
    }
    const float dut = nu < 1e-24f ? guh * 1e12f : fmaf(-uhj, ugu, guh) * iu;
    const float dka = nk < 1e-24f ? aga * 1e12f : fmaf(-khj, kga, aga) * ik;
    du[j] = dut;
    const float dkt = __ldcg(dk + j) + dka;  // the S part, written by the other CTA of a pair
    dk[j] = dkt;
    return fmaf(dut, 0.f, dkt * 0.f);
}

// S side of the reverse sweep for head bh of BH. fin: the forward's final S
// [BH][D][D] | A | z^key [BH][D]. rflag: the A side's progress counter.
template <int D, typename TIn>
__device__ __forceinline__ void s_sweep(const Params& p, int bh, size_t BH, const float* dO, const float* dST,
                                        const float* dzkT, float* dq, float* dk, float* dv, float* dS0,
                                        float* dzk0, float* tape, const float* ckpt, const float* fin,
                                        uint32_t rflag) {
    using L = SLay<D, TIn>;
    constexpr int RW = L::RW, CL = L::CL, NW = L::NW, NB = L::NB;
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* ring = smem + L::RING;
    float* P1 = reinterpret_cast<float*>(smem + L::P1);
    float* C1 = reinterpret_cast<float*>(smem + L::C1);
    float* R1 = reinterpret_cast<float*>(smem + L::R1);
    float* P2 = reinterpret_cast<float*>(smem + L::P2);
    float* DP = reinterpret_cast<float*>(smem + L::DP);
    float* DS = reinterpret_cast<float*>(smem + L::DS);
    float* RED = reinterpret_cast<float*>(smem + L::RED);

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int r0 = w * RW, rr = r0 + (l >> 2);
    const int T = p.T;
    const size_t hin = (size_t)bh * T * D, hdd = (size_t)bh * D * D;
    const TIn* gq = static_cast<const TIn*>(p.q) + hin;
    const TIn* gk = static_cast<const TIn*>(p.k) + hin;
    const float* go_h = dO ? dO + hin : nullptr;
    float* tp = tape + (size_t)bh * T * L::TREC;
    const float* cp = ckpt + (size_t)bh * ((T + CK - 1) / CK + 1) * L::CREC;
    float gchk = 0.f;  // fma(x, 0, .) of every gradient and g_a written: 0 unless one is NaN or Inf

    // S and gS: rows r0 + 2 rp (.x) and r0 + 2 rp + 1 (.y), columns l + 32 c,
    // updated by packed FP32 FMAs (two rows per instruction)
    float2 S2[RW / 2][CL], gS2[RW / 2][CL];
    float zk[CL], gzk[CL];
#pragma unroll
    for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const size_t e = hdd + (size_t)(r0 + 2 * rp) * D + l + 32 * c;
            S2[rp][c] = T > 0 ? make_float2(fin[e], fin[e + D]) : dup2(0.f);
            gS2[rp][c] = dST ? make_float2(dST[e], dST[e + D]) : dup2(0.f);
        }
#pragma unroll
    for (int c = 0; c < CL; ++c) {
        const size_t e = (size_t)bh * D + l + 32 * c;
        zk[c] = T > 0 ? fin[2 * BH * D * D + e] : 0.f;
        gzk[c] = dzkT ? dzkT[e] : 0.f;
    }
    if (!dO)
        for (int i = tid; i < NB * D; i += L::THREADS)
            reinterpret_cast<float*>(ring + (i / D) * L::SLOT_B + L::G)[i % D] = 0.f;
    for (int s = 0; s < 3; ++s) {
        const int tok = T - 1 - s;
        if (tok >= 0) prefetch_s<D, TIn>(ring + (tok % NB) * L::SLOT_B, gk, gq, go_h, tp, tok);
        cp_commit();
    }
    cp_wait<1>();
    __syncthreads();
    const bool ku_warp = w >= NW - CL;
    const int jw = w - (NW - CL);
    float j_ege = 0.f, j_nk = 1.f;  // scalars of the token whose dL/dk is pending
    for (int t = T - 1; t >= 0; --t) {
        const unsigned char* sl = ring + (t % NB) * L::SLOT_B;
        const float* rec = reinterpret_cast<const float*>(sl + L::TP);
        const float* gov = reinterpret_cast<const float*>(sl + L::G);
        float* r1 = R1 + (t & 1) * D;
        const float na = rec[3 * D + 1], dsg = rec[3 * D + 2], nk = rec[3 * D + 4];
        const bool clamped = dsg < 0.f;
        const float rden = rcpa(clamped ? -dsg : dsg), ik = inv_norm(nk);
        const bool tiny = na < 1e-12f;
        const float ina = rcpa(fmaxf(na, 1e-12f));
        const size_t orow = ((size_t)bh * T + t) * D;

        float kh[CL], pq[CL], al[CL];
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const int j = l + 32 * c;
            kh[c] = lds_in<TIn>(sl + L::K, j) * ik;
            pq[c] = phi(lds_in<TIn>(sl + L::Q, j));
            al[c] = rec[D + j];
        }
        // product pass 1: rows gS alpha^; columns gS^T e, S_t^T dL/do
        float d4[4] = {0.f, 0.f, 0.f, 0.f};
        {
            float pg[RW];
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp) {
                float2 a = dup2(0.f);
#pragma unroll
                for (int c = 0; c < CL; ++c) a = __ffma2_rn(gS2[rp][c], dup2(al[c]), a);
                pg[2 * rp] = a.x;
                pg[2 * rp + 1] = a.y;
            }
            const float gsal = rowsum8(pg);
            if ((l & 3) == 0) r1[rr] = gsal;
            float er[RW], gor[RW], qe[CL], qo[CL];
            lds8f(rec + 2 * D, r0, er);
            lds8f(gov, r0, gor);
            {
                float2 qe2[CL], qo2[CL];
#pragma unroll
                for (int c = 0; c < CL; ++c) qe2[c] = qo2[c] = dup2(0.f);
#pragma unroll
                for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
                    for (int c = 0; c < CL; ++c) {
                        qe2[c] = __ffma2_rn(gS2[rp][c], pair2(er, 2 * rp), qe2[c]);
                        qo2[c] = __ffma2_rn(S2[rp][c], pair2(gor, 2 * rp), qo2[c]);
                    }
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    qe[c] = qe2[c].x + qe2[c].y;
                    qo[c] = qo2[c].x + qo2[c].y;
                }
            }
            // token dots phi_q . alpha^, dL/do . e; this warp's shares of phi_q . S_t^T dL/do, alpha^ . gS^T e
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                const int j = l + 32 * c;
                P1[(w * 2 + 0) * D + j] = qe[c];
                P1[(w * 2 + 1) * D + j] = qo[c];
                d4[0] = fmaf(pq[c], al[c], d4[0]);
                d4[1] = fmaf(gov[j], rec[2 * D + j], d4[1]);
                d4[2] = fmaf(pq[c], qo[c], d4[2]);
                d4[3] = fmaf(al[c], qe[c], d4[3]);
            }
        }
        allreduce<4, 16>(d4);
        if (l == 0) {
            DP[w] = d4[2];
            DP[NW + w] = d4[3];
        }
        cp_wait<1>();
        __syncthreads();  // B1 (also publishes token t-1's slot)
        if (tid == PairLay<D, TIn>::PUB && !p.stall_producer) pair_publish(rflag, t + 1);  // the step for t+1 is done
        if (t >= 3) prefetch_s<D, TIn>(ring + ((t - 3) % NB) * L::SLOT_B, gk, gq, go_h, tp, t - 3);
        cp_commit();
        if (tid < 2 * D) {
            const int x = tid / D, j = tid - x * D;
            float s = 0.f;
#pragma unroll
            for (int v = 0; v < NW; ++v) s += P1[(v * 2 + x) * D + j];
            C1[x * D + j] = s;
        } else {
            if (w == 2 * CL && l < 2) {
                float s = 0.f;
#pragma unroll
                for (int v = 0; v < NW; ++v) s += DP[l * NW + v];
                DS[l] = s;
            }
            if (ku_warp && t + 1 < T)
                gchk += k_grad_s<D, TIn>(ring + ((t + 1) % NB) * L::SLOT_B, P2, RED, jw, pick<CL>(gzk, jw), j_ege,
                                         j_nk, dk + orow + D);
        }
        __syncthreads();  // B2

        const float c1n = d4[0], c2n = d4[1];
        const float c1 = c1n * rden, c2 = c2n * rden;
        const float s_o = DS[0], s_ae = DS[1];
        const float gden = clamped ? 0.f : -s_o * rden * rden;  // -(dL/do . o) / den
        const float al_gal = fmaf(c2, c1n, s_ae);                // alpha^ . g_alpha
        const float e_ge = fmaf(c1, c2n, s_ae);                  // e . g_e
        // columns: g_a (over the tape's e_t), dL/dq, the z^key adjoint
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const int j = l + 32 * c;
            const float gal = fmaf(pq[c], c2, C1[j]);
            const float ga = (tiny ? gal : fmaf(-al[c], al_gal, gal)) * ina;
            const float gpq = fmaf(gden, zk[c], C1[D + j] * rden);
            gzk[c] = fmaf(gden, pq[c], gzk[c]);
            if (w == 0) {
                const float x = gpq * phi_d(lds_in<TIn>(sl + L::Q, j));
                dq[orow + j] = x;
                tp[(size_t)t * L::TREC + 2 * D + j] = ga;
                gchk = fmaf(x, 0.f, fmaf(ga, 0.f, gchk));
            }
        }
        // rows: g_e = gS alpha^ + dL/do (phi_q . alpha^) / den = dL/dv
        float ger[RW], gor[RW];
        {
            float a8[RW];
            lds8f(r1, r0, a8);
            lds8f(gov, r0, gor);
#pragma unroll
            for (int r = 0; r < RW; ++r) ger[r] = fmaf(gor[r], c1, a8[r]);
        }
        if (l < RW) {
            const float x = pick<RW>(ger, l);
            dv[orow + r0 + l] = x;
            gchk = fmaf(x, 0.f, gchk);
        }
        // product pass 2: columns S_t^T g_e
        {
            float2 qg2[CL];
#pragma unroll
            for (int c = 0; c < CL; ++c) qg2[c] = dup2(0.f);
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
                for (int c = 0; c < CL; ++c) qg2[c] = __ffma2_rn(S2[rp][c], pair2(ger, 2 * rp), qg2[c]);
#pragma unroll
            for (int c = 0; c < CL; ++c) P2[w * D + l + 32 * c] = qg2[c].x + qg2[c].y;
        }
        // gS += dL/do phi_q^T / den - g_e k^^T
#pragma unroll
        for (int rp = 0; rp < RW / 2; ++rp) {
            const float2 gs = make_float2(gor[2 * rp] * rden, gor[2 * rp + 1] * rden);
            const float2 mg = make_float2(-ger[2 * rp], -ger[2 * rp + 1]);
#pragma unroll
            for (int c = 0; c < CL; ++c)
                gS2[rp][c] = __ffma2_rn(gs, dup2(pq[c]), __ffma2_rn(mg, dup2(kh[c]), gS2[rp][c]));
        }
        // S_{t-1} = S_t - e alpha^^T, z^key_{t-1} = z^key_t - phi(k_t); exact copies at checkpoints
        if (t % CK == 0) {
            const float* c = cp + (size_t)(t / CK) * L::CREC;
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
                for (int cc = 0; cc < CL; ++cc) {
                    const int e = (r0 + 2 * rp) * D + l + 32 * cc;
                    S2[rp][cc] = make_float2(c[e], c[e + D]);
                }
#pragma unroll
            for (int cc = 0; cc < CL; ++cc) zk[cc] = c[2 * D * D + l + 32 * cc];
        } else {
            float er[RW];
            lds8f(rec + 2 * D, r0, er);
#pragma unroll
            for (int rp = 0; rp < RW / 2; ++rp) {
                const float2 me = make_float2(-er[2 * rp], -er[2 * rp + 1]);
#pragma unroll
                for (int c = 0; c < CL; ++c) S2[rp][c] = __ffma2_rn(me, dup2(al[c]), S2[rp][c]);
            }
#pragma unroll
            for (int c = 0; c < CL; ++c) zk[c] -= phi(lds_in<TIn>(sl + L::K, l + 32 * c));
        }
        j_ege = e_ge, j_nk = nk;
    }
    __syncthreads();  // pass-2 partials of token 0 visible
    if (tid == PairLay<D, TIn>::PUB && !p.stall_producer) pair_publish(rflag, 0);  // every step done
    if (T > 0 && ku_warp) gchk += k_grad_s<D, TIn>(ring, P2, RED, jw, pick<CL>(gzk, jw), j_ege, j_nk, dk + (size_t)bh * T * D);
    __syncthreads();
    if (tid == PairLay<D, TIn>::PUB && !p.stall_producer) pair_publish(rflag, -1);  // dL/dk_0's S part is written
    cp_wait<0>();
#pragma unroll
    for (int rp = 0; rp < RW / 2; ++rp)
#pragma unroll
        for (int c = 0; c < CL; ++c)
            if (dS0) {
                const size_t e = hdd + (size_t)(r0 + 2 * rp) * D + l + 32 * c;
                dS0[e] = gS2[rp][c].x;
                dS0[e + D] = gS2[rp][c].y;
            }
    if (w == 0 && dzk0)
#pragma unroll
        for (int c = 0; c < CL; ++c) dzk0[(size_t)bh * D + l + 32 * c] = gzk[c];
    if (gchk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_S, bh, -1);
}

// A side of the reverse sweep for head bh of BH, behind the S side: g_a_t is
// in the tape's e_t slot once the counter `flag` is at most t.
template <int D, typename TIn>
__device__ __forceinline__ void a_sweep(const Params& p, int bh, size_t BH, const float* dAT, float* dk, float* du,
                                        float* dA0, const float* tape, const float* ckpt, const float* fin,
                                        const int* flag) {
    using L = ALay<D, TIn>;
    constexpr int RW = L::RW, CL = L::CL, NW = L::NW, NB = L::NB;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* ring = smem + L::RING;
    float* P1 = reinterpret_cast<float*>(smem + L::P1);
    float* C1 = reinterpret_cast<float*>(smem + L::C1);
    float* R1 = reinterpret_cast<float*>(smem + L::R1);
    float* R2 = reinterpret_cast<float*>(smem + L::R2);
    float* DP = reinterpret_cast<float*>(smem + L::DP);
    float* DS = reinterpret_cast<float*>(smem + L::DS);
    float* RED = reinterpret_cast<float*>(smem + L::RED);

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int r0 = w * RW, rr = r0 + (l >> 2);
    const int T = p.T;
    const size_t hin = (size_t)bh * T * D, hdd = (size_t)bh * D * D;
    const TIn* gu = static_cast<const TIn*>(p.u) + hin;
    const TIn* gk = static_cast<const TIn*>(p.k) + hin;
    const float* tp = tape + (size_t)bh * T * L::TREC;
    const float* cp = ckpt + (size_t)bh * ((T + CK - 1) / CK + 1) * L::CREC;
    float gchk = 0.f;  // fma(x, 0, .) of every gradient written: 0 unless one is NaN or Inf
    bool gave_up = false;  // thread 0: a wait for the S side ran out of time
    auto wait_s = [&](int target) {  // thread 0: the S side's writes for tokens >= target are done
        if (!gave_up && !pair_wait(flag, target, p.wait_ns)) {
            gave_up = true;
            record_failure(p.status, BIT_TIMEOUT, ROLE_A, bh, target);
        }
    };

    float A[RW][CL], gA[RW][CL];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const size_t e = hdd + (size_t)(r0 + r) * D + l + 32 * c;
            A[r][c] = T > 0 ? fin[BH * D * D + e] : 0.f;
            gA[r][c] = dAT ? dAT[e] : 0.f;
        }
    if (tid == 0 && T > 0) wait_s(max(T - 3, 0));
    __syncthreads();
    for (int s = 0; s < 3; ++s) {
        const int tok = T - 1 - s;
        if (tok >= 0) prefetch_a<D, TIn>(ring + (tok % NB) * L::SLOT_B, gu, gk, tp, tok);
        cp_commit();
    }
    cp_wait<1>();
    __syncthreads();
    const bool ku_warp = w >= NW - CL;
    const int jw = w - (NW - CL);
    float j_kz = 0.f, j_gdl = 0.f, j_zgz = 0.f, j_az = 0.f, j_nac = 1.f, j_dl = 1.f, j_nu = 1.f, j_nk = 1.f;
    for (int t = T - 1; t >= 0; --t) {
        const unsigned char* sl = ring + (t % NB) * L::SLOT_B;
        const float* rec = reinterpret_cast<const float*>(sl + L::TP);
        float* r1 = R1 + (t & 1) * D;
        const float dl = rec[3 * D], na = rec[3 * D + 1], nu = rec[3 * D + 3], nk = rec[3 * D + 4];
        const float rdl = rcpa(dl), iu = inv_norm(nu), ik = inv_norm(nk);
        const float nac = fmaxf(na, 1e-12f);
        const size_t orow = ((size_t)bh * T + t) * D;

        float uh[CL], kh[CL], zc[CL], gac[CL];
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const int j = l + 32 * c;
            uh[c] = lds_in<TIn>(sl + L::U, j) * iu;
            kh[c] = lds_in<TIn>(sl + L::K, j) * ik;
            zc[c] = rec[j];
            gac[c] = rec[2 * D + j];  // g_a, written over e_t by the S side
        }
        // product pass 1: rows gA z; columns gA^T z
        float d3[3] = {0.f, 0.f, 0.f};
        {
            float pz[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                pz[r] = 0.f;
#pragma unroll
                for (int c = 0; c < CL; ++c) pz[r] = fmaf(gA[r][c], zc[c], pz[r]);
            }
            const float gaz = rowsum8(pz);
            if ((l & 3) == 0) r1[rr] = gaz;
            float zr[RW], qz[CL];
            lds8f(rec, r0, zr);
#pragma unroll
            for (int c = 0; c < CL; ++c) qz[c] = 0.f;
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int c = 0; c < CL; ++c) qz[c] = fmaf(gA[r][c], zr[r], qz[c]);
            // token dots k^ . z, g_a . z; this warp's share of z . gA^T z
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                P1[w * D + l + 32 * c] = qz[c];
                d3[0] = fmaf(kh[c], zc[c], d3[0]);
                d3[1] = fmaf(gac[c], zc[c], d3[1]);
                d3[2] = fmaf(zc[c], qz[c], d3[2]);
            }
        }
        allreduce<3, 16>(d3);
        if (l == 0) DP[w] = d3[2];
        if (tid == 0 && t >= 3) wait_s(t - 3);  // before token t-3's record is prefetched
        cp_wait<1>();
        __syncthreads();  // B1
        if (t >= 3) prefetch_a<D, TIn>(ring + ((t - 3) % NB) * L::SLOT_B, gu, gk, tp, t - 3);
        cp_commit();
        if (tid < D) {
            float s = 0.f;
#pragma unroll
            for (int v = 0; v < NW; ++v) s += P1[v * D + tid];
            C1[tid] = s;
        } else {
            if (w == CL && l == 0) {
                float s = 0.f;
#pragma unroll
                for (int v = 0; v < NW; ++v) s += DP[v];
                DS[0] = s;
            }
            if (ku_warp && t + 1 < T)
                gchk += ku_grad_a<D, TIn>(ring + ((t + 1) % NB) * L::SLOT_B, R2, RED, jw, j_kz, j_gdl, j_zgz, j_az,
                                          j_nac, j_dl, j_nu, j_nk, dk + orow + D, du + orow + D);
        }
        __syncthreads();  // B2

        const float kz = d3[0], az = d3[1];
        const float zgz = fmaf(az, kz, DS[0]);  // z^T (gA + g_a k^^T) z
        const float gdl = zgz * rdl * rdl;      // dL/d delta
        // columns: w1 = (gA + gA^T) z, g_z = -((gA + g_a k^^T) z + (gA + g_a k^^T)^T z) / delta + g_delta u^
        float w1c[CL], gzc[CL];
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            const int j = l + 32 * c;
            w1c[c] = r1[j] + C1[j];
            gzc[c] = fmaf(gdl, uh[c], -(w1c[c] + fmaf(gac[c], kz, kh[c] * az)) * rdl);
        }
        // product pass 2: rows A_t g_a, A_t w1
        {
            float pa[RW], pw[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                pa[r] = pw[r] = 0.f;
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    pa[r] = fmaf(A[r][c], gac[c], pa[r]);
                    pw[r] = fmaf(A[r][c], w1c[c], pw[r]);
                }
            }
            const float aga = rowsum8(pa), aw1 = rowsum8(pw);
            if ((l & 3) == 0) {
                R2[rr] = aga;
                R2[D + rr] = aw1;
            }
        }
        // gA += g_a k^^T + g_z u^^T (rows r0 .. r0+7 are columns of lanes r0 mod 32 .. +7, slot r0 / 32)
        {
            const int cs = r0 >> 5, lb = r0 & 31;
            const float ga_s = pick<CL>(gac, cs), gz_s = pick<CL>(gzc, cs);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float gar = __shfl_sync(FULL, ga_s, lb + r), gzr = __shfl_sync(FULL, gz_s, lb + r);
#pragma unroll
                for (int c = 0; c < CL; ++c) gA[r][c] = fmaf(gar, kh[c], fmaf(gzr, uh[c], gA[r][c]));
            }
        }
        // A_{t-1} = A_t + z z^T / delta; exact copies at checkpoints
        if (t % CK == 0) {
            const float* c = cp + (size_t)(t / CK) * L::CREC;
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int cc = 0; cc < CL; ++cc) A[r][cc] = c[D * D + (r0 + r) * D + l + 32 * cc];
        } else {
            float zr[RW];
            lds8f(rec, r0, zr);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float zs = zr[r] * rdl;
#pragma unroll
                for (int c = 0; c < CL; ++c) A[r][c] = fmaf(zs, zc[c], A[r][c]);
            }
        }
        j_kz = kz, j_gdl = gdl, j_zgz = zgz, j_az = az, j_nac = nac, j_dl = dl, j_nu = nu, j_nk = nk;
    }
    if (tid == 0) wait_s(-1);  // the S part of dL/dk_0
    __syncthreads();  // pass-2 products of token 0 visible
    if (T > 0 && ku_warp)
        gchk += ku_grad_a<D, TIn>(ring, R2, RED, jw, j_kz, j_gdl, j_zgz, j_az, j_nac, j_dl, j_nu, j_nk,
                                  dk + (size_t)bh * T * D, du + (size_t)bh * T * D);
    cp_wait<0>();
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int c = 0; c < CL; ++c)
            if (dA0) dA0[hdd + (r0 + r) * D + l + 32 * c] = gA[r][c];
    if (gchk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_A, bh, -1);
}

// Both sides at once: a cluster of two CTAs per head (grid 2 BH), CTA 0 the S
// side, CTA 1 the A side.
template <int D, typename TIn>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(SLay<D, TIn>::THREADS, 1)
    vla_backward_pair_kernel(const Params p, const float* dO, const float* dST, const float* dAT, const float* dzkT,
                             float* dq, float* dk, float* dv, float* du, float* dS0, float* dA0, float* dzk0,
                             float* tape, const float* ckpt, const float* fin) {
    extern __shared__ __align__(16) unsigned char smem[];
    int* flag = reinterpret_cast<int*>(smem + PairLay<D, TIn>::FLAG);
    const uint32_t rank = pair_rank();
    const int bh = blockIdx.x >> 1;
    const size_t BH = gridDim.x >> 1;
    if (rank == 1 && threadIdx.x == 0) *flag = p.T;  // no step of the S side done yet
    pair_sync();
    if (rank == 0)
        s_sweep<D, TIn>(p, bh, BH, dO, dST, dzkT, dq, dk, dv, dS0, dzk0, tape, ckpt, fin, pair_peer(flag, 1));
    else
        a_sweep<D, TIn>(p, bh, BH, dAT, dk, du, dA0, tape, ckpt, fin, flag);
    pair_sync();  // neither CTA leaves while the other may still write into its shared memory
}

}  // namespace bw
