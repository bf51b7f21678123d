// vla_decode.cuh -- the VLA forward recurrence ("Variational Linear
// Attention", arXiv 2605.11196, §3.3 eq. 9-11) for short sequences with a
// carried state: decode (T = 1) and a few tokens per call. Also the fixed-A
// variant of the §3.5 ablation (A held at its initial value, eq. 9 skipped).
// Included by vla_forward.cu inside namespace vla.
//
// At small T the cost is moving the state: S and A are read and written once
// per call (2 d^2 floats each way per head), so the kernel is laid out to
// stream them. One persistent CTA per SM runs heads b, b + gridDim.x, ...;
// while a head computes, TMA bulk copies bring the next head's state and
// first-token inputs into shared memory. Warp w owns rows 8w .. 8w+7 of S and
// A and lane l owns columns l, l+32, .. in registers. Per token: one pass of row products
// (A u^, A k^, S k^, S phi(q), with the states before the token), a
// warp-shuffle halving exchange for the row sums, one block barrier to share
// z and A k^, then scalars by warp butterflies and the rank-1 updates in
// registers. The readout uses S_t phi = S_{t-1} phi + e (alpha^ . phi). For
// d <= 96 the finished head's S and A go back through shared memory and two
// bulk copies, which overlap the next head's work.

namespace dec {

template <int D, typename TIn>
struct DLay {
    static constexpr int RW = 8;             // rows per warp
    static constexpr int NW = D / RW;        // warps
    static constexpr int THREADS = 32 * NW;  // 384 at d = 96
    static constexpr int CL = D / 32;        // columns per lane
    static constexpr int IN_B = D * (int)sizeof(TIn);
    // shared memory (bytes): [2 parities][z | A k^] | mbarrier | the next
    // head's S | A | z^key | first-token u, k, q, v rows (TMA bulk copies)
    static constexpr int X = 0;
    static constexpr int BAR = X + 2 * 2 * D * 4;
    static constexpr int IS = BAR + 16;
    static constexpr int IA = IS + D * D * 4;
    static constexpr int IZ = IA + D * D * 4;
    static constexpr int IU = IZ + D * 4;
    static constexpr int IK = IU + IN_B, IQ = IK + IN_B, IV = IQ + IN_B;
    // the finished head's S | A, written out by two bulk copies (when both
    // areas fit: d <= 96; larger d stores from registers)
    static constexpr int OS = (IV + IN_B + 127) / 128 * 128, OA = OS + D * D * 4;
    static constexpr bool BULK_OUT = OA + D * D * 4 <= 227 * 1024;
    static constexpr int SMEM = BULK_OUT ? OA + D * D * 4 : IV + IN_B;
    static_assert(D % 32 == 0 && D <= 128, "register tiles hold 8 rows x d/32 columns of S and A");
    static_assert(IS % 16 == 0 && IN_B % 16 == 0, "bulk copy alignment");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Row sums of a warp's 8 rows (p[r]: this lane's partial sum of row r); the
// sum of row (lane >> 2) ends in this lane.
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

__device__ __forceinline__ float inv_norm(float n2) { return fminf(rsqrtf(n2), 1e12f); }  // 1 / max(sqrt(n2), 1e-12)

// bulk copy shared -> global (both addresses 16-byte aligned, size a multiple
// of 16), tracked by this thread's bulk async-groups
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk copies have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk copies are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Thread 0: bulk copies of head h's carried state and first-token inputs into
// the IN area, completing on `bar`. Every copied pointer is 16-byte aligned
// (the host checks) and every size is a multiple of 16.
template <int D, typename TIn, bool FIXED>
__device__ __forceinline__ void issue_head(const Params& p, unsigned char* sm, uint64_t* bar, int h) {
    using L = DLay<D, TIn>;
    const size_t hdd = (size_t)h * D * D, hin = (size_t)h * p.T * D;
    uint32_t bytes = 0;
    if (p.S0) bytes += D * D * 4;
    if (p.A0) bytes += D * D * 4;
    if (p.zk0) bytes += D * 4;
    if (p.T > 0) bytes += (FIXED ? 3 : 4) * L::IN_B;
    mbar_arrive_expect_tx(bar, bytes);
    if (p.S0) bulk_g2s(sm + L::IS, p.S0 + hdd, D * D * 4, bar);
    if (p.A0) bulk_g2s(sm + L::IA, p.A0 + hdd, D * D * 4, bar);
    if (p.zk0) bulk_g2s(sm + L::IZ, p.zk0 + (size_t)h * D, D * 4, bar);
    if (p.T > 0) {
        if (!FIXED) bulk_g2s(sm + L::IU, static_cast<const TIn*>(p.u) + hin, L::IN_B, bar);
        bulk_g2s(sm + L::IK, static_cast<const TIn*>(p.k) + hin, L::IN_B, bar);
        bulk_g2s(sm + L::IQ, static_cast<const TIn*>(p.q) + hin, L::IN_B, bar);
        bulk_g2s(sm + L::IV, static_cast<const TIn*>(p.v) + hin, L::IN_B, bar);
    }
}

// Persistent: CTA b runs heads b, b + gridDim.x, ...; with `bulk`, the next
// head's state is copied into shared memory while the current head computes.
// FIXED: the fixed-A variant (u is not read, A stays at its initial value).
template <int D, typename TIn, bool FIXED>
__global__ void __launch_bounds__(DLay<D, TIn>::THREADS, 1) vla_decode_kernel(const Params p, int BH, int bulk) {
    constexpr bool fixed_a = FIXED;
    using L = DLay<D, TIn>;
    constexpr int RW = L::RW, CL = L::CL;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char sm[];
    float* X = reinterpret_cast<float*>(sm + L::X);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
    const float* inS = reinterpret_cast<const float*>(sm + L::IS);
    const float* inA = reinterpret_cast<const float*>(sm + L::IA);
    const float* inZ = reinterpret_cast<const float*>(sm + L::IZ);

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int r0 = w * RW, rr = r0 + (l >> 2);
    const int T = p.T;
    bool bad = false;
    float ochk = 0.f;  // fma(o, 0, .) of every output: 0 unless one is NaN or Inf (branch-free)

    if (bulk) {
        if (tid == 0) {
            mbar_init(bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        // test hook: copy nothing, so that the wait below runs out
        if (tid == 0 && (int)blockIdx.x < BH && !p.stall_producer) issue_head<D, TIn, FIXED>(p, sm, bar, blockIdx.x);
    }
    int it = 0;
    for (int bh = blockIdx.x; bh < BH; bh += gridDim.x, ++it) {
        const size_t hin = (size_t)bh * T * D, hdd = (size_t)bh * D * D;
        const TIn* gq = static_cast<const TIn*>(p.q) + hin;
        const TIn* gk = static_cast<const TIn*>(p.k) + hin;
        const TIn* gv = static_cast<const TIn*>(p.v) + hin;
        const TIn* gu = static_cast<const TIn*>(p.u) + hin;

        float S[RW][CL], A[RW][CL], zk[CL];
        // raw u, k, q of the current token (this lane's columns), v of row rr
        float uc[CL], kc[CL], qc[CL], vr = 0.f;
        if (bulk) {
            const bool timed_out = !mbar_wait(bar, it & 1, nullptr, p.wait_ns);
            if (__syncthreads_or(timed_out)) {
                if (tid == 0) {
                    record_failure(p.status, BIT_TIMEOUT, ROLE_S, bh, 0);
                    // the copies issue_head started for this head may still be in
                    // flight: let them land (bounded wait) before the CTA can exit
                    (void)mbar_wait(bar, it & 1, nullptr, p.wait_ns);
                    if (L::BULK_OUT) bulk_wait_all();  // earlier heads' stores leave shared memory first
                }
                return;
            }
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    const int i = r0 + r, j = l + 32 * c;
                    A[r][c] = p.A0 ? inA[i * D + j] : (i == j ? p.inv_lambda0 : 0.f);
                    S[r][c] = p.S0 ? inS[i * D + j] : 0.f;
                }
#pragma unroll
            for (int c = 0; c < CL; ++c) zk[c] = p.zk0 ? inZ[l + 32 * c] : 0.f;
            if (T > 0) {
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    uc[c] = fixed_a ? 0.f : bw::lds_in<TIn>(sm + L::IU, l + 32 * c);
                    kc[c] = bw::lds_in<TIn>(sm + L::IK, l + 32 * c);
                    qc[c] = bw::lds_in<TIn>(sm + L::IQ, l + 32 * c);
                }
                vr = bw::lds_in<TIn>(sm + L::IV, rr);
            }
            __syncthreads();  // the IN area is free
            if (tid == 0 && bh + (int)gridDim.x < BH) {
                fence_proxy_async_smem();
                issue_head<D, TIn, FIXED>(p, sm, bar, bh + gridDim.x);
            }
        } else {
            __syncthreads();  // the previous head's reads of X are done
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    const int i = r0 + r, j = l + 32 * c;
                    A[r][c] = p.A0 ? p.A0[hdd + i * D + j] : (i == j ? p.inv_lambda0 : 0.f);
                    S[r][c] = p.S0 ? p.S0[hdd + i * D + j] : 0.f;
                }
#pragma unroll
            for (int c = 0; c < CL; ++c) zk[c] = p.zk0 ? p.zk0[(size_t)bh * D + l + 32 * c] : 0.f;
            if (T > 0) {
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    uc[c] = fixed_a ? 0.f : ld_in<TIn>(gu, l + 32 * c);
                    kc[c] = ld_in<TIn>(gk, l + 32 * c);
                    qc[c] = ld_in<TIn>(gq, l + 32 * c);
                }
                vr = ld_in<TIn>(gv, rr);
            }
        }
        float nu = 0.f, nk = 0.f;
        if (T > 0) {
            float nn[2] = {0.f, 0.f};
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                nn[0] = fmaf(uc[c], uc[c], nn[0]);
                nn[1] = fmaf(kc[c], kc[c], nn[1]);
            }
            allreduce<2, 16>(nn);
            nu = nn[0];
            nk = nn[1];
        }
        for (int t = 0; t < T; ++t) {
            const float iu = inv_norm(nu), ik = inv_norm(nk);
            float uh[CL], kh[CL], pq[CL];
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                uh[c] = uc[c] * iu;
                kh[c] = kc[c] * ik;
                pq[c] = phi(qc[c]);
                zk[c] += phi(kc[c]);  // z^key_t (eq. 11), on raw k
            }
            // products with the states before the token
            float pa[RW], pk[RW], ps[RW], po[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                pa[r] = pk[r] = ps[r] = po[r] = 0.f;
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    if (!fixed_a) pa[r] = fmaf(A[r][c], uh[c], pa[r]);
                    pk[r] = fmaf(A[r][c], kh[c], pk[r]);
                    ps[r] = fmaf(S[r][c], kh[c], ps[r]);
                    po[r] = fmaf(S[r][c], pq[c], po[r]);
                }
            }
            const float za = fixed_a ? 0.f : rowsum8(pa);
            const float ka = rowsum8(pk), sk = rowsum8(ps), sphi = rowsum8(po);
            float* x = X + (t & 1) * 2 * D;
            if ((l & 3) == 0) {
                x[rr] = za;
                x[D + rr] = ka;
            }
            const float erow = vr - sk;  // e = v - S_{t-1} k^ for row rr
            // next token's inputs (overlap the loads with the barrier)
            const bool more = t + 1 < T;
            if (more) {
                const size_t nx = (size_t)(t + 1) * D;
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    uc[c] = fixed_a ? 0.f : ld_in<TIn>(gu + nx, l + 32 * c);
                    kc[c] = ld_in<TIn>(gk + nx, l + 32 * c);
                    qc[c] = ld_in<TIn>(gq + nx, l + 32 * c);
                }
                vr = ld_in<TIn>(gv + nx, rr);
            }
            __syncthreads();
            // delta, z.k^, den and the next token's norms
            float zc[CL], d5[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                zc[c] = x[l + 32 * c];
                d5[0] = fmaf(uh[c], zc[c], d5[0]);
                d5[1] = fmaf(kh[c], zc[c], d5[1]);
                d5[2] = fmaf(pq[c], zk[c], d5[2]);
                if (more) {
                    d5[3] = fmaf(uc[c], uc[c], d5[3]);
                    d5[4] = fmaf(kc[c], kc[c], d5[4]);
                }
            }
            allreduce<5, 16>(d5);
            const float dl = 1.f + d5[0], kz = d5[1], pd = d5[2];
            const float rdl = 1.f / dl;
            // a = A_t k^ = A_{t-1} k^ - z (z.k^) / delta; ||a||^2 and a . phi(q)
            float al[CL], d2[2] = {0.f, 0.f};
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                al[c] = fmaf(-zc[c], kz * rdl, x[D + l + 32 * c]);
                d2[0] = fmaf(al[c], al[c], d2[0]);
                d2[1] = fmaf(al[c], pq[c], d2[1]);
            }
            allreduce<2, 16>(d2);
            const float ina = inv_norm(d2[0]);
            const float den = fmaxf(pd, p.eps);
            // o_t = S_t phi / den = (S_{t-1} phi + e (alpha^ . phi)) / den
            const float orow = fmaf(erow, d2[1] * ina, sphi) / den;
            if ((l & 3) == 0) {
                p.o[(size_t)bh * p.o_stride + (size_t)t * D + rr] = orow;
                ochk = fmaf(orow, 0.f, ochk);
            }
            if (l == 0 && w == 0 && (!isfinite(dl) || !isfinite(d2[0]) || !isfinite(pd))) bad = true;
#pragma unroll
            for (int c = 0; c < CL; ++c) al[c] *= ina;
            // A_t = A_{t-1} - z z^T / delta;  S_t = S_{t-1} + e alpha^^T
            float zr[RW];
            {
                const float4 a = reinterpret_cast<const float4*>(x)[r0 / 4];
                const float4 b = reinterpret_cast<const float4*>(x)[r0 / 4 + 1];
                zr[0] = a.x, zr[1] = a.y, zr[2] = a.z, zr[3] = a.w, zr[4] = b.x, zr[5] = b.y, zr[6] = b.z,
                zr[7] = b.w;
            }
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float er = __shfl_sync(FULL, erow, 4 * r);
                const float zs = -zr[r] * rdl;
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    if (!fixed_a) A[r][c] = fmaf(zs, zc[c], A[r][c]);
                    S[r][c] = fmaf(er, al[c], S[r][c]);
                }
            }
            nu = d5[3];
            nk = d5[4];
        }
        if constexpr (L::BULK_OUT) {
            // the state through shared memory and two bulk copies: the previous
            // head's copies have read the OUT area before it is rewritten
            float* oS = reinterpret_cast<float*>(sm + L::OS);
            float* oA = reinterpret_cast<float*>(sm + L::OA);
            if (it > 0) {
                if (tid == 0) bulk_wait_read();
                __syncthreads();
            }
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    const int e = (r0 + r) * D + l + 32 * c;
                    oS[e] = S[r][c];
                    oA[e] = A[r][c];
                }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                bulk_s2g(p.S_out + hdd, oS, D * D * 4);
                bulk_s2g(p.A_out + hdd, oA, D * D * 4);
                bulk_commit();
            }
        } else {
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    const size_t e = hdd + (size_t)(r0 + r) * D + l + 32 * c;
                    p.S_out[e] = S[r][c];
                    p.A_out[e] = A[r][c];
                }
        }
        if (w == 0 && p.zk_out)
#pragma unroll
            for (int c = 0; c < CL; ++c) p.zk_out[(size_t)bh * D + l + 32 * c] = zk[c];
        if (bad || ochk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_S, bh, -1);
        bad = false;
        ochk = 0.f;
    }
    if (L::BULK_OUT && tid == 0) bulk_wait_all();
}

}  // namespace dec
