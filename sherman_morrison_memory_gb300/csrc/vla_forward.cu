// vla_forward.cu -- GB300 (sm_103a) kernels and C ABI for the Variational
// Linear Attention forward recurrence ("Variational Linear Attention", arXiv
// 2605.11196, §3.3 eq. 9-11).
//
// One CTA runs one (batch, head) stream over all T tokens. Its warps split
// the per-token work into four roles that run concurrently and hand data to
// each other through shared-memory rings guarded by mbarriers:
//
//   staging warp  TMA bulk copies of q, k, v, u chunks into shared memory;
//                 per token: u^ = u/||u||, k^ = k/||k||, phi(q), v (fp32),
//                 z^key += phi(k) and den = max(phi(q) . z^key, eps)  (eq. 11)
//   A warps       A (d x d fp32) resident in registers, split into
//                 RA x CA blocks. Per token one pass over A applies the
//                 pending Sherman-Morrison update of the previous token and
//                 forms z = A u^ and w = A k^ (eq. 9); row sums are reduced
//                 with shuffles, then one named barrier per token publishes
//                 z, w and the partial sums of delta = 1 + u^ . z and
//                 z . k^ to the other A warps and to the gate warp.
//   gate warp     alpha^ = a / ||a|| with a = A_t k^ = w - z (z . k^)/delta
//                 (eq. 10, the updated A_t) and s = alpha^ . phi(q).
//   S warps       S (d x d fp32) resident in registers; rows are independent,
//                 so each warp owns whole rows. Per token: S k^ and S phi(q)
//                 from S_{t-1}, e = v - S k^, S += e alpha^^T (eq. 10), and
//                 o = (S_{t-1} phi(q) + e s) / den = S_t phi(q) / den (eq. 11).
//
// The A chain is the only strictly serial dependence; the S warps lag a few
// tokens behind it and fill the FMA pipes while the A warps wait on their
// per-token reduction. All waits are bounded (see vla_device.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "vla.h"
#include "vla_device.cuh"

namespace vla {

// ---------------------------------------------------------------------------
// Per-head-dimension configuration.
//   NA/NS   A and S warps;  CBA/CBS  column blocks per row (lanes sharing a row)
//   NG      gate warps (token t goes to gate warp t mod NG)
//   CH      tokens per staged chunk;  TB  tokens the staging warp prepares at once
//   NP      prepped chunk slots;  NRAW  raw chunk slots
//   RZ/RG   token slots of the A->gate and gate->S rings
//   PAD     pad shared vectors by 4 floats per 32 (bank spread for the
//           column-block strides of these layouts)
//   MINB    CTAs per SM the register budget is sized for
// ---------------------------------------------------------------------------
template <int D>
struct Cfg;
template <>
struct Cfg<32> {
    static constexpr int NA = 1, CBA = 4, NS = 1, CBS = 4, NG = 1, CH = 8, TB = 4, NP = 6, NRAW = 3, RZ = 16,
                         RG = 16, PAD = 1, MINB = 4;
};
template <>
struct Cfg<64> {
    static constexpr int NA = 4, CBA = 8, NS = 2, CBS = 4, NG = 1, CH = 8, TB = 4, NP = 4, NRAW = 3, RZ = 16,
                         RG = 16, PAD = 1, MINB = 2;
};
template <>
struct Cfg<96> {
    static constexpr int NA = 4, CBA = 8, NS = 4, CBS = 8, NG = 2, CH = 8, TB = 4, NP = 8, NRAW = 3, RZ = 16,
                         RG = 16, PAD = 0, MINB = 1;
};
template <>
struct Cfg<128> {
    static constexpr int NA = 8, CBA = 8, NS = 8, CBS = 4, NG = 1, CH = 8, TB = 2, NP = 6, NRAW = 2, RZ = 16,
                         RG = 16, PAD = 1, MINB = 1;
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int D, typename TIn>
struct Layout {
    using C = Cfg<D>;
    // padded length of a d-vector in shared memory
    static constexpr int VD = D + (C::PAD ? 4 * (D / 32) : 0);
    static constexpr int NA4 = (C::NA + 3) / 4 * 4;
    // prepped token record: u^ | k^ | phi(q) (padded) | v | den, pad
    static constexpr int P_U = 0, P_K = VD, P_Q = 2 * VD, P_V = 3 * VD, P_DEN = 3 * VD + D;
    static constexpr int PSTRIDE = 3 * VD + D + 4;
    // A -> gate record: z | w (padded) | per-warp partials of u^.z and k^.z
    static constexpr int Z_Z = 0, Z_W = VD, Z_DD = 2 * VD, Z_DK = 2 * VD + NA4;
    static constexpr int ZSTRIDE = 2 * VD + 2 * NA4;
    // gate -> S record: alpha^ (padded) | s = alpha^ . phi(q), pad
    static constexpr int G_A = 0, G_S = VD;
    static constexpr int GSTRIDE = VD + 4;
    // warp roles
    static constexpr int W_PROD = 0, W_GATE = 1, W_A0 = 1 + C::NG, W_S0 = 1 + C::NG + C::NA;
    static constexpr int NWARPS = 1 + C::NG + C::NA + C::NS, THREADS = 32 * NWARPS;
    // shared memory map (bytes)
    static constexpr int NBAR = C::NRAW + 2 * C::NP + 2 * C::RZ + 2 * C::RG;
    static constexpr size_t OFF_FLAG = 8 * (size_t)NBAR;
    static constexpr size_t RAW_TENSOR = (size_t)C::CH * D * sizeof(TIn);
    static constexpr size_t OFF_RAW = align_up(OFF_FLAG + 16, 128);
    static constexpr size_t OFF_PREP = align_up(OFF_RAW + (size_t)C::NRAW * 4 * RAW_TENSOR, 128);
    static constexpr size_t OFF_Z = align_up(OFF_PREP + (size_t)C::NP * C::CH * PSTRIDE * 4, 128);
    static constexpr size_t OFF_G = align_up(OFF_Z + (size_t)C::RZ * ZSTRIDE * 4, 128);
    static constexpr size_t SMEM = align_up(OFF_G + (size_t)C::RG * GSTRIDE * 4, 128);

    static_assert(VD % 4 == 0 && PSTRIDE % 4 == 0 && ZSTRIDE % 4 == 0 && GSTRIDE % 4 == 0, "float4 records");
    static_assert(RAW_TENSOR % 16 == 0, "bulk-copy granularity");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

template <int D>
__device__ __forceinline__ int vidx(int j) {
    return Cfg<D>::PAD ? j + 4 * (j >> 5) : j;
}

struct Params {
    const void* q;
    const void* k;
    const void* v;
    const void* u;
    const float* S0;
    const float* A0;
    const float* zk0;
    float* o;
    float* S_out;
    float* A_out;
    float* zk_out;
    DeviceStatus* status;
    int T;
    float inv_lambda0;
    float eps;
    unsigned long long wait_ns;
    int stall_producer;
    unsigned long long* trace;
};

// Per-token clock stamps of head 0 for pipeline analysis (-DVLA_TRACE builds only).
#ifdef VLA_TRACE
#define VLA_TRACE_AT(p, role, t)                                                              \
    do {                                                                                      \
        if ((p).trace && blockIdx.x == 0) (p).trace[(size_t)(role) * (p).T + (t)] = clock64(); \
    } while (0)
// sub-step stamps of one thread (rows 5.. of the trace buffer)
#define VLA_TRACE_PT(p, row, t) VLA_TRACE_AT(p, row, t)
#else
#define VLA_TRACE_AT(p, role, t) \
    do {                         \
    } while (0)
#define VLA_TRACE_PT(p, row, t) \
    do {                        \
    } while (0)
#endif

struct Smem {
    uint64_t* full_r;   // raw chunk landed (TMA tx)
    uint64_t* full_p;   // prepped chunk published
    uint64_t* empty_p;  // prepped chunk released by the S warps (its last readers)
    uint64_t* full_z;   // z/w of a token published by the A warps
    uint64_t* empty_z;  // ... released by the gate
    uint64_t* full_g;   // alpha^ of a token published by the gate
    uint64_t* empty_g;  // ... released by the S warps
    volatile int* abort;
    unsigned char* raw;
    float* prep;
    float* zr;
    float* gr;
};

__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : expf(x); }

template <typename TIn>
__device__ __forceinline__ float ld_in(const TIn* p, int j);
template <>
__device__ __forceinline__ float ld_in<float>(const float* p, int j) {
    return p[j];
}
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p, int j) {
    return __bfloat162float(p[j]);
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

enum Role { ROLE_STAGE = 0, ROLE_GATE = 1, ROLE_A = 2, ROLE_S = 3 };

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

// Sum of N per-warp partials stored contiguously (N a multiple of 4 is read
// with float4 loads), in a fixed tree order so every reader gets the same bits.
template <int N>
__device__ __forceinline__ float sum_partials(const float* p) {
    if constexpr (N % 4 == 0) {
        float4 acc = ld4(p);
#pragma unroll
        for (int i = 4; i < N; i += 4) {
            const float4 x = ld4(p + i);
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
        }
        return (acc.x + acc.y) + (acc.z + acc.w);
    } else {
        float s = p[0];
#pragma unroll
        for (int i = 1; i < N; ++i) s += p[i];
        return s;
    }
}

// ---------------------------------------------------------------------------
// staging warp: TMA bulk copies of raw q, k, v, u chunks, then per token
// u^, k^ (unit), phi(q), v (fp32), z^key += phi(k), den = max(phi(q).z^key, eps)
// (§3.2-3.3, eq. 11). Tokens are processed TB at a time so that the
// cross-lane reductions of several tokens overlap.
// ---------------------------------------------------------------------------
template <int D, typename TIn>
__device__ __forceinline__ void stage_role(const Params& p, const Smem& sm, int bh, int lane) {
    using C = Cfg<D>;
    using LY = Layout<D, TIn>;
    constexpr int E = D / 32;
    constexpr int TB = C::TB;
    static_assert(C::CH % TB == 0, "token batch divides the chunk");
    const int T = p.T;
    const int nch = (T + C::CH - 1) / C::CH;
    const size_t head = (size_t)bh * T * D;
    const TIn* src[4] = {static_cast<const TIn*>(p.q) + head, static_cast<const TIn*>(p.k) + head,
                         static_cast<const TIn*>(p.v) + head, static_cast<const TIn*>(p.u) + head};

    // testing hook: publish nothing and raise no flag, so that every consumer
    // runs into its own wait limit
    if (p.stall_producer) return;

    float zk[E];
#pragma unroll
    for (int m = 0; m < E; ++m) zk[m] = p.zk0 ? p.zk0[(size_t)bh * D + lane + 32 * m] : 0.f;

    auto issue = [&](int c) {  // lane 0 only
        const int rs = c % C::NRAW;
        const int nt = min(C::CH, T - c * C::CH);
        const uint32_t bytes = (uint32_t)(nt * D * sizeof(TIn));
        mbar_arrive_expect_tx(sm.full_r + rs, 4 * bytes);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            bulk_g2s(sm.raw + (size_t)(rs * 4 + i) * LY::RAW_TENSOR, src[i] + (size_t)c * C::CH * D, bytes,
                     sm.full_r + rs);
    };

    bool abort = false;
    int issued = min(C::NRAW, nch), landed = 0, c = 0;
    if (lane == 0)
        for (int i = 0; i < issued; ++i) issue(i);
    for (; c < nch; ++c) {
        const int rs = c % C::NRAW, ps = c % C::NP;
        if (!mbar_wait(sm.full_r + rs, (c / C::NRAW) & 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        landed = c + 1;
        if (lane == 0) VLA_TRACE_PT(p, 14, c * C::CH);
        if (!mbar_wait(sm.empty_p + ps, ((c / C::NP) & 1) ^ 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        if (lane == 0) VLA_TRACE_PT(p, 15, c * C::CH);
        const int nt = min(C::CH, T - c * C::CH);
        const TIn* raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[i] = reinterpret_cast<const TIn*>(sm.raw + (size_t)(rs * 4 + i) * LY::RAW_TENSOR);
        float* P0 = sm.prep + (size_t)ps * C::CH * LY::PSTRIDE;
        for (int tb = 0; tb < nt; tb += TB) {
            float qv[TB][E], kv[TB][E], vv[TB][E], uv[TB][E];
            float red[3 * TB];  // per token: ||u||^2, ||k||^2, phi(q) . z^key
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                const bool live = tb + b < nt;
                float uu = 0.f, kk = 0.f, qz = 0.f;
#pragma unroll
                for (int m = 0; m < E; ++m) {
                    const int j = (tb + b) * D + lane + 32 * m;
                    qv[b][m] = live ? ld_in<TIn>(raw[0], j) : 0.f;
                    kv[b][m] = live ? ld_in<TIn>(raw[1], j) : 0.f;
                    vv[b][m] = live ? ld_in<TIn>(raw[2], j) : 0.f;
                    uv[b][m] = live ? ld_in<TIn>(raw[3], j) : 0.f;
                    uu = fmaf(uv[b][m], uv[b][m], uu);
                    kk = fmaf(kv[b][m], kv[b][m], kk);
                    if (live) zk[m] += phi(kv[b][m]);
                    qv[b][m] = phi(qv[b][m]);
                    qz = fmaf(qv[b][m], zk[m], qz);
                }
                red[3 * b] = uu;
                red[3 * b + 1] = kk;
                red[3 * b + 2] = qz;
            }
            allreduce<3 * TB, 16>(red);
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                if (tb + b < nt) {
                    const float iu = rsqrtf(fmaxf(red[3 * b], 1e-24f));  // 1 / max(||u||, 1e-12)
                    const float ik = rsqrtf(fmaxf(red[3 * b + 1], 1e-24f));
                    float* P = P0 + (tb + b) * LY::PSTRIDE;
#pragma unroll
                    for (int m = 0; m < E; ++m) {
                        const int j = lane + 32 * m;
                        P[LY::P_U + vidx<D>(j)] = uv[b][m] * iu;
                        P[LY::P_K + vidx<D>(j)] = kv[b][m] * ik;
                        P[LY::P_Q + vidx<D>(j)] = qv[b][m];
                        P[LY::P_V + j] = vv[b][m];
                    }
                    if (lane == 0) P[LY::P_DEN] = fmaxf(red[3 * b + 2], p.eps);
                }
            }
        }
        // our generic-proxy reads of raw slot rs are done before the TMA refill
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(sm.full_p + ps);
            VLA_TRACE_AT(p, 0, c * C::CH);
            if (c + C::NRAW < nch) issue(c + C::NRAW);
        }
        issued = min(c + 1 + C::NRAW, nch);
    }
    if (abort) {
        if (lane == 0) record_failure(p.status, BIT_TIMEOUT, ROLE_STAGE, bh, c * C::CH);
        *sm.abort = 1;
        // let copies already in flight land before the CTA can exit
        for (int cc = landed; cc < issued; ++cc)
            (void)mbar_wait(sm.full_r + cc % C::NRAW, (cc / C::NRAW) & 1, nullptr, p.wait_ns);
        return;
    }
    if (p.zk_out) {
#pragma unroll
        for (int m = 0; m < E; ++m) p.zk_out[(size_t)bh * D + lane + 32 * m] = zk[m];
    }
}

// ---------------------------------------------------------------------------
// gate warps: alpha^_t = A_t k^ / ||A_t k^|| (eq. 10) from the published z, w,
// with A_t k^ = w - z (z . k^) / delta. Gate warp g handles tokens t = g mod NG.
// ---------------------------------------------------------------------------
template <int D, typename TIn>
__device__ __forceinline__ void gate_role(const Params& p, const Smem& sm, int bh, int g, int lane) {
    using C = Cfg<D>;
    using LY = Layout<D, TIn>;
    constexpr int E = D / 32;
    bool abort = false, nonfinite = false;
    int t = g;
    for (; t < p.T; t += C::NG) {
        const int zs = t % C::RZ;
        if (!mbar_wait(sm.full_z + zs, (t / C::RZ) & 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        const int chunk = t / C::CH, tc = t - chunk * C::CH, ps = chunk % C::NP;
        if (tc < C::NG && !mbar_wait(sm.full_p + ps, (chunk / C::NP) & 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        const float* Z = sm.zr + (size_t)zs * LY::ZSTRIDE;
        const float* P = sm.prep + (size_t)(ps * C::CH + tc) * LY::PSTRIDE;
        if (lane == 0 && g == 0) VLA_TRACE_PT(p, 11, t);
        const float delta = 1.f + sum_partials<C::NA>(Z + LY::Z_DD);
        const float zkd = sum_partials<C::NA>(Z + LY::Z_DK);
        const float cf = zkd * __frcp_rn(delta);
        float av[E];
        float red[2] = {0.f, 0.f};  // ||a||^2, a . phi(q)
#pragma unroll
        for (int m = 0; m < E; ++m) {
            const int j = vidx<D>(lane + 32 * m);
            av[m] = fmaf(-cf, Z[LY::Z_Z + j], Z[LY::Z_W + j]);
            red[0] = fmaf(av[m], av[m], red[0]);
            red[1] = fmaf(av[m], P[LY::P_Q + j], red[1]);
        }
        allreduce<2, 16>(red);
        if (lane == 0 && g == 0) VLA_TRACE_PT(p, 12, t);
        const float inv = rsqrtf(fmaxf(red[0], 1e-24f));  // 1 / max(||a||, 1e-12)
        if (!(isfinite(delta) && isfinite(red[0]) && isfinite(red[1]))) nonfinite = true;
        const int gs = t % C::RG;
        if (!mbar_wait(sm.empty_g + gs, ((t / C::RG) & 1) ^ 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        if (lane == 0 && g == 0) VLA_TRACE_PT(p, 13, t);
        float* G = sm.gr + (size_t)gs * LY::GSTRIDE;
#pragma unroll
        for (int m = 0; m < E; ++m) G[LY::G_A + vidx<D>(lane + 32 * m)] = av[m] * inv;
        if (lane == 0) G[LY::G_S] = red[1] * inv;
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(sm.full_g + gs);
            VLA_TRACE_AT(p, 2, t);
            mbar_arrive(sm.empty_z + zs);
        }
    }
    if (abort) {
        if (lane == 0) record_failure(p.status, BIT_TIMEOUT, ROLE_GATE, bh, t);
        *sm.abort = 1;
    }
    if (nonfinite && lane == 0) record_failure(p.status, BIT_NONFINITE, ROLE_GATE, bh, -1);
}

// ---------------------------------------------------------------------------
// A warps: Sherman-Morrison chain (eq. 9), A resident in registers as float2
// pairs (packed fp32 FMA). Per token one pass over A applies the pending
// update of the previous token, A -= (z/delta) z^T, and accumulates
// z = A u^ and w = A k^.
// ---------------------------------------------------------------------------
template <int D, typename TIn>
__device__ __forceinline__ void a_role(const Params& p, const Smem& sm, int bh, int warp, int lane) {
    using C = Cfg<D>;
    using LY = Layout<D, TIn>;
    constexpr int RPW = 32 / C::CBA;              // row groups per warp
    constexpr int RA = D / (C::NA * RPW);         // rows per thread
    constexpr int CA = D / C::CBA;                // columns per thread
    constexpr int C2 = CA / 2;                    // float2 columns
    constexpr int NV = 2 * RA + 2;                // z rows, w rows, u^.z and k^.z partials
    constexpr int HR = C::CBA / 2;
    constexpr int NOUT = rs_count<NV, HR>();
    static_assert(RA * C::NA * RPW == D && CA * C::CBA == D && CA % 4 == 0, "A layout");

    const int wa = warp - LY::W_A0;
    const int cb = lane % C::CBA, rgl = lane / C::CBA;
    const int row0 = (wa * RPW + rgl) * RA, col0 = cb * CA;

    float2 a[RA][C2];
    {
        const float* A0 = p.A0 ? p.A0 + (size_t)bh * D * D : nullptr;
#pragma unroll
        for (int r = 0; r < RA; ++r)
#pragma unroll
            for (int c = 0; c < C2; ++c) {
                const int i = row0 + r, j = col0 + 2 * c;
                a[r][c] = A0 ? f2(A0[(size_t)i * D + j], A0[(size_t)i * D + j + 1])
                             : f2(i == j ? p.inv_lambda0 : 0.f, i == j + 1 ? p.inv_lambda0 : 0.f);
            }
    }
    // pending rank-1 update of the previous token: A -= (z/delta) z^T
    float2 nyr[RA], zj[C2];
#pragma unroll
    for (int r = 0; r < RA; ++r) nyr[r] = f2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < C2; ++c) zj[c] = f2(0.f, 0.f);

    // this token's u^, k^ (columns, and rows for the scalar partials)
    float2 uj[C2], kj[C2];
    float ui[RA], ki[RA];
    auto load_token = [&](const float* P) {
#pragma unroll
        for (int c4 = 0; c4 < CA; c4 += 4) {
            const float4 u4 = ld4(P + LY::P_U + vidx<D>(col0 + c4));
            const float4 k4 = ld4(P + LY::P_K + vidx<D>(col0 + c4));
            uj[c4 / 2] = f2(u4.x, u4.y);
            uj[c4 / 2 + 1] = f2(u4.z, u4.w);
            kj[c4 / 2] = f2(k4.x, k4.y);
            kj[c4 / 2 + 1] = f2(k4.z, k4.w);
        }
#pragma unroll
        for (int r = 0; r < RA; ++r) {
            ui[r] = P[LY::P_U + vidx<D>(row0 + r)];
            ki[r] = P[LY::P_K + vidx<D>(row0 + r)];
        }
    };

    bool abort = false;
    int t = 0;
    if (p.T > 0) {
        if (!mbar_wait(sm.full_p, 0, sm.abort, p.wait_ns)) abort = true;
        load_token(sm.prep);
    }
    for (; t < p.T; ++t) {
        const bool tr0 = (wa == 0 && lane == 0);
        if (tr0) VLA_TRACE_PT(p, 5, t);

        // one pass over A: apply the pending update, then z = A u^, w = A k^
        float2 pz[RA], pw[RA];
#pragma unroll
        for (int r = 0; r < RA; ++r) pz[r] = pw[r] = f2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < C2; ++c)
#pragma unroll
            for (int r = 0; r < RA; ++r) {
                const float2 x = __ffma2_rn(nyr[r], zj[c], a[r][c]);
                a[r][c] = x;
                pz[r] = __ffma2_rn(x, uj[c], pz[r]);
                pw[r] = __ffma2_rn(x, kj[c], pw[r]);
            }
        float vals[NV];
        float dd = 0.f, dk = 0.f;
#pragma unroll
        for (int r = 0; r < RA; ++r) {
            const float z = pz[r].x + pz[r].y;
            vals[r] = z;
            vals[RA + r] = pw[r].x + pw[r].y;
            dd = fmaf(ui[r], z, dd);
            dk = fmaf(ki[r], z, dk);
        }
        vals[2 * RA] = dd;
        vals[2 * RA + 1] = dk;
        if (tr0) VLA_TRACE_PT(p, 6, t);
        reduce_scatter<NV, HR>(vals, lane);
        // the two scalar partials also need the sum over this warp's row groups
        float sc[NOUT];
#pragma unroll
        for (int j = 0; j < NOUT; ++j) sc[j] = vals[j];
#pragma unroll
        for (int h = C::CBA; h < 32; h <<= 1)
#pragma unroll
            for (int j = 0; j < NOUT; ++j) sc[j] += __shfl_xor_sync(0xffffffffu, sc[j], h);

        const int zs = t % C::RZ;
        if (tr0) VLA_TRACE_PT(p, 7, t);
        if (!abort && !mbar_wait(sm.empty_z + zs, ((t / C::RZ) & 1) ^ 1, sm.abort, p.wait_ns)) abort = true;
        if (tr0) VLA_TRACE_PT(p, 8, t);
        float* Z = sm.zr + (size_t)zs * LY::ZSTRIDE;
#pragma unroll
        for (int j = 0; j < NOUT; ++j) {
            const int idx = rs_index<NV, HR>(cb, j);
            if (idx < 0)
                continue;
            else if (idx < RA)
                Z[LY::Z_Z + vidx<D>(row0 + idx)] = vals[j];
            else if (idx < 2 * RA)
                Z[LY::Z_W + vidx<D>(row0 + idx - RA)] = vals[j];
            else if (rgl == 0 && idx == 2 * RA)
                Z[LY::Z_DD + wa] = sc[j];
            else if (rgl == 0 && idx == 2 * RA + 1)
                Z[LY::Z_DK + wa] = sc[j];
        }
        // prefetch the next token's vectors while the other A warps catch up
        if (t + 1 < p.T) {
            const int t1 = t + 1, chunk1 = t1 / C::CH, tc1 = t1 - chunk1 * C::CH, ps1 = chunk1 % C::NP;
            if (tc1 == 0 && !abort && !mbar_wait(sm.full_p + ps1, (chunk1 / C::NP) & 1, sm.abort, p.wait_ns))
                abort = true;
            load_token(sm.prep + (size_t)(ps1 * C::CH + tc1) * LY::PSTRIDE);
        }
        // publish among the A warps; every A thread takes the same abort decision
        if (bar_red_or(1, C::NA * 32, abort || (*sm.abort != 0))) {
            abort = true;
            break;
        }
        if (tr0) VLA_TRACE_PT(p, 9, t);
        if (wa == 0 && lane == 0) {
            mbar_arrive(sm.full_z + zs);
            VLA_TRACE_AT(p, 1, t);
        }
        const float delta = 1.f + sum_partials<C::NA>(Z + LY::Z_DD);
        const float inv = __frcp_rn(delta);
#pragma unroll
        for (int r = 0; r < RA; ++r) {
            const float y = -Z[LY::Z_Z + vidx<D>(row0 + r)] * inv;
            nyr[r] = f2(y, y);
        }
#pragma unroll
        for (int c4 = 0; c4 < CA; c4 += 4) {
            const float4 z4 = ld4(Z + LY::Z_Z + vidx<D>(col0 + c4));
            zj[c4 / 2] = f2(z4.x, z4.y);
            zj[c4 / 2 + 1] = f2(z4.z, z4.w);
        }
        if (tr0) VLA_TRACE_PT(p, 10, t);
    }
    if (abort) {
        if (wa == 0 && lane == 0) record_failure(p.status, BIT_TIMEOUT, ROLE_A, bh, t);
        *sm.abort = 1;
        return;
    }
    float* Ao = p.A_out + (size_t)bh * D * D;
#pragma unroll
    for (int r = 0; r < RA; ++r)
#pragma unroll
        for (int c = 0; c < C2; c += 2) {
            const float2 x0 = __ffma2_rn(nyr[r], zj[c], a[r][c]);
            const float2 x1 = __ffma2_rn(nyr[r], zj[c + 1], a[r][c + 1]);
            *reinterpret_cast<float4*>(Ao + (size_t)(row0 + r) * D + col0 + 2 * c) = make_float4(x0.x, x0.y, x1.x, x1.y);
        }
}

// ---------------------------------------------------------------------------
// S warps: residual write and readout (eq. 10-11), S resident in registers as
// float2 pairs; each warp owns whole rows.
// ---------------------------------------------------------------------------
template <int D, typename TIn>
__device__ __forceinline__ void s_role(const Params& p, const Smem& sm, int bh, int warp, int lane) {
    using C = Cfg<D>;
    using LY = Layout<D, TIn>;
    constexpr int RPW = 32 / C::CBS;
    constexpr int RS = D / (C::NS * RPW);
    constexpr int CS = D / C::CBS;
    constexpr int C2 = CS / 2;
    constexpr int HS = C::CBS / 2;
    constexpr int NOUT = rs_count<RS, HS>();
    static_assert(RS * C::NS * RPW == D && CS * C::CBS == D && CS % 4 == 0, "S layout");

    const int ws = warp - LY::W_S0;
    const int cb = lane % C::CBS, rgl = lane / C::CBS;
    const int row0 = (ws * RPW + rgl) * RS, col0 = cb * CS;

    float2 s[RS][C2];
    {
        const float* S0 = p.S0 ? p.S0 + (size_t)bh * D * D : nullptr;
#pragma unroll
        for (int r = 0; r < RS; ++r)
#pragma unroll
            for (int c = 0; c < C2; ++c)
                s[r][c] = S0 ? f2(S0[(size_t)(row0 + r) * D + col0 + 2 * c], S0[(size_t)(row0 + r) * D + col0 + 2 * c + 1])
                             : f2(0.f, 0.f);
    }
    float* o = p.o + (size_t)bh * p.T * D;

    bool abort = false;
    int t = 0;
    for (; t < p.T; ++t) {
        const int chunk = t / C::CH, tc = t - chunk * C::CH, ps = chunk % C::NP;
        if (tc == 0 && !mbar_wait(sm.full_p + ps, (chunk / C::NP) & 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        const float* P = sm.prep + (size_t)(ps * C::CH + tc) * LY::PSTRIDE;
        // S_{t-1} k^ and S_{t-1} phi(q)
        float2 sk2[RS], sq2[RS];
#pragma unroll
        for (int r = 0; r < RS; ++r) sk2[r] = sq2[r] = f2(0.f, 0.f);
#pragma unroll
        for (int c4 = 0; c4 < CS; c4 += 4) {
            const float4 k4 = ld4(P + LY::P_K + vidx<D>(col0 + c4));
            const float4 q4 = ld4(P + LY::P_Q + vidx<D>(col0 + c4));
            const float2 ka = f2(k4.x, k4.y), kb = f2(k4.z, k4.w);
            const float2 qa = f2(q4.x, q4.y), qb = f2(q4.z, q4.w);
#pragma unroll
            for (int r = 0; r < RS; ++r) {
                sk2[r] = __ffma2_rn(s[r][c4 / 2], ka, sk2[r]);
                sk2[r] = __ffma2_rn(s[r][c4 / 2 + 1], kb, sk2[r]);
                sq2[r] = __ffma2_rn(s[r][c4 / 2], qa, sq2[r]);
                sq2[r] = __ffma2_rn(s[r][c4 / 2 + 1], qb, sq2[r]);
            }
        }
        float sk[RS], sq[RS];
#pragma unroll
        for (int r = 0; r < RS; ++r) {
            sk[r] = sk2[r].x + sk2[r].y;
            sq[r] = sq2[r].x + sq2[r].y;
        }
        // reduce both over the row group's lanes with one mapping: slot j of this
        // lane holds row idx_j of S k^ and of S phi(q)
        reduce_scatter<RS, HS>(sk, lane);
        reduce_scatter<RS, HS>(sq, lane);
        float ej[NOUT];
#pragma unroll
        for (int j = 0; j < NOUT; ++j) {
            const int idx = rs_index<RS, HS>(cb, j);
            ej[j] = idx >= 0 ? P[LY::P_V + row0 + idx] - sk[j] : 0.f;
        }

        const int gs = t % C::RG;
        if (!mbar_wait(sm.full_g + gs, (t / C::RG) & 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        const float* G = sm.gr + (size_t)gs * LY::GSTRIDE;
        const float st = G[LY::G_S];
        const float rden = __frcp_rn(P[LY::P_DEN]);
        // o_t = (S_{t-1} phi(q) + e (alpha^ . phi(q))) / den = S_t phi(q) / den
#pragma unroll
        for (int j = 0; j < NOUT; ++j) {
            const int idx = rs_index<RS, HS>(cb, j);
            if (idx >= 0) o[(size_t)t * D + row0 + idx] = fmaf(ej[j], st, sq[j]) * rden;
        }
        // every lane of the row group needs the whole residual for the write
        float2 e2[RS];
        const int gbase = lane & ~(C::CBS - 1);
#pragma unroll
        for (int r = 0; r < RS; ++r) {
            const float er = __shfl_sync(0xffffffffu, ej[rs_owner_slot<RS, HS>(r)], gbase | rs_owner_lane<RS, HS>(r));
            e2[r] = f2(er, er);
        }
#pragma unroll
        for (int c4 = 0; c4 < CS; c4 += 4) {
            const float4 a4 = ld4(G + LY::G_A + vidx<D>(col0 + c4));
            const float2 aa = f2(a4.x, a4.y), ab = f2(a4.z, a4.w);
#pragma unroll
            for (int r = 0; r < RS; ++r) {
                s[r][c4 / 2] = __ffma2_rn(e2[r], aa, s[r][c4 / 2]);
                s[r][c4 / 2 + 1] = __ffma2_rn(e2[r], ab, s[r][c4 / 2 + 1]);
            }
        }
        __syncwarp();
        if (lane == 0) {
            if (ws == 0) VLA_TRACE_AT(p, 3, t);
            if (ws == C::NS - 1) VLA_TRACE_AT(p, 4, t);
            mbar_arrive(sm.empty_g + gs);
            if (tc == C::CH - 1 || t == p.T - 1) mbar_arrive(sm.empty_p + ps);
        }
    }
    if (abort) {
        if (ws == 0 && lane == 0) record_failure(p.status, BIT_TIMEOUT, ROLE_S, bh, t);
        *sm.abort = 1;
        return;
    }
    float* So = p.S_out + (size_t)bh * D * D;
#pragma unroll
    for (int r = 0; r < RS; ++r)
#pragma unroll
        for (int c = 0; c < C2; c += 2)
            *reinterpret_cast<float4*>(So + (size_t)(row0 + r) * D + col0 + 2 * c) =
                make_float4(s[r][c].x, s[r][c].y, s[r][c + 1].x, s[r][c + 1].y);
}

template <int D, typename TIn>
__global__ void __launch_bounds__(Layout<D, TIn>::THREADS, Cfg<D>::MINB) vla_fused_kernel(const Params p) {
    using C = Cfg<D>;
    using LY = Layout<D, TIn>;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    Smem sm;
    sm.full_r = bars;
    sm.full_p = sm.full_r + C::NRAW;
    sm.empty_p = sm.full_p + C::NP;
    sm.full_z = sm.empty_p + C::NP;
    sm.empty_z = sm.full_z + C::RZ;
    sm.full_g = sm.empty_z + C::RZ;
    sm.empty_g = sm.full_g + C::RG;
    sm.abort = reinterpret_cast<volatile int*>(smem + LY::OFF_FLAG);
    sm.raw = smem + LY::OFF_RAW;
    sm.prep = reinterpret_cast<float*>(smem + LY::OFF_PREP);
    sm.zr = reinterpret_cast<float*>(smem + LY::OFF_Z);
    sm.gr = reinterpret_cast<float*>(smem + LY::OFF_G);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NRAW; ++i) mbar_init(sm.full_r + i, 1);
        for (int i = 0; i < C::NP; ++i) {
            mbar_init(sm.full_p + i, 1);
            mbar_init(sm.empty_p + i, C::NS);  // the S warps are the last readers of a chunk
        }
        for (int i = 0; i < C::RZ; ++i) {
            mbar_init(sm.full_z + i, 1);
            mbar_init(sm.empty_z + i, 1);
        }
        for (int i = 0; i < C::RG; ++i) {
            mbar_init(sm.full_g + i, 1);
            mbar_init(sm.empty_g + i, C::NS);
        }
        *sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == LY::W_PROD)
        stage_role<D, TIn>(p, sm, bh, lane);
    else if (warp < LY::W_A0)
        gate_role<D, TIn>(p, sm, bh, warp - LY::W_GATE, lane);
    else if (warp < LY::W_S0)
        a_role<D, TIn>(p, sm, bh, warp, lane);
    else
        s_role<D, TIn>(p, sm, bh, warp, lane);
}

// ---------------------------------------------------------------------------
// plain cumulative linear-attention state S = sum_t v_t phi(k_t)^T (§4.1)
// ---------------------------------------------------------------------------
constexpr int LA_THREADS = 256, LA_TT = 16;

template <typename TIn>
__global__ void __launch_bounds__(LA_THREADS) la_state_kernel(const TIn* k, const TIn* v, int T, int D,
                                                              float* S_out) {
    __shared__ float sv[LA_TT][128], sk[LA_TT][128];
    const size_t base = (size_t)blockIdx.x * T * D;
    const int DD = D * D;
    float acc[64];
#pragma unroll
    for (int m = 0; m < 64; ++m) acc[m] = 0.f;
    for (int t0 = 0; t0 < T; t0 += LA_TT) {
        const int nt = min(LA_TT, T - t0);
        for (int i = threadIdx.x; i < nt * D; i += LA_THREADS) {
            const int tt = i / D, j = i - tt * D;
            sv[tt][j] = ld_in<TIn>(v + base + (size_t)t0 * D, i);
            sk[tt][j] = phi(ld_in<TIn>(k + base + (size_t)t0 * D, i));
        }
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
#pragma unroll
            for (int m = 0; m < 64; ++m) {
                const int e = threadIdx.x + LA_THREADS * m;
                if (e < DD) acc[m] = fmaf(sv[tt][e / D], sk[tt][e % D], acc[m]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int m = 0; m < 64; ++m) {
        const int e = threadIdx.x + LA_THREADS * m;
        if (e < DD) S_out[(size_t)blockIdx.x * DD + e] = acc[m];
    }
}

}  // namespace vla

// ===========================================================================
// C ABI
// ===========================================================================
namespace {

constexpr size_t kWorkspaceBytes = 256;
constexpr unsigned kDefaultWaitUs = 2000000u;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

template <int D, typename TIn>
vla_status launch_fused(const vla::Params& p, int BH, cudaStream_t s) {
    using LY = vla::Layout<D, TIn>;
    auto kern = vla::vla_fused_kernel<D, TIn>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::SMEM) != cudaSuccess)
        return VLA_ERR_CUDA;
    kern<<<BH, LY::THREADS, LY::SMEM, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

template <typename TIn>
vla_status launch_d(int d, const vla::Params& p, int BH, cudaStream_t s) {
    switch (d) {
        case 32: return launch_fused<32, TIn>(p, BH, s);
        case 64: return launch_fused<64, TIn>(p, BH, s);
        case 96: return launch_fused<96, TIn>(p, BH, s);
        case 128: return launch_fused<128, TIn>(p, BH, s);
        default: return VLA_ERR_UNSUPPORTED;
    }
}

}  // namespace

extern "C" {

size_t vla_workspace_bytes(void) { return kWorkspaceBytes; }

vla_status vla_workspace_reset(void* workspace, void* stream) {
    if (!workspace || !aligned16(workspace)) return VLA_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, sizeof(vla::DeviceStatus), static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? VLA_OK
               : VLA_ERR_CUDA;
}

vla_status vla_forward_ex(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B,
                          int H, int T, int d, float lambda0, float eps, const float* S0, const float* A0,
                          const float* zk0, float* o, float* S_out, float* A_out, float* zk_out,
                          void* workspace, size_t workspace_bytes, void* stream, const vla_options* opts) {
    if (B < 0 || H < 0 || T < 0) return VLA_ERR_INVALID_ARG;
    if (dtype != VLA_F32 && dtype != VLA_BF16) return VLA_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 96 && d != 128) return VLA_ERR_UNSUPPORTED;
    if (!(lambda0 > 0.f) || !std::isfinite(lambda0)) return VLA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !std::isfinite(eps)) return VLA_ERR_INVALID_ARG;
    const long long BH = (long long)B * H;
    if (BH > 2147483647LL) return VLA_ERR_INVALID_ARG;
    if ((unsigned long long)BH * (unsigned long long)T * (unsigned long long)d > (1ULL << 60))
        return VLA_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < kWorkspaceBytes) return VLA_ERR_INVALID_ARG;
    if (BH == 0) return VLA_OK;
    if (T > 0) {
        if (!q || !k || !v || !u || !o) return VLA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(u) || !aligned16(o))
            return VLA_ERR_INVALID_ARG;
    }
    if (!S_out || !A_out || !aligned16(S_out) || !aligned16(A_out)) return VLA_ERR_INVALID_ARG;
    if ((S0 && !aligned4(S0)) || (A0 && !aligned4(A0)) || (zk0 && !aligned4(zk0)) ||
        (zk_out && !aligned4(zk_out)))
        return VLA_ERR_INVALID_ARG;

    vla::Params p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.u = u;
    p.S0 = S0;
    p.A0 = A0;
    p.zk0 = zk0;
    p.o = o;
    p.S_out = S_out;
    p.A_out = A_out;
    p.zk_out = zk_out;
    p.status = static_cast<vla::DeviceStatus*>(workspace);
    p.T = T;
    p.inv_lambda0 = 1.0f / lambda0;
    p.eps = eps;
    const unsigned wait_us = (opts && opts->wait_limit_us) ? opts->wait_limit_us : kDefaultWaitUs;
    p.wait_ns = 1000ull * wait_us;
    p.stall_producer = (opts && opts->test_stall_producer) ? 1 : 0;
    p.trace = opts ? opts->trace : nullptr;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == VLA_BF16 ? launch_d<__nv_bfloat16>(d, p, (int)BH, s) : launch_d<float>(d, p, (int)BH, s);
}

vla_status vla_forward(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B, int H,
                       int T, int d, float lambda0, float eps, const float* S0, const float* A0,
                       const float* zk0, float* o, float* S_out, float* A_out, float* zk_out, void* workspace,
                       size_t workspace_bytes, void* stream) {
    return vla_forward_ex(q, k, v, u, dtype, B, H, T, d, lambda0, eps, S0, A0, zk0, o, S_out, A_out, zk_out,
                          workspace, workspace_bytes, stream, nullptr);
}

vla_status vla_get_last_device_status(void* workspace, void* stream, int* detail) {
    if (detail) detail[0] = detail[1] = detail[2] = -1;
    if (!workspace || !aligned16(workspace)) return VLA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    vla::DeviceStatus h;
    if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return VLA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VLA_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(h), s) != cudaSuccess) return VLA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VLA_ERR_CUDA;
    if (h.bits == 0) return VLA_OK;
    if (detail) {
        detail[0] = h.role;
        detail[1] = h.head;
        detail[2] = h.token;
    }
    if (h.bits & vla::BIT_TIMEOUT) return VLA_ERR_TIMEOUT;
    return VLA_ERR_NONFINITE;
}

const char* vla_status_string(vla_status st) {
    switch (st) {
        case VLA_OK: return "ok";
        case VLA_ERR_INVALID_ARG: return "invalid argument";
        case VLA_ERR_UNSUPPORTED: return "unsupported head dimension (use 32, 64, 96 or 128)";
        case VLA_ERR_CUDA: return "CUDA runtime error";
        case VLA_ERR_TIMEOUT: return "in-kernel wait timed out; outputs are invalid";
        case VLA_ERR_NONFINITE: return "non-finite value in delta or the gate norm";
        default: return "unknown status";
    }
}

vla_status vla_linear_attention_state(const void* k, const void* v, vla_dtype dtype, int B, int H, int T, int d,
                                      float* S_out, void* stream) {
    if (B < 0 || H < 0 || T < 0) return VLA_ERR_INVALID_ARG;
    if (dtype != VLA_F32 && dtype != VLA_BF16) return VLA_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 96 && d != 128) return VLA_ERR_UNSUPPORTED;
    const long long BH = (long long)B * H;
    if (BH > 2147483647LL) return VLA_ERR_INVALID_ARG;
    if (BH == 0) return VLA_OK;
    if (!S_out || !aligned4(S_out)) return VLA_ERR_INVALID_ARG;
    if (T > 0 && (!k || !v || !aligned4(k) || !aligned4(v))) return VLA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == VLA_BF16)
        vla::la_state_kernel<__nv_bfloat16><<<(int)BH, vla::LA_THREADS, 0, s>>>(
            static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), T, d, S_out);
    else
        vla::la_state_kernel<float><<<(int)BH, vla::LA_THREADS, 0, s>>>(
            static_cast<const float*>(k), static_cast<const float*>(v), T, d, S_out);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

}  // extern "C"
