// vla_fused.cuh -- the per-token forward kernel of the Variational Linear
// Attention recurrence ("Variational Linear Attention", arXiv 2605.11196,
// §3.3 eq. 9-11), the parameter block every forward kernel takes, and the
// plain linear-attention state of §4.1. Included by vla_forward.cu inside
// namespace vla.
//
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

// ---------------------------------------------------------------------------
// Per-head-dimension configuration.
//   NA/NS   A and S warps;  CBA/CBS  column blocks per row (lanes sharing a row)
//   NG      gate warps (token t goes to gate warp t mod NG)
//   NSTG    staging warps (chunk c goes to staging warp c mod NSTG)
//   CH      tokens per staged chunk;  TB  tokens the staging warp prepares at once
//   NP      prepped chunk slots;  NRAW  raw chunk slots
//   CB      tokens per A step (blocked Sherman-Morrison update)
//   RZ      A-step slots of the A->gate ring;  RG  token slots of gate->S
//   PAD     pad shared vectors by 4 floats per 32 (bank spread for the
//           column-block strides of these layouts)
//   MINB    CTAs per SM the register budget is sized for
// ---------------------------------------------------------------------------
template <int D>
struct Cfg;
template <>
struct Cfg<32> {
    static constexpr int NA = 1, CBA = 4, NS = 1, CBS = 4, NG = 1, NSTG = 1, CB = 2, CH = 8, TB = 4, NP = 6, NRAW = 3, RZ = 8,
                         RG = 16, PAD = 1, MINB = 4;
};
template <>
struct Cfg<64> {
    static constexpr int NA = 4, CBA = 8, NS = 2, CBS = 4, NG = 1, NSTG = 1, CB = 2, CH = 8, TB = 4, NP = 4, NRAW = 3, RZ = 8,
                         RG = 16, PAD = 1, MINB = 2;
};
template <>
struct Cfg<96> {
    static constexpr int NA = 4, CBA = 8, NS = 4, CBS = 8, NG = 2, NSTG = 2, CB = 2, CH = 8, TB = 4, NP = 8, NRAW = 4, RZ = 8,
                         RG = 16, PAD = 0, MINB = 1;
};
template <>
struct Cfg<128> {
    static constexpr int NA = 8, CBA = 8, NS = 8, CBS = 4, NG = 1, NSTG = 1, CB = 2, CH = 8, TB = 2, NP = 6, NRAW = 2, RZ = 8,
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
    // A -> gate record of one step (CB tokens): z'_0..z'_{CB-1} | w'_0..w'_{CB-1}
    // (padded) | per-warp parts of the Gram upper triangles Guu, Guk ([2*NP2][NA4])
    static constexpr int NP2 = C::CB * (C::CB + 1) / 2;
    static constexpr int Z_Z0 = 0, Z_W0 = C::CB * VD, Z_SC = 2 * C::CB * VD;
    static constexpr int ZSTRIDE = 2 * C::CB * VD + 2 * NP2 * NA4;
    // gate -> S record: alpha^ (padded) | s = alpha^ . phi(q), pad
    static constexpr int G_A = 0, G_S = VD;
    static constexpr int GSTRIDE = VD + 4;
    // warp roles
    static constexpr int NSTG = C::NSTG;
    static constexpr int W_PROD = 0, W_GATE = NSTG, W_A0 = NSTG + C::NG, W_S0 = NSTG + C::NG + C::NA;
    static constexpr int NWARPS = NSTG + C::NG + C::NA + C::NS, THREADS = 32 * NWARPS;
    // shared memory map (bytes)
    static constexpr int NBAR = C::NRAW + 2 * C::NP + 2 * C::RZ + 2 * C::RG + 2;
    static constexpr size_t OFF_FLAG = 8 * (size_t)NBAR;
    static constexpr size_t OFF_ZK = align_up(OFF_FLAG + 16, 16);  // z^key hand-off ring [2][D]
    static constexpr size_t RAW_TENSOR = (size_t)C::CH * D * sizeof(TIn);
    static constexpr size_t OFF_RAW = align_up(OFF_ZK + 2 * D * 4, 128);
    static constexpr size_t OFF_PREP = align_up(OFF_RAW + (size_t)C::NRAW * 4 * RAW_TENSOR, 128);
    static constexpr size_t OFF_Z = align_up(OFF_PREP + (size_t)C::NP * C::CH * PSTRIDE * 4, 128);
    static constexpr size_t OFF_G = align_up(OFF_Z + (size_t)C::RZ * ZSTRIDE * 4, 128);
    // per-warp transpose scratch for the cross-lane reductions: row v holds the
    // 32 lanes' copies of item v (stride RST floats keeps the reads conflict-free)
    static constexpr int RST = 36;
    static constexpr int A_ROWS = 2 * C::CB * (D / (C::NA * (32 / C::CBA))) + C::CB * (C::CB + 1);
    static constexpr int S_ROWS = 2 * (D / (C::NS * (32 / C::CBS))) + 1;
    static constexpr size_t OFF_ARED = align_up(OFF_G + (size_t)C::RG * GSTRIDE * 4, 128);
    static constexpr size_t OFF_SRED = align_up(OFF_ARED + (size_t)C::NA * A_ROWS * RST * 4, 128);
    static constexpr size_t SMEM = align_up(OFF_SRED + (size_t)C::NS * S_ROWS * RST * 4, 128);

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
    size_t o_stride;  // elements from one head's o rows to the next (T * d when o is [B, H, T, d])
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
    int fixed_a;  // the fixed-A variant: A stays A0 and eq. 9 is skipped
    float* tape;  // chunked kernel with TAPE (the backward pass's forward): per-token records
    float* ckpt;  //   and the states before every 64th token; else null
    // read by the single-CTA chunked kernel only (the segmented path runs it on
    // parts of the sequence); zero-filled fields give the plain layout
    size_t in_stride;  // elements from one head's q, k, v, u rows to the next (0: T * d)
    int s0_shared;     // nonzero: every head starts from the same S0 (one d x d matrix)
    int v_shared;      // nonzero: every head reads the same v rows (at p.v)
};

// Per-token clock stamps of head 0 for pipeline analysis (-DVLA_TRACE builds only).
#ifdef VLA_TRACE
#define VLA_TRACE_AT(p, role, t)                                                              \
    do {                                                                                      \
        if ((p).trace && blockIdx.x == 0) (p).trace[(size_t)(role) * (p).T + (t)] = clock64(); \
    } while (0)
// sub-step stamps of one thread (rows 5.. of the trace buffer)
#define VLA_TRACE_PT(p, row, t) VLA_TRACE_AT(p, row, t)
// stamp from the CTAs for which `cond` holds (e.g. both CTAs of head 0's cluster)
#define VLA_TRACE_IF(p, cond, row, t)                                                   \
    do {                                                                                \
        if ((p).trace && (cond)) (p).trace[(size_t)(row) * (p).T + (t)] = clock64();   \
    } while (0)
#else
#define VLA_TRACE_IF(p, cond, row, t) \
    do {                              \
    } while (0)
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
    uint64_t* full_z;   // an A step (CB tokens) published by the A warps
    uint64_t* empty_z;  // ... released by the gate warp that handled it
    uint64_t* full_g;   // alpha^ of a token published by the gate
    uint64_t* empty_g;  // ... released by the S warps
    uint64_t* zk_full;  // z^key at the end of a chunk handed to the next chunk's staging warp
    float* zkr;
    volatile int* abort;
    unsigned char* raw;
    float* prep;
    float* zr;
    float* gr;
    float* ared;  // A warps' transpose scratch
    float* sred;  // S warps' transpose scratch
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

// Sum of item v over the CBW lanes of row group g (columns g*CBW .. g*CBW+CBW-1
// of row v of a per-warp transpose scratch), in a fixed order.
template <int CBW, int RST>
__device__ __forceinline__ float rowgroup_sum(const float* red, int v, int g) {
    const float* q = red + v * RST + g * CBW;
    if constexpr (CBW == 8) {
        const float4 x = ld4(q), y = ld4(q + 4);
        return ((x.x + x.y) + (x.z + x.w)) + ((y.x + y.y) + (y.z + y.w));
    } else {
        static_assert(CBW == 4, "row groups of 4 or 8 lanes");
        const float4 x = ld4(q);
        return (x.x + x.y) + (x.z + x.w);
    }
}

// Sum of item v over all 32 lanes of a per-warp transpose scratch.
template <int RST>
__device__ __forceinline__ float warp_row_sum(const float* red, int v) {
    const float* q = red + v * RST;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 x = ld4(q + 4 * i);
        acc[0] += x.x;
        acc[1] += x.y;
        acc[2] += x.z;
        acc[3] += x.w;
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// ---------------------------------------------------------------------------
// staging warps: TMA bulk copies of raw q, k, v, u chunks, then per token
// u^, k^ (unit), phi(q), v (fp32) and den = max(phi(q) . z^key, eps) with
// z^key += phi(k) (§3.2-3.3, eq. 11). Staging warp s handles chunks c = s mod NSTG.
// Everything but the key sum is independent per token; the running z^key
// is handed from chunk to chunk through a shared ring guarded by mbarriers.
// ---------------------------------------------------------------------------
template <int D, typename TIn>
__device__ __forceinline__ void stage_role(const Params& p, const Smem& sm, int bh, int sw, int lane) {
    using C = Cfg<D>;
    using LY = Layout<D, TIn>;
    constexpr int E = D / 32;
    constexpr int TB = C::TB;
    constexpr int NSTG = LY::NSTG;
    constexpr int RPW = C::NRAW / NSTG;  // raw slots per staging warp
    static_assert(C::CH % TB == 0 && C::NRAW % NSTG == 0, "staging layout");
    const int T = p.T;
    const int nch = (T + C::CH - 1) / C::CH;
    const size_t head = (size_t)bh * T * D;
    const TIn* src[4] = {static_cast<const TIn*>(p.q) + head, static_cast<const TIn*>(p.k) + head,
                         static_cast<const TIn*>(p.v) + head, static_cast<const TIn*>(p.u) + head};

    // testing hook: publish nothing and raise no flag, so that every consumer
    // runs into its own wait limit
    if (p.stall_producer) return;

    auto issue = [&](int c) {  // lane 0 only; chunk c goes to raw slot c % NRAW
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
    float dchk = 0.f;  // fma(phi(q) . z^key, 0, .) per token: stays 0 unless q made it NaN or Inf
    // this warp's chunks are sw, sw + NSTG, ...; keep RPW of them in flight
    int issued = sw, landed = sw, c = sw;
    if (lane == 0)
        for (int i = 0; i < RPW && sw + i * NSTG < nch; ++i) issue(sw + i * NSTG);
    for (int i = 0; i < RPW && sw + i * NSTG < nch; ++i) issued = sw + (i + 1) * NSTG;
    float zk[E];
    for (; c < nch; c += NSTG) {
        const int rs = c % C::NRAW, ps = c % C::NP, use = c / C::NRAW;
        if (!mbar_wait(sm.full_r + rs, use & 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        landed = c + NSTG;
        if (lane == 0 && sw == 0) VLA_TRACE_PT(p, 14, c * C::CH);
        if (!mbar_wait(sm.empty_p + ps, ((c / C::NP) & 1) ^ 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        if (lane == 0 && sw == 0) VLA_TRACE_PT(p, 15, c * C::CH);
        const int nt = min(C::CH, T - c * C::CH);
        const TIn* raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            raw[i] = reinterpret_cast<const TIn*>(sm.raw + (size_t)(rs * 4 + i) * LY::RAW_TENSOR);
        float* P0 = sm.prep + (size_t)ps * C::CH * LY::PSTRIDE;
        float pk[C::CH][E], pq[C::CH][E];  // phi(k), phi(q) of the chunk's tokens
#pragma unroll
        for (int tb = 0; tb < C::CH; tb += TB) {
            if (tb >= nt) break;
            float qv[TB][E], kv[TB][E], vv[TB][E], uv[TB][E];
            float red[2 * TB];  // per token ||u||^2, ||k||^2
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                const bool live = tb + b < nt;
                float uu = 0.f, kk = 0.f;
#pragma unroll
                for (int m = 0; m < E; ++m) {
                    const int j = (tb + b) * D + lane + 32 * m;
                    qv[b][m] = live ? ld_in<TIn>(raw[0], j) : 0.f;
                    kv[b][m] = live ? ld_in<TIn>(raw[1], j) : 0.f;
                    vv[b][m] = live ? ld_in<TIn>(raw[2], j) : 0.f;
                    uv[b][m] = live ? ld_in<TIn>(raw[3], j) : 0.f;
                    uu = fmaf(uv[b][m], uv[b][m], uu);
                    kk = fmaf(kv[b][m], kv[b][m], kk);
                    pk[tb + b][m] = live ? phi(kv[b][m]) : 0.f;
                    pq[tb + b][m] = phi(qv[b][m]);
                }
                red[2 * b] = uu;
                red[2 * b + 1] = kk;
            }
            // reduce-scatter the 2*TB squared norms, invert on the owner lane, gather back
            reduce_scatter<2 * TB, 16>(red, lane);
            float inv[rs_count<2 * TB, 16>()];
#pragma unroll
            for (int j = 0; j < rs_count<2 * TB, 16>(); ++j) inv[j] = rsqrtf(fmaxf(red[j], 1e-24f));
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                constexpr int dummy = 0;
                (void)dummy;
                const float iu = __shfl_sync(0xffffffffu, inv[rs_owner_slot<2 * TB, 16>(2 * b)],
                                             rs_owner_lane<2 * TB, 16>(2 * b));
                const float ik = __shfl_sync(0xffffffffu, inv[rs_owner_slot<2 * TB, 16>(2 * b + 1)],
                                             rs_owner_lane<2 * TB, 16>(2 * b + 1));
                if (tb + b < nt) {
                    float* P = P0 + (tb + b) * LY::PSTRIDE;
#pragma unroll
                    for (int m = 0; m < E; ++m) {
                        const int j = lane + 32 * m;
                        P[LY::P_U + vidx<D>(j)] = uv[b][m] * iu;
                        P[LY::P_K + vidx<D>(j)] = kv[b][m] * ik;
                        P[LY::P_Q + vidx<D>(j)] = pq[tb + b][m];
                        P[LY::P_V + j] = vv[b][m];
                    }
                }
            }
        }
        // a tail that ends inside an A step leaves the rest of the step empty:
        // give those tokens zero u^ and k^ so that the A warps read them unconditionally
        for (int tp = nt; tp < C::CH && tp % C::CB != 0; ++tp) {
            float* P = P0 + tp * LY::PSTRIDE;
#pragma unroll
            for (int m = 0; m < E; ++m) {
                P[LY::P_U + vidx<D>(lane + 32 * m)] = 0.f;
                P[LY::P_K + vidx<D>(lane + 32 * m)] = 0.f;
            }
        }
        // the running key sum: z^key at the start of this chunk
        if (c == 0) {
#pragma unroll
            for (int m = 0; m < E; ++m) zk[m] = p.zk0 ? p.zk0[(size_t)bh * D + lane + 32 * m] : 0.f;
        } else {
            const int cp = c - 1;
            if (!mbar_wait(sm.zk_full + (cp % 2), (cp / 2) & 1, sm.abort, p.wait_ns)) {
                abort = true;
                break;
            }
#pragma unroll
            for (int m = 0; m < E; ++m) zk[m] = sm.zkr[(cp % 2) * D + lane + 32 * m];
        }
        float qz[C::CH];
#pragma unroll
        for (int t = 0; t < C::CH; ++t) {
            float s = 0.f;
            if (t < nt) {  // tokens past the end of a partial chunk were never loaded
#pragma unroll
                for (int m = 0; m < E; ++m) {
                    zk[m] += pk[t][m];
                    s = fmaf(pq[t][m], zk[m], s);
                }
            }
            qz[t] = s;
        }
        // hand z^key at the end of this chunk to the next one
#pragma unroll
        for (int m = 0; m < E; ++m) sm.zkr[(c % 2) * D + lane + 32 * m] = zk[m];
        reduce_scatter<C::CH, 16>(qz, lane);
#pragma unroll
        for (int j = 0; j < rs_count<C::CH, 16>(); ++j) {
            const int t = rs_index<C::CH, 16>(lane, j);
            if (t >= 0 && t < nt) {
                P0[t * LY::PSTRIDE + LY::P_DEN] = fmaxf(qz[j], p.eps);
                dchk = fmaf(qz[j], 0.f, dchk);
            }
        }
        // our generic-proxy reads of raw slot rs are done before the TMA refill
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(sm.zk_full + (c % 2));
            mbar_arrive(sm.full_p + ps);
            if (sw == 0) VLA_TRACE_AT(p, 0, c * C::CH);
            if (c + C::NRAW < nch) issue(c + C::NRAW);
        }
        if (c + C::NRAW < nch) issued = c + C::NRAW + NSTG;
        if (c + NSTG >= nch && p.zk_out) {
#pragma unroll
            for (int m = 0; m < E; ++m) p.zk_out[(size_t)bh * D + lane + 32 * m] = zk[m];
        }
    }
    if (dchk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_STAGE, bh, -1);
    if (abort) {
        if (lane == 0) record_failure(p.status, BIT_TIMEOUT, ROLE_STAGE, bh, c * C::CH);
        *sm.abort = 1;
        // let copies already in flight land before the CTA can exit
        for (int cc = landed; cc < issued; cc += NSTG)
            (void)mbar_wait(sm.full_r + cc % C::NRAW, (cc / C::NRAW) & 1, nullptr, p.wait_ns);
        return;
    }
    if (T == 0 && sw == 0 && p.zk_out) {
#pragma unroll
        for (int m = 0; m < E; ++m) p.zk_out[(size_t)bh * D + lane + 32 * m] = p.zk0 ? p.zk0[(size_t)bh * D + lane + 32 * m] : 0.f;
    }
}

// ---------------------------------------------------------------------------
// Blocked Sherman-Morrison step over CB tokens. For the step's starting A and
// unit vectors u^_s, k^_s (s < CB), with z'_s = A u^_s, w'_s = A k^_s and the
// Gram entries Guu[s][t] = u^_s . z'_t, Guk[s][t] = u^_s . w'_t (s <= t),
// the sequential updates of eq. 9 give z_t = sum_s c[t][s] z'_s with
//   c[t] = e_t - sum_{r<t} ((z_r . u^_t) / delta_r) c[r],
//   delta_t = 1 + z_t . u^_t,      z_r . u^_t = sum_s c[r][s] Guu[s][t],
// so that A after the step is A - Z' Q Z'^T with Q = sum_r c[r] c[r]^T / delta_r,
// and the gate direction of token t (eq. 10) is
//   A_t k^_t = w'_t - sum_{s<=t} beta[s][t] z'_s,
//   beta[s][t] = sum_{r=s..t} c[r][s] (sum_{s'<=r} c[r][s'] Guk[s'][t]) / delta_r.
// ---------------------------------------------------------------------------
template <int CB>
__host__ __device__ constexpr int upair(int s, int t) {  // index of (s <= t) in row-major upper triangle
    return s * CB - s * (s - 1) / 2 + (t - s);
}

template <int CB>
__device__ __forceinline__ void block_coeffs(const float* Guu, float (&c)[CB][CB], float (&rd)[CB]) {
#pragma unroll
    for (int t = 0; t < CB; ++t)
#pragma unroll
        for (int s = 0; s < CB; ++s) c[t][s] = (s == t) ? 1.f : 0.f;
#pragma unroll
    for (int t = 0; t < CB; ++t) {
#pragma unroll
        for (int r = 0; r < t; ++r) {
            float g = 0.f;
#pragma unroll
            for (int s = 0; s <= r; ++s) g = fmaf(c[r][s], Guu[upair<CB>(s, t)], g);
            g *= rd[r];
#pragma unroll
            for (int s = 0; s <= r; ++s) c[t][s] = fmaf(-g, c[r][s], c[t][s]);
        }
        float dl = 1.f;
#pragma unroll
        for (int s = 0; s <= t; ++s) dl = fmaf(c[t][s], Guu[upair<CB>(s, t)], dl);
        rd[t] = __frcp_rn(dl);
    }
}

// Sum NK scalars, each stored as NA per-warp parts at base[k * NA4 + w], with
// the lanes of the warp: lane l reads part (l + 32 m) and a butterfly over NA
// lanes adds the parts; the result for every k is broadcast to all lanes.
// Every caller uses the same order of additions.
template <int NK, int NA, int NA4>
__device__ __forceinline__ void gather_scalars(const float* base, int lane, float (&out)[NK]) {
    constexpr int NV = NK * NA, R = (NV + 31) / 32;
    float v[R];
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int i = lane + 32 * m;
        v[m] = i < NV ? base[(i / NA) * NA4 + (i % NA)] : 0.f;
    }
#pragma unroll
    for (int h = 1; h < NA; h <<= 1)
#pragma unroll
        for (int m = 0; m < R; ++m) v[m] += __shfl_xor_sync(0xffffffffu, v[m], h);
#pragma unroll
    for (int k = 0; k < NK; ++k) out[k] = __shfl_sync(0xffffffffu, v[(k * NA) / 32], (k * NA) % 32);
}

// ---------------------------------------------------------------------------
// gate warps: alpha^_t = A_t k^_t / ||A_t k^_t|| (eq. 10) and s_t = alpha^_t . phi(q_t)
// for the tokens of published A steps; gate warp g handles steps b = g mod NG.
// ---------------------------------------------------------------------------
template <int D, typename TIn>
__device__ __forceinline__ void gate_role(const Params& p, const Smem& sm, int bh, int g, int lane) {
    using C = Cfg<D>;
    using LY = Layout<D, TIn>;
    constexpr int E = D / 32, CB = C::CB, NP2 = CB * (CB + 1) / 2;
    bool abort = false, nonfinite = false;
    int t = g * CB;
    const int nsteps = (p.T + CB - 1) / CB;
    for (int b = g; b < nsteps && !abort; b += C::NG) {
        const int zs = b % C::RZ;
        t = b * CB;
        if (!mbar_wait(sm.full_z + zs, (b / C::RZ) & 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        const int chunk = t / C::CH, ps = chunk % C::NP;
        if (!mbar_wait(sm.full_p + ps, (chunk / C::NP) & 1, sm.abort, p.wait_ns)) {
            abort = true;
            break;
        }
        const float* Z = sm.zr + (size_t)zs * LY::ZSTRIDE;
        float G2[2 * NP2];  // Guu then Guk (upper triangles)
        gather_scalars<2 * NP2, C::NA, LY::NA4>(Z + LY::Z_SC, lane, G2);
        float c[CB][CB], rd[CB];
        block_coeffs<CB>(G2, c, rd);
#pragma unroll
        for (int s = 0; s < CB; ++s)
            if (!isfinite(rd[s])) nonfinite = true;
#pragma unroll
        for (int j = 0; j < CB; ++j) {
            const int tj = t + j;
            if (tj >= p.T) break;
            // beta[s][j] for s <= j
            float beta[CB];
#pragma unroll
            for (int s = 0; s < CB; ++s) beta[s] = 0.f;
#pragma unroll
            for (int r = 0; r <= j; ++r) {
                float zk = 0.f;
#pragma unroll
                for (int s2 = 0; s2 <= r; ++s2) zk = fmaf(c[r][s2], G2[NP2 + upair<CB>(s2, j)], zk);
                zk *= rd[r];
#pragma unroll
                for (int s = 0; s <= r; ++s) beta[s] = fmaf(c[r][s], zk, beta[s]);
            }
            if (lane == 0 && g == 0) VLA_TRACE_PT(p, 11, tj);
            const int tc = tj - chunk * C::CH;
            const float* P = sm.prep + (size_t)(ps * C::CH + tc) * LY::PSTRIDE;
            float av[E];
            float red[2] = {0.f, 0.f};  // ||a||^2, a . phi(q)
#pragma unroll
            for (int m = 0; m < E; ++m) {
                const int jv = vidx<D>(lane + 32 * m);
                float x = Z[LY::Z_W0 + j * LY::VD + jv];
#pragma unroll
                for (int s = 0; s <= j; ++s) x = fmaf(-beta[s], Z[LY::Z_Z0 + s * LY::VD + jv], x);
                av[m] = x;
                red[0] = fmaf(x, x, red[0]);
                red[1] = fmaf(x, P[LY::P_Q + jv], red[1]);
            }
            allreduce<2, 16>(red);
            if (lane == 0 && g == 0) VLA_TRACE_PT(p, 12, tj);
            const float inv = rsqrtf(fmaxf(red[0], 1e-24f));  // 1 / max(||a||, 1e-12)
            if (!(isfinite(red[0]) && isfinite(red[1]))) nonfinite = true;
            const int gs = tj % C::RG;
            if (!mbar_wait(sm.empty_g + gs, ((tj / C::RG) & 1) ^ 1, sm.abort, p.wait_ns)) {
                abort = true;
                t = tj;
                break;
            }
            if (lane == 0 && g == 0) VLA_TRACE_PT(p, 13, tj);
            float* Gp = sm.gr + (size_t)gs * LY::GSTRIDE;
#pragma unroll
            for (int m = 0; m < E; ++m) Gp[LY::G_A + vidx<D>(lane + 32 * m)] = av[m] * inv;
            if (lane == 0) Gp[LY::G_S] = red[1] * inv;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sm.full_g + gs);
                VLA_TRACE_AT(p, 2, tj);
            }
        }
        if (!abort && lane == 0) mbar_arrive(sm.empty_z + zs);
    }
    if (abort) {
        if (lane == 0) record_failure(p.status, BIT_TIMEOUT, ROLE_GATE, bh, t);
        *sm.abort = 1;
    }
    if (nonfinite && lane == 0) record_failure(p.status, BIT_NONFINITE, ROLE_GATE, bh, -1);
}

// ---------------------------------------------------------------------------
// A warps: the Sherman-Morrison chain (eq. 9), CB tokens per step. A is
// resident in registers as float2 pairs. One step: sub-pass 1 applies the
// previous step's update A -= Z' Q Z'^T (as A += nm_s z'_s^T) and forms
// z'_t = A u^_t; sub-pass 2 forms w'_t = A k^_t; the row sums and this thread's
// parts of the Gram entries are reduced across the lanes of a row and
// published with one named barrier per step.
// ---------------------------------------------------------------------------
template <int D, typename TIn>
__device__ __forceinline__ void a_role(const Params& p, const Smem& sm, int bh, int warp, int lane) {
    using C = Cfg<D>;
    using LY = Layout<D, TIn>;
    constexpr int CB = C::CB, NP2 = CB * (CB + 1) / 2;
    constexpr int RPW = 32 / C::CBA;              // row groups per warp
    constexpr int RA = D / (C::NA * RPW);         // rows per thread
    constexpr int CA = D / C::CBA;                // columns per thread
    constexpr int C2 = CA / 2;                    // float2 columns
    constexpr int NVV = 2 * CB * RA;              // z' and w' rows
    constexpr int NV = NVV + 2 * NP2;             // + Guu, Guk parts
    static_assert(RA * C::NA * RPW == D && CA * C::CBA == D && CA % 4 == 0, "A layout");
    static_assert(C::CH % CB == 0, "steps stay inside a chunk");
    static_assert(NV == LY::A_ROWS && 2 * NP2 <= 32, "A transpose scratch");

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
    // pending update of the previous step: A += sum_s nm[s] (x) z'_s at this
    // thread's columns (read from the previous step's slot; zeros before step 0)
    float2 nm[CB][RA];
#pragma unroll
    for (int s = 0; s < CB; ++s)
#pragma unroll
        for (int r = 0; r < RA; ++r) nm[s][r] = f2(0.f, 0.f);
    const float* Zprev = sm.zr + (size_t)(C::RZ - 1) * LY::ZSTRIDE;
    {
        float* Zw = sm.zr + (size_t)(C::RZ - 1) * LY::ZSTRIDE;
        for (int i = wa * 32 + lane; i < CB * LY::VD; i += C::NA * 32) Zw[LY::Z_Z0 + i] = 0.f;
        bar_red_or(1, C::NA * 32, false);
    }

    bool abort = false;
    int t = 0;
    if (p.T > 0 && !mbar_wait(sm.full_p, 0, sm.abort, p.wait_ns)) abort = true;
    for (int b = 0; t < p.T; ++b, t += CB) {
        const bool tr0 = (wa == 0 && lane == 0);
        if (tr0) VLA_TRACE_PT(p, 5, t);
        const int chunk = t / C::CH, tc = t - chunk * C::CH, ps = chunk % C::NP;
        const float* P0 = sm.prep + (size_t)(ps * C::CH + tc) * LY::PSTRIDE;  // tokens past T hold zeros

        // sub-pass 1: pending update, then z'_s = A u^_s
        float zr[CB][RA];
        {
            float2 pz[CB][RA];
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int r = 0; r < RA; ++r) pz[s][r] = f2(0.f, 0.f);
#pragma unroll
            for (int c4 = 0; c4 < CA; c4 += 4) {
                const int jv = vidx<D>(col0 + c4);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float2 zc[CB], uc[CB];
#pragma unroll
                    for (int s = 0; s < CB; ++s) {
                        zc[s] = *reinterpret_cast<const float2*>(Zprev + LY::Z_Z0 + s * LY::VD + jv + 2 * h);
                        uc[s] = *reinterpret_cast<const float2*>(P0 + s * LY::PSTRIDE + LY::P_U + jv + 2 * h);
                    }
#pragma unroll
                    for (int r = 0; r < RA; ++r) {
                        const int c = c4 / 2 + h;
                        float2 x = a[r][c];
#pragma unroll
                        for (int s = 0; s < CB; ++s) x = __ffma2_rn(nm[s][r], zc[s], x);
                        a[r][c] = x;
#pragma unroll
                        for (int s = 0; s < CB; ++s) pz[s][r] = __ffma2_rn(x, uc[s], pz[s][r]);
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int r = 0; r < RA; ++r) zr[s][r] = pz[s][r].x + pz[s][r].y;
        }
        // sub-pass 2: w'_s = A k^_s
        float wr[CB][RA];
        {
            float2 pw[CB][RA];
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int r = 0; r < RA; ++r) pw[s][r] = f2(0.f, 0.f);
#pragma unroll
            for (int c4 = 0; c4 < CA; c4 += 4) {
                const int jv = vidx<D>(col0 + c4);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float2 kc[CB];
#pragma unroll
                    for (int s = 0; s < CB; ++s)
                        kc[s] = *reinterpret_cast<const float2*>(P0 + s * LY::PSTRIDE + LY::P_K + jv + 2 * h);
#pragma unroll
                    for (int r = 0; r < RA; ++r) {
                        const int c = c4 / 2 + h;
#pragma unroll
                        for (int s = 0; s < CB; ++s) pw[s][r] = __ffma2_rn(a[r][c], kc[s], pw[s][r]);
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int r = 0; r < RA; ++r) wr[s][r] = pw[s][r].x + pw[s][r].y;
        }
        // row sums and Gram parts, reduced across the lanes of each row
        float vals[NV];
#pragma unroll
        for (int s = 0; s < CB; ++s)
#pragma unroll
            for (int r = 0; r < RA; ++r) {
                vals[s * RA + r] = zr[s][r];
                vals[(CB + s) * RA + r] = wr[s][r];
            }
        {
            float ur[CB][RA];
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int r = 0; r < RA; ++r) ur[s][r] = P0[s * LY::PSTRIDE + LY::P_U + vidx<D>(row0 + r)];
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int tt = s; tt < CB; ++tt) {
                    float gu = 0.f, gk = 0.f;
#pragma unroll
                    for (int r = 0; r < RA; ++r) {
                        gu = fmaf(ur[s][r], zr[tt][r], gu);
                        gk = fmaf(ur[s][r], wr[tt][r], gk);
                    }
                    vals[NVV + upair<CB>(s, tt)] = gu;
                    vals[NVV + NP2 + upair<CB>(s, tt)] = gk;
                }
        }
        if (tr0) VLA_TRACE_PT(p, 6, t);
        // reduce the row sums and Gram parts through this warp's transpose scratch:
        // row v holds the 32 lanes' copies of item v
        float* red = sm.ared + (size_t)wa * LY::A_ROWS * LY::RST;
        __syncwarp();
#pragma unroll
        for (int v = 0; v < NV; ++v) red[v * LY::RST + lane] = vals[v];
        __syncwarp();
        const int zs = b % C::RZ;
        if (tr0) VLA_TRACE_PT(p, 7, t);
        if (!abort && !mbar_wait(sm.empty_z + zs, ((b / C::RZ) & 1) ^ 1, sm.abort, p.wait_ns)) abort = true;
        if (tr0) VLA_TRACE_PT(p, 8, t);
        float* Z = sm.zr + (size_t)zs * LY::ZSTRIDE;
        // row items: lane (row group, cb) finishes items cb, cb + CBA, ... of its row group
#pragma unroll
        for (int j = 0; j < (NVV + C::CBA - 1) / C::CBA; ++j) {
            const int v = cb + j * C::CBA;
            if (v < NVV) {
                const float sum = rowgroup_sum<C::CBA, LY::RST>(red, v, rgl);
                const int vec = v / RA, r = v - vec * RA;
                Z[vec * LY::VD + vidx<D>(row0 + r)] = sum;
            }
        }
        // Gram parts: lane l finishes item NVV + l over the whole warp
        if (lane < 2 * NP2) Z[LY::Z_SC + lane * LY::NA4 + wa] = warp_row_sum<LY::RST>(red, NVV + lane);
        // the next step may start a new chunk
        if (t + CB < p.T) {
            const int t2 = t + CB, chunk2 = t2 / C::CH;
            if (t2 - chunk2 * C::CH == 0 && !abort &&
                !mbar_wait(sm.full_p + chunk2 % C::NP, (chunk2 / C::NP) & 1, sm.abort, p.wait_ns))
                abort = true;
        }
        // publish among the A warps; every A thread takes the same abort decision
        if (bar_red_or(1, C::NA * 32, abort || (*sm.abort != 0))) {
            abort = true;
            break;
        }
        if (tr0) VLA_TRACE_PT(p, 9, t);
        if (wa == 0 && lane == 0) {
            mbar_arrive(sm.full_z + zs);
#pragma unroll
            for (int j = 0; j < CB; ++j)
                if (t + j < p.T) VLA_TRACE_AT(p, 1, t + j);
        }
        {
            float Guu[NP2];
            gather_scalars<NP2, C::NA, LY::NA4>(Z + LY::Z_SC, lane, Guu);
            float c[CB][CB], rd[CB];
            block_coeffs<CB>(Guu, c, rd);
            float Q[CB][CB];
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int s2 = 0; s2 < CB; ++s2) {
                    float q = 0.f;
#pragma unroll
                    for (int r = (s > s2 ? s : s2); r < CB; ++r) q = fmaf(c[r][s] * rd[r], c[r][s2], q);
                    Q[s][s2] = q;
                }
            float zrow[CB][RA];
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int r = 0; r < RA; ++r) zrow[s][r] = Z[LY::Z_Z0 + s * LY::VD + vidx<D>(row0 + r)];
#pragma unroll
            for (int s = 0; s < CB; ++s)
#pragma unroll
                for (int r = 0; r < RA; ++r) {
                    float m = 0.f;
#pragma unroll
                    for (int s2 = 0; s2 < CB; ++s2) m = fmaf(Q[s][s2], zrow[s2][r], m);
                    nm[s][r] = f2(-m, -m);
                }
        }
        Zprev = Z;
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
        for (int c4 = 0; c4 < CA; c4 += 4) {
            const int jv = vidx<D>(col0 + c4);
            float2 x0 = a[r][c4 / 2], x1 = a[r][c4 / 2 + 1];
#pragma unroll
            for (int s = 0; s < CB; ++s) {
                const float4 z4 = ld4(Zprev + LY::Z_Z0 + s * LY::VD + jv);
                x0 = __ffma2_rn(nm[s][r], f2(z4.x, z4.y), x0);
                x1 = __ffma2_rn(nm[s][r], f2(z4.z, z4.w), x1);
            }
            *reinterpret_cast<float4*>(Ao + (size_t)(row0 + r) * D + col0 + c4) = make_float4(x0.x, x0.y, x1.x, x1.y);
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
    static_assert(RS * C::NS * RPW == D && CS * C::CBS == D && CS % 4 == 0, "S layout");
    static_assert(RS <= C::CBS && 2 * RS + 1 == LY::S_ROWS, "S transpose scratch");

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
    float* o = p.o + (size_t)bh * p.o_stride;

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
        // reduce S k^ and S phi(q) through this warp's transpose scratch; lane cb < RS
        // of a row group finishes row cb of it
        float* red = sm.sred + (size_t)ws * LY::S_ROWS * LY::RST;
        __syncwarp();
#pragma unroll
        for (int r = 0; r < RS; ++r) {
            red[r * LY::RST + lane] = sk2[r].x + sk2[r].y;
            red[(RS + r) * LY::RST + lane] = sq2[r].x + sq2[r].y;
        }
        __syncwarp();
        const bool own = cb < RS;
        float e_own = 0.f, sq_own = 0.f;
        if (own) {
            const float sk_own = rowgroup_sum<C::CBS, LY::RST>(red, cb, rgl);
            sq_own = rowgroup_sum<C::CBS, LY::RST>(red, RS + cb, rgl);
            e_own = P[LY::P_V + row0 + cb] - sk_own;
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
        if (own) {
            const float ov = fmaf(e_own, st, sq_own) * rden;
            o[(size_t)t * D + row0 + cb] = ov;
            red[2 * RS * LY::RST + rgl * C::CBS + cb] = e_own;
        }
        __syncwarp();
        // every lane of the row group needs the whole residual for the write
        float2 e2[RS];
        {
            const float* er = red + 2 * RS * LY::RST + rgl * C::CBS;
#pragma unroll
            for (int r4 = 0; r4 < RS; r4 += 4) {
                const float4 x = ld4(er + r4);
                const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (r4 + i < RS) e2[r4 + i] = f2(xs[i], xs[i]);
            }
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
    // Non-finite outputs are detected where they can arise rather than per
    // output (a check on every o cost this kernel 18%): through q in the
    // staging warps' phi(q) . z^key, through k and u in the gate and delta
    // checks, and through v in S, whose row stays non-finite to the end.
    float* So = p.S_out + (size_t)bh * D * D;
    float schk = 0.f;
#pragma unroll
    for (int r = 0; r < RS; ++r)
#pragma unroll
        for (int c = 0; c < C2; c += 2) {
            *reinterpret_cast<float4*>(So + (size_t)(row0 + r) * D + col0 + 2 * c) =
                make_float4(s[r][c].x, s[r][c].y, s[r][c + 1].x, s[r][c + 1].y);
            schk = fmaf(s[r][c].x + s[r][c].y + s[r][c + 1].x + s[r][c + 1].y, 0.f, schk);
        }
    if (schk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_S, bh, -1);
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
    sm.zk_full = sm.empty_g + C::RG;
    sm.zkr = reinterpret_cast<float*>(smem + LY::OFF_ZK);
    sm.abort = reinterpret_cast<volatile int*>(smem + LY::OFF_FLAG);
    sm.raw = smem + LY::OFF_RAW;
    sm.prep = reinterpret_cast<float*>(smem + LY::OFF_PREP);
    sm.zr = reinterpret_cast<float*>(smem + LY::OFF_Z);
    sm.gr = reinterpret_cast<float*>(smem + LY::OFF_G);
    sm.ared = reinterpret_cast<float*>(smem + LY::OFF_ARED);
    sm.sred = reinterpret_cast<float*>(smem + LY::OFF_SRED);

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
        mbar_init(sm.zk_full, 1);
        mbar_init(sm.zk_full + 1, 1);
        *sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp < LY::W_GATE)
        stage_role<D, TIn>(p, sm, bh, warp - LY::W_PROD, lane);
    else if (warp < LY::W_A0)
        gate_role<D, TIn>(p, sm, bh, warp - LY::W_GATE, lane);
    else if (warp < LY::W_S0)
        a_role<D, TIn>(p, sm, bh, warp, lane);
    else
        s_role<D, TIn>(p, sm, bh, warp, lane);
}

// ---------------------------------------------------------------------------
// plain cumulative linear-attention state S = sum_t v_t phi(k_t)^T (§4.1).
// One CTA per head; thread (ti, tj) of a 16 x 16 grid accumulates the
// (D/16) x (D/16) block of S at rows ti*R.., columns tj*R.. from tokens staged
// in shared memory LA_TT at a time.
// ---------------------------------------------------------------------------
constexpr int LA_THREADS = 256, LA_TT = 32;

template <int D, typename TIn>
__global__ void __launch_bounds__(LA_THREADS) la_state_kernel(const TIn* k, const TIn* v, int T, float* S_out) {
    constexpr int R = D / 16;
    __shared__ float sv[LA_TT][D], sk[LA_TT][D];
    const size_t base = (size_t)blockIdx.x * T * D;
    const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
    float acc[R][R];
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
        for (int b = 0; b < R; ++b) acc[a][b] = 0.f;
    for (int t0 = 0; t0 < T; t0 += LA_TT) {
        const int nt = min(LA_TT, T - t0);
        for (int i = threadIdx.x; i < LA_TT * D; i += LA_THREADS) {
            const int tt = i / D, j = i - tt * D;
            const bool live = tt < nt;
            sv[tt][j] = live ? ld_in<TIn>(v + base + (size_t)t0 * D, i) : 0.f;
            sk[tt][j] = live ? phi(ld_in<TIn>(k + base + (size_t)t0 * D, i)) : 0.f;
        }
        __syncthreads();
        for (int tt = 0; tt < LA_TT; ++tt) {
            float vi[R], kj[R];
#pragma unroll
            for (int a = 0; a < R; ++a) {
                vi[a] = sv[tt][ti * R + a];
                kj[a] = sk[tt][tj * R + a];
            }
#pragma unroll
            for (int a = 0; a < R; ++a)
#pragma unroll
                for (int b = 0; b < R; ++b) acc[a][b] = fmaf(vi[a], kj[b], acc[a][b]);
        }
        __syncthreads();
    }
    float* So = S_out + (size_t)blockIdx.x * D * D;
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
        for (int b = 0; b < R; ++b) So[(size_t)(ti * R + a) * D + tj * R + b] = acc[a][b];
}
