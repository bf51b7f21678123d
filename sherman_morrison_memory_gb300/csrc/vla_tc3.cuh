// vla_tc3.cuh -- the chunked tensor-core recurrence of vla_tc.cuh on a
// thread-block cluster of 1 + NS CTAs per (batch, head), with the rows of S
// split over NS CTAs. Included by vla_forward.cu inside namespace vla, after
// vla_tc2.cuh (it reuses that file's cluster helpers and staging warps and
// vla_tc.cuh's chunk arithmetic).
//
// "Variational Linear Attention" (arXiv 2605.11196), §3.3 eq. 9-11, C = 16
// tokens at a time. The residual write of eq. 10, S_t = S_{t-1} + e_t
// alpha^_t^T with e_t = v_t - S_{t-1} k^_t, acts on each row of S on its own:
// row i of S needs only row i of v, the key k^_t and the gate alpha^_t. So
//
//   CTA rank 0          the A-pass (eq. 9 and a_t = A_t k^_t of eq. 10) as in
//                       vla_tc2.cuh, A and its tf32 lo part in its tensor
//                       memory; per chunk it sends the gate (the rows a_t,
//                       the K-major hi / lo tiles of their transpose and
//                       ||a_t||^2) to every S rank: one set of bulk copies
//                       (cp.async.bulk shared::cta -> shared::cluster) per
//                       peer, completing on that peer's barrier; no multicast
//   CTA rank r = 1..NS  rows [(r-1) R, r R) of S (R = d / NS) in its tensor
//                       memory: per chunk [S k | S phi] for its rows, the
//                       residual writes and readout of those rows (eq. 10,
//                       11) and their update S += E' A
//
// Each CTA has eight team warps. A row's per-chunk work is split between two
// threads of different warps that reach the same tensor-memory lane (warps w
// and w + 4): in rank 0, the product columns, the gate sums and the lo
// refresh of A; in an S rank, the products (S k for the solve, S phi for the
// readout), the lo refresh, and the readout, which runs beside the update.
// In an S rank the chunk's products are issued before the gate arrives, and
// all eight warps form the chunk's 16 x 16 Gram matrices once it has.
//
// Every wait is bounded; a role that gives up raises the abort flag of every
// CTA of the cluster.

namespace tc3 {

using tc2::bulk_to_peer;
using tc2::cluster_rank;
using tc2::cluster_sync_all;
using tc2::mbar_arrive_peer;
using tc2::mbar_expect_tx_peer;
using tc2::mbar_wait_cl;
using tc2::peer_addr;
using tc2::st_peer_u32;

// arm a peer's barrier for `bytes` of bulk copies (one arrival), with relaxed
// ordering: the data reach the peer through the copies, whose completion the
// peer's wait observes, so this thread's earlier writes need no release
__device__ __forceinline__ void mbar_expect_tx_peer_relaxed(uint32_t rbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(rbar), "r"(bytes)
                 : "memory");
}

// -DVLA_TRACE builds: per-chunk clock stamps of head 0's cluster, stamp k of
// chunk c at trace[row][k * nch + c] (row 4 + rank)
#define TC3_STAMP(p, rank, k, c, nch) \
    VLA_TRACE_IF(p, blockIdx.x < (unsigned)(1 + NS) && threadIdx.x == 0, 4 + (rank), (k) * (nch) + (c))
// the same from thread `tid` of the CTA
#define TC3_STAMP_T(p, rank, k, c, nch, tid) \
    VLA_TRACE_IF(p, blockIdx.x < (unsigned)(1 + NS) && threadIdx.x == (tid), 4 + (rank), (k) * (nch) + (c))

constexpr int C = tc::C;
constexpr int NSTAGE = 4;
constexpr int THREADS = 32 * 12;
constexpr int NTEAM = 256;  // team warps 0-7
// named barriers: 1 team, 3 staging, 8-11 row hand-offs
constexpr int ID_T = 1, ID_ST = 3, ID_Y = 8, ID_M = 9, ID_E = 10, ID_EM = 11;
constexpr int FACTOR_WARP = 4;
constexpr int NISS = 4;  // warps that issue the d x 2C chunk products, one accumulator each
constexpr size_t MIN_SMEM = 116 * 1024;

template <int D, typename TIn, int NS>
struct Lay3 {
    static constexpr bool F32IN = sizeof(TIn) == 4;
    static constexpr int NRW = D / 32;             // rank 0 row warps (and as many helpers, warps 4..)
    static constexpr int R = D / NS;               // rows of S per S rank
    static constexpr int NRS = (R + 31) / 32;      // S-rank row warps
    static_assert(D % NS == 0 && R % 16 == 0 && R <= 64, "S rows per rank");
    static constexpr int NP = F32IN ? 2 : 3;       // prepared chunk slots
    static constexpr int NRAW = F32IN ? 1 : 2;     // raw chunk slots
    static constexpr int HI_ROWS = 2 * C;
    static constexpr int LO_ROWS = F32IN ? 2 * C : C;
    static constexpr int SBO_D = (D / 4) * 128;
    static constexpr int SBO_C = (C / 4) * 128;
    static constexpr int SC_IU = 0, SC_IK = C, SC_RDEN = 2 * C;
    static constexpr int SLOT = (HI_ROWS + LO_ROWS) * D + 64;  // floats
    static constexpr int SCR_STRIDE = D + 4;
    static constexpr int GSTR = C + 4;
    static constexpr int XS = D + 4;
    // tensor memory of every rank: state | its lo part | NISS product accumulators
    static constexpr uint32_t T_X = 0, T_XL = D, T_P = 2 * D;
    static constexpr uint32_t TNEED = 2 * D + NISS * 2 * C;
    static constexpr uint32_t TCOLS = TNEED <= 128 ? 128 : (TNEED <= 256 ? 256 : 512);
    static_assert(TNEED <= 512, "TMEM columns");
    // the gate of one chunk (one mailbox buffer), bytes; ||a_t||^2 (MB_LAA) is
    // formed by each S rank from the rows
    static constexpr uint32_t MB_ALR = C * XS * 4, MB_G = D * C * 4, MB_LAA = C * 4;
    static constexpr uint32_t MB_BYTES = MB_ALR + 2 * MB_G;
    static_assert(MB_ALR % 16 == 0 && MB_G % 16 == 0 && MB_LAA % 16 == 0, "bulk-copy granularity");

    static constexpr size_t al(size_t x) { return (x + 127) / 128 * 128; }
    static constexpr int NBAR = NRAW + 2 * NP + 2 + 2 + 2;
    static constexpr size_t OFF_BAR = 0;
    static constexpr size_t OFF_MISC = al(8 * NBAR);  // abort flag, TMEM base, mailbox counts
    static constexpr size_t OFF_PREP = al(OFF_MISC + 16);
    static constexpr size_t OFF_RAW = al(OFF_PREP + (size_t)NP * SLOT * 4);
    static constexpr size_t RAW_T = (size_t)C * D * sizeof(TIn);
    static constexpr size_t OFF_SCR = al(OFF_RAW + (size_t)NRAW * 2 * RAW_T);
    static constexpr size_t OFF_ZP = al(OFF_SCR + (size_t)2 * C * SCR_STRIDE * 4);  // staging phi(k) sums
    // the mailbox: the same offsets in every rank, so that rank 0 finds a peer's copy by mapa
    static constexpr size_t OFF_AL = al(OFF_ZP + (size_t)NSTAGE * D * 4);  // a rows [2][C x XS]
    static constexpr size_t OFF_GH = OFF_AL + 2 * (size_t)MB_ALR;           // a^T hi [2][D x C]
    static constexpr size_t OFF_GL = OFF_GH + 2 * (size_t)MB_G;             // a^T lo [2][D x C]
    static constexpr size_t OFF_LAA = OFF_GL + 2 * (size_t)MB_G;            // ||a||^2 [2][C] (S ranks)
    static constexpr size_t OFF_SM = al(OFF_LAA + 2 * (size_t)MB_LAA);
    // small matrices, rank 0: Guu, Guk, 1/sqrt(delta), L^T, X = L^-1 Guk, 1/delta; S ranks: Lk^T, Lq (two partials each)
    static constexpr int MS = C * GSTR;
    static constexpr int SM_GUU = 0, SM_GUK = MS, SM_RS = 2 * MS, SM_LMT = 3 * MS, SM_X = 4 * MS,
                         SM_RD = 5 * MS, SM_LKT = 0, SM_LQ = 2 * MS;
    static constexpr size_t OFF_U = al(OFF_SM + (size_t)(5 * MS + C) * 4);
    // rank 0: xr (z' | w rows, then y = z / delta | w) [2C x XS], -N hi / lo
    // [128 x C], N hi / lo [D x C], Gram partials of quarters 1..3 [2][3][32 x 8]
    static constexpr size_t OFF_XR = OFF_U;
    static constexpr size_t OFF_PH = al(OFF_XR + (size_t)2 * C * XS * 4);
    static constexpr size_t OFF_PL = OFF_PH + 128 * C * 4;
    static constexpr size_t OFF_ZH = OFF_PL + 128 * C * 4;
    static constexpr size_t OFF_ZL = OFF_ZH + (size_t)D * C * 4;
    static constexpr size_t OFF_GP = OFF_ZL + (size_t)D * C * 4;
    static constexpr size_t END_A = OFF_GP + (size_t)2 * 3 * 256 * 4;
    // S ranks: E' hi / lo [128 x C], Gram partials of quarters 1..3 [2][3][32 x 8]
    static constexpr size_t OFF_EH = OFF_U;
    static constexpr size_t OFF_EL = OFF_EH + 128 * C * 4;
    static constexpr size_t OFF_GPS = OFF_EL + 128 * C * 4;
    static constexpr size_t END_S = OFF_GPS + (size_t)2 * 3 * 256 * 4;
    static constexpr size_t SMEM = al(END_A > END_S ? END_A : END_S);
    static constexpr size_t SMEM_LAUNCH = SMEM > MIN_SMEM ? SMEM : MIN_SMEM;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(RAW_T % 16 == 0 && (D * sizeof(TIn)) % 16 == 0, "bulk-copy granularity");
};

struct Bars3 {
    uint64_t* full_r;    // [NRAW] raw chunk landed
    uint64_t* full_p;    // [NP] prepared chunk published
    uint64_t* empty_p;   // [NP] released by the team
    uint64_t* full_al;   // [2] S ranks: mailbox buffer filled by rank 0 (tx bytes)
    uint64_t* empty_al;  // [2] rank 0: every S rank done with the mailbox buffer (count NS)
    uint64_t* mma_x;     // state update committed
    uint64_t* mma_p;     // chunk products issued by NISS warps (count NISS)
};

template <int D, typename TIn, int NS>
struct Ctx3 {
    using L = Lay3<D, TIn, NS>;
    unsigned char* base;
    Bars3 b;
    volatile int* abort;
    uint32_t* tmem_base;
    int* n_sent;  // rank 0: mailbox buffers sent; S ranks: the same count, written by rank 0 at the end
    int* n_recv;  // S ranks: mailbox buffers received
    __device__ float* slot(int s) const { return reinterpret_cast<float*>(base + L::OFF_PREP) + (size_t)s * L::SLOT; }
    __device__ float* hi(int s) const { return slot(s); }
    __device__ float* lo(int s) const { return slot(s) + L::HI_ROWS * D; }
    __device__ float* sc(int s) const { return slot(s) + (L::HI_ROWS + L::LO_ROWS) * D; }
    __device__ unsigned char* raw(int r) const { return base + L::OFF_RAW + (size_t)r * 2 * L::RAW_T; }
    __device__ float* f(size_t off) const { return reinterpret_cast<float*>(base + off); }
    __device__ float* sm() const { return f(L::OFF_SM); }
    // raise the abort flag here and in every other CTA of the cluster
    __device__ void abort_peers(uint32_t rank) const {
        *abort = 1;
#pragma unroll 1
        for (uint32_t r = 0; r <= (uint32_t)NS; ++r)
            if (r != rank) st_peer_u32(peer_addr((const void*)abort, r), 1u);
    }
};

// columns [col0, col0 + C) of a row (this warp's TMEM lanes) summed over the NISS accumulators
__device__ __forceinline__ void ld_prod_cols(uint32_t tp, uint32_t col0, float (&v)[16]) {
    float x1[16], x2[16], x3[16];
    static_assert(NISS == 4, "four accumulators");
    tc_ld16(tp + col0, v);
    tc_ld16(tp + 2 * C + col0, x1);
    tc_ld16(tp + 4 * C + col0, x2);
    tc_ld16(tp + 6 * C + col0, x3);
    tc_wait_ld();
#pragma unroll
    for (int t = 0; t < 16; ++t) v[t] = (v[t] + x1[t]) + (x2[t] + x3[t]);
}

// lo parts of TMEM columns [c0, c0 + N) of this warp's lanes: column col + j -> dst + j
template <int N>
__device__ __forceinline__ void refresh_cols(uint32_t lanebase, uint32_t col, uint32_t dst, int c0) {
    static_assert(N % 16 == 0, "16-column blocks");
    if constexpr (N % 32 == 0) {
#pragma unroll 1
        for (int j = c0; j < c0 + N; j += 32) {
            float v[16], w[16];
            tc_ld16(lanebase + col + j, v);
            tc_ld16(lanebase + col + j + 16, w);
            tc_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                v[k] = tf32_lo(v[k]);
                w[k] = tf32_lo(w[k]);
            }
            tc_st16(lanebase + dst + j, v);
            tc_st16(lanebase + dst + j + 16, w);
        }
    } else {
#pragma unroll 1
        for (int j = c0; j < c0 + N; j += 16) {
            float v[16];
            tc_ld16(lanebase + col + j, v);
            tc_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = tf32_lo(v[k]);
            tc_st16(lanebase + dst + j, v);
        }
    }
    tc_wait_st();
}

// a_t[i] = w_t[i] - sum_{q<=t} y_q[i] X[q][t] (eq. 10, a_t = A_t k^_t) for the
// 16 tokens of row i, q outermost so that the 16 sums advance side by side;
// tokens t >= n are zero
__device__ __forceinline__ void gate16(const float* xr, int xs, const float* xm, int gstr, int i, int n, bool fixed,
                                       const float (&y)[C], float (&av)[C]) {
#pragma unroll
    for (int t = 0; t < C; ++t) av[t] = xr[(C + t) * xs + i];  // w_t
    if (!fixed) {
#pragma unroll
        for (int q = 0; q < C; ++q) {
            float lr[C];
            tc::ld_row16(xm + q * gstr, lr);  // X[q][t]
#pragma unroll
            for (int t = q; t < C; ++t) av[t] = fmaf(-y[q], lr[t], av[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < C; ++t) av[t] = t < n ? av[t] : 0.f;
}

// ---------------------------------------------------------------------------
// rank 0, team warps 0-7: Sherman-Morrison steps of eq. 9 and the gate of
// eq. 10, one chunk at a time (the arithmetic of tc::tc_a_team). Row i < D is
// owned by thread i of warps 0-3 ("primary": z' columns, the substitution,
// the rows of N and -N, lo refresh of columns [0, D/2)) and by thread i of
// warps 4-7 ("helper": w columns, the gate row, lo refresh of columns
// [D/2, D)); the helper forms the gate while the primary writes the update's
// operands.
// Warp 4 also factors I + Guu and sends the gate to the S ranks.
// ---------------------------------------------------------------------------
template <int D, typename TIn, int NS>
__device__ void a_rank(const Params& p, const Ctx3<D, TIn, NS>& x, int bh, int warp, int lane) {
    using L = Lay3<D, TIn, NS>;
    constexpr int XS = L::XS, NRW = L::NRW;
    const int ta = threadIdx.x;
    const bool prim = warp < NRW;
    const bool help = warp >= 4 && warp < 4 + NRW;
    const int i = 32 * (warp & 3) + lane;  // row (TMEM lane) of a primary or helper thread
    const uint32_t tm = __shfl_sync(0xffffffffu, *x.tmem_base, 0);
    const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    const int T = p.T, nch = (T + C - 1) / C;
    float* sm = x.sm();
    float* xr = x.f(L::OFF_XR);
    float* ph = x.f(L::OFF_PH);
    float* pl = x.f(L::OFF_PL);
    float* zh = x.f(L::OFF_ZH);
    float* zl = x.f(L::OFF_ZL);
    float* gp = x.f(L::OFF_GP);
    bool bad = false, nonfinite = false;
    const bool fixed = p.fixed_a != 0;
    int sent = 0;

    // A_0 = I / lambda0 unless carried in (eq. 9), and its lo part
    if (prim) {
        const float* A0 = p.A0 ? p.A0 + ((size_t)bh * D + i) * D : nullptr;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16], w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                v[j] = A0 ? A0[c0 + j] : (i == c0 + j ? p.inv_lambda0 : 0.f);
                w[j] = tf32_lo(v[j]);
            }
            tc_st16(tl + L::T_X + c0, v);
            tc_st16(tl + L::T_XL + c0, w);
        }
        tc_wait_st();
    }
    // rows D..127 of the -N operand stay zero
    for (int e = ta; e < (128 - D) * C; e += NTEAM) {
        ph[cm_off(D + e / C, e % C, C)] = 0.f;
        pl[cm_off(D + e / C, e % C, C)] = 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(ID_T, NTEAM);

    uint32_t pa = 0;
    int c = 0;
    for (; c < nch; ++c) {
        const int s = c % L::NP, n = min(C, T - c * C), b = c & 1;
        bad = !mbar_wait(x.b.full_p + s, (c / L::NP) & 1, x.abort, p.wait_ns);
        if (bar_red_or(ID_T, NTEAM, bad || *x.abort != 0)) {
            bad = true;
            break;
        }
        TC3_STAMP(p, 0, 0, c, nch);
        const float* hi = x.hi(s);
        const float* sc = x.sc(s);
        // [Z' | W] = A_c [u | k]^T; warp q < NISS issues K steps q, q + NISS, ... into accumulator q
        if (warp < NISS && tc::elect_one()) {
            tc_fence_after();
            const uint32_t id = tc_idesc_tf32(128, 2 * C);
            const uint32_t bh0 = smem_u32(hi), bl0 = smem_u32(x.lo(s));
            const uint32_t dst = tm + L::T_P + warp * 2 * C;
#pragma unroll 1
            for (int ks = warp; ks < D / 8; ks += NISS) {
                const uint64_t bd = tc_sdesc(bh0 + ks * 256, 128, L::SBO_D);
                tc_mma_ts(dst, tm + L::T_X + 8 * ks, bd, id, ks >= NISS);
                tc_mma_ts(dst, tm + L::T_XL + 8 * ks, bd, id, 1);
                if constexpr (L::F32IN)
                    tc_mma_ts(dst, tm + L::T_X + 8 * ks, tc_sdesc(bl0 + ks * 256, 128, L::SBO_D), id, 1);
            }
            tc_commit(x.b.mma_p);
        }
        bool ok = mbar_wait(x.b.mma_p, c & 1, nullptr, p.wait_ns);
        TC3_STAMP(p, 0, 1, c, nch);
        tc_fence_after();
        if (prim) {
            float v[16];
            ld_prod_cols(tl + L::T_P, 0, v);
#pragma unroll
            for (int t = 0; t < C; ++t) {
                v[t] *= sc[L::SC_IU + t];  // z'_t = A_c u^_t
                xr[t * XS + i] = v[t];
            }
        } else if (help) {
            float v[16];
            ld_prod_cols(tl + L::T_P, C, v);
#pragma unroll
            for (int t = 0; t < C; ++t) xr[(C + t) * XS + i] = v[t] * sc[L::SC_IK + t];  // w_t = A_c k^_t
        }
        named_bar(ID_T, NTEAM);
        TC3_STAMP(p, 0, 2, c, nch);
        if (!fixed) {
            // Guu[s][t] = u^_s . z'_t, Guk[s][t] = u^_s . w_t: warp = (matrix, quarter of D);
            // quarters 1-3 leave their partial sums, warps 0-1 add them
            const int mat = warp & 1, qtr = warp >> 1;
            float acc[2][4];
            tc::gram16<D, true>(hi, 0, xr + mat * C * XS, XS, qtr * (D / 4), (qtr + 1) * (D / 4), lane, acc,
                                !L::F32IN);
            float* part = gp + (size_t)(mat * 3) * 256 + lane * 8;
            if (qtr > 0) {
#pragma unroll
                for (int m = 0; m < 2; ++m)
                    *reinterpret_cast<float4*>(part + (qtr - 1) * 256 + 4 * m) =
                        make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
            }
            named_bar(ID_T, NTEAM);
            if (qtr == 0) {
#pragma unroll
                for (int k = 0; k < 3; ++k)
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const float4 o = ld4(part + k * 256 + 4 * m);
                        acc[m][0] += o.x;
                        acc[m][1] += o.y;
                        acc[m][2] += o.z;
                        acc[m][3] += o.w;
                    }
                tc::put_gram16(sm + (mat ? L::SM_GUK : L::SM_GUU), L::GSTR, acc, lane, sc + L::SC_IU, false);
            }
            named_bar(ID_T, NTEAM);
        }
        TC3_STAMP(p, 0, 3, c, nch);
        if (ta == 0) mbar_arrive(x.b.empty_p + s);  // done with the chunk's u, k rows
        if (warp == FACTOR_WARP && !fixed) {
            // LDL^T of I + Guu by Gaussian elimination of the augmented
            // [I + Guu | Guk]: lane j < C holds column j, lane C + j column j of
            // Guk. delta_t = pivot t (eq. 9's 1 + u^_t . z_t), L[r][t] = the
            // multipliers, and the Guk columns end as X = L^-1 Guk.
            const int j = lane & (C - 1);
            const bool mcol = lane < C;
            const float* src = sm + (mcol ? L::SM_GUU : L::SM_GUK);
            float col[C];
#pragma unroll
            for (int r = 0; r < C; ++r) col[r] = src[r * L::GSTR + j] + ((mcol && r == j) ? 1.f : 0.f);
            float myrd = 0.f, mydl = 1.f;
#pragma unroll 16
            for (int t = 0; t < C; ++t) {
                const float piv = __shfl_sync(0xffffffffu, col[t], t);
                const float rdt = tc::rcp_approx(piv);
                if (lane == t) {
                    myrd = rdt;
                    mydl = piv;  // delta_t; its 1/sqrt is taken after the elimination, off its chain
                }
                if (!(piv > 0.f) || !isfinite(rdt)) nonfinite = true;
                const bool live = !mcol || lane > t;
                const float ct = col[t] * rdt;
#pragma unroll
                for (int r = 0; r < C; ++r)
                    if (r > t) {
                        const float m = __shfl_sync(0xffffffffu, col[r], t);
                        if (live) col[r] = fmaf(-m, ct, col[r]);
                    }
            }
            if (mcol) {
                sm[L::SM_RD + j] = myrd;
                sm[L::SM_RS + j] = rsqrtf(mydl);
#pragma unroll
                for (int r = 0; r < C; ++r)  // L[r][j] below the unit diagonal, stored transposed
                    sm[L::SM_LMT + j * L::GSTR + r] = r > j ? col[r] * myrd : 0.f;
            } else {
#pragma unroll
                for (int r = 0; r < C; ++r) sm[L::SM_X + r * L::GSTR + j] = col[r];  // X[r][j]
            }
        } else if (c >= 2) {
            // every S rank is done with mailbox buffer b (chunk c - 2), so its
            // local source can be rewritten
            ok = ok && mbar_wait_cl(x.b.empty_al + b, ((c >> 1) & 1) ^ 1, x.abort, p.wait_ns);
        }
        if (bar_red_or(ID_T, NTEAM, !ok || *x.abort != 0)) {
            bad = true;
            break;
        }
        TC3_STAMP(p, 0, 4, c, nch);
        float* alr = x.f(L::OFF_AL) + (size_t)b * C * XS;
        float* gh = x.f(L::OFF_GH) + (size_t)b * D * C;
        float* gl = x.f(L::OFF_GL) + (size_t)b * D * C;
        // every S rank is done with buffer b: arm its barrier for this chunk's
        // bytes now (the phase completes when the bulk copies below land), so
        // that the send after the gate only issues the copies
        if (warp == FACTOR_WARP && lane < NS)
            mbar_expect_tx_peer_relaxed(peer_addr(x.b.full_al + b, (uint32_t)lane + 1u), L::MB_BYTES);
        float y[C];
        if (prim) {
            float nv[C];
            if (!fixed) {
                // y = z_i = z'_i L^-T (forward substitution, in place), then y D^-1;
                // published in xr rows 0..C-1 for the helper's gate row
                float lr[C];
#pragma unroll
                for (int t = 0; t < C; ++t) y[t] = xr[t * XS + i];
#pragma unroll
                for (int r = 0; r < C - 1; ++r) {
                    tc::ld_row16(sm + L::SM_LMT + r * L::GSTR, lr);  // L[t][r], t > r
#pragma unroll
                    for (int t = r + 1; t < C; ++t) y[t] = fmaf(-lr[t], y[r], y[t]);
                }
                // row i of N = Z D^-1/2: A_{c+1} = A_c - N N^T (symmetric by construction)
                tc::ld_row16(sm + L::SM_RS, lr);
#pragma unroll
                for (int t = 0; t < C; ++t) nv[t] = y[t] * lr[t];
                tc::ld_row16(sm + L::SM_RD, lr);
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    y[t] *= lr[t];
                    xr[t * XS + i] = y[t];
                }
            }
            TC3_STAMP(p, 0, 8, c, nch);
            tc::bar_arrive(ID_Y, 64 * NRW);
            if (!fixed) {
                tc::put_row16(zh, i, nv, false);
                tc::put_row16(zl, i, nv, true);
#pragma unroll
                for (int t = 0; t < C; ++t) nv[t] = -nv[t];
                tc::put_row16(ph, i, nv, false);
                tc::put_row16(pl, i, nv, true);
                fence_proxy_async_smem();
            }
            TC3_STAMP(p, 0, 9, c, nch);
            // A_{c+1} = A_c - N N^T once every row's -N and N are in place
            named_bar(ID_M, 32 * NRW);
            if (warp == 0 && !fixed && tc::elect_one()) {
                tc_fence_after();
                const uint32_t id = tc_idesc_tf32(128, D);
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks) {
                    const uint64_t ah = tc_sdesc(smem_u32(ph) + ks * 256, 128, L::SBO_C);
                    const uint64_t alo = tc_sdesc(smem_u32(pl) + ks * 256, 128, L::SBO_C);
                    const uint64_t bhd = tc_sdesc(smem_u32(zh) + ks * 256, 128, L::SBO_C);
                    const uint64_t bld = tc_sdesc(smem_u32(zl) + ks * 256, 128, L::SBO_C);
                    tc_mma_ss(tm + L::T_X, ah, bhd, id, 1);
                    tc_mma_ss(tm + L::T_X, ah, bld, id, 1);
                    tc_mma_ss(tm + L::T_X, alo, bhd, id, 1);
                }
                tc_commit(x.b.mma_x);
            }
            TC3_STAMP(p, 0, 10, c, nch);
        } else if (help) {
            named_bar(ID_Y, 64 * NRW);
            TC3_STAMP_T(p, 0, 12, c, nch, 128);
            // the gate row, with y = z / delta from xr
#pragma unroll
            for (int t = 0; t < C; ++t) y[t] = !fixed ? xr[t * XS + i] : 0.f;
            float av[C];
            gate16(xr, XS, sm + L::SM_X, L::GSTR, i, n, fixed, y, av);
#pragma unroll
            for (int t = 0; t < C; ++t) alr[t * XS + i] = av[t];
            tc::put_row16(gh, i, av, false);
            tc::put_row16(gl, i, av, true);
            TC3_STAMP_T(p, 0, 13, c, nch, 128);
        }
        fence_proxy_async_smem();
        named_bar(ID_T, NTEAM);
        TC3_STAMP(p, 0, 5, c, nch);
        if (warp == FACTOR_WARP) {
            // the chunk's gate into every S rank's mailbox (its barrier was armed above)
            if (lane < NS) {
                const uint32_t peer = (uint32_t)lane + 1u;
                const uint32_t rbar = peer_addr(x.b.full_al + b, peer);
                const uint32_t r_al = peer_addr(x.f(L::OFF_AL), peer);
                bulk_to_peer(r_al + (uint32_t)(b * L::MB_ALR), alr, L::MB_ALR, rbar);
                bulk_to_peer(r_al + (uint32_t)(L::OFF_GH - L::OFF_AL) + b * L::MB_G, gh, L::MB_G, rbar);
                bulk_to_peer(r_al + (uint32_t)(L::OFF_GL - L::OFF_AL) + b * L::MB_G, gl, L::MB_G, rbar);
            }
            ++sent;
        }
        if (!fixed) {
            bad = !mbar_wait(x.b.mma_x, pa, nullptr, p.wait_ns);
            pa ^= 1;
        }
        TC3_STAMP(p, 0, 6, c, nch);
        tc_fence_after();
        if (!fixed) {
            if (prim) refresh_cols<D / 2>(tl, L::T_X, L::T_XL, 0);
            if (help) refresh_cols<D / 2>(tl, L::T_X, L::T_XL, D / 2);
        }
        tc_fence_before();
        if (bar_red_or(ID_T, NTEAM, bad)) {
            bad = true;
            ++c;
            break;
        }
        TC3_STAMP(p, 0, 7, c, nch);
    }
    if (warp == FACTOR_WARP && lane == 0) {
        *x.n_sent = sent;
#pragma unroll 1
        for (int r = 1; r <= NS; ++r) st_peer_u32(peer_addr(x.n_sent, (uint32_t)r), (uint32_t)sent);
    }
    if (bad) {
        if (ta == 0) {
            record_failure(p.status, BIT_TIMEOUT, ROLE_A, bh, c * C);
            x.abort_peers(0u);
        }
    } else if (prim) {
        float* Ao = p.A_out + ((size_t)bh * D + i) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
            tc_ld16(tl + L::T_X + c0, v);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(Ao + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    if (nonfinite) record_failure(p.status, BIT_NONFINITE, ROLE_A, bh, -1);
}

// ---------------------------------------------------------------------------
// S rank r = 1..NS, team warps 0-7: residual writes and readout of eq. 10-11
// for rows [R0, R0 + R) of S (R0 = (r - 1) R), local row i at TMEM lane i.
// Row i is owned by thread i of warp i / 32 ("primary": S k^ columns, the
// unit-triangular solve, the E' row, lo refresh of columns [0, D/2)) and of
// warp 4 + i / 32 ("helper": S phi columns, the readout o_t, lo refresh of
// columns [D/2, D)). The chunk's products are issued before the gate
// arrives; once it has arrived, all eight warps form the Gram matrices Lk, Lq
// (the row warps have read their products by then).
// ---------------------------------------------------------------------------
template <int D, typename TIn, int NS>
__device__ void s_rank(const Params& p, const Ctx3<D, TIn, NS>& x, int bh, int warp, int lane, uint32_t rank) {
    using L = Lay3<D, TIn, NS>;
    constexpr int XS = L::XS, R = L::R, NRS = L::NRS;
    const int ts = threadIdx.x;
    const int i = 32 * (warp & 3) + lane;  // local row (TMEM lane) of a primary or helper thread
    // tcgen05.ld / st are warp-wide (.sync.aligned): whole primary and helper
    // warps take part in them (lanes i >= R of a partial warp read and refresh
    // rows that stay zero); prim / help select the threads whose row is real
    const bool prim_w = warp < NRS, help_w = warp >= 4 && warp < 4 + NRS;
    const bool prim = prim_w && i < R;
    const bool help = help_w && i < R;
    const bool gram = (warp & 3) >= 2;
    const int R0 = ((int)rank - 1) * R;
    const int gi = R0 + i;  // global row of S
    const uint32_t tm = __shfl_sync(0xffffffffu, *x.tmem_base, 0);
    const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    const int T = p.T, nch = (T + C - 1) / C;
    float* sm = x.sm();
    float* eh = x.f(L::OFF_EH);
    float* el = x.f(L::OFF_EL);
    const TIn* gv = static_cast<const TIn*>(p.v) + (size_t)bh * T * D;
    float* go = p.o + (size_t)bh * p.o_stride;
    const uint32_t r_empty_al = peer_addr(x.b.empty_al, 0u);
    bool bad = false, nonfinite = false;
    float nfchk = 0.f;  // fma(o, 0, .) of every output (branch-free)
    int recv = 0;

    // S_0 rows (0 unless carried in) and their lo part; lanes R..127 hold zeros
    if (warp < 4) {
        const float* S0 = (p.S0 && i < R) ? p.S0 + ((size_t)bh * D + gi) * D : nullptr;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16], w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                v[j] = S0 ? S0[c0 + j] : 0.f;
                w[j] = tf32_lo(v[j]);
            }
            tc_st16(tl + L::T_X + c0, v);
            tc_st16(tl + L::T_XL + c0, w);
        }
        tc_wait_st();
    }
    // rows R..127 of the E' operand stay zero
    for (int e = ts; e < (128 - R) * C; e += NTEAM) {
        eh[cm_off(R + e / C, e % C, C)] = 0.f;
        el[cm_off(R + e / C, e % C, C)] = 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(ID_T, NTEAM);

    uint32_t ps = 0;
    int c = 0;
    for (; c < nch; ++c) {
        const int s = c % L::NP, n = min(C, T - c * C), b = c & 1;
        typename tc::RawIn<TIn>::type vr[C];
        if (prim) tc::load_v_raw<D, TIn>(gv + (size_t)c * C * D, gi, n, vr);
        TC3_STAMP(p, rank, 0, c, nch);
        bad = !mbar_wait(x.b.full_p + s, (c / L::NP) & 1, x.abort, p.wait_ns);
        if (bar_red_or(ID_T, NTEAM, bad || *x.abort != 0)) {
            bad = true;
            break;
        }
        TC3_STAMP(p, rank, 1, c, nch);
        const float* hi = x.hi(s);
        const float* sc = x.sc(s);
        const float* alr = x.f(L::OFF_AL) + (size_t)b * C * XS;
        // [S_c k | S_c phi] for this rank's rows, issued before the gate arrives;
        // warp q < NISS issues K steps q, q + NISS, ... into accumulator q
        if (warp < NISS && tc::elect_one()) {
            tc_fence_after();
            const uint32_t id32 = tc_idesc_tf32(128, 2 * C), id16 = tc_idesc_tf32(128, C);
            const uint32_t bh0 = smem_u32(hi), bl0 = smem_u32(x.lo(s));
            const uint32_t dst = tm + L::T_P + warp * 2 * C;
#pragma unroll 1
            for (int ks = warp; ks < D / 8; ks += NISS) {
                const uint64_t bd = tc_sdesc(bh0 + ks * 256, 128, L::SBO_D);
                const uint64_t bld = tc_sdesc(bl0 + ks * 256, 128, L::SBO_D);
                tc_mma_ts(dst, tm + L::T_X + 8 * ks, bd, id32, ks >= NISS);
                tc_mma_ts(dst, tm + L::T_XL + 8 * ks, bd, id32, 1);
                if constexpr (L::F32IN)
                    tc_mma_ts(dst, tm + L::T_X + 8 * ks, bld, id32, 1);
                else
                    tc_mma_ts(dst + C, tm + L::T_X + 8 * ks, bld, id16, 1);
            }
            tc_commit(x.b.mma_p);
        }
        bool ok = true;
        float sk[C], sq[C];
        if (!gram) {
            ok = mbar_wait(x.b.mma_p, c & 1, nullptr, p.wait_ns);
            TC3_STAMP(p, rank, 8, c, nch);
            tc_fence_after();
            if (prim_w) {
                ld_prod_cols(tl + L::T_P, 0, sk);
#pragma unroll
                for (int t = 0; t < C; ++t) sk[t] *= sc[L::SC_IK + t];  // S_c k^_t
            } else if (help_w) {
                ld_prod_cols(tl + L::T_P, C, sq);  // S_c phi_t
            }
        }
        ok = mbar_wait_cl(x.b.full_al + b, (c >> 1) & 1, x.abort, p.wait_ns) && ok;
        TC3_STAMP(p, rank, 9, c, nch);
        {
            // Lk[t][s] = k^_t . a_s, Lq[t][s] = phi_t . a_s on all eight warps
            // (matrix, quarter of D); quarters 1-3 leave their partial sums,
            // warps 0-1 add them (a failed wait leaves garbage here, which the
            // vote below discards)
            const int mat = warp & 1, qtr = warp >> 1;
            float acc[2][4];
            tc::gram16<D, true>(hi + (mat ? C : 0) * D, 0, alr, XS, qtr * (D / 4), (qtr + 1) * (D / 4), lane, acc,
                                !L::F32IN && mat == 0);
            float* part = x.f(L::OFF_GPS) + (size_t)(mat * 3) * 256 + lane * 8;
            if (qtr > 0) {
#pragma unroll
                for (int m = 0; m < 2; ++m)
                    *reinterpret_cast<float4*>(part + (qtr - 1) * 256 + 4 * m) =
                        make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
            }
            if (warp == 4 && lane < C) {
                // ||a_t||^2 from the gate rows that arrived
                float2 a2 = f2(0.f, 0.f);
#pragma unroll 8
                for (int k4 = 0; k4 < D / 4; ++k4) {
                    const float4 a = ld4(alr + lane * XS + 4 * k4);
                    a2 = __ffma2_rn(f2(a.x, a.y), f2(a.x, a.y), a2);
                    a2 = __ffma2_rn(f2(a.z, a.w), f2(a.z, a.w), a2);
                }
                x.f(L::OFF_LAA)[b * C + lane] = a2.x + a2.y;
            }
            named_bar(ID_T, NTEAM);
            if (qtr == 0) {
#pragma unroll
                for (int k = 0; k < 3; ++k)
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const float4 o = ld4(part + k * 256 + 4 * m);
                        acc[m][0] += o.x;
                        acc[m][1] += o.y;
                        acc[m][2] += o.z;
                        acc[m][3] += o.w;
                    }
                if (mat)
                    tc::put_gram16(sm + L::SM_LQ, L::GSTR, acc, lane, nullptr, false);
                else
                    tc::put_gram16(sm + L::SM_LKT, L::GSTR, acc, lane, sc + L::SC_IK, true);
            }
            TC3_STAMP_T(p, rank, 7, c, nch, 64);
        }
        if (bar_red_or(ID_T, NTEAM, !ok || *x.abort != 0)) {
            bad = true;
            break;
        }
        recv = c + 1;
        TC3_STAMP(p, rank, 2, c, nch);
        if (warp < NRS) {
            // primary warps (rows i >= R of a partial warp take part in the barriers only)
            if (prim) {
                float lr[C], nr[C], vv[C];
                // e_t = v_t - S_c k^_t - sum_{s<t} (k^_t . alpha^_s) e_s, kept (in place)
                // as e'_t = e_t / ||a_t||
                tc::ld_row16(x.f(L::OFF_LAA) + b * C, nr);
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    vv[t] = tc::raw_f32(vr[t]) - sk[t];
                    nr[t] = rsqrtf(fmaxf(nr[t], 1e-24f));
                }
#pragma unroll
                for (int r = 0; r < C; ++r) {
                    vv[r] *= nr[r];
                    if (r < C - 1) {
                        tc::ld_row16(sm + L::SM_LKT + r * L::GSTR, lr);  // Lk[t][r], t > r
#pragma unroll
                        for (int t = r + 1; t < C; ++t) vv[t] = fmaf(-lr[t], vv[r], vv[t]);
                    }
                }
                tc::put_row16(eh, i, vv, false);
                tc::put_row16(el, i, vv, true);
            }
            TC3_STAMP(p, rank, 10, c, nch);
            fence_proxy_async_smem();
            tc::bar_arrive(ID_E, 64 * NRS);
            // S_{c+1} = S_c + E' A once every row's E' is in place (rows a_t from the mailbox)
            named_bar(ID_EM, 32 * NRS);
            if (warp == 0 && tc::elect_one()) {
                tc_fence_after();
                const uint32_t id = tc_idesc_tf32(128, D);
                const float* gh = x.f(L::OFF_GH) + (size_t)b * D * C;
                const float* gl = x.f(L::OFF_GL) + (size_t)b * D * C;
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks) {
                    const uint64_t ah = tc_sdesc(smem_u32(eh) + ks * 256, 128, L::SBO_C);
                    const uint64_t alo = tc_sdesc(smem_u32(el) + ks * 256, 128, L::SBO_C);
                    const uint64_t bhd = tc_sdesc(smem_u32(gh) + ks * 256, 128, L::SBO_C);
                    const uint64_t bld = tc_sdesc(smem_u32(gl) + ks * 256, 128, L::SBO_C);
                    tc_mma_ss(tm + L::T_X, ah, bhd, id, 1);
                    tc_mma_ss(tm + L::T_X, ah, bld, id, 1);
                    tc_mma_ss(tm + L::T_X, alo, bhd, id, 1);
                }
                tc_commit(x.b.mma_x);
            }
            TC3_STAMP(p, rank, 3, c, nch);
        } else if (warp >= 4 && warp < 4 + NRS) {
            // helper warps (rows i >= R of a partial warp take part in the barriers only)
            named_bar(ID_E, 64 * NRS);
            if (help) {
                // o_t = (S_c phi_t + sum_{s<=t} e_s (alpha^_s . phi_t)) / den_t = S_t phi_t / den_t (eq. 11)
                float ev[C], lr[C], rd[C];
#pragma unroll
                for (int g = 0; g < C / 4; ++g) {
                    const float4 e4 = ld4(eh + cm_off(i, 4 * g, C));
                    ev[4 * g] = e4.x;
                    ev[4 * g + 1] = e4.y;
                    ev[4 * g + 2] = e4.z;
                    ev[4 * g + 3] = e4.w;
                }
                tc::ld_row16(sc + L::SC_RDEN, rd);
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    tc::ld_row16(sm + L::SM_LQ + t * L::GSTR, lr);
                    float a = sq[t];
#pragma unroll
                    for (int q = 0; q <= t; ++q) a = fmaf(lr[q], ev[q], a);
                    const float ov = a * rd[t];
                    if (t < n) {
                        go[(size_t)(c * C + t) * D + gi] = ov;
                        nfchk = fmaf(ov, 0.f, nfchk);  // stays 0 unless an o is NaN or Inf
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(x.b.empty_p + s);  // done with the chunk's k, phi rows and den
            TC3_STAMP_T(p, rank, 6, c, nch, 128);
        }
        ok = mbar_wait(x.b.mma_x, ps, nullptr, p.wait_ns);
        ps ^= 1;
        TC3_STAMP(p, rank, 4, c, nch);
        tc_fence_after();
        if (ts == 0) mbar_arrive_peer(r_empty_al + 8u * b);  // mailbox buffer b back to rank 0
        if (prim_w) refresh_cols<D / 2>(tl, L::T_X, L::T_XL, 0);
        if (help_w) refresh_cols<D / 2>(tl, L::T_X, L::T_XL, D / 2);
        tc_fence_before();
        if (bar_red_or(ID_T, NTEAM, !ok)) {
            bad = true;
            ++c;
            break;
        }
        TC3_STAMP(p, rank, 5, c, nch);
    }
    if (ts == 0) *x.n_recv = recv;
    if (bad) {
        if (ts == 0) {
            record_failure(p.status, BIT_TIMEOUT, ROLE_S, bh, c * C);
            x.abort_peers(rank);
        }
    } else if (prim_w) {
        float* So = p.S_out + ((size_t)bh * D + (prim ? gi : 0)) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
            tc_ld16(tl + L::T_X + c0, v);  // the whole warp (see prim_w)
            tc_wait_ld();
            if (prim) {
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4*>(So + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
    }
    if (nonfinite || nfchk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_S, bh, -1);
}

}  // namespace tc3

template <int D, typename TIn, int NS>
__global__ void __launch_bounds__(tc3::THREADS, 1) vla_tc3_kernel(const Params p) {
    using L = tc3::Lay3<D, TIn, NS>;
    extern __shared__ __align__(1024) unsigned char smem[];
    tc3::Ctx3<D, TIn, NS> x;
    x.base = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
    x.b.full_r = bars;
    x.b.full_p = x.b.full_r + L::NRAW;
    x.b.empty_p = x.b.full_p + L::NP;
    x.b.full_al = x.b.empty_p + L::NP;
    x.b.empty_al = x.b.full_al + 2;
    x.b.mma_x = x.b.empty_al + 2;
    x.b.mma_p = x.b.mma_x + 1;
    x.abort = reinterpret_cast<volatile int*>(smem + L::OFF_MISC);
    x.tmem_base = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC + 4);
    x.n_sent = reinterpret_cast<int*>(smem + L::OFF_MISC + 8);
    x.n_recv = reinterpret_cast<int*>(smem + L::OFF_MISC + 12);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const uint32_t rank = tc3::cluster_rank();
    const int bh = blockIdx.x / (1 + NS);
    if (threadIdx.x == 0) {
        for (int r = 0; r < L::NRAW; ++r) mbar_init(x.b.full_r + r, 1);
        for (int s = 0; s < L::NP; ++s) {
            mbar_init(x.b.full_p + s, 1);
            // rank 0: one arrival after the Gram matrices; S ranks: one per helper warp after the readout
            mbar_init(x.b.empty_p + s, rank == 0 ? 1 : L::NRS);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(x.b.full_al + s, 1);
            mbar_init(x.b.empty_al + s, NS);
        }
        mbar_init(x.b.mma_x, 1);
        mbar_init(x.b.mma_p, tc3::NISS);
        *x.abort = 0;
        *x.n_sent = 0;
        *x.n_recv = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc_alloc(x.tmem_base, L::TCOLS);
    tc_fence_before();
    // every rank's barriers are initialised before any rank arrives on them
    tc3::cluster_sync_all();
    tc_fence_after();
    if (warp < 8) {
        if (rank == 0)
            tc3::a_rank<D, TIn, NS>(p, x, bh, warp, lane);
        else
            tc3::s_rank<D, TIn, NS>(p, x, bh, warp, lane, rank);
    } else if (rank == 0) {
        tc2::stage2<D, TIn, true>(p, x, bh, warp - 8, lane, rank);
    } else {
        tc2::stage2<D, TIn, false>(p, x, bh, warp - 8, lane, rank, rank == 1);
    }
    tc_fence_before();
    __syncthreads();
    // rank 0 has sent its last mailbox buffer and written the count into every S rank
    tc3::cluster_sync_all();
    if (rank != 0 && threadIdx.x == 0) {
        // after a failure: let the buffers that rank 0 sent but this rank did
        // not consume land before the CTA can exit
        for (int j = *x.n_recv; j < *x.n_sent; ++j)
            (void)tc3::mbar_wait_cl(x.b.full_al + (j & 1), (j >> 1) & 1, nullptr, p.wait_ns);
    }
    tc3::cluster_sync_all();
    tc_fence_after();
    if (warp == 0) tc_dealloc(*x.tmem_base, L::TCOLS);
}
