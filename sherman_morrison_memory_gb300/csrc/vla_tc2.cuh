// vla_tc2.cuh -- the chunked tensor-core recurrence of vla_tc.cuh split over a
// cluster of two CTAs per (batch, head). Included by vla_forward.cu inside
// namespace vla, after vla_tc.cuh (it reuses that file's chunk arithmetic
// helpers: gram16, put_row16, refresh_lo, ...).
//
// "Variational Linear Attention" (arXiv 2605.11196), §3.3 eq. 9-11, C = 16
// tokens at a time, exactly as in vla_tc.cuh, but the two recurrences of a
// head run on two SMs:
//
//   CTA rank 0 (A-pass)  stages u, k; A and its tf32 lo part in its own tensor
//                        memory; per chunk [A u | A k] on the tensor cores,
//                        the Gram matrices, the LDL^T of I + U^ A U^^T, the
//                        state update A -= N N^T (eq. 9) and the gate rows
//                        a_t = A_t k^_t (eq. 10), which it sends to rank 1
//   CTA rank 1 (S-pass)  stages q, k; S and its lo part in its own tensor
//                        memory; per chunk [S k | S phi] on the tensor cores,
//                        the residual writes e_t and the readout o_t (eq. 10,
//                        11) and S += E' A on the tensor cores
//
// The hand-off is the gate of a chunk: its rows a_t (row-major, for the S
// side's Gram matrices), the K-major hi / lo tiles of its transpose (the B
// operand of S's update) and ||a_t||^2. Rank 0 builds them in its own shared
// memory and moves them into rank 1's shared memory with one bulk copy each
// (cp.async.bulk shared::cta -> shared::cluster), completing on a barrier of
// rank 1; rank 1 hands each of the two mailbox buffers back with a remote
// mbarrier arrive once its update has read it.
//
// Each SM holds a whole tensor memory and shared memory for one state, so the
// split also runs d = 128 (A, S and their lo parts need 4 d = 512 columns, all
// of one SM's tensor memory), and heads that are fewer than the SMs use twice
// as many SMs.
//
// Warps (both ranks launch 12): rank 0: 0-3 A rows (TMEM lane quarters) and
// the Gram matrices, 4 the LDL^T factorisation and the hand-off, 8-11 staging;
// rank 1: 0-3 S rows and the Gram matrices, 8-11 staging. Every wait is
// bounded; a role that gives up raises the abort flag of both ranks.

namespace tc2 {

// -DVLA_TRACE builds: per-chunk clock stamps of head 0's cluster, stamp k of
// chunk c at trace[row][k * nch + c] (row 4: rank 0, row 5: rank 1)
#define TC2_STAMP(p, row, k, c, nch) \
    VLA_TRACE_IF(p, blockIdx.x < 2 && threadIdx.x == 0, row, (k) * (nch) + (c))

constexpr int C = tc::C;
constexpr int NSTAGE = 4;
constexpr int THREADS = 32 * 12;
constexpr int NT_A = 160, NT_S = 128;        // threads of the rank-0 / rank-1 team barrier
constexpr int ID_T = 1, ID_ST = 3;           // team and staging named barriers (4, 5: Gram pairs)
constexpr int FACTOR_WARP = 4;
// warps that issue the d x 2C chunk products (one thread each, into their own
// accumulator): issuing a tcgen05.mma costs a thread about 100 clocks at
// N = 2C, so the K steps are spread over four issuers
constexpr int NISS = 4;
// one CTA per SM: a second CTA's tensor-memory request could otherwise wait
// for a CTA whose cluster peer waits for it
constexpr size_t MIN_SMEM = 116 * 1024;

// ---------------------------------------------------------------------------
// cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_peer(uint32_t rbar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_peer(uint32_t rbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(rbar),
                 "r"(bytes)
                 : "memory");
}
// bulk copy from this CTA's shared memory into a peer's, completing on the peer's barrier
__device__ __forceinline__ void bulk_to_peer(uint32_t rdst, const void* src, uint32_t bytes, uint32_t rbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     rdst),
                 "r"(smem_u32(src)), "r"(bytes), "r"(rbar)
                 : "memory");
}
__device__ __forceinline__ void st_peer_u32(uint32_t raddr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(raddr), "r"(v) : "memory");
}
// every thread of both CTAs
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// waits on barriers that the peer CTA arrives on: acquire at cluster scope
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __noinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                          uint64_t limit_ns) {
    if (mbar_try_wait_cl(bar, parity, 0u)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait_cl(bar, parity, 20000u)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// row i of the chunk products summed over the NISS accumulators: columns
// [0, C) into a, [C, 2C) into b (this warp's TMEM lanes)
__device__ __forceinline__ void ld_products(uint32_t tp, float (&a)[16], float (&b)[16]) {
    tc_ld16(tp, a);
    tc_ld16(tp + C, b);
    tc_wait_ld();
#pragma unroll 1
    for (int q = 1; q < NISS; ++q) {
        float x[16], y[16];
        tc_ld16(tp + q * 2 * C, x);
        tc_ld16(tp + q * 2 * C + C, y);
        tc_wait_ld();
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            a[t] += x[t];
            b[t] += y[t];
        }
    }
}

// ---------------------------------------------------------------------------
// layout (the same offsets in both ranks, so that the mailbox and the
// barriers of the peer are found by mapa)
// ---------------------------------------------------------------------------
template <int D, typename TIn>
struct Lay2 {
    static constexpr bool F32IN = sizeof(TIn) == 4;
    static constexpr int NRW = D / 32;          // row warps
    static constexpr int NP = F32IN ? 2 : 3;    // prepared chunk slots
    static constexpr int NRAW = F32IN ? 1 : 2;  // raw chunk slots
    // prepared chunk: HI tile rows 0..C-1 | C..2C-1 = u | k (rank 0) or k | phi
    // (rank 1); LO tile: rank 0 fp32 u_lo | k_lo; rank 1 fp32 k_lo | phi_lo,
    // bf16 phi_lo (bf16 u, k are exact in tf32)
    static constexpr int HI_ROWS = 2 * C;
    static constexpr int LO_ROWS = F32IN ? 2 * C : C;
    static constexpr int SBO_D = (D / 4) * 128;
    static constexpr int SBO_C = (C / 4) * 128;
    static constexpr int SC_IU = 0, SC_IK = C, SC_RDEN = 2 * C;
    static constexpr int SLOT = (HI_ROWS + LO_ROWS) * D + 64;  // floats
    static constexpr int SCR_STRIDE = D + 4;
    static constexpr int GSTR = C + 4;
    static constexpr int XS = D + 4;
    // tensor memory of each rank: state | its lo part | chunk products (K
    // step ks in accumulator ks mod NISS, 2C columns each)
    static constexpr uint32_t T_X = 0, T_XL = D, T_P = 2 * D;
    static constexpr uint32_t TNEED = 2 * D + NISS * 2 * C;
    static constexpr uint32_t TCOLS = TNEED <= 128 ? 128 : (TNEED <= 256 ? 256 : 512);
    static_assert(TNEED <= 512, "TMEM columns");
    // mailbox buffer sizes (bytes)
    static constexpr uint32_t MB_ALR = C * XS * 4, MB_G = D * C * 4, MB_LAA = C * 4;
    static constexpr uint32_t MB_BYTES = MB_ALR + 2 * MB_G + MB_LAA;
    static_assert(MB_ALR % 16 == 0 && MB_G % 16 == 0 && MB_LAA % 16 == 0, "bulk-copy granularity");

    static constexpr size_t al(size_t x) { return (x + 127) / 128 * 128; }
    static constexpr int NBAR = NRAW + 2 * NP + 2 + 2 + 2;
    static constexpr size_t OFF_BAR = 0;
    static constexpr size_t OFF_MISC = al(8 * NBAR);  // abort flag, TMEM base, mailbox counts
    static constexpr size_t OFF_PREP = al(OFF_MISC + 16);
    static constexpr size_t OFF_RAW = al(OFF_PREP + (size_t)NP * SLOT * 4);
    static constexpr size_t RAW_T = (size_t)C * D * sizeof(TIn);
    static constexpr size_t OFF_SCR = al(OFF_RAW + (size_t)NRAW * 2 * RAW_T);
    static constexpr size_t OFF_AL = al(OFF_SCR + (size_t)2 * C * SCR_STRIDE * 4);  // a rows [2][C x XS]
    static constexpr size_t OFF_GH = OFF_AL + 2 * (size_t)MB_ALR;                    // a^T hi [2][D x C]
    static constexpr size_t OFF_GL = OFF_GH + 2 * (size_t)MB_G;                      // a^T lo [2][D x C]
    static constexpr size_t OFF_LAA = OFF_GL + 2 * (size_t)MB_G;                     // ||a||^2 [2][C]
    static constexpr size_t OFF_SM = al(OFF_LAA + 2 * (size_t)MB_LAA);
    // small matrices, rank 0: Guu, Guk (two partials each), 1/sqrt(delta), L^T, X^T, 1/delta;
    // rank 1: Lk^T, Lq (two partials each)
    static constexpr int MS = C * GSTR;
    static constexpr int SM_GUU = 0, SM_GUK = 2 * MS, SM_RS = 4 * MS, SM_LMT = 5 * MS, SM_XGT = 6 * MS,
                         SM_RD = 7 * MS, SM_LKT = 0, SM_LQ = 2 * MS;
    static constexpr size_t OFF_U = al(OFF_SM + (size_t)(7 * MS + C) * 4);
    // role-specific region: rank 0 xr (z' | w rows) [2C x XS], -N hi/lo
    // [128 x C], N hi/lo [D x C]; rank 1 E' hi/lo [128 x C], staging phi(k) sums
    static constexpr size_t OFF_XR = OFF_U;
    static constexpr size_t OFF_PH = al(OFF_XR + (size_t)2 * C * XS * 4);
    static constexpr size_t OFF_PL = OFF_PH + 128 * C * 4;
    static constexpr size_t OFF_ZH = OFF_PL + 128 * C * 4;
    static constexpr size_t OFF_ZL = OFF_ZH + (size_t)D * C * 4;
    static constexpr size_t END_A = OFF_ZL + (size_t)D * C * 4;
    static constexpr size_t OFF_EH = OFF_U;
    static constexpr size_t OFF_EL = OFF_EH + 128 * C * 4;
    static constexpr size_t OFF_ZP = OFF_EL + 128 * C * 4;
    static constexpr size_t END_S = OFF_ZP + (size_t)NSTAGE * D * 4;
    static constexpr size_t SMEM = al(END_A > END_S ? END_A : END_S);
    static constexpr size_t SMEM_LAUNCH = SMEM > MIN_SMEM ? SMEM : MIN_SMEM;
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(RAW_T % 16 == 0 && (D * sizeof(TIn)) % 16 == 0, "bulk-copy granularity");
};

struct Bars2 {
    uint64_t* full_r;    // [NRAW] raw chunk landed
    uint64_t* full_p;    // [NP] prepared chunk published
    uint64_t* empty_p;   // [NP] released by the team
    uint64_t* full_al;   // [2] rank 1: mailbox buffer filled by rank 0 (tx bytes)
    uint64_t* empty_al;  // [2] rank 0: rank 1 done with the mailbox buffer
    uint64_t* mma_x;     // state update committed
    uint64_t* mma_p;     // chunk products issued by NISS warps (count NISS)
};

template <int D, typename TIn>
struct Ctx2 {
    using L = Lay2<D, TIn>;
    unsigned char* base;
    Bars2 b;
    volatile int* abort;
    uint32_t* tmem_base;
    int* n_sent;      // rank 0: mailbox buffers sent; rank 1: the same count, written by rank 0 at the end
    int* n_recv;      // rank 1: mailbox buffers received
    __device__ float* slot(int s) const { return reinterpret_cast<float*>(base + L::OFF_PREP) + (size_t)s * L::SLOT; }
    __device__ float* hi(int s) const { return slot(s); }
    __device__ float* lo(int s) const { return slot(s) + L::HI_ROWS * D; }
    __device__ float* sc(int s) const { return slot(s) + (L::HI_ROWS + L::LO_ROWS) * D; }
    __device__ unsigned char* raw(int r) const { return base + L::OFF_RAW + (size_t)r * 2 * L::RAW_T; }
    __device__ float* f(size_t off) const { return reinterpret_cast<float*>(base + off); }
    __device__ float* sm() const { return f(L::OFF_SM); }
    // raise the abort flag here and in the peer CTA
    __device__ void abort_peers(uint32_t rank) const {
        *abort = 1;
        st_peer_u32(peer_addr((const void*)abort, rank ^ 1u), 1u);
    }
};

// ---------------------------------------------------------------------------
// staging warps (4) of either rank: per chunk, TMA bulk copies of two raw
// tensors (A side: u, k; S side: q, k); warp w handles tokens 4w..4w+3.
// A side (RANK0): 1/||u||, 1/||k|| and the u | k operand tiles. S side:
// phi(q), 1/||k||, z^key += phi(k) and den = max(phi(q) . z^key, eps)
// (eq. 11), the k | phi operand tiles; `write_zk`: this CTA writes the final
// z^key. X is the cluster kernel's context (its layout X::L has the fields
// used here; x.abort_peers(rank) raises the abort flag of every CTA of the
// cluster). TAPE (the backward pass's forward): rank 0 also writes ||u_t||^2
// and ||k_t||^2 into each token's tape record, rank 1 den_t (negative where
// the eps floor is taken) and z^key before every 64th token.
// ---------------------------------------------------------------------------
template <int D, typename TIn, bool RANK0, typename X, bool TAPE = false>
__device__ __forceinline__ void stage2(const Params& p, const X& x, int bh, int sw, int lane, uint32_t rank,
                                       bool write_zk = true) {
    using L = typename X::L;
    constexpr int E = D / 32, TW = C / NSTAGE;
    const int T = p.T, nch = (T + C - 1) / C;
    const TIn* g0 = static_cast<const TIn*>(RANK0 ? p.u : p.q) + (size_t)bh * T * D;
    const TIn* gk = static_cast<const TIn*>(p.k) + (size_t)bh * T * D;
    const TIn* gv = static_cast<const TIn*>(p.v) + (size_t)bh * T * D;
    float zk[E];  // z^key before the chunk (rank 1; identical in every staging warp)
#pragma unroll
    for (int m = 0; m < E; ++m) zk[m] = (!RANK0 && p.zk0) ? p.zk0[(size_t)bh * D + lane + 32 * m] : 0.f;

    auto issue = [&](int c) {
        const int n = min(C, T - c * C);
        const uint32_t bytes = (uint32_t)n * D * sizeof(TIn);
        unsigned char* r = x.raw(c % L::NRAW);
        mbar_arrive_expect_tx(x.b.full_r + c % L::NRAW, 2 * bytes);
        bulk_g2s(r, g0 + (size_t)c * C * D, bytes, x.b.full_r + c % L::NRAW);
        bulk_g2s(r + L::RAW_T, gk + (size_t)c * C * D, bytes, x.b.full_r + c % L::NRAW);
    };
    // test hook: publish nothing, so that every consumer's bounded wait runs out
    if (p.stall_producer) return;
    const bool leader = sw == 0 && lane == 0;
    int issued = min(L::NRAW, nch), c = 0;
    if (leader)
        for (int cc = 0; cc < issued; ++cc) issue(cc);
    float* scr = x.f(L::OFF_SCR);
    float* zpart = x.f(L::OFF_ZP);
    bool bad = false;
    for (c = 0; c < nch; ++c) {
        const int s = c % L::NP, rs = c % L::NRAW, n = min(C, T - c * C);
        bool ok = c < L::NP || mbar_wait(x.b.empty_p + s, ((c / L::NP) & 1) ^ 1, x.abort, p.wait_ns);
        ok = ok && mbar_wait(x.b.full_r + rs, (c / L::NRAW) & 1, x.abort, p.wait_ns);
        if (bar_red_or(ID_ST, 32 * NSTAGE, !ok || *x.abort != 0)) {
            bad = true;
            break;
        }
        // rank 1's S rows read this chunk's v from global memory a few chunks from now
        if constexpr (!RANK0) tc::prefetch_v_l2<D, TIn>(gv + (size_t)c * C * D, n, sw * 32 + lane);
        if constexpr (TAPE && !RANK0) {
            if ((c & 3) == 0 && sw == 0) {  // z^key before token 16 c (= 64 (c / 4))
                float* ck = tc::ckpt_slot<D>(p, bh, c >> 2) + 2 * D * D;
#pragma unroll
                for (int m = 0; m < E; ++m) ck[lane + 32 * m] = zk[m];
            }
        }
        const TIn* r0 = reinterpret_cast<const TIn*>(x.raw(rs));
        const TIn* rk = reinterpret_cast<const TIn*>(x.raw(rs) + L::RAW_T);
        float fq[TW][E], pk[TW][E], red[TW][3];
        float zsum[E];
#pragma unroll
        for (int m = 0; m < E; ++m) zsum[m] = 0.f;
#pragma unroll
        for (int j = 0; j < TW; ++j) {
            const int t = sw * TW + j;
            red[j][0] = red[j][1] = red[j][2] = 0.f;
#pragma unroll
            for (int m = 0; m < E; ++m) {
                const int e = lane + 32 * m;
                float xv = 0.f, kv = 0.f;
                if (t < n) {
                    xv = ld_in<TIn>(r0 + (size_t)t * D, e);
                    kv = ld_in<TIn>(rk + (size_t)t * D, e);
                }
                red[j][1] = fmaf(kv, kv, red[j][1]);
                if constexpr (RANK0) {
                    red[j][0] = fmaf(xv, xv, red[j][0]);
                    scr[(0 * C + t) * L::SCR_STRIDE + e] = xv;  // u
                    scr[(1 * C + t) * L::SCR_STRIDE + e] = kv;  // k
                } else {
                    fq[j][m] = t < n ? tc::phi_bf(xv) : 0.f;
                    zsum[m] += t < n ? tc::phi_bf(kv) : 0.f;
                    pk[j][m] = zsum[m];  // this warp's phi(k) prefix, inclusive
                    scr[(0 * C + t) * L::SCR_STRIDE + e] = kv;        // k
                    scr[(1 * C + t) * L::SCR_STRIDE + e] = fq[j][m];  // phi(q)
                }
            }
        }
        if constexpr (!RANK0) {
#pragma unroll
            for (int m = 0; m < E; ++m) zpart[sw * D + lane + 32 * m] = zsum[m];
            named_bar(ID_ST, 32 * NSTAGE);
            // z^key before this warp's tokens, and before the next chunk
#pragma unroll
            for (int m = 0; m < E; ++m) {
                float pre = zk[m], all = zk[m];
#pragma unroll
                for (int w = 0; w < NSTAGE; ++w) {
                    const float zp = zpart[w * D + lane + 32 * m];
                    if (w < sw) pre += zp;
                    all += zp;
                }
#pragma unroll
                for (int j = 0; j < TW; ++j) red[j][2] = fmaf(fq[j][m], pre + pk[j][m], red[j][2]);
                zk[m] = all;
            }
        }
        allreduce<3 * TW, 16>(&red[0][0]);
        float* sc = x.sc(s);
        if (lane < TW) {
            float r0v = red[0][0], r1v = red[0][1], r2v = red[0][2];
#pragma unroll
            for (int j = 1; j < TW; ++j)
                if (lane == j) {
                    r0v = red[j][0];
                    r1v = red[j][1];
                    r2v = red[j][2];
                }
            const int t = sw * TW + lane;
            sc[L::SC_IK + t] = t < n ? rsqrtf(fmaxf(r1v, 1e-24f)) : 0.f;
            if constexpr (RANK0)
                sc[L::SC_IU + t] = t < n ? rsqrtf(fmaxf(r0v, 1e-24f)) : 0.f;
            else
                sc[L::SC_RDEN + t] = t < n ? __frcp_rn(fmaxf(r2v, p.eps)) : 1.f;  // 1 / den
            if constexpr (TAPE) {
                if (t < n) {
                    float* rec = tc::tape_rec<D>(p, bh, c * C + t) + 3 * D;
                    if constexpr (RANK0) {
                        rec[3] = r0v;  // ||u_t||^2
                        rec[4] = r1v;  // ||k_t||^2
                    } else {
                        rec[2] = r2v < p.eps ? -p.eps : r2v;  // den, negative where the eps floor is taken
                    }
                }
            }
        }
        named_bar(ID_ST, 32 * NSTAGE);
        // scratch rows -> operand tiles, one 8-row group per unit: lane =
        // (row, 16-byte chunk). Units 0..3: HI rows (row type unit / 2, half
        // unit % 2); then LO rows: fp32 both row types, bf16 rank 1 phi only.
        {
            float* hi = x.hi(s);
            float* lo = x.lo(s);
            const int r8 = lane & 7;
            constexpr int NLO = L::F32IN ? 4 : (RANK0 ? 0 : 2);
            for (int unit = sw; unit < 4 + NLO; unit += NSTAGE) {
                int y, row0;
                float* dst;
                bool lopart;
                const int half = unit & 1;
                if (unit < 4) {
                    y = unit >> 1;
                    row0 = y * C + half * 8;
                    dst = hi;
                    lopart = false;
                } else {
                    const int lu = unit - 4;
                    y = L::F32IN ? (lu >> 1) : 1;  // bf16: the phi rows only
                    row0 = (L::F32IN ? y * C : 0) + half * 8;
                    dst = lo;
                    lopart = true;
                }
                for (int g = lane >> 3; g < D / 4; g += 4) {
                    float4 v = ld4(scr + (y * C + half * 8 + r8) * L::SCR_STRIDE + 4 * g);
                    if (lopart) v = make_float4(tf32_lo(v.x), tf32_lo(v.y), tf32_lo(v.z), tf32_lo(v.w));
                    *reinterpret_cast<float4*>(dst + cm_off(row0 + r8, 4 * g, D)) = v;
                }
            }
        }
        // the tiles are read by the tensor cores (async proxy); our generic
        // reads of the raw slot are done before its refill by the TMA
        fence_proxy_async_smem();
        named_bar(ID_ST, 32 * NSTAGE);
        if (leader) {
            mbar_arrive(x.b.full_p + s);
            if (c + L::NRAW < nch) issue(c + L::NRAW);
        }
        if (c + L::NRAW < nch) issued = c + L::NRAW + 1;
    }
    if (bad) {
        if (leader) {
            record_failure(p.status, BIT_TIMEOUT, ROLE_STAGE, bh, c * C);
            x.abort_peers(rank);
            // let copies already in flight land before the CTA can exit
            for (int cc = c; cc < issued; ++cc)
                    (void)mbar_wait(x.b.full_r + cc % L::NRAW, (cc / L::NRAW) & 1, nullptr, p.wait_ns);
        }
        return;
    }
    if (!RANK0 && write_zk && p.zk_out && sw == 0) {
#pragma unroll
        for (int m = 0; m < E; ++m) p.zk_out[(size_t)bh * D + lane + 32 * m] = zk[m];
    }
}

// ---------------------------------------------------------------------------
// rank 0, warps 0-4: Sherman-Morrison steps of eq. 9 and the gate of eq. 10,
// one chunk at a time (the arithmetic of tc::tc_a_team). Thread i < D of
// warps 0-3 owns row i of A (TMEM lane i) and of every d x C intermediate;
// warp 4 factors I + Guu and sends the gate to rank 1. TAPE: also z_t,
// delta_t and ||a_t|| into the tape, and A before every 64th token.
// ---------------------------------------------------------------------------
template <int D, typename TIn, bool TAPE = false>
__device__ void a_rank(const Params& p, const Ctx2<D, TIn>& x, int bh, int warp, int lane, uint32_t rank) {
    using L = Lay2<D, TIn>;
    constexpr int XS = L::XS;
    const int ta = threadIdx.x;
    const bool rw = warp < L::NRW;
    const int i = ta;
    const uint32_t tm = __shfl_sync(0xffffffffu, *x.tmem_base, 0);
    const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    const int T = p.T, nch = (T + C - 1) / C;
    float* sm = x.sm();
    float* xr = x.f(L::OFF_XR);
    float* ph = x.f(L::OFF_PH);
    float* pl = x.f(L::OFF_PL);
    float* zh = x.f(L::OFF_ZH);
    float* zl = x.f(L::OFF_ZL);
    bool bad = false, nonfinite = false;
    const bool fixed = p.fixed_a != 0;
    // the peer's mailbox and barriers
    const uint32_t r_full_al = peer_addr(x.b.full_al, 1u);
    const uint32_t r_al = peer_addr(x.f(L::OFF_AL), 1u);
    int sent = 0;

    // A_0 = I / lambda0 unless carried in (eq. 9), and its lo part
    if (rw) {
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
    for (int e = ta; e < (128 - D) * C; e += NT_A) {
        ph[cm_off(D + e / C, e % C, C)] = 0.f;
        pl[cm_off(D + e / C, e % C, C)] = 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(ID_T, NT_A);

    uint32_t pa = 0;
    int c = 0;
    for (; c < nch; ++c) {
        const int s = c % L::NP, n = min(C, T - c * C), b = c & 1;
        bad = !mbar_wait(x.b.full_p + s, (c / L::NP) & 1, x.abort, p.wait_ns);
        if (bar_red_or(ID_T, NT_A, bad || *x.abort != 0)) {
            bad = true;
            break;
        }
        TC2_STAMP(p, 4, 0, c, nch);
        if (TAPE && (c & 3) == 0 && rw) {  // A before token 16 c
            tc_fence_after();
            tc::tmem_row_out<D>(tl, L::T_X, tc::ckpt_slot<D>(p, bh, c >> 2) + D * D + (size_t)i * D);
        }
        const float* hi = x.hi(s);
        const float* sc = x.sc(s);
        // [Z' | W] = A_c [u | k]^T (rows u, k of the chunk; scaled by 1/||.|| below);
        // warp q < NISS issues the K steps ks = q mod NISS into accumulator q
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
        TC2_STAMP(p, 4, 1, c, nch);
        tc_fence_after();
        if (rw) {
            float v0[16], v1[16];
            ld_products(tl + L::T_P, v0, v1);
#pragma unroll
            for (int t = 0; t < C; ++t) {
                v0[t] *= sc[L::SC_IU + t];  // z'_t = A_c u^_t
                v1[t] *= sc[L::SC_IK + t];  // w_t = A_c k^_t
                xr[t * XS + i] = v0[t];
                xr[(C + t) * XS + i] = v1[t];
            }
        }
        named_bar(ID_T, NT_A);
        TC2_STAMP(p, 4, 2, c, nch);
        if (!fixed) {
            // Guu[s][t] = u^_s . z'_t, Guk[s][t] = u^_s . w_t; warps 0-3 = (matrix, half of D)
            if (warp < 4) {
                const int mat = warp & 1, half = warp >> 1;
                float acc[2][4];
                tc::gram16<D, true>(hi, 0, xr + mat * C * XS, XS, half * (D / 2), (half + 1) * (D / 2), lane, acc,
                                    !L::F32IN);
                tc::gram_pair_sum(sm + (mat ? L::SM_GUK : L::SM_GUU), L::MS, L::GSTR, acc, lane, half, 4 + mat,
                                  sc + L::SC_IU, false);
            }
            named_bar(ID_T, NT_A);
        }
        TC2_STAMP(p, 4, 3, c, nch);
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
                if (TAPE && j < n) tc::tape_rec<D>(p, bh, c * C + j)[3 * D] = mydl;  // delta_t = 1 + u^_t . z_t
            } else {
#pragma unroll
                for (int r = 0; r < C; ++r) sm[L::SM_XGT + j * L::GSTR + r] = col[r];
            }
        } else if (c >= 2) {
            // rank 1 is done with mailbox buffer b (chunk c - 2), so its local
            // source can be rewritten
            ok = ok && mbar_wait_cl(x.b.empty_al + b, ((c >> 1) & 1) ^ 1, x.abort, p.wait_ns);
        }
        if (bar_red_or(ID_T, NT_A, !ok || *x.abort != 0)) {
            bad = true;
            break;
        }
        TC2_STAMP(p, 4, 4, c, nch);
        float* alr = x.f(L::OFF_AL) + (size_t)b * C * XS;
        float* gh = x.f(L::OFF_GH) + (size_t)b * D * C;
        float* gl = x.f(L::OFF_GL) + (size_t)b * D * C;
        float* laa = x.f(L::OFF_LAA) + (size_t)b * C;
        // the update's operands first: the state update is issued before the gate
        float y[C], lr[C];
        if (rw && !fixed) {
            // y = z_i = z'_i L^-T (forward substitution, in place), then y D^-1
#pragma unroll
            for (int t = 0; t < C; ++t) y[t] = xr[t * XS + i];
#pragma unroll
            for (int r = 0; r < C - 1; ++r) {
                tc::ld_row16(sm + L::SM_LMT + r * L::GSTR, lr);  // L[t][r], t > r
#pragma unroll
                for (int t = r + 1; t < C; ++t) y[t] = fmaf(-lr[t], y[r], y[t]);
            }
            if (TAPE) {  // z_t = A_{t-1} u^_t of eq. 9
#pragma unroll
                for (int t = 0; t < C; ++t)
                    if (t < n) tc::tape_rec<D>(p, bh, c * C + t)[i] = y[t];
            }
            // row i of N = Z D^-1/2: A_{c+1} = A_c - N N^T (symmetric by construction)
            float nv[C];
            tc::ld_row16(sm + L::SM_RS, lr);
#pragma unroll
            for (int t = 0; t < C; ++t) nv[t] = y[t] * lr[t];
            tc::ld_row16(sm + L::SM_RD, lr);
#pragma unroll
            for (int t = 0; t < C; ++t) y[t] *= lr[t];
            tc::put_row16(zh, i, nv, false);
            tc::put_row16(zl, i, nv, true);
#pragma unroll
            for (int t = 0; t < C; ++t) nv[t] = -nv[t];
            tc::put_row16(ph, i, nv, false);
            tc::put_row16(pl, i, nv, true);
        }
        fence_proxy_async_smem();
        named_bar(ID_T, NT_A);
        TC2_STAMP(p, 4, 5, c, nch);
        // A_{c+1} = A_c - N N^T
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
        if (rw) {
            // a_t = A_t k^_t = w_t - sum_{s<=t} z_s (z_s . k^_t) / delta_s (eq. 10)
            float av[C];
#pragma unroll
            for (int t = 0; t < C; ++t) {
                float a = xr[(C + t) * XS + i];
                if (!fixed) {
                    tc::ld_row16(sm + L::SM_XGT + t * L::GSTR, lr);  // X[q][t]
#pragma unroll
                    for (int q = 0; q <= t; ++q) a = fmaf(-y[q], lr[q], a);
                }
                av[t] = t < n ? a : 0.f;
                alr[t * XS + i] = av[t];
            }
            tc::put_row16(gh, i, av, false);
            tc::put_row16(gl, i, av, true);
        }
        fence_proxy_async_smem();
        named_bar(ID_T, NT_A);
        TC2_STAMP(p, 4, 6, c, nch);
        if (warp == FACTOR_WARP) {
            // ||a_t||^2 for rank 1, then the chunk's gate into rank 1's mailbox
            if (lane < C) {
                float2 acc = f2(0.f, 0.f);
#pragma unroll 8
                for (int k4 = 0; k4 < D / 4; ++k4) {
                    const float4 a = ld4(alr + lane * XS + 4 * k4);
                    acc = __ffma2_rn(f2(a.x, a.y), f2(a.x, a.y), acc);
                    acc = __ffma2_rn(f2(a.z, a.w), f2(a.z, a.w), acc);
                }
                laa[lane] = acc.x + acc.y;
                if (TAPE && lane < n) tc::tape_rec<D>(p, bh, c * C + lane)[3 * D + 1] = sqrtf(acc.x + acc.y);  // ||a_t||
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const uint32_t rbar = r_full_al + 8u * b;
                mbar_expect_tx_peer(rbar, L::MB_BYTES);
                bulk_to_peer(r_al + (uint32_t)(b * L::MB_ALR), alr, L::MB_ALR, rbar);
                bulk_to_peer(r_al + (uint32_t)(L::OFF_GH - L::OFF_AL) + b * L::MB_G, gh, L::MB_G, rbar);
                bulk_to_peer(r_al + (uint32_t)(L::OFF_GL - L::OFF_AL) + b * L::MB_G, gl, L::MB_G, rbar);
                bulk_to_peer(r_al + (uint32_t)(L::OFF_LAA - L::OFF_AL) + b * L::MB_LAA, laa, L::MB_LAA, rbar);
                ++sent;
            }
        }
        if (!fixed) {
            bad = !mbar_wait(x.b.mma_x, pa, nullptr, p.wait_ns);
            pa ^= 1;
        }
        TC2_STAMP(p, 4, 7, c, nch);
        tc_fence_after();
        if (rw && !fixed) tc::refresh_lo<D>(tl, L::T_X, L::T_XL);
        tc_fence_before();
        if (bar_red_or(ID_T, NT_A, bad)) {
            bad = true;
            ++c;
            break;
        }
        TC2_STAMP(p, 4, 8, c, nch);
    }
    if (warp == FACTOR_WARP && lane == 0) {
        *x.n_sent = sent;
        st_peer_u32(peer_addr(x.n_sent, 1u), (uint32_t)sent);
    }
    if (bad) {
        if (ta == 0) {
            record_failure(p.status, BIT_TIMEOUT, ROLE_A, bh, c * C);
            x.abort_peers(rank);
        }
    } else if (rw) {
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
// rank 1, warps 0-3: residual writes and readout of eq. 10-11 for the chunk
// rank 0 sent (the arithmetic of tc::tc_s_team). Thread i < D owns row i of S.
// TAPE: also alpha^_t and e_t into the tape, and S before every 64th token.
// ---------------------------------------------------------------------------
template <int D, typename TIn, bool TAPE = false>
__device__ void s_rank(const Params& p, const Ctx2<D, TIn>& x, int bh, int warp, int lane, uint32_t rank) {
    using L = Lay2<D, TIn>;
    constexpr int XS = L::XS;
    const int ts = threadIdx.x;
    const bool rw = warp < L::NRW;
    const int i = ts;
    const uint32_t tm = __shfl_sync(0xffffffffu, *x.tmem_base, 0);
    const uint32_t tl = tm + ((uint32_t)(32 * warp) << 16);
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

    // S_0 = 0 unless carried in, and its lo part
    if (rw) {
        const float* S0 = p.S0 ? p.S0 + ((size_t)bh * D + i) * D : nullptr;
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
    for (int e = ts; e < (128 - D) * C; e += NT_S) {
        eh[cm_off(D + e / C, e % C, C)] = 0.f;
        el[cm_off(D + e / C, e % C, C)] = 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(ID_T, NT_S);

    uint32_t ps = 0;
    int c = 0;
    for (; c < nch; ++c) {
        const int s = c % L::NP, n = min(C, T - c * C), b = c & 1;
        float vv[C];
        typename tc::RawIn<TIn>::type vr[C];
        if (rw) tc::load_v_raw<D, TIn>(gv + (size_t)c * C * D, i, n, vr);
        TC2_STAMP(p, 5, 0, c, nch);
        bad = !mbar_wait(x.b.full_p + s, (c / L::NP) & 1, x.abort, p.wait_ns) ||
              !mbar_wait_cl(x.b.full_al + b, (c >> 1) & 1, x.abort, p.wait_ns);
        if (bar_red_or(ID_T, NT_S, bad || *x.abort != 0)) {
            bad = true;
            break;
        }
        TC2_STAMP(p, 5, 1, c, nch);
        recv = c + 1;
        if (TAPE && (c & 3) == 0 && rw) {  // S before token 16 c
            tc_fence_after();
            tc::tmem_row_out<D>(tl, L::T_X, tc::ckpt_slot<D>(p, bh, c >> 2) + (size_t)i * D);
        }
        const float* hi = x.hi(s);
        const float* sc = x.sc(s);
        const float* alr = x.f(L::OFF_AL) + (size_t)b * C * XS;
        // [S_c k | S_c phi] (rows k, phi of the chunk); warp q < NISS issues the
        // K steps ks = q mod NISS into accumulator q
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
        bool ok = mbar_wait(x.b.mma_p, c & 1, nullptr, p.wait_ns);
        TC2_STAMP(p, 5, 2, c, nch);
        tc_fence_after();
        float sk[C], sq[C];
        if (rw) {
            ld_products(tl + L::T_P, sk, sq);
#pragma unroll
            for (int t = 0; t < C; ++t) sk[t] *= sc[L::SC_IK + t];  // S_c k^_t; sq = S_c phi_t
        }
        TC2_STAMP(p, 5, 3, c, nch);
        // Lk[t][s] = k^_t . a_s, Lq[t][s] = phi_t . a_s; warp = (matrix, half of D)
        {
            const int mat = warp & 1, half = warp >> 1;
            float acc[2][4];
            tc::gram16<D, true>(hi + (mat ? C : 0) * D, 0, alr, XS, half * (D / 2), (half + 1) * (D / 2), lane, acc,
                                !L::F32IN && mat == 0);
            if (mat)
                tc::gram_pair_sum(sm + L::SM_LQ, L::MS, L::GSTR, acc, lane, half, 4 + mat, nullptr, false);
            else
                tc::gram_pair_sum(sm + L::SM_LKT, L::MS, L::GSTR, acc, lane, half, 4 + mat, sc + L::SC_IK, true);
        }
        named_bar(ID_T, NT_S);
        TC2_STAMP(p, 5, 4, c, nch);
        if (rw) {
            float lr[C], nr[C];
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
            TC2_STAMP(p, 5, 5, c, nch);
            if (TAPE) {  // alpha^_t = a_t / ||a_t|| and e_t = e'_t ||a_t|| (eq. 10)
#pragma unroll
                for (int t = 0; t < C; ++t)
                    if (t < n) {
                        float* rec = tc::tape_rec<D>(p, bh, c * C + t);
                        rec[D + i] = alr[t * XS + i] * nr[t];
                        rec[2 * D + i] = vv[t] / nr[t];
                    }
            }
            // o_t = (S_c phi_t + sum_{s<=t} e_s (alpha^_s . phi_t)) / den_t = S_t phi_t / den_t (eq. 11)
            tc::ld_row16(sc + L::SC_RDEN, nr);
#pragma unroll
            for (int t = 0; t < C; ++t) {
                tc::ld_row16(sm + L::SM_LQ + t * L::GSTR, lr);
                float a = sq[t];
#pragma unroll
                for (int q = 0; q <= t; ++q) a = fmaf(lr[q], vv[q], a);
                const float ov = a * nr[t];
                if (t < n) {
                    go[(size_t)(c * C + t) * D + i] = ov;
                    nfchk = fmaf(ov, 0.f, nfchk);  // stays 0 unless an o is NaN or Inf
                }
            }
            tc::put_row16(eh, i, vv, false);
            tc::put_row16(el, i, vv, true);
        }
        fence_proxy_async_smem();
        named_bar(ID_T, NT_S);
        TC2_STAMP(p, 5, 6, c, nch);
        // S_{c+1} = S_c + E' A (rows a_t from the mailbox, columns scaled into E')
        if (warp == 0 && tc::elect_one()) {
            mbar_arrive(x.b.empty_p + s);  // done with the chunk's k, phi rows and den
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
        ok = mbar_wait(x.b.mma_x, ps, nullptr, p.wait_ns) && ok;
        TC2_STAMP(p, 5, 7, c, nch);
        ps ^= 1;
        tc_fence_after();
        if (ts == 0) mbar_arrive_peer(r_empty_al + 8u * b);  // mailbox buffer b back to rank 0
        if (rw) tc::refresh_lo<D>(tl, L::T_X, L::T_XL);
        tc_fence_before();
        if (bar_red_or(ID_T, NT_S, !ok)) {
            bad = true;
            ++c;
            break;
        }
        TC2_STAMP(p, 5, 8, c, nch);
    }
    if (ts == 0) *x.n_recv = recv;
    if (bad) {
        if (ts == 0) {
            record_failure(p.status, BIT_TIMEOUT, ROLE_S, bh, c * C);
            x.abort_peers(rank);
        }
    } else if (rw) {
        float* So = p.S_out + ((size_t)bh * D + i) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
            tc_ld16(tl + L::T_X + c0, v);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(So + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    if (nonfinite || nfchk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_S, bh, -1);
}

}  // namespace tc2

// TAPE: the backward pass's forward, which also writes the tape and the
// 64-token checkpoints that the reverse sweep reads (as vla_tc_kernel does)
template <int D, typename TIn, bool TAPE = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(tc2::THREADS, 1) vla_tc2_kernel(const Params p) {
    using L = tc2::Lay2<D, TIn>;
    extern __shared__ __align__(1024) unsigned char smem[];
    tc2::Ctx2<D, TIn> x;
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
    const uint32_t rank = tc2::cluster_rank();
    const int bh = blockIdx.x >> 1;
    if (threadIdx.x == 0) {
        for (int r = 0; r < L::NRAW; ++r) mbar_init(x.b.full_r + r, 1);
        for (int s = 0; s < L::NP; ++s) {
            mbar_init(x.b.full_p + s, 1);
            mbar_init(x.b.empty_p + s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(x.b.full_al + s, 1);
            mbar_init(x.b.empty_al + s, 1);
        }
        mbar_init(x.b.mma_x, 1);
        mbar_init(x.b.mma_p, tc2::NISS);
        *x.abort = 0;
        *x.n_sent = 0;
        *x.n_recv = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc_alloc(x.tmem_base, L::TCOLS);
    tc_fence_before();
    // the peer's barriers are initialised before either rank arrives on them
    tc2::cluster_sync_all();
    tc_fence_after();
    if (warp < 8) {
        if (rank == 0 && warp <= tc2::FACTOR_WARP)
            tc2::a_rank<D, TIn, TAPE>(p, x, bh, warp, lane, rank);
        else if (rank == 1 && warp < 4)
            tc2::s_rank<D, TIn, TAPE>(p, x, bh, warp, lane, rank);
    } else if (rank == 0) {
        tc2::stage2<D, TIn, true, tc2::Ctx2<D, TIn>, TAPE>(p, x, bh, warp - 8, lane, rank);
    } else {
        tc2::stage2<D, TIn, false, tc2::Ctx2<D, TIn>, TAPE>(p, x, bh, warp - 8, lane, rank);
    }
    tc_fence_before();
    __syncthreads();
    // rank 0 has sent its last mailbox buffer and written the count into rank 1
    tc2::cluster_sync_all();
    if (rank == 1 && threadIdx.x == 0) {
        // after a failure: let the buffers that rank 0 sent but this rank did
        // not consume land before the CTA can exit
        for (int j = *x.n_recv; j < *x.n_sent; ++j)
            (void)tc2::mbar_wait_cl(x.b.full_al + (j & 1), (j >> 1) & 1, nullptr, p.wait_ns);
    }
    tc2::cluster_sync_all();
    tc_fence_after();
    if (warp == 0) tc_dealloc(*x.tmem_base, L::TCOLS);
}
