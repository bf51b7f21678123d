// vla_tc.cuh -- chunked VLA forward on the 5th-generation tensor cores
// (tcgen05, TMEM) of sm_103a. Included by vla_forward.cu inside namespace vla.
//
// "Variational Linear Attention" (arXiv 2605.11196), §3.3 eq. 9-11, computed
// C = 16 tokens at a time. For a chunk with starting state A_c, S_c and raw
// rows u_s, k_t (unit vectors u^ = u / ||u||, k^ = k / ||k||):
//
//   A-pass   Z' = A_c U^T, W = A_c K^T              (tensor cores, d x d x 2C)
//            Guu = U^ Z', Guk = U^ W                 (C x C Gram matrices)
//            I + Guu = L D L^T (eliminated together with Guk: X = L^-1 Guk)
//            per row i:  z_i = Z'_i L^-T  (the Sherman-Morrison vectors of
//            eq. 9 for the chunk's tokens), n_i = z_i D^-1/2,
//            a_t[i] = w_t[i] - sum_{s<=t} z_s[i] X[s][t] / delta_s
//            (a_t = A_t k^_t, the unnormalised gate of eq. 10)
//            A_{c+1} = A_c - N N^T                   (tensor cores, rank C)
//            (Woodbury: Z' (L D L^T)^-1 Z'^T = N N^T, so the update is
//            symmetric by construction and A keeps no antisymmetric rounding
//            error, which the downdates would not damp while A shrinks)
//   S-pass   S_c K^T, S_c Phi^T                      (tensor cores)
//            Lk[t][s] = k^_t . a_s, Lq[t][s] = phi_t . a_s, ||a_s||^2
//            per row i: e_t = v_t - S_c k^_t - sum_{s<t} (k^_t . alpha^_s) e_s,
//            o_t = (S_c phi_t + sum_{s<=t} (phi_t . alpha^_s) e_s) / den_t
//            S_{c+1} = S_c + E Alpha                 (tensor cores, rank C)
//
// The sequential recurrence of eq. 9-11 and this chunk form are the same
// arithmetic up to rounding order: the Sherman-Morrison steps of a chunk are
// the LDL^T factorisation of I + U^ A_c U^^T, and the residual writes of eq. 10
// are a unit lower-triangular solve.
//
// Tensor-core products run in tf32 with the 3-term split x = hi(x) + lo(x)
// (hi*hi + hi*lo + lo*hi), which keeps them at fp32 accuracy. A, S and their
// lo parts live in TMEM for the whole sequence (lane = row); the chunk's
// vectors are MMA operands in shared memory.
//
// Warps: 0-3 A team (row warps own TMEM lane quarters, warp 3 also factors
// I + Guu), 4-7 S team (row warps; 6-7 form the gate), 8-11 staging (TMA bulk
// copies of q, k, u; phi, norms, z^key, den, operand tiles). The A team runs up
// to two chunks ahead of the S team's gate. All waits are bounded.

namespace tc {

constexpr int C = 16;           // tokens per chunk
constexpr int NSTAGE = 4;        // staging warps
constexpr int THREADS = 32 * (8 + NSTAGE);
constexpr int ID_A = 1, ID_S = 2, ID_ST = 3;  // named barriers of the A team, S team, staging warps
constexpr int ID_M = 9;  // A-team rows (arrive) -> warp 3 (sync): -N, N of a chunk are in place
constexpr int ID_G = 8;  // S-team warps 6 and 7: the chunk's gate rows are in place

// true on one lane of a converged warp (elect.sync). Issuing tcgen05 work
// from a warp-uniform branch through it, with operands the compiler can prove
// warp-uniform (warp index and TMEM base broadcast from lane 0), keeps them
// out of a per-lane path.
__device__ __forceinline__ bool elect_one() {
    uint32_t e;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
    return e != 0;
}

template <int D, typename TIn>
struct Lay {
    static constexpr bool F32IN = sizeof(TIn) == 4;
    static constexpr int NRW = D / 32;          // row warps per team
    // prepared and raw chunk slots: three and two, so that the staging warps
    // run up to two chunks ahead of the A team; fp32 inputs at d = 96 leave
    // room for only two and one
    static constexpr int NP = (F32IN && D > 64) ? 2 : 3;
    static constexpr int NRAW = (F32IN && D > 64) ? 1 : 2;
    // prepared chunk: HI tile rows u (0..C-1) | k (C..2C-1) | phi (2C..3C-1)
    // (raw values; bf16 u, k are exact in tf32), LO tile rows = lo parts that
    // are nonzero: phi_lo only for bf16 inputs, u_lo | k_lo | phi_lo for fp32
    static constexpr int HI_ROWS = 3 * C;
    static constexpr int LO_ROWS = F32IN ? 3 * C : C;
    static constexpr int SBO_D = (D / 4) * 128;   // bytes between 8-row groups, rows of D
    static constexpr int SBO_C = (C / 4) * 128;   // rows of C
    static constexpr int SC_IU = 0, SC_IK = C, SC_RDEN = 2 * C;  // per-token scalars: 1/||u||, 1/||k||, 1/den
    static constexpr int SLOT = (HI_ROWS + LO_ROWS) * D + 64;   // floats
    static constexpr int SCR_STRIDE = D + 4;
    static constexpr int GSTR = C + 4;            // row stride of the small C x C matrices (16-byte rows)
    static constexpr int XS = D + 4;              // row stride of the row-major d-vectors (z' | w, a)

    // TMEM columns
    // (the chunk products [A u | A k] and [S k | S phi] accumulate their even
    // and odd K steps in two column blocks each, summed when read)
    static constexpr uint32_t T_A = 0, T_AL = D, T_S = 2 * D, T_SL = 3 * D, T_XA = 4 * D, T_XS = 4 * D + 2 * C,
                              T_XA2 = 4 * D + 4 * C, T_XS2 = 4 * D + 6 * C;
    static constexpr uint32_t TCOLS = (4 * D + 8 * C) <= 256 ? 256 : 512;
    static_assert(4 * D + 8 * C <= 512, "TMEM columns");

    // shared memory map (bytes)
    static constexpr size_t al(size_t x) { return (x + 127) / 128 * 128; }
    static constexpr int NBAR = NRAW + 2 * NP + 4 + 4;
    static constexpr size_t OFF_BAR = 0;
    static constexpr size_t OFF_MISC = al(8 * NBAR);             // abort flag, TMEM base
    static constexpr size_t OFF_PREP = al(OFF_MISC + 16);
    static constexpr size_t OFF_RAW = al(OFF_PREP + (size_t)NP * SLOT * 4);
    static constexpr size_t RAW_T = (size_t)C * D * sizeof(TIn);  // one tensor of a raw chunk
    static constexpr size_t OFF_SCR = al(OFF_RAW + (size_t)NRAW * 3 * RAW_T);
    static constexpr size_t OFF_ZP = al(OFF_SCR + (size_t)3 * C * SCR_STRIDE * 4);   // staging phi(k) sums
    static constexpr size_t OFF_XR = al(OFF_ZP + (size_t)NSTAGE * D * 4);
    static constexpr size_t OFF_PH = al(OFF_XR + (size_t)2 * C * XS * 4);  // -N hi/lo, 128 x C
    static constexpr size_t OFF_PL = OFF_PH + 128 * C * 4;
    static constexpr size_t OFF_ZH = OFF_PL + 128 * C * 4;                  // N hi/lo, D x C
    static constexpr size_t OFF_ZL = OFF_ZH + (size_t)D * C * 4;
    static constexpr size_t OFF_EH = OFF_ZL + (size_t)D * C * 4;            // E hi/lo, 128 x C
    static constexpr size_t OFF_EL = OFF_EH + 128 * C * 4;
    // the gate of a chunk, formed by the S team: a rows [C x XS], a^T hi/lo [D x C]
    static constexpr size_t OFF_AL = OFF_EL + 128 * C * 4;
    static constexpr size_t OFF_GH = OFF_AL + (size_t)C * XS * 4;
    static constexpr size_t OFF_GL = OFF_GH + (size_t)D * C * 4;
    // what the A team hands the S team for a chunk's gate, two buffers each:
    // w rows [C x D], y rows (z / delta) [C x D], X [C x GSTR]
    static constexpr size_t OFF_WP = OFF_GL + (size_t)D * C * 4;
    static constexpr size_t OFF_YP = OFF_WP + (size_t)2 * C * D * 4;
    static constexpr size_t OFF_XP = OFF_YP + (size_t)2 * C * D * 4;
    static constexpr size_t OFF_SM = OFF_XP + (size_t)2 * C * GSTR * 4;    // small matrices
    // small matrices: Guu, Guk (two partial sums each, over the halves of
    // D), 1/sqrt(delta) (one row), L^T, Lk^T, Lq (two partials each),
    // 1/delta, ||a||^2
    static constexpr int MS = C * GSTR;
    static constexpr int SM_GUU = 0, SM_GUK = 2 * MS, SM_RS = 4 * MS, SM_LMT = 5 * MS, SM_LKT = 6 * MS,
                         SM_LQ = 8 * MS, SM_RD = 10 * MS, SM_LAA = SM_RD + C;
    static constexpr size_t SMEM = al(OFF_SM + (size_t)(10 * MS + 2 * C) * 4);
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(RAW_T % 16 == 0 && (D * sizeof(TIn)) % 16 == 0, "bulk-copy granularity");
};

struct Bars {
    uint64_t* full_r;    // [NRAW] raw chunk landed
    uint64_t* full_p;    // [NP] prepared chunk published
    uint64_t* empty_p;   // [NP] released by both teams (count 2)
    uint64_t* full_al;   // [2] A team published w, z / delta and X of a chunk
    uint64_t* empty_al;  // [2] S team has formed the chunk's gate from them
    uint64_t* mma_a;     // A-team tcgen05 commits (state update)
    uint64_t* mma_s;     // S-team tcgen05 commits (state update)
    uint64_t* mma_xa;    // [A u | A k] issued by two A warps (count 2)
    uint64_t* mma_xs;    // [S k | S phi] issued by two S warps (count 2)
};

template <int D, typename TIn>
struct Ctx {
    using L = Lay<D, TIn>;
    unsigned char* base;
    Bars b;
    volatile int* abort;
    uint32_t* tmem_base;
    __device__ float* slot(int s) const { return reinterpret_cast<float*>(base + L::OFF_PREP) + (size_t)s * L::SLOT; }
    __device__ float* hi(int s) const { return slot(s); }
    __device__ float* lo(int s) const { return slot(s) + L::HI_ROWS * D; }
    __device__ float* sc(int s) const { return slot(s) + (L::HI_ROWS + L::LO_ROWS) * D; }
    __device__ unsigned char* raw(int r) const { return base + L::OFF_RAW + (size_t)r * 3 * L::RAW_T; }
    __device__ float* f(size_t off) const { return reinterpret_cast<float*>(base + off); }
    __device__ float* sm() const { return f(L::OFF_SM); }
};

// ---------------------------------------------------------------------------
// staging warps (4): per chunk, TMA bulk copies of the raw q, k, u rows; then
// warp w handles tokens 4w..4w+3: phi(q), phi(k), 1/||u||, 1/||k||, and
// den = max(phi(q) . z^key, eps) with z^key += phi(k) (eq. 11). z^key is a
// running sum over tokens: each warp publishes the sum of its 4 phi(k) rows
// and adds the sums of the warps before it. The raw u, k rows and phi(q)
// pass through a row-major scratch into the K-major operand tiles.
// ---------------------------------------------------------------------------
// The S rows' v loads leave their values unconverted in registers: a bf16 ->
// fp32 conversion (or a select) right after a global load would make the
// thread wait for the load there, at the top of the chunk, instead of where
// the residual first uses it.
template <typename TIn>
struct RawIn;
template <>
struct RawIn<float> {
    using type = float;
};
template <>
struct RawIn<__nv_bfloat16> {
    using type = unsigned short;
};
__device__ __forceinline__ float raw_f32(float x) { return x; }
__device__ __forceinline__ float raw_f32(unsigned short x) { return __uint_as_float((uint32_t)x << 16); }

// rows t < n of column i of a chunk of v (row stride D), unconverted; rows >= n are zero
template <int D, typename TIn>
__device__ __forceinline__ void load_v_raw(const TIn* vrow, int i, int n, typename RawIn<TIn>::type (&vr)[16]) {
    using R = typename RawIn<TIn>::type;
    const R* p = reinterpret_cast<const R*>(vrow) + i;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        vr[t] = R(0);
        if (t < n) vr[t] = p[(size_t)t * D];
    }
}

// prefetch the n rows of a chunk of v into L2 (one 128-byte line per staging
// thread; a chunk of v is at most 16 x 128 x 4 bytes = 64 lines)
template <int D, typename TIn>
__device__ __forceinline__ void prefetch_v_l2(const TIn* vrow, int n, int tid) {
    const int bytes = n * D * (int)sizeof(TIn);
    if (tid * 128 < bytes)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const unsigned char*>(vrow) + tid * 128));
}

__device__ __forceinline__ float phi_bf(float x) {  // ELU + 1, branch-free; NaN stays NaN
    const float e = __expf(x);
    return x > 0.f ? x + 1.f : e;
}

// record of token t of head bh in the backward pass's tape, and the checkpoint
// slot of the state before token 64 k (layouts of vla_backward.cuh)
template <int D>
__device__ __forceinline__ float* tape_rec(const Params& p, int bh, int t) {
    return p.tape + ((size_t)bh * p.T + t) * (size_t)(3 * D + 8);
}
template <int D>
__device__ __forceinline__ float* ckpt_slot(const Params& p, int bh, int k) {
    return p.ckpt + ((size_t)bh * ((p.T + 63) / 64 + 1) + k) * (size_t)(2 * D * D + D);
}
// row i (this thread's TMEM lane) of a d x d state in TMEM columns [col, col + D) to dst[0..D)
template <int D>
__device__ __forceinline__ void tmem_row_out(uint32_t lanebase, uint32_t col, float* dst) {
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 16) {
        float v[16];
        tc_ld16(lanebase + col + c0, v);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    }
}

// TAPE (the backward pass's forward): also write, per token, the record the
// reverse sweep reads (z_t, alpha^_t, e_t, delta_t, ||a_t||, den_t with the
// sign of the eps floor, ||u_t||^2, ||k_t||^2: 3d + 8 floats) to p.tape, and
// the state before every 64th token (S, A, z^key) to p.ckpt.
template <int D, typename TIn, bool TAPE>
__device__ __forceinline__ void tc_stage(const Params& p, const Ctx<D, TIn>& x, int bh, int sw, int lane) {
    using L = Lay<D, TIn>;
    constexpr int E = D / 32, TW = C / NSTAGE;
    const int T = p.T, nch = (T + C - 1) / C;
    const size_t hs = p.in_stride ? p.in_stride : (size_t)T * D;
    const TIn* gq = static_cast<const TIn*>(p.q) + (size_t)bh * hs;
    const TIn* gk = static_cast<const TIn*>(p.k) + (size_t)bh * hs;
    const TIn* gu = static_cast<const TIn*>(p.u) + (size_t)bh * hs;
    const TIn* gv = static_cast<const TIn*>(p.v) + (p.v_shared ? 0 : (size_t)bh * hs);
    float zk[E];  // z^key before the chunk (identical in every staging warp)
#pragma unroll
    for (int m = 0; m < E; ++m) zk[m] = p.zk0 ? p.zk0[(size_t)bh * D + lane + 32 * m] : 0.f;

    auto issue = [&](int c) {
        const int n = min(C, T - c * C);
        const uint32_t bytes = (uint32_t)n * D * sizeof(TIn);
        unsigned char* r = x.raw(c % L::NRAW);
        mbar_arrive_expect_tx(x.b.full_r + c % L::NRAW, 3 * bytes);
        bulk_g2s(r, gq + (size_t)c * C * D, bytes, x.b.full_r + c % L::NRAW);
        bulk_g2s(r + L::RAW_T, gk + (size_t)c * C * D, bytes, x.b.full_r + c % L::NRAW);
        bulk_g2s(r + 2 * L::RAW_T, gu + (size_t)c * C * D, bytes, x.b.full_r + c % L::NRAW);
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
        // the S rows read this chunk's v from global memory a few chunks from now
        prefetch_v_l2<D, TIn>(gv + (size_t)c * C * D, n, sw * 32 + lane);
        if (TAPE && (c & 3) == 0 && sw == 0) {  // z^key before token 16 c (= 64 (c / 4))
            float* ck = ckpt_slot<D>(p, bh, c >> 2) + 2 * D * D;
#pragma unroll
            for (int m = 0; m < E; ++m) ck[lane + 32 * m] = zk[m];
        }
        const TIn* rq = reinterpret_cast<const TIn*>(x.raw(rs));
        const TIn* rk = reinterpret_cast<const TIn*>(x.raw(rs) + L::RAW_T);
        const TIn* ru = reinterpret_cast<const TIn*>(x.raw(rs) + 2 * L::RAW_T);
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
                float qv = 0.f, kv = 0.f, uv = 0.f;
                if (t < n) {
                    qv = ld_in<TIn>(rq + (size_t)t * D, e);
                    kv = ld_in<TIn>(rk + (size_t)t * D, e);
                    uv = ld_in<TIn>(ru + (size_t)t * D, e);
                }
                fq[j][m] = t < n ? phi_bf(qv) : 0.f;
                zsum[m] += t < n ? phi_bf(kv) : 0.f;
                pk[j][m] = zsum[m];  // this warp's phi(k) prefix, inclusive
                red[j][0] = fmaf(uv, uv, red[j][0]);
                red[j][1] = fmaf(kv, kv, red[j][1]);
                scr[(0 * C + t) * L::SCR_STRIDE + e] = uv;
                scr[(1 * C + t) * L::SCR_STRIDE + e] = kv;
                scr[(2 * C + t) * L::SCR_STRIDE + e] = fq[j][m];
            }
        }
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
        allreduce<3 * TW, 16>(&red[0][0]);
        float* sc = x.sc(s);
        if (lane < TW) {
            float r0 = red[0][0], r1 = red[0][1], r2 = red[0][2];
#pragma unroll
            for (int j = 1; j < TW; ++j)
                if (lane == j) {
                    r0 = red[j][0];
                    r1 = red[j][1];
                    r2 = red[j][2];
                }
            const int t = sw * TW + lane;
            sc[L::SC_IU + t] = t < n ? rsqrtf(fmaxf(r0, 1e-24f)) : 0.f;
            sc[L::SC_IK + t] = t < n ? rsqrtf(fmaxf(r1, 1e-24f)) : 0.f;
            sc[L::SC_RDEN + t] = t < n ? __frcp_rn(fmaxf(r2, p.eps)) : 1.f;  // 1 / den
            if (TAPE && t < n) {
                float* rec = tape_rec<D>(p, bh, c * C + t) + 3 * D;
                rec[2] = r2 < p.eps ? -p.eps : r2;  // den, negative where the eps floor is taken
                rec[3] = r0;                         // ||u_t||^2
                rec[4] = r1;                         // ||k_t||^2
            }
        }
        named_bar(ID_ST, 32 * NSTAGE);
        // scratch rows -> operand tiles, one 8-row group per unit: lane =
        // (row, 16-byte chunk); units are (row type, half chunk) split over warps
        {
            float* hi = x.hi(s);
            float* lo = x.lo(s);
            const int r8 = lane & 7;
            for (int unit = sw; unit < 3 * 2 + L::LO_ROWS / 8; unit += NSTAGE) {
                // units 0..5: HI rows (type unit / 2, half unit % 2); then LO rows
                int y, half, row0;
                float* dst;
                bool lopart;
                if (unit < 6) {
                    y = unit >> 1;
                    half = unit & 1;
                    row0 = y * C + half * 8;
                    dst = hi;
                    lopart = false;
                } else {
                    const int lu = unit - 6;
                    half = lu & 1;
                    y = L::F32IN ? (lu >> 1) : 2;  // fp32: u, k, phi lo parts; bf16: phi lo only
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
            VLA_TRACE_AT(p, 3, c);
            mbar_arrive(x.b.full_p + s);
            if (c + L::NRAW < nch) issue(c + L::NRAW);
        }
        if (c + L::NRAW < nch) issued = c + L::NRAW + 1;
    }
    if (bad) {
        if (leader) record_failure(p.status, BIT_TIMEOUT, ROLE_STAGE, bh, c * C);
        *x.abort = 1;
        // let copies already in flight land before the CTA can exit
        if (leader)
            for (int cc = c; cc < issued; ++cc)
                (void)mbar_wait(x.b.full_r + cc % L::NRAW, (cc / L::NRAW) & 1, nullptr, p.wait_ns);
        return;
    }
    if (p.zk_out && sw == 0) {
#pragma unroll
        for (int m = 0; m < E; ++m) p.zk_out[(size_t)bh * D + lane + 32 * m] = zk[m];
    }
}

// 16 consecutive floats (16-byte aligned) into registers
__device__ __forceinline__ void ld_row16(const float* p, float (&v)[C]) {
#pragma unroll
    for (int g = 0; g < C / 4; ++g) {
        const float4 x = ld4(p + 4 * g);
        v[4 * g] = x.x;
        v[4 * g + 1] = x.y;
        v[4 * g + 2] = x.z;
        v[4 * g + 3] = x.w;
    }
}

// 1 / x to within about 1 ulp (one MUFU reciprocal); used for the Sherman-
// Morrison pivots delta >= 1
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// v[idx] for a per-lane index without dynamic register indexing
template <int N>
__device__ __forceinline__ float col_pick(const float (&v)[N], int idx) {
    float r = v[0];
#pragma unroll
    for (int k = 1; k < N; ++k) r = idx == k ? v[k] : r;
    return r;
}

// ---------------------------------------------------------------------------
// 16 x 16 Gram block on the warp-level tensor-core path (mma.sync m16n8k8
// tf32, 3-term split): G[s][t] += sum_{k in [k0, k1)} a_s[k] b_t[k]. Row s of
// `a` is read from a K-major operand tile (rows of D) when A_CM, else from a
// row-major matrix with row stride `as`; row t of `b` from a row-major matrix
// with row stride `bs`. Lane (g, q) = (lane / 4, lane % 4) ends with
// acc[n][0..3] = G[g][8n + 2q], G[g][8n + 2q + 1], G[g + 8][8n + 2q], G[g + 8][8n + 2q + 1].
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t tf32_hi_bits(float x) { return __float_as_uint(x) & 0xFFFFE000u; }
__device__ __forceinline__ uint32_t tf32_lo_bits(float x) { return __float_as_uint(tf32_lo(x)); }

// a_exact: every a value is exact in tf32 (raw bf16 inputs), so its lo part is
// zero and the lo(a) x hi(b) term is skipped.
template <int D, bool A_CM>
__device__ __forceinline__ void gram16(const float* a, int as, const float* b, int bs, int k0, int k1, int lane,
                                       float (&acc)[2][4], bool a_exact = false) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
#pragma unroll 2
    for (int k = k0; k < k1; k += 8) {
        float av[4];
        if constexpr (A_CM) {
            av[0] = a[cm_off(g, k + q, D)];
            av[1] = a[cm_off(g + 8, k + q, D)];
            av[2] = a[cm_off(g, k + q + 4, D)];
            av[3] = a[cm_off(g + 8, k + q + 4, D)];
        } else {
            av[0] = a[g * as + k + q];
            av[1] = a[(g + 8) * as + k + q];
            av[2] = a[g * as + k + q + 4];
            av[3] = a[(g + 8) * as + k + q + 4];
        }
        float bv[2][2];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            bv[n][0] = b[(8 * n + g) * bs + k + q];
            bv[n][1] = b[(8 * n + g) * bs + k + q + 4];
        }
        const uint32_t ah0 = tf32_hi_bits(av[0]), ah1 = tf32_hi_bits(av[1]), ah2 = tf32_hi_bits(av[2]),
                       ah3 = tf32_hi_bits(av[3]);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const uint32_t bh0 = tf32_hi_bits(bv[n][0]), bh1 = tf32_hi_bits(bv[n][1]);
            mma_tf32(acc[n], ah0, ah1, ah2, ah3, tf32_lo_bits(bv[n][0]), tf32_lo_bits(bv[n][1]));
            if (!a_exact)
                mma_tf32(acc[n], tf32_lo_bits(av[0]), tf32_lo_bits(av[1]), tf32_lo_bits(av[2]), tf32_lo_bits(av[3]),
                         bh0, bh1);
            mma_tf32(acc[n], ah0, ah1, ah2, ah3, bh0, bh1);
        }
    }
}

// store a gram16 result (scaled by rs[row] if rs) to G[row][col] (or transposed)
__device__ __forceinline__ void put_gram16(float* G, int gs, const float (&acc)[2][4], int lane, const float* rs,
                                           bool transpose) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = g + 8 * (e >> 1), c = 8 * n + 2 * q + (e & 1);
            const float v = rs ? acc[n][e] * rs[r] : acc[n][e];
            if (transpose)
                G[c * gs + r] = v;
            else
                G[r * gs + c] = v;
        }
}

// Sum of the gram16 partials of a warp pair (halves 0 and 1 of D): half 1
// stores its accumulators in the scratch copy G + ms, the pair meets at named
// barrier `bar_id` (64 threads), half 0 adds them and stores the result
// (scaled by rs[row] if rs) to G[row][col] (transposed if asked).
__device__ __forceinline__ void gram_pair_sum(float* G, int ms, int gs, float (&acc)[2][4], int lane, int half,
                                              int bar_id, const float* rs, bool transpose) {
    float* part = G + ms + lane * 8;
    if (half) {
#pragma unroll
        for (int n = 0; n < 2; ++n)
            *reinterpret_cast<float4*>(part + 4 * n) = make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
    }
    named_bar(bar_id, 64);
    if (!half) {
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const float4 o = ld4(part + 4 * n);
            acc[n][0] += o.x;
            acc[n][1] += o.y;
            acc[n][2] += o.z;
            acc[n][3] += o.w;
        }
        put_gram16(G, gs, acc, lane, rs, transpose);
    }
}

// 16 values -> four float4 stores at the K-major operand positions (row, 0..15)
// of a tile with rows of C elements; `lo` selects the tf32 lo parts
__device__ __forceinline__ void put_row16(float* tile, int row, const float (&v)[C], bool lo) {
#pragma unroll
    for (int g = 0; g < C / 4; ++g) {
        float4 x = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        if (lo) x = make_float4(tf32_lo(x.x), tf32_lo(x.y), tf32_lo(x.z), tf32_lo(x.w));
        *reinterpret_cast<float4*>(tile + cm_off(row, 4 * g, C)) = x;
    }
}

// lo part of TMEM columns [col, col + D) of this warp's lanes -> columns [dst, dst + D)
template <int D>
__device__ __forceinline__ void refresh_lo(uint32_t lanebase, uint32_t col, uint32_t dst) {
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 16) {
        float v[16];
        tc_ld16(lanebase + col + c0, v);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = tf32_lo(v[j]);
        tc_st16(lanebase + dst + c0, v);
    }
    tc_wait_st();
}

// arrive at named barrier `id` (of `nthreads`) without waiting for it
__device__ __forceinline__ void bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// A team (warps 0-3): Sherman-Morrison steps of eq. 9 and what the gate of
// eq. 10 is formed from, one chunk at a time. Thread i < D of the row warps
// owns row i of A (TMEM lane i) and of every d x C intermediate.
// ---------------------------------------------------------------------------
template <int D, typename TIn, bool TAPE>
__device__ void tc_a_team(const Params& p, const Ctx<D, TIn>& x, int bh, int warp, int lane) {
    using L = Lay<D, TIn>;
    constexpr int XS = L::XS;
    const int ta = threadIdx.x;
    const bool rw = warp < L::NRW;
    const int i = ta;
    const uint32_t tm = __shfl_sync(0xffffffffu, *x.tmem_base, 0);
    const uint32_t tl = tm + ((uint32_t)(32 * warp) << 16);
    const int T = p.T, nch = (T + C - 1) / C;
    float* sm = x.sm();
    float* xr = x.f(L::OFF_XR);
    float* ph = x.f(L::OFF_PH);
    float* pl = x.f(L::OFF_PL);
    float* zh = x.f(L::OFF_ZH);
    float* zl = x.f(L::OFF_ZL);
    bool bad = false, nonfinite = false;
    // the fixed-A variant: A stays A_0, the gate is a_t = A_0 k^_t, and the
    // Sherman-Morrison steps (Grams, LDL^T, update, lo refresh) are skipped
    const bool fixed = p.fixed_a != 0;

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
            tc_st16(tl + L::T_A + c0, v);
            tc_st16(tl + L::T_AL + c0, w);
        }
        tc_wait_st();
    }
    // rows D..127 of the -N operand stay zero
    for (int e = ta; e < (128 - D) * C; e += 128) {
        ph[cm_off(D + e / C, e % C, C)] = 0.f;
        pl[cm_off(D + e / C, e % C, C)] = 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(ID_A, 128);

    uint32_t pa = 0;
    int c = 0;
    for (; c < nch; ++c) {
        const int s = c % L::NP, n = min(C, T - c * C), b = c & 1;
        bad = !mbar_wait(x.b.full_p + s, (c / L::NP) & 1, x.abort, p.wait_ns);
        // the S team has formed the gate of chunk c - 2 from the hand-over buffers
        if (c >= 2 && !bad) bad = !mbar_wait(x.b.empty_al + b, ((c >> 1) & 1) ^ 1, x.abort, p.wait_ns);
        if (bar_red_or(ID_A, 128, bad || *x.abort != 0)) {
            bad = true;
            break;
        }
        if (ta == 0) VLA_TRACE_AT(p, 4, c);
        if (TAPE && (c & 3) == 0 && rw) {  // A before token 16 c
            tc_fence_after();
            tmem_row_out<D>(tl, L::T_A, ckpt_slot<D>(p, bh, c >> 2) + D * D + (size_t)i * D);
        }
        const float* hi = x.hi(s);
        const float* sc = x.sc(s);
        // [Z' | W] = A_c [u | k]^T (rows u, k of the chunk; scaled by 1/||.|| below);
        // warps 0 and 1 issue the even and odd K steps into separate accumulators
        if (warp < 2 && elect_one()) {
            tc_fence_after();
            const uint32_t id = tc_idesc_tf32(128, 2 * C);
            const uint32_t bh0 = smem_u32(hi), bl0 = smem_u32(x.lo(s));
#pragma unroll 1
            for (int ks = warp; ks < D / 8; ks += 2) {
                const uint32_t dst = tm + ((ks & 1) ? L::T_XA2 : L::T_XA);
                const uint64_t bd = tc_sdesc(bh0 + ks * 256, 128, L::SBO_D);
                tc_mma_ts(dst, tm + L::T_A + 8 * ks, bd, id, ks > 1);
                tc_mma_ts(dst, tm + L::T_AL + 8 * ks, bd, id, 1);
                if constexpr (L::F32IN)
                    tc_mma_ts(dst, tm + L::T_A + 8 * ks, tc_sdesc(bl0 + ks * 256, 128, L::SBO_D), id, 1);
            }
            tc_commit(x.b.mma_xa);
        }
        bool ok = mbar_wait(x.b.mma_xa, c & 1, nullptr, p.wait_ns);
        if (ta == 0) VLA_TRACE_AT(p, 5, c);
        tc_fence_after();
        float* wp = x.f(L::OFF_WP) + (size_t)b * C * D;
        float* yp = x.f(L::OFF_YP) + (size_t)b * C * D;
        if (rw) {
            float v0[16], v1[16], v2[16], v3[16];
            tc_ld16(tl + L::T_XA, v0);
            tc_ld16(tl + L::T_XA + C, v1);
            tc_ld16(tl + L::T_XA2, v2);
            tc_ld16(tl + L::T_XA2 + C, v3);
            tc_wait_ld();
#pragma unroll
            for (int t = 0; t < C; ++t) {
                v0[t] = (v0[t] + v2[t]) * sc[L::SC_IU + t];  // z'_t = A_c u^_t
                v1[t] = (v1[t] + v3[t]) * sc[L::SC_IK + t];  // w_t = A_c k^_t
                xr[t * XS + i] = v0[t];
                xr[(C + t) * XS + i] = v1[t];
                wp[t * D + i] = v1[t];
            }
        }
        named_bar(ID_A, 128);
        if (!fixed) {
            // Guu[s][t] = u^_s . z'_t, Guk[s][t] = u^_s . w_t; warp = (matrix, half of D),
            // the half-D partials of a warp pair summed through shared memory
            const int mat = warp & 1, half = warp >> 1;
            float acc[2][4];
            gram16<D, true>(hi, 0, xr + mat * C * XS, XS, half * (D / 2), (half + 1) * (D / 2), lane, acc,
                            !L::F32IN);
            gram_pair_sum(sm + (mat ? L::SM_GUK : L::SM_GUU), L::MS, L::GSTR, acc, lane, half, 4 + mat,
                          sc + L::SC_IU, false);
            named_bar(ID_A, 128);
        }
        if (ta == 0) VLA_TRACE_AT(p, 6, c);
        if (ta == 0) mbar_arrive(x.b.empty_p + s);  // done with the chunk's u, k rows
        float mypiv = 1.f;  // delta of token `lane` (warp 3, taped)
        if (warp == 3 && !fixed) {
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
                const float rdt = rcp_approx(piv);
                if (lane == t) {
                    myrd = rdt;
                    mydl = piv;  // delta_t; its 1/sqrt is taken after the elimination, off its chain
                }
                if (TAPE && lane == t) mypiv = piv;
                if (!(piv > 0.f) || !isfinite(rdt)) nonfinite = true;
                // eliminate below pivot t in the columns not yet factored (M
                // columns j > t, every Guk column); a factored column j keeps
                // its entries below the diagonal: delta_j L[r][j]
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
                float* xp = x.f(L::OFF_XP) + (size_t)b * C * L::GSTR;  // X for the S team's gate
#pragma unroll
                for (int r = 0; r < C; ++r) xp[r * L::GSTR + j] = col[r];
            }
            if (lane == 0) VLA_TRACE_AT(p, 1, c);
        }
        if (bar_red_or(ID_A, 128, !ok || *x.abort != 0)) {
            bad = true;
            break;
        }
        if (ta == 0) VLA_TRACE_AT(p, 7, c);
        float y[C], lr[C];
        if (rw && !fixed) {
            // y = z_i = z'_i L^-T (forward substitution, in place), then y D^-1
#pragma unroll
            for (int t = 0; t < C; ++t) y[t] = xr[t * XS + i];
#pragma unroll
            for (int r = 0; r < C - 1; ++r) {
                ld_row16(sm + L::SM_LMT + r * L::GSTR, lr);  // L[t][r], t > r
#pragma unroll
                for (int t = r + 1; t < C; ++t) y[t] = fmaf(-lr[t], y[r], y[t]);
            }
            if (TAPE) {  // z_t = A_{t-1} u^_t of eq. 9
#pragma unroll
                for (int t = 0; t < C; ++t)
                    if (t < n) tape_rec<D>(p, bh, c * C + t)[i] = y[t];
            }
            // row i of N = Z D^-1/2: the rank-C update is A_c - N N^T (Woodbury
            // with I + Guu = L D L^T), symmetric by construction
            float nv[C];
            ld_row16(sm + L::SM_RS, lr);
#pragma unroll
            for (int t = 0; t < C; ++t) nv[t] = y[t] * lr[t];
            ld_row16(sm + L::SM_RD, lr);
#pragma unroll
            for (int t = 0; t < C; ++t) {
                y[t] *= lr[t];
                yp[t * D + i] = y[t];  // z_t / delta_t for the S team's gate
            }
            put_row16(zh, i, nv, false);
            put_row16(zl, i, nv, true);
#pragma unroll
            for (int t = 0; t < C; ++t) nv[t] = -nv[t];
            put_row16(ph, i, nv, false);
            put_row16(pl, i, nv, true);
        }
        fence_proxy_async_smem();
        // A_{c+1} = A_c - N N^T, issued by warp 3 (not a row warp for d <= 96) once
        // the rows have -N, N and z / delta in place; then the chunk's hand-over
        // buffers go to the S team, which forms the gate (eq. 10) off this chain
        if (warp < 3)
            bar_arrive(ID_M, 128);
        else
            named_bar(ID_M, 128);
        if (warp == 3) {
            if (!fixed && elect_one()) {
                VLA_TRACE_AT(p, 8, c);
                tc_fence_after();
                const uint32_t id = tc_idesc_tf32(128, D);
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks) {
                    const uint64_t ah = tc_sdesc(smem_u32(ph) + ks * 256, 128, L::SBO_C);
                    const uint64_t alo = tc_sdesc(smem_u32(pl) + ks * 256, 128, L::SBO_C);
                    const uint64_t bhd = tc_sdesc(smem_u32(zh) + ks * 256, 128, L::SBO_C);
                    const uint64_t bld = tc_sdesc(smem_u32(zl) + ks * 256, 128, L::SBO_C);
                    tc_mma_ss(tm + L::T_A, ah, bhd, id, 1);
                    tc_mma_ss(tm + L::T_A, ah, bld, id, 1);
                    tc_mma_ss(tm + L::T_A, alo, bhd, id, 1);
                }
                tc_commit(x.b.mma_a);
            }
            if (lane == 0) mbar_arrive(x.b.full_al + b);
            if (TAPE && lane < n) tape_rec<D>(p, bh, c * C + lane)[3 * D] = mypiv;  // delta_t = 1 + u^_t . z_t
        }
        if (!fixed) {
            bad = !mbar_wait(x.b.mma_a, pa, nullptr, p.wait_ns);
            pa ^= 1;
        }
        if (ta == 0) VLA_TRACE_AT(p, 9, c);
        tc_fence_after();
        if (rw && !fixed) refresh_lo<D>(tl, L::T_A, L::T_AL);
        if (ta == 0) VLA_TRACE_AT(p, 10, c);
        tc_fence_before();
        if (bar_red_or(ID_A, 128, bad)) {
            bad = true;
            ++c;
            break;
        }
    }
    if (bad) {
        if (ta == 0) record_failure(p.status, BIT_TIMEOUT, ROLE_A, bh, c * C);
        *x.abort = 1;
    } else if (rw) {
        float* Ao = p.A_out + ((size_t)bh * D + i) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
            tc_ld16(tl + L::T_A + c0, v);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(Ao + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    if (nonfinite) record_failure(p.status, BIT_NONFINITE, ROLE_A, bh, -1);
}

// ---------------------------------------------------------------------------
// S team (warps 4-7): the gate, residual writes and readout of eq. 10-11 for
// the chunk the A team published. Thread i < D of the row warps owns row i of S.
// ---------------------------------------------------------------------------
template <int D, typename TIn, bool TAPE>
__device__ void tc_s_team(const Params& p, const Ctx<D, TIn>& x, int bh, int warp, int lane) {
    using L = Lay<D, TIn>;
    constexpr int XS = L::XS;
    const int ts = threadIdx.x - 128, wq = warp - 4;
    const bool rw = wq < L::NRW;
    const int i = ts;
    const uint32_t tm = __shfl_sync(0xffffffffu, *x.tmem_base, 0);
    const uint32_t tl = tm + ((uint32_t)(32 * wq) << 16);
    const int T = p.T, nch = (T + C - 1) / C;
    float* sm = x.sm();
    float* eh = x.f(L::OFF_EH);
    float* el = x.f(L::OFF_EL);
    float* alr = x.f(L::OFF_AL);
    float* gh = x.f(L::OFF_GH);
    float* gl = x.f(L::OFF_GL);
    const bool fixed = p.fixed_a != 0;
    const TIn* gv = static_cast<const TIn*>(p.v) + (p.v_shared ? 0 : (size_t)bh * (p.in_stride ? p.in_stride : (size_t)T * D));
    float* go = p.o + (size_t)bh * p.o_stride;
    bool bad = false, nonfinite = false;
    float nfchk = 0.f;  // fma(o, 0, .) of every output (branch-free)

    // S_0 = 0 unless carried in, and its lo part
    if (rw) {
        const float* S0 = p.S0 ? p.S0 + ((p.s0_shared ? 0 : (size_t)bh * D) + i) * D : nullptr;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16], w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                v[j] = S0 ? S0[c0 + j] : 0.f;
                w[j] = tf32_lo(v[j]);
            }
            tc_st16(tl + L::T_S + c0, v);
            tc_st16(tl + L::T_SL + c0, w);
        }
        tc_wait_st();
    }
    for (int e = ts; e < (128 - D) * C; e += 128) {
        eh[cm_off(D + e / C, e % C, C)] = 0.f;
        el[cm_off(D + e / C, e % C, C)] = 0.f;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(ID_S, 128);

    uint32_t ps = 0;
    int c = 0;
    for (; c < nch; ++c) {
        const int s = c % L::NP, n = min(C, T - c * C), b = c & 1;
        float vv[C];
        typename RawIn<TIn>::type vr[C];
        if (rw) load_v_raw<D, TIn>(gv + (size_t)c * C * D, i, n, vr);
        bad = !mbar_wait(x.b.full_p + s, (c / L::NP) & 1, x.abort, p.wait_ns) ||
              !mbar_wait(x.b.full_al + b, (c >> 1) & 1, x.abort, p.wait_ns);
        if (bar_red_or(ID_S, 128, bad || *x.abort != 0)) {
            bad = true;
            break;
        }
        const float* hi = x.hi(s);
        const float* sc = x.sc(s);
        if (ts == 0) VLA_TRACE_AT(p, 11, c);
        if (TAPE && (c & 3) == 0 && rw) {  // S before token 16 c
            tc_fence_after();
            tmem_row_out<D>(tl, L::T_S, ckpt_slot<D>(p, bh, c >> 2) + (size_t)i * D);
        }
        // [S_c k | S_c phi] (rows k, phi of the chunk)
        if (wq < 2 && elect_one()) {
            tc_fence_after();
            const uint32_t id32 = tc_idesc_tf32(128, 2 * C), id16 = tc_idesc_tf32(128, C);
            const uint32_t bh0 = smem_u32(hi) + 2 * L::SBO_D;
            const uint32_t bl0 = smem_u32(x.lo(s)) + (L::F32IN ? 2 * L::SBO_D : 0);
#pragma unroll 1
            for (int ks = wq; ks < D / 8; ks += 2) {
                const uint32_t dst = tm + ((ks & 1) ? L::T_XS2 : L::T_XS);
                const uint64_t bd = tc_sdesc(bh0 + ks * 256, 128, L::SBO_D);
                const uint64_t bld = tc_sdesc(bl0 + ks * 256, 128, L::SBO_D);
                tc_mma_ts(dst, tm + L::T_S + 8 * ks, bd, id32, ks > 1);
                tc_mma_ts(dst, tm + L::T_SL + 8 * ks, bd, id32, 1);
                if constexpr (L::F32IN)
                    tc_mma_ts(dst, tm + L::T_S + 8 * ks, bld, id32, 1);
                else
                    tc_mma_ts(dst + C, tm + L::T_S + 8 * ks, bld, id16, 1);
            }
            tc_commit(x.b.mma_xs);
        }
        // while warps 4 and 5 issue the products (about 100 clocks per MMA),
        // warps 6 and 7 form the gate a_t = A_t k^_t = w_t - sum_{q<=t}
        // (z_q / delta_q) X[q][t] (eq. 10; a_t = A_0 k^_t with A fixed), zero
        // past the end of the sequence, from the A team's hand-over buffers:
        // thread g of the two warps takes rows g and g + 64
        if (wq >= 2) {
            const float* wp = x.f(L::OFF_WP) + (size_t)b * C * D;
            const float* yp = x.f(L::OFF_YP) + (size_t)b * C * D;
            const float* xp = x.f(L::OFF_XP) + (size_t)b * C * L::GSTR;
#pragma unroll 1
            for (int r = ts - 64; r < D; r += 64) {
                float lr[C], av[C];
#pragma unroll
                for (int t = 0; t < C; ++t) av[t] = wp[t * D + r];
                if (!fixed) {
                    // q outermost: the 16 sums advance side by side, each in
                    // ascending q
#pragma unroll
                    for (int q = 0; q < C; ++q) {
                        const float yq = yp[q * D + r];
                        ld_row16(xp + q * L::GSTR, lr);  // X[q][t]
#pragma unroll
                        for (int t = q; t < C; ++t) av[t] = fmaf(-yq, lr[t], av[t]);
                    }
                }
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    av[t] = t < n ? av[t] : 0.f;
                    alr[t * XS + r] = av[t];
                }
                put_row16(gh, r, av, false);
                put_row16(gl, r, av, true);
            }
        }
        if (wq >= 2) {
            named_bar(ID_G, 64);
            if (wq == 3 && lane < C) {
                // ||a_t||^2
                float2 acc = f2(0.f, 0.f);
#pragma unroll 8
                for (int k4 = 0; k4 < D / 4; ++k4) {
                    const float4 a = ld4(alr + lane * XS + 4 * k4);
                    acc = __ffma2_rn(f2(a.x, a.y), f2(a.x, a.y), acc);
                    acc = __ffma2_rn(f2(a.z, a.w), f2(a.z, a.w), acc);
                }
                sm[L::SM_LAA + lane] = acc.x + acc.y;
                if (TAPE && lane < n) tape_rec<D>(p, bh, c * C + lane)[3 * D + 1] = sqrtf(acc.x + acc.y);  // ||a_t||
            }
        }
        named_bar(ID_S, 128);
        if (ts == 0) mbar_arrive(x.b.empty_al + b);  // the hand-over buffers are free
        // Lk[t][s] = k^_t . a_s, Lq[t][s] = phi_t . a_s; warp = (matrix, half of D)
        {
            const int mat = wq & 1, half = wq >> 1;
            float acc[2][4];
            gram16<D, true>(hi + (mat ? 32 : 16) * D, 0, alr, XS, half * (D / 2), (half + 1) * (D / 2), lane, acc,
                            !L::F32IN && mat == 0);
            if (mat)
                gram_pair_sum(sm + L::SM_LQ, L::MS, L::GSTR, acc, lane, half, 6 + mat, nullptr, false);
            else
                gram_pair_sum(sm + L::SM_LKT, L::MS, L::GSTR, acc, lane, half, 6 + mat, sc + L::SC_IK, true);
        }
        bool ok = mbar_wait(x.b.mma_xs, c & 1, nullptr, p.wait_ns);
        if (ts == 0) VLA_TRACE_AT(p, 12, c);
        tc_fence_after();
        float sk[C], sq[C];
        if (rw) {
            float v0[16], v1[16], v2[16], v3[16];
            tc_ld16(tl + L::T_XS, v0);
            tc_ld16(tl + L::T_XS + C, v1);
            tc_ld16(tl + L::T_XS2, v2);
            tc_ld16(tl + L::T_XS2 + C, v3);
            tc_wait_ld();
#pragma unroll
            for (int t = 0; t < C; ++t) {
                sk[t] = (v0[t] + v2[t]) * sc[L::SC_IK + t];  // S_c k^_t
                sq[t] = v1[t] + v3[t];                        // S_c phi_t
            }
        }
        named_bar(ID_S, 128);
        if (ts == 0) VLA_TRACE_AT(p, 13, c);
        if (rw) {
            float lr[C], nr[C];
            // e_t = v_t - S_c k^_t - sum_{s<t} (k^_t . alpha^_s) e_s, kept (in place)
            // as e'_t = e_t / ||a_t||
            ld_row16(sm + L::SM_LAA, nr);
#pragma unroll
            for (int t = 0; t < C; ++t) {
                vv[t] = raw_f32(vr[t]) - sk[t];
                nr[t] = rsqrtf(fmaxf(nr[t], 1e-24f));
            }
#pragma unroll
            for (int r = 0; r < C; ++r) {
                vv[r] *= nr[r];
                if (r < C - 1) {
                    ld_row16(sm + L::SM_LKT + r * L::GSTR, lr);  // Lk[t][r], t > r
#pragma unroll
                    for (int t = r + 1; t < C; ++t) vv[t] = fmaf(-lr[t], vv[r], vv[t]);
                }
            }
            if (ts == 0) VLA_TRACE_AT(p, 0, c);
            if (TAPE) {  // alpha^_t = a_t / ||a_t|| and e_t = e'_t ||a_t|| (eq. 10)
#pragma unroll
                for (int t = 0; t < C; ++t)
                    if (t < n) {
                        float* rec = tape_rec<D>(p, bh, c * C + t);
                        rec[D + i] = alr[t * XS + i] * nr[t];
                        rec[2 * D + i] = vv[t] / nr[t];
                    }
            }
            // o_t = (S_c phi_t + sum_{s<=t} e_s (alpha^_s . phi_t)) / den_t = S_t phi_t / den_t (eq. 11)
            ld_row16(sc + L::SC_RDEN, nr);
#pragma unroll
            for (int t = 0; t < C; ++t) {
                ld_row16(sm + L::SM_LQ + t * L::GSTR, lr);
                float a = sq[t];
#pragma unroll
                for (int q = 0; q <= t; ++q) a = fmaf(lr[q], vv[q], a);
                const float ov = a * nr[t];
                if (t < n) {
                    go[(size_t)(c * C + t) * D + i] = ov;
                    nfchk = fmaf(ov, 0.f, nfchk);  // stays 0 unless an o is NaN or Inf
                }
            }
            if (ts == 0) VLA_TRACE_AT(p, 2, c);
            put_row16(eh, i, vv, false);
            put_row16(el, i, vv, true);
        }
        fence_proxy_async_smem();
        named_bar(ID_S, 128);
        // S_{c+1} = S_c + E' A (rows a_t, columns scaled into E')
        if (wq == 0 && elect_one()) {
            mbar_arrive(x.b.empty_p + s);  // done with the chunk's k, phi rows and den
            tc_fence_after();
            const uint32_t id = tc_idesc_tf32(128, D);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks) {
                const uint64_t ah = tc_sdesc(smem_u32(eh) + ks * 256, 128, L::SBO_C);
                const uint64_t alo = tc_sdesc(smem_u32(el) + ks * 256, 128, L::SBO_C);
                const uint64_t bhd = tc_sdesc(smem_u32(gh) + ks * 256, 128, L::SBO_C);
                const uint64_t bld = tc_sdesc(smem_u32(gl) + ks * 256, 128, L::SBO_C);
                tc_mma_ss(tm + L::T_S, ah, bhd, id, 1);
                tc_mma_ss(tm + L::T_S, ah, bld, id, 1);
                tc_mma_ss(tm + L::T_S, alo, bhd, id, 1);
            }
            tc_commit(x.b.mma_s);
        }
        if (ts == 0) VLA_TRACE_AT(p, 14, c);
        ok = mbar_wait(x.b.mma_s, ps, nullptr, p.wait_ns) && ok;
        ps ^= 1;
        if (ts == 0) VLA_TRACE_AT(p, 15, c);
        tc_fence_after();
        if (rw) refresh_lo<D>(tl, L::T_S, L::T_SL);
        tc_fence_before();
        if (bar_red_or(ID_S, 128, !ok)) {
            bad = true;
            ++c;
            break;
        }
    }
    if (bad) {
        if (ts == 0) record_failure(p.status, BIT_TIMEOUT, ROLE_S, bh, c * C);
        *x.abort = 1;
    } else if (rw) {
        float* So = p.S_out + ((size_t)bh * D + i) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float v[16];
            tc_ld16(tl + L::T_S + c0, v);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(So + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    if (nonfinite || nfchk != 0.f) record_failure(p.status, BIT_NONFINITE, ROLE_S, bh, -1);
}

}  // namespace tc

// one head (bh) of the chunked kernel on this CTA
template <int D, typename TIn, bool TAPE>
__device__ __forceinline__ void tc_head(const Params& p, int bh) {
    using L = tc::Lay<D, TIn>;
    static_assert(D % 32 == 0 && D <= 96, "row warps of a team fit in warps 0-2 / 4-6");
    extern __shared__ __align__(1024) unsigned char smem[];
    tc::Ctx<D, TIn> x;
    x.base = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
    x.b.full_r = bars;
    x.b.full_p = x.b.full_r + L::NRAW;
    x.b.empty_p = x.b.full_p + L::NP;
    x.b.full_al = x.b.empty_p + L::NP;
    x.b.empty_al = x.b.full_al + 2;
    x.b.mma_a = x.b.empty_al + 2;
    x.b.mma_s = x.b.mma_a + 1;
    x.b.mma_xa = x.b.mma_s + 1;
    x.b.mma_xs = x.b.mma_xa + 1;
    x.abort = reinterpret_cast<volatile int*>(smem + L::OFF_MISC);
    x.tmem_base = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC + 8);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int r = 0; r < L::NRAW; ++r) mbar_init(x.b.full_r + r, 1);
        for (int s = 0; s < L::NP; ++s) {
            mbar_init(x.b.full_p + s, 1);
            mbar_init(x.b.empty_p + s, 2);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(x.b.full_al + s, 1);
            mbar_init(x.b.empty_al + s, 1);
        }
        mbar_init(x.b.mma_a, 1);
        mbar_init(x.b.mma_s, 1);
        mbar_init(x.b.mma_xa, 2);
        mbar_init(x.b.mma_xs, 2);
        *x.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc_alloc(x.tmem_base, L::TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp < 4)
        tc::tc_a_team<D, TIn, TAPE>(p, x, bh, warp, lane);
    else if (warp < 8)
        tc::tc_s_team<D, TIn, TAPE>(p, x, bh, warp, lane);
    else
        tc::tc_stage<D, TIn, TAPE>(p, x, bh, warp - 8, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tc_dealloc(*x.tmem_base, L::TCOLS);
}

template <int D, typename TIn, bool TAPE = false>
__global__ void __launch_bounds__(tc::THREADS, 1) vla_tc_kernel(const Params p) {
    tc_head<D, TIn, TAPE>(p, blockIdx.x);
}
