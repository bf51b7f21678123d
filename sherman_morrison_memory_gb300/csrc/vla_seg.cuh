// vla_seg.cuh -- the two-segment form of the recurrence: the second half of
// the sequence runs beside the first. Included by vla_forward.cu inside
// namespace vla, after vla_tc.cuh.
//
// "Variational Linear Attention" (arXiv 2605.11196). With the sequence cut
// at token L:
//
//  * A. The penalty M_t = lambda0 I + sum_{s<=t} u^_s u^_s^T of §3.2 is a
//    prefix sum, and A_t = M_t^-1 (eq. 9 is Sherman-Morrison on it). So
//    A_L = (A_0^-1 + sum_{s<L} u^_s u^_s^T)^-1 without running the first
//    half; likewise z^key_L = z^key_0 + sum_{s<L} phi(k_s) (eq. 11).
//  * S. Eq. 12, read on the transposed state, composes associatively:
//    S_t = S_{t-1} P_t + v_t alpha^_t^T with P_t = I - k^_t alpha^_t^T, so for
//    t >= L, S_t = S_L Pi_t + G_t. G_t is the second half's recurrence from
//    S = 0, and Pi_t the same recurrence from S = I with v = 0; the gates of
//    both come from A_L alone. The readout is
//    o_t = (G_t phi_t + S_L Pi_t phi_t) / den_t.
//
// One call therefore runs three launches of the chunked kernel side by side
// (first half; second half from S = 0; second half from S = I with v = 0),
// the first at once, the other two after two small kernels that form A_L
// and z^key_L, and then a combine kernel that forms S_T = S_L Pi_T + G_T
// and adds S_L (Pi_t phi_t / den_t) to the second half's o_t.

namespace seg {

constexpr int THREADS = 256;
constexpr int NSPLIT = 16;  // at most this many CTAs per head share the prefix sums
constexpr int TILE = 128;   // tokens staged per step of the prefix sums

// Per (head, split): the partial sums of u^_s u^_s^T and phi(k_s) over its
// share of tokens [0, L) (the u^ sums are skipped for the fixed-A variant).
struct PrefixParams {
    const void* u;
    const void* k;
    size_t in_stride;  // elements between heads' rows
    int L;             // tokens of the first segment
    int nsplit;        // CTAs per head, 1 .. NSPLIT
    int fixed_a;
    float* dpart;      // [heads][NSPLIT][D][D], the first nsplit of each head written
    float* zpart;      // [heads][NSPLIT][D]
};

// 8 consecutive input elements (16-byte aligned for bf16, 32 for fp32), as
// loaded (Raw8) and as float (cvt8), so that a thread's loads can all be in
// flight before the first is used
template <typename TIn>
struct Raw8;
template <>
struct Raw8<float> {
    float4 a, b;
};
template <>
struct Raw8<__nv_bfloat16> {
    uint4 a;
};
__device__ __forceinline__ void ld8(const float* p, Raw8<float>& r) {
    r.a = *reinterpret_cast<const float4*>(p);
    r.b = *reinterpret_cast<const float4*>(p + 4);
}
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, Raw8<__nv_bfloat16>& r) {
    r.a = *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ void cvt8(const Raw8<float>& r, float (&x)[8]) {
    x[0] = r.a.x, x[1] = r.a.y, x[2] = r.a.z, x[3] = r.a.w, x[4] = r.b.x, x[5] = r.b.y, x[6] = r.b.z, x[7] = r.b.w;
}
__device__ __forceinline__ void cvt8(const Raw8<__nv_bfloat16>& r, float (&x)[8]) {
    const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// R consecutive floats of shared memory (R even; 16-byte aligned when R is a
// multiple of 4, else 8-byte aligned), in the widest loads that keep a
// 16-thread row of them free of bank conflicts
template <int R>
__device__ __forceinline__ void lds_run(const float* p, float (&x)[R]) {
    static_assert(R % 2 == 0, "pairs of floats");
    if constexpr (R % 4 == 0) {
#pragma unroll
        for (int h = 0; h < R / 4; ++h) {
            const float4 v = reinterpret_cast<const float4*>(p)[h];
            x[4 * h] = v.x, x[4 * h + 1] = v.y, x[4 * h + 2] = v.z, x[4 * h + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int h = 0; h < R / 2; ++h) {
            const float2 v = reinterpret_cast<const float2*>(p)[h];
            x[2 * h] = v.x, x[2 * h + 1] = v.y;
        }
    }
}

template <int D, typename TIn>
__global__ void __launch_bounds__(THREADS, 2) vla_seg_prefix_kernel(const PrefixParams pp) {
    constexpr int R = D / 16;             // each thread owns an R x R block of the D x D sum
    constexpr int US = D + 4;             // row stride of the staged rows (16-byte rows)
    constexpr int NC = D / 8;             // 8-element chunks per row
    constexpr int NG = THREADS / NC;      // token groups of the staging map
    constexpr int NIT = (TILE + NG - 1) / NG;
    constexpr int NB = sizeof(TIn) == 4 ? (NIT + 1) / 2 : NIT;  // loads in flight per batch
    static_assert(D % 16 == 0, "16 x 16 thread grid");
    extern __shared__ __align__(16) float psh[];
    float* ur = psh;                      // TILE x US: u^ rows
    float* zs = ur + TILE * US;           // NG x D: phi(k) sums per token group
    const int bh = blockIdx.x / pp.nsplit, sp = blockIdx.x % pp.nsplit;
    const int per = (pp.L + pp.nsplit - 1) / pp.nsplit;
    const int t0 = sp * per, t1 = min(pp.L, t0 + per);
    const TIn* gu = static_cast<const TIn*>(pp.u) + (size_t)bh * pp.in_stride;
    const TIn* gk = static_cast<const TIn*>(pp.k) + (size_t)bh * pp.in_stride;
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int warp = tid / 32, lane = tid % 32;
    // staging map: thread tid < NG * NC takes column chunk j8 of tokens g, g + NG, ...
    const bool stager = tid < NG * NC;
    const int j8 = tid % NC, g = tid / NC;
    float acc[R][R];
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
        for (int b = 0; b < R; ++b) acc[a][b] = 0.f;
    float zk[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // phi(k) sums of this thread's column chunk
    for (int tb = t0; tb < t1; tb += TILE) {
        const int nt = min(TILE, t1 - tb);
        __syncthreads();  // the previous tile's rows are consumed
        if (stager) {
#pragma unroll
            for (int i0 = 0; i0 < NIT; i0 += NB) {
                Raw8<TIn> ru[NB], rk[NB];
#pragma unroll
                for (int i = 0; i < NB; ++i) {
                    const int t = g + NG * (i0 + i);
                    if (i0 + i < NIT && t < nt) {
                        if (!pp.fixed_a) ld8(gu + (size_t)(tb + t) * D + 8 * j8, ru[i]);
                        ld8(gk + (size_t)(tb + t) * D + 8 * j8, rk[i]);
                    }
                }
#pragma unroll
                for (int i = 0; i < NB; ++i) {
                    const int t = g + NG * (i0 + i);
                    if (i0 + i < NIT && t < nt) {
                        float x[8], kx[8];
                        cvt8(rk[i], kx);
#pragma unroll
                        for (int e = 0; e < 8; ++e) zk[e] += phi(kx[e]);
                        if (!pp.fixed_a) {
                            cvt8(ru[i], x);
                            float4* dst = reinterpret_cast<float4*>(ur + t * US + 8 * j8);
                            dst[0] = make_float4(x[0], x[1], x[2], x[3]);
                            dst[1] = make_float4(x[4], x[5], x[6], x[7]);
                        }
                    }
                }
            }
        }
        if (pp.fixed_a) continue;
        __syncthreads();
        // warp w scales tokens w, w + 8, ... to unit length (1 / max(||u||, 1e-12))
        for (int t = warp; t < nt; t += THREADS / 32) {
            float s2 = 0.f;
            for (int j = lane; j < D; j += 32) s2 = fmaf(ur[t * US + j], ur[t * US + j], s2);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
            const float rn = 1.f / fmaxf(sqrtf(s2), 1e-12f);
            for (int j = lane; j < D; j += 32) ur[t * US + j] *= rn;
        }
        __syncthreads();
        // rows ty R .. ty R + R - 1 and columns tx R .. tx R + R - 1 of the sum
#pragma unroll 4
        for (int t = 0; t < nt; ++t) {
            float ra[R], rb[R];
            lds_run<R>(ur + t * US + ty * R, ra);
            lds_run<R>(ur + t * US + tx * R, rb);
#pragma unroll
            for (int a = 0; a < R; ++a)
#pragma unroll
                for (int b = 0; b < R; ++b) acc[a][b] = fmaf(ra[a], rb[b], acc[a][b]);
        }
    }
    // the token groups' phi(k) sums, added in a fixed order
    __syncthreads();
    if (stager) {
#pragma unroll
        for (int e = 0; e < 8; ++e) zs[g * D + 8 * j8 + e] = zk[e];
    }
    __syncthreads();
    if (tid < D) {
        float z = 0.f;
        for (int w = 0; w < NG; ++w) z += zs[w * D + tid];
        pp.zpart[((size_t)bh * NSPLIT + sp) * D + tid] = z;
    }
    float* dp = pp.dpart + ((size_t)bh * NSPLIT + sp) * D * D;
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
        for (int b = 0; b < R; ++b) dp[(ty * R + a) * D + tx * R + b] = acc[a][b];
}

// dynamic shared memory of vla_seg_prefix_kernel<D>
template <int D>
constexpr int prefix_smem() {
    return (TILE * (D + 4) + (THREADS / (D / 8)) * D) * 4;
}

// Per head: z^key_L, and A_L = (A_0^-1 + sum_s u^_s u^_s^T)^-1 by in-place
// Gauss-Jordan elimination (no pivoting: the matrices are symmetric positive
// definite), symmetrised; A_L = A_0 for the fixed-A variant. Block 0 also
// writes the identity that the second half's transition starts from.
struct InvertParams {
    const float* dpart;
    const float* zpart;
    int nsplit;
    const float* A0;   // nullable: A_0 = I / lambda0
    const float* zk0;  // nullable
    float lambda0, inv_lambda0;
    int fixed_a;
    float* A_cut;  // [heads][D][D]
    float* zk_cut; // [heads][D]
    float* ident;  // [D][D]
    DeviceStatus* status;
};

// In-place inverse of a D x D matrix held in registers, by Gauss-Jordan
// elimination without pivoting (the matrices here are symmetric positive
// definite). Thread (ty, tx) = (tid / 16, tid % 16) holds rows ty + 16 a and
// columns tx + 16 b in x[a][b]. Pivot k = 16 ka + kr sits in register slot ka
// of the threads with ty == kr (its row) or tx == kr (its column), so with
// ka a compile-time index every step is one fused multiply-add per element
// plus the fix-up of the pivot row and column. Step k reads pivot column and
// row k from one of two shared buffers (cr[k & 1]); the owners of column and
// row k + 1 write those into the other, so one barrier separates the steps.
// cr: 4 x D floats. Returns false if a pivot was not positive.
template <int D>
__device__ __forceinline__ bool gauss_jordan(float (&x)[D / 16][D / 16], float* cr) {
    constexpr int R = D / 16;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    bool ok = true;
    __syncthreads();  // earlier readers of cr are done
    if (tx == 0) {
#pragma unroll
        for (int a = 0; a < R; ++a) cr[ty + 16 * a] = x[a][0];  // column 0
    }
    if (ty == 0) {
#pragma unroll
        for (int b = 0; b < R; ++b) cr[D + tx + 16 * b] = x[0][b];  // row 0
    }
    __syncthreads();
#pragma unroll
    for (int ka = 0; ka < R; ++ka) {
#pragma unroll 1
        for (int kr = 0; kr < 16; ++kr) {
            const int k = 16 * ka + kr;
            const float* col = cr + (k & 1) * 2 * D;
            const float* row = col + D;
            float* ncol = cr + ((k + 1) & 1) * 2 * D;
            float* nrow = ncol + D;
            const float piv = row[k];
            if (!(piv > 0.f)) ok = false;
            const float rp = 1.f / piv;
            float r[R], c[R];
#pragma unroll
            for (int b = 0; b < R; ++b) r[b] = row[tx + 16 * b];
#pragma unroll
            for (int a = 0; a < R; ++a) c[a] = col[ty + 16 * a] * rp;
#pragma unroll
            for (int a = 0; a < R; ++a)
#pragma unroll
                for (int b = 0; b < R; ++b) x[a][b] = fmaf(-c[a], r[b], x[a][b]);
            if (ty == kr) {  // the pivot row
#pragma unroll
                for (int b = 0; b < R; ++b) x[ka][b] = r[b] * rp;
            }
            if (tx == kr) {  // the pivot column
#pragma unroll
                for (int a = 0; a < R; ++a) x[a][ka] = -c[a];
                if (ty == kr) x[ka][ka] = rp;
            }
            // publish column and row k + 1: slot ka at residue kr + 1, or slot ka + 1 at residue 0
            if (kr < 15) {
                if (tx == kr + 1) {
#pragma unroll
                    for (int a = 0; a < R; ++a) ncol[ty + 16 * a] = x[a][ka];
                }
                if (ty == kr + 1) {
#pragma unroll
                    for (int b = 0; b < R; ++b) nrow[tx + 16 * b] = x[ka][b];
                }
            } else if (ka + 1 < R) {
                if (tx == 0) {
#pragma unroll
                    for (int a = 0; a < R; ++a) ncol[ty + 16 * a] = x[a][ka + 1];
                }
                if (ty == 0) {
#pragma unroll
                    for (int b = 0; b < R; ++b) nrow[tx + 16 * b] = x[ka + 1][b];
                }
            }
            __syncthreads();
        }
    }
    return ok;
}

template <int D>
__global__ void __launch_bounds__(THREADS) vla_seg_invert_kernel(const InvertParams ip) {
    constexpr int R = D / 16, MS = D + 1;
    extern __shared__ __align__(16) float sh[];
    float* m = sh;           // D x MS: the summed partials, then the inverse
    float* cr = m + D * MS;  // 4 x D: pivot columns and rows
    const int bh = blockIdx.x, tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    if (bh == 0)
        for (int e = tid; e < D * D; e += THREADS) ip.ident[e] = (e / D == e % D) ? 1.f : 0.f;
    if (tid < D) {
        float z = ip.zk0 ? ip.zk0[(size_t)bh * D + tid] : 0.f;
        for (int sp = 0; sp < ip.nsplit; ++sp) z += ip.zpart[((size_t)bh * NSPLIT + sp) * D + tid];
        ip.zk_cut[(size_t)bh * D + tid] = z;
    }
    float* out = ip.A_cut + (size_t)bh * D * D;
    const float* A0 = ip.A0 ? ip.A0 + (size_t)bh * D * D : nullptr;
    if (ip.fixed_a) {
        for (int e = tid; e < D * D; e += THREADS)
            out[e] = A0 ? A0[e] : ((e / D == e % D) ? ip.inv_lambda0 : 0.f);
        return;
    }
    // the split partials, summed in a fixed order (16-byte loads, all splits in flight)
    const float4* dp = reinterpret_cast<const float4*>(ip.dpart + (size_t)bh * NSPLIT * D * D);
    for (int f = tid; f < D * D / 4; f += THREADS) {
        float4 v[NSPLIT];
#pragma unroll
        for (int sp = 0; sp < NSPLIT; ++sp)
            if (sp < ip.nsplit) v[sp] = dp[(size_t)sp * (D * D / 4) + f];
        float4 acc = v[0];
#pragma unroll
        for (int sp = 1; sp < NSPLIT; ++sp)
            if (sp < ip.nsplit) acc.x += v[sp].x, acc.y += v[sp].y, acc.z += v[sp].z, acc.w += v[sp].w;
        const int i = (4 * f) / D, j = 4 * f - i * D;
        m[i * MS + j] = acc.x, m[i * MS + j + 1] = acc.y, m[i * MS + j + 2] = acc.z, m[i * MS + j + 3] = acc.w;
    }
    float x[R][R];
    bool ok = true;
    if (A0) {
#pragma unroll
        for (int a = 0; a < R; ++a)
#pragma unroll
            for (int b = 0; b < R; ++b) x[a][b] = A0[(ty + 16 * a) * D + tx + 16 * b];
        ok = gauss_jordan<D>(x, cr);  // A_0^-1 (its first barrier also orders the sums above)
    } else {
#pragma unroll
        for (int a = 0; a < R; ++a)
#pragma unroll
            for (int b = 0; b < R; ++b) x[a][b] = (ty + 16 * a == tx + 16 * b) ? ip.lambda0 : 0.f;
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
        for (int b = 0; b < R; ++b) x[a][b] += m[(ty + 16 * a) * MS + tx + 16 * b];
    ok = gauss_jordan<D>(x, cr) && ok;
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
        for (int b = 0; b < R; ++b) m[(ty + 16 * a) * MS + tx + 16 * b] = x[a][b];
    __syncthreads();
    for (int e = tid; e < D * D; e += THREADS) {
        const int i = e / D, j = e % D;
        out[e] = 0.5f * (m[i * MS + j] + m[j * MS + i]);
    }
    if (!ok && tid == 0) record_failure(ip.status, BIT_NONFINITE, ROLE_A, bh, -1);
}

// S_T = S_L Pi_T + G_T (blockIdx.y == the last tile), and
// o_t += S_L (Pi_t phi_t / den_t) for the second half's tokens, OT per CTA
struct CombineParams {
    const float* G0;   // S_L [heads][D][D]
    const float* F1;   // Pi_T
    const float* G1;   // G_T
    const float* fphi; // Pi_t phi_t / den_t [heads][L1][D]
    float* o;          // the second half's o rows: head h, token t at o + h * o_stride + t * D
    size_t o_stride;
    int L1;
    float* S_out;
};

constexpr int OT = 64;  // tokens per CTA of the o correction

// Shared-memory tiles are stored transposed (the contraction index m outer),
// so that a thread's operands are runs of consecutive floats: thread
// (tt, io) = (tid / 16, tid % 16) forms tokens 4 tt .. 4 tt + 3 of outputs
// io R .. io R + R - 1 (R = D / 16) from one 16-byte load and R / 2 or R / 4
// wider loads per m. The transposing copies map lane l of a warp to 8
// consecutive columns and 4 rows (m0 + l / 4, r0 + l % 4): with row strides
// of 4 mod 32 words the 32 stores fall in 32 banks, and each global read is a
// full 32-byte sector.
template <int D>
__global__ void __launch_bounds__(THREADS) vla_seg_combine_kernel(const CombineParams cp) {
    constexpr int R = D / 16, DS = D + 4, FS = OT + 4;
    static_assert(DS % 32 == 4 && FS % 32 == 4, "transposing stores across all banks");
    extern __shared__ __align__(16) float sh[];
    float* gT = sh;  // S_L transposed: gT[m * DS + i] = S_L[i][m]
    const int bh = blockIdx.x, tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const float* G0 = cp.G0 + (size_t)bh * D * D;
    {
        // all of a thread's loads in flight before its stores
        constexpr int NBK = (D / 4) * (D / 8) / (THREADS / 32);
        static_assert((D / 4) * (D / 8) % (THREADS / 32) == 0, "whole blocks per warp");
        float v[NBK];
#pragma unroll
        for (int j = 0; j < NBK; ++j) {
            const int blk = warp + (THREADS / 32) * j;
            v[j] = G0[((blk % (D / 4)) * 4 + lane % 4) * D + (blk / (D / 4)) * 8 + lane / 4];
        }
#pragma unroll
        for (int j = 0; j < NBK; ++j) {
            const int blk = warp + (THREADS / 32) * j;
            gT[((blk / (D / 4)) * 8 + lane / 4) * DS + (blk % (D / 4)) * 4 + lane % 4] = v[j];
        }
    }
    const int ntile = (cp.L1 + OT - 1) / OT;
    if ((int)blockIdx.y == ntile) {
        // rows ty R .., columns tx R .. of S_L Pi_T; Pi_T's rows read through the read-only path
        __syncthreads();
        const float* F1 = cp.F1 + (size_t)bh * D * D;
        const int ty = tid / 16, tx = tid % 16;
        float acc[R][R];
#pragma unroll
        for (int a = 0; a < R; ++a)
#pragma unroll
            for (int b = 0; b < R; ++b) acc[a][b] = 0.f;
#pragma unroll 2
        for (int mm = 0; mm < D; ++mm) {
            float ga[R], fb[R];
            lds_run<R>(gT + mm * DS + ty * R, ga);
#pragma unroll
            for (int h = 0; h < R / 2; ++h) {
                const float2 v = __ldg(reinterpret_cast<const float2*>(F1 + mm * D + tx * R) + h);
                fb[2 * h] = v.x, fb[2 * h + 1] = v.y;
            }
#pragma unroll
            for (int a = 0; a < R; ++a)
#pragma unroll
                for (int b = 0; b < R; ++b) acc[a][b] = fmaf(ga[a], fb[b], acc[a][b]);
        }
        const float* G1 = cp.G1 + (size_t)bh * D * D;
        float* So = cp.S_out + (size_t)bh * D * D;
#pragma unroll
        for (int a = 0; a < R; ++a)
#pragma unroll
            for (int b = 0; b < R; ++b) {
                const int e = (ty * R + a) * D + tx * R + b;
                So[e] = G1[e] + acc[a][b];
            }
        return;
    }
    float* fT = gT + D * DS;  // this tile's Pi_t phi_t / den_t, transposed: fT[m * FS + t]
    const int tb = blockIdx.y * OT, nt = min(OT, cp.L1 - tb);
    const float* F = cp.fphi + ((size_t)bh * cp.L1 + tb) * D;
    {
        constexpr int NBK = (OT / 4) * (D / 8) / (THREADS / 32);
        static_assert((OT / 4) * (D / 8) % (THREADS / 32) == 0, "whole blocks per warp");
        float v[NBK];
#pragma unroll
        for (int j = 0; j < NBK; ++j) {
            const int blk = warp + (THREADS / 32) * j;
            const int t = (blk % (OT / 4)) * 4 + lane % 4, mm = (blk / (OT / 4)) * 8 + lane / 4;
            v[j] = t < nt ? F[(size_t)t * D + mm] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < NBK; ++j) {
            const int blk = warp + (THREADS / 32) * j;
            fT[((blk / (OT / 4)) * 8 + lane / 4) * FS + (blk % (OT / 4)) * 4 + lane % 4] = v[j];
        }
    }
    __syncthreads();
    const int tt = tid / 16, io = tid % 16;
    float acc[4][R];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < R; ++b) acc[a][b] = 0.f;
#pragma unroll 2
    for (int mm = 0; mm < D; ++mm) {
        const float4 f4 = *reinterpret_cast<const float4*>(fT + mm * FS + 4 * tt);
        const float fa[4] = {f4.x, f4.y, f4.z, f4.w};
        float gb[R];
        lds_run<R>(gT + mm * DS + io * R, gb);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < R; ++b) acc[a][b] = fmaf(gb[b], fa[a], acc[a][b]);
    }
    float* o = cp.o + (size_t)bh * cp.o_stride + (size_t)tb * D;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int t = 4 * tt + a;
        if (t < nt) {
#pragma unroll
            for (int b = 0; b < R; ++b) o[(size_t)t * D + io * R + b] += acc[a][b];
        }
    }
}

// dynamic shared memory of vla_seg_combine_kernel<D>
template <int D>
constexpr int combine_smem() {
    return (D * (D + 4) + D * (OT + 4)) * 4;
}

}  // namespace seg
