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
constexpr int NSPLIT = 16;  // CTAs per head that share the prefix sums
constexpr int TILE = 128;   // tokens staged per step of the prefix sums

// Per (head, split): the partial sums of u^_s u^_s^T and phi(k_s) over its
// share of tokens [0, L) (the u^ sums are skipped for the fixed-A variant).
struct PrefixParams {
    const void* u;
    const void* k;
    size_t in_stride;  // elements between heads' rows
    int L;             // tokens of the first segment
    int fixed_a;
    float* dpart;      // [heads][NSPLIT][D][D]
    float* zpart;      // [heads][NSPLIT][D]
};

// 8 consecutive input elements (16-byte aligned for bf16, 32 for fp32) as float
template <typename TIn>
__device__ __forceinline__ void ld8_in(const TIn* p, float (&x)[8]);
template <>
__device__ __forceinline__ void ld8_in<float>(const float* p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
template <>
__device__ __forceinline__ void ld8_in<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <int D, typename TIn>
__global__ void __launch_bounds__(THREADS) vla_seg_prefix_kernel(const PrefixParams pp) {
    constexpr int R = D / 16;             // each thread owns an R x R block of the D x D sum
    constexpr int US = D + 4;             // row stride of the staged rows (16-byte rows)
    constexpr int NC = D / 8;             // 8-element chunks per row
    constexpr int NG = THREADS / NC;      // token groups of the staging map
    static_assert(D % 16 == 0, "16 x 16 thread grid");
    extern __shared__ __align__(16) float psh[];
    float* ur = psh;                      // TILE x US: u rows
    float* inv2 = ur + TILE * US;         // TILE: 1 / max(||u||, 1e-12)^2
    float* zs = inv2 + TILE;              // NG x D: phi(k) sums per token group
    const int bh = blockIdx.x / NSPLIT, sp = blockIdx.x % NSPLIT;
    const int per = (pp.L + NSPLIT - 1) / NSPLIT;
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
            for (int t = g; t < nt; t += NG) {
                float x[8], kx[8];
                if (!pp.fixed_a) ld8_in<TIn>(gu + (size_t)(tb + t) * D + 8 * j8, x);
                ld8_in<TIn>(gk + (size_t)(tb + t) * D + 8 * j8, kx);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    ur[t * US + 8 * j8 + e] = pp.fixed_a ? 0.f : x[e];
                    zk[e] += phi(kx[e]);
                }
            }
        }
        __syncthreads();
        if (!pp.fixed_a) {
            // warp w: 1 / max(||u||, 1e-12)^2 of tokens w, w + 8, ...
            for (int t = warp; t < nt; t += THREADS / 32) {
                float s2 = 0.f;
                for (int j = lane; j < D; j += 32) s2 = fmaf(ur[t * US + j], ur[t * US + j], s2);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                if (lane == 0) inv2[t] = 1.f / fmaxf(s2, 1e-24f);
            }
            __syncthreads();
            for (int t = 0; t < nt; ++t) {
                const float w = inv2[t];
                float ra[R], rb[R];
#pragma unroll
                for (int a = 0; a < R; ++a) {
                    ra[a] = ur[t * US + ty * R + a] * w;
                    rb[a] = ur[t * US + tx * R + a];
                }
#pragma unroll
                for (int a = 0; a < R; ++a)
#pragma unroll
                    for (int b = 0; b < R; ++b) acc[a][b] = fmaf(ra[a], rb[b], acc[a][b]);
            }
        }
    }
    // the token groups' phi(k) sums, added in a fixed order
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
    return (TILE * (D + 4) + TILE + (THREADS / (D / 8)) * D) * 4;
}

// Per head: z^key_L, and A_L = (A_0^-1 + sum_s u^_s u^_s^T)^-1 by in-place
// Gauss-Jordan elimination (no pivoting: the matrices are symmetric positive
// definite), symmetrised; A_L = A_0 for the fixed-A variant. Block 0 also
// writes the identity that the second half's transition starts from.
struct InvertParams {
    const float* dpart;
    const float* zpart;
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
// definite). Thread tid holds elements e = tid + THREADS r (row e / D, column
// e % D) in x[r]. Step k updates them from pivot column and row k, read from
// one of two shared buffers (cr[k & 1]), and the owners of column and row
// k + 1 write those into the other, so one barrier separates the steps.
// cr: 4 x D floats. Returns false if a pivot was not positive.
template <int D>
__device__ __forceinline__ bool gauss_jordan(float (&x)[D * D / THREADS], float* cr) {
    constexpr int NE = D * D / THREADS;
    static_assert(D * D % THREADS == 0, "whole elements per thread");
    const int tid = threadIdx.x;
    bool ok = true;
    __syncthreads();  // earlier readers of cr are done
#pragma unroll
    for (int r = 0; r < NE; ++r) {
        const int e = tid + THREADS * r, i = e / D, j = e - i * D;
        if (j == 0) cr[i] = x[r];      // column 0
        if (i == 0) cr[D + j] = x[r];  // row 0
    }
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < D; ++k) {
        const float* col = cr + (k & 1) * 2 * D;
        const float* row = col + D;
        float* ncol = cr + ((k + 1) & 1) * 2 * D;
        float* nrow = ncol + D;
        const float piv = row[k];
        if (!(piv > 0.f)) ok = false;
        const float rp = 1.f / piv;
#pragma unroll
        for (int r = 0; r < NE; ++r) {
            const int e = tid + THREADS * r, i = e / D, j = e - i * D;
            float v;
            if (i == k)
                v = (j == k) ? rp : row[j] * rp;
            else
                v = (j == k) ? -col[i] * rp : fmaf(-col[i] * rp, row[j], x[r]);
            x[r] = v;
            if (j == k + 1) ncol[i] = v;
            if (i == k + 1) nrow[j] = v;
        }
        __syncthreads();
    }
    return ok;
}

template <int D>
__global__ void __launch_bounds__(THREADS) vla_seg_invert_kernel(const InvertParams ip) {
    constexpr int NE = D * D / THREADS, MS = D + 1;
    extern __shared__ __align__(16) float sh[];
    float* m = sh;           // D x MS: the inverse, for the symmetrised copy
    float* cr = m + D * MS;  // 4 x D: pivot columns and rows
    const int bh = blockIdx.x, tid = threadIdx.x;
    if (bh == 0)
        for (int e = tid; e < D * D; e += THREADS) ip.ident[e] = (e / D == e % D) ? 1.f : 0.f;
    if (tid < D) {
        float z = ip.zk0 ? ip.zk0[(size_t)bh * D + tid] : 0.f;
        for (int sp = 0; sp < NSPLIT; ++sp) z += ip.zpart[((size_t)bh * NSPLIT + sp) * D + tid];
        ip.zk_cut[(size_t)bh * D + tid] = z;
    }
    float* out = ip.A_cut + (size_t)bh * D * D;
    const float* A0 = ip.A0 ? ip.A0 + (size_t)bh * D * D : nullptr;
    if (ip.fixed_a) {
        for (int e = tid; e < D * D; e += THREADS)
            out[e] = A0 ? A0[e] : ((e / D == e % D) ? ip.inv_lambda0 : 0.f);
        return;
    }
    float x[NE];
    bool ok = true;
    if (A0) {
#pragma unroll
        for (int r = 0; r < NE; ++r) x[r] = A0[tid + THREADS * r];
        ok = gauss_jordan<D>(x, cr);  // A_0^-1
    } else {
#pragma unroll
        for (int r = 0; r < NE; ++r) {
            const int e = tid + THREADS * r;
            x[r] = (e / D == e % D) ? ip.lambda0 : 0.f;
        }
    }
#pragma unroll
    for (int r = 0; r < NE; ++r) {
        const int e = tid + THREADS * r;
        float a = 0.f;
        for (int sp = 0; sp < NSPLIT; ++sp) a += ip.dpart[((size_t)bh * NSPLIT + sp) * D * D + e];
        x[r] += a;
    }
    ok = gauss_jordan<D>(x, cr) && ok;
#pragma unroll
    for (int r = 0; r < NE; ++r) {
        const int e = tid + THREADS * r, i = e / D, j = e - i * D;
        m[i * MS + j] = x[r];
    }
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

// Each thread forms a 4 x (D / 16) block: tokens 4 (tid / 16) .. + 3 and
// outputs tid % 16 + 16 r (or, for S_T, rows and columns of an R x R block),
// so that each pair of shared-memory loads feeds several fused multiply-adds.
template <int D>
__global__ void __launch_bounds__(THREADS) vla_seg_combine_kernel(const CombineParams cp) {
    constexpr int MS = D + 1, R = D / 16;
    extern __shared__ __align__(16) float sh[];
    float* g0 = sh;  // S_L, row stride MS
    const int bh = blockIdx.x, tid = threadIdx.x;
    const float* G0 = cp.G0 + (size_t)bh * D * D;
    for (int e = tid; e < D * D; e += THREADS) g0[(e / D) * MS + e % D] = G0[e];
    const int ntile = (cp.L1 + OT - 1) / OT;
    if ((int)blockIdx.y == ntile) {
        float* f1 = g0 + D * MS;  // Pi_T
        const float* F1 = cp.F1 + (size_t)bh * D * D;
        for (int e = tid; e < D * D; e += THREADS) f1[(e / D) * MS + e % D] = F1[e];
        __syncthreads();
        const int ty = tid / 16, tx = tid % 16;  // rows ty + 16 a, columns tx + 16 b
        float acc[R][R];
#pragma unroll
        for (int a = 0; a < R; ++a)
#pragma unroll
            for (int b = 0; b < R; ++b) acc[a][b] = 0.f;
#pragma unroll 4
        for (int m = 0; m < D; ++m) {
            float ga[R], fb[R];
#pragma unroll
            for (int a = 0; a < R; ++a) {
                ga[a] = g0[(ty + 16 * a) * MS + m];
                fb[a] = f1[m * MS + tx + 16 * a];
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
                const int e = (ty + 16 * a) * D + tx + 16 * b;
                So[e] = G1[e] + acc[a][b];
            }
        return;
    }
    float* fp = g0 + D * MS;  // OT rows of Pi_t phi_t / den_t, row stride D + 4
    constexpr int FS = D + 4;
    const int tb = blockIdx.y * OT, nt = min(OT, cp.L1 - tb);
    const float* F = cp.fphi + ((size_t)bh * cp.L1 + tb) * D;
    for (int e = tid; e < OT * D; e += THREADS) fp[(e / D) * FS + e % D] = e < nt * D ? F[e] : 0.f;
    __syncthreads();
    const int tt = tid / 16, io = tid % 16;
    float acc[4][R];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < R; ++b) acc[a][b] = 0.f;
#pragma unroll 4
    for (int m = 0; m < D; ++m) {
        float fa[4], gb[R];
#pragma unroll
        for (int a = 0; a < 4; ++a) fa[a] = fp[(4 * tt + a) * FS + m];
#pragma unroll
        for (int b = 0; b < R; ++b) gb[b] = g0[(io + 16 * b) * MS + m];
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
            for (int b = 0; b < R; ++b) o[(size_t)t * D + io + 16 * b] += acc[a][b];
        }
    }
}

// dynamic shared memory of vla_seg_combine_kernel<D>
template <int D>
constexpr int combine_smem() {
    return (D * (D + 1) + (OT * (D + 4) > D * (D + 1) ? OT * (D + 4) : D * (D + 1))) * 4;
}

}  // namespace seg
