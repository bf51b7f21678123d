// vla_forward.cu -- host side of the GB300 (sm_103a) library for the
// Variational Linear Attention recurrence ("Variational Linear Attention",
// arXiv 2605.11196, §3.3 eq. 9-11): the launch code of every kernel, the
// choice between them, the fork and join of the segmented path, and the
// C ABI of include/vla.h. The kernels are in the headers included below,
// inside namespace vla: vla_fused.cuh (the per-token kernel and the
// parameter block), vla_tc.cuh, vla_tc2.cuh, vla_tc3.cuh (the chunked
// tensor-core kernels), vla_seg.cuh (the segmented path's prefix sums,
// inverse and combine), vla_backward.cuh, vla_backward_split.cuh (the
// reverse sweeps) and vla_decode.cuh (the register-resident decode kernel).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <algorithm>
#include <mutex>

#include "vla.h"
#include "vla_device.cuh"
#include "vla_internal.h"

namespace vla {

#include "vla_fused.cuh"
#include "vla_tc.cuh"
#include "vla_tc2.cuh"
#include "vla_tc3.cuh"
#include "vla_seg.cuh"
#include "vla_backward.cuh"
#include "vla_backward_split.cuh"
#include "vla_decode.cuh"

}  // namespace vla

// ===========================================================================
// C ABI
// ===========================================================================
namespace {

constexpr size_t kWorkspaceBytes = 256;
constexpr unsigned kDefaultWaitUs = 2000000u;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
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

template <int D, typename TIn>
vla_status launch_tc(const vla::Params& p, int BH, cudaStream_t s) {
    using LY = vla::tc::Lay<D, TIn>;
    auto kern = vla::vla_tc_kernel<D, TIn>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::SMEM) != cudaSuccess)
        return VLA_ERR_CUDA;
    kern<<<BH, vla::tc::THREADS, LY::SMEM, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

// the chunked recurrence on a cluster of two CTAs per head (rank 0 the A-pass,
// rank 1 the S-pass)
template <int D, typename TIn>
vla_status launch_tc2(const vla::Params& p, int BH, cudaStream_t s) {
    using LY = vla::tc2::Lay2<D, TIn>;
    auto kern = vla::vla_tc2_kernel<D, TIn>;
    if ((long long)BH * 2 > 2147483647LL) return VLA_ERR_INVALID_ARG;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::SMEM_LAUNCH) != cudaSuccess)
        return VLA_ERR_CUDA;
    kern<<<2 * BH, vla::tc2::THREADS, LY::SMEM_LAUNCH, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

// the chunked recurrence on a cluster of 1 + NS CTAs per head: rank 0 the
// A-pass, ranks 1..NS the rows of S split in NS equal blocks
template <int D, typename TIn, int NS>
vla_status launch_tc3(const vla::Params& p, int BH, cudaStream_t s) {
    using LY = vla::tc3::Lay3<D, TIn, NS>;
    auto kern = vla::vla_tc3_kernel<D, TIn, NS>;
    if ((long long)BH * (1 + NS) > 2147483647LL) return VLA_ERR_INVALID_ARG;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::SMEM_LAUNCH) != cudaSuccess)
        return VLA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((1 + NS) * BH), 1, 1);
    cfg.blockDim = dim3(vla::tc3::THREADS, 1, 1);
    cfg.dynamicSmemBytes = LY::SMEM_LAUNCH;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1 + NS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return VLA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

template <int D, typename TIn>
vla_status launch_dec(const vla::Params& p, int BH, bool fixed_a, cudaStream_t s) {
    using DL = vla::dec::DLay<D, TIn>;
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0)
        return VLA_ERR_CUDA;
    const int grid = BH < n_sm ? BH : n_sm;  // one persistent CTA per SM
    // bulk copies of the carried state need 16-byte aligned state pointers
    const int bulk = ((!p.S0 || aligned16(p.S0)) && (!p.A0 || aligned16(p.A0)) && (!p.zk0 || aligned16(p.zk0))) ? 1 : 0;
    auto kern = fixed_a ? vla::dec::vla_decode_kernel<D, TIn, true> : vla::dec::vla_decode_kernel<D, TIn, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DL::SMEM) != cudaSuccess)
        return VLA_ERR_CUDA;
    kern<<<grid, DL::THREADS, DL::SMEM, s>>>(p, BH, bulk);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

// sequences up to this length go to the decode kernel under VLA_ALGO_AUTO
constexpr int kDecodeMaxT = 4;
// VLA_ALGO_AUTO takes the segmented path from this length on (d <= 96, heads
// that fit on the SMs three CTAs each, and a workspace that holds its buffers)
constexpr int kSegMinT = 1024;

// SMs of the current device (0 if the query fails)
int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

// The segmented path's buffers in the workspace, after the status record:
// the prefix partial sums, the state at the cut (A, z^key), the identity the
// transition starts from, the three groups' final states (the first half's
// S = S_L; the second half's G_T and Pi_T; scratch for the state outputs the
// combine does not read), Pi_t phi_t / den_t for the second half's tokens and
// the zero rows that the transition reads as its v.
struct SegPlan {
    int L0 = 0, L1 = 0;
    size_t dpart = 0, zpart = 0, A_cut = 0, zk_cut = 0, ident = 0, G0 = 0, A_s0 = 0, zk_s0 = 0, G1 = 0, F1 = 0,
           A_s2 = 0, zk_s2 = 0, fphi = 0, vzero = 0, total = 0;
};

// Tokens of the first segment. The second half's two runs start only after
// the prefix sums and the inverse at the cut, the first half at once, so the
// cut sits past T / 2 by about (prefix + inverse time) / (2 x the chunked
// kernel's time per token): delta = alpha_d T + gamma_d tokens, fitted to the
// measured best cut on GB300 (T = 4096 and 16384; d = 64: 0.545 T and 0.52 T,
// d = 96: 0.56 T at T = 4096). A multiple of 16, one chunk at least each side.
int seg_cut(int T, int d) {
    const double alpha = d == 96 ? 0.0218 : d == 64 ? 0.0117 : 0.003;
    const double gamma = d == 96 ? 157.0 : d == 64 ? 136.0 : 100.0;
    const int L0 = (int)(0.5 * T + alpha * T + gamma) / 16 * 16;
    return std::max(16, std::min(L0, (T - 1) / 16 * 16));
}

bool seg_plan(long long BH, int T, int d, SegPlan* sp) {
    if (BH <= 0 || T < 32 || (d != 32 && d != 64 && d != 96)) return false;
    sp->L0 = seg_cut(T, d);
    sp->L1 = T - sp->L0;
    const size_t bh = (size_t)BH, dd = (size_t)d * d, dv = (size_t)d;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    size_t off = al(kWorkspaceBytes);
    auto take = [&](size_t floats) {
        const size_t at = off;
        off += al(floats * 4);
        return at;
    };
    sp->dpart = take(bh * vla::seg::NSPLIT * dd);
    sp->zpart = take(bh * vla::seg::NSPLIT * dv);
    sp->A_cut = take(bh * dd);
    sp->zk_cut = take(bh * dv);
    sp->ident = take(dd);
    sp->G0 = take(bh * dd);
    sp->A_s0 = take(bh * dd);
    sp->zk_s0 = take(bh * dv);
    sp->G1 = take(bh * dd);
    sp->F1 = take(bh * dd);
    sp->A_s2 = take(bh * dd);
    sp->zk_s2 = take(bh * dv);
    sp->fphi = take(bh * (size_t)sp->L1 * dv);
    sp->vzero = take((size_t)sp->L1 * dv);
    sp->total = off;
    return true;
}

// the segmented path would serve these sizes under VLA_ALGO_AUTO on a device with n_sm SMs
bool seg_auto(long long BH, int T, int d, int n_sm) { return d <= 96 && T >= kSegMinT && 3LL * BH <= (long long)n_sm; }

// Side streams and events of the segmented path, one set per host thread and
// device, created on the thread's first call there and destroyed when the
// thread exits. Per thread, so that a stream capture on one thread (which
// takes the side streams into its graph until the capture ends) leaves the
// calls of other threads alone, and calls from different threads never share
// an event in flight; calls of one thread enqueue one after another.
constexpr int kSegMaxDevices = 64;
struct SegFork {
    bool ready = false;
    cudaStream_t side[2] = {};
    cudaEvent_t start = nullptr, cut = nullptr, done[2] = {};
    ~SegFork() {
        if (!ready) return;
        // work still queued on the side streams completes before they are released
        cudaStreamDestroy(side[0]);
        cudaStreamDestroy(side[1]);
        cudaEventDestroy(start);
        cudaEventDestroy(cut);
        cudaEventDestroy(done[0]);
        cudaEventDestroy(done[1]);
    }
};
thread_local SegFork g_seg[kSegMaxDevices];

vla_status seg_fork_for(SegFork** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSegMaxDevices) return VLA_ERR_CUDA;
    SegFork& F = g_seg[dev];
    if (!F.ready) {
        const unsigned ef = cudaEventDisableTiming;
        SegFork n;
        const bool ok = cudaStreamCreateWithFlags(&n.side[0], cudaStreamNonBlocking) == cudaSuccess &&
                        cudaStreamCreateWithFlags(&n.side[1], cudaStreamNonBlocking) == cudaSuccess &&
                        cudaEventCreateWithFlags(&n.start, ef) == cudaSuccess &&
                        cudaEventCreateWithFlags(&n.cut, ef) == cudaSuccess &&
                        cudaEventCreateWithFlags(&n.done[0], ef) == cudaSuccess &&
                        cudaEventCreateWithFlags(&n.done[1], ef) == cudaSuccess;
        if (!ok) {
            // release what was created (nullptr handles are skipped)
            for (cudaStream_t x : n.side)
                if (x) cudaStreamDestroy(x);
            for (cudaEvent_t x : {n.start, n.cut, n.done[0], n.done[1]})
                if (x) cudaEventDestroy(x);
            return VLA_ERR_CUDA;
        }
        F.side[0] = n.side[0];
        F.side[1] = n.side[1];
        F.start = n.start;
        F.cut = n.cut;
        F.done[0] = n.done[0];
        F.done[1] = n.done[1];
        F.ready = true;
    }
    *out = &F;
    return VLA_OK;
}

// The two-segment form (vla_seg.cuh) as a fork and join on `s`: the first
// half starts at once on a side stream; the prefix sums and the inverse at
// the cut run on `s`, then the second half's transition on the other side
// stream and its run from S = 0 on `s`; `s` waits for both side streams and
// runs the combine. Every launch is the single-CTA chunked kernel or a small
// kernel of vla_seg.cuh.
template <int D, typename TIn>
vla_status launch_seg(const vla::Params& p, int BH, unsigned char* ws, const SegPlan& sp, cudaStream_t s) {
    using LY = vla::tc::Lay<D, TIn>;
    const int T = p.T;
    auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const size_t hs = (size_t)T * D;
    auto tk = vla::vla_tc_kernel<D, TIn>;
    auto pk = vla::seg::vla_seg_prefix_kernel<D, TIn>;
    auto ik = vla::seg::vla_seg_invert_kernel<D>;
    auto ck = vla::seg::vla_seg_combine_kernel<D>;
    constexpr int p_smem = vla::seg::prefix_smem<D>();
    constexpr int i_smem = (D * (D + 1) + 4 * D) * 4;
    constexpr int c_smem = vla::seg::combine_smem<D>();
    if (cudaFuncSetAttribute(tk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, p_smem) != cudaSuccess ||
        cudaFuncSetAttribute(ik, cudaFuncAttributeMaxDynamicSharedMemorySize, i_smem) != cudaSuccess ||
        cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, c_smem) != cudaSuccess)
        return VLA_ERR_CUDA;
    // the three runs of the chunked kernel
    vla::Params g0 = p;  // first half, from the given state
    g0.T = sp.L0;
    g0.in_stride = hs;
    g0.S_out = F(sp.G0);
    g0.A_out = F(sp.A_s0);
    g0.zk_out = F(sp.zk_s0);
    vla::Params g1 = p;  // second half from S = 0, A and z^key at the cut
    g1.T = sp.L1;
    g1.in_stride = hs;
    g1.q = static_cast<const TIn*>(p.q) + (size_t)sp.L0 * D;
    g1.k = static_cast<const TIn*>(p.k) + (size_t)sp.L0 * D;
    g1.v = static_cast<const TIn*>(p.v) + (size_t)sp.L0 * D;
    g1.u = static_cast<const TIn*>(p.u) + (size_t)sp.L0 * D;
    g1.o = p.o + (size_t)sp.L0 * D;
    g1.S0 = nullptr;
    g1.A0 = F(sp.A_cut);
    g1.zk0 = F(sp.zk_cut);
    g1.S_out = F(sp.G1);
    vla::Params g2 = g1;  // the transition: second half from S = I with v = 0 (zero rows shared by every head)
    g2.v = ws + sp.vzero;
    g2.v_shared = 1;
    g2.S0 = F(sp.ident);
    g2.s0_shared = 1;
    g2.o = F(sp.fphi);
    g2.o_stride = (size_t)sp.L1 * D;
    g2.S_out = F(sp.F1);
    g2.A_out = F(sp.A_s2);
    g2.zk_out = F(sp.zk_s2);
    vla::seg::PrefixParams pp{};
    pp.u = p.u;
    pp.k = p.k;
    pp.in_stride = hs;
    pp.L = sp.L0;
    pp.fixed_a = p.fixed_a;
    // one wave of prefix CTAs beside the first half's BH CTAs, 16 tokens at least per CTA
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, pk, vla::seg::THREADS, p_smem) != cudaSuccess) return VLA_ERR_CUDA;
    const int free_slots = std::max(1, sm_count() - BH) * std::max(occ, 1);
    pp.nsplit = std::max(1, std::min({vla::seg::NSPLIT, free_slots / BH, sp.L0 / 16}));
    pp.dpart = F(sp.dpart);
    pp.zpart = F(sp.zpart);
    vla::seg::InvertParams ip{};
    ip.dpart = F(sp.dpart);
    ip.zpart = F(sp.zpart);
    ip.nsplit = pp.nsplit;
    ip.A0 = p.A0;
    ip.zk0 = p.zk0;
    ip.lambda0 = 1.0f / p.inv_lambda0;
    ip.inv_lambda0 = p.inv_lambda0;
    ip.fixed_a = p.fixed_a;
    ip.A_cut = F(sp.A_cut);
    ip.zk_cut = F(sp.zk_cut);
    ip.ident = F(sp.ident);
    ip.status = p.status;
    vla::seg::CombineParams cp{};
    cp.G0 = F(sp.G0);
    cp.F1 = F(sp.F1);
    cp.G1 = F(sp.G1);
    cp.fphi = F(sp.fphi);
    cp.o = p.o + (size_t)sp.L0 * D;
    cp.o_stride = p.o_stride;
    cp.L1 = sp.L1;
    cp.S_out = p.S_out;
    const int ntile = (sp.L1 + vla::seg::OT - 1) / vla::seg::OT;

    SegFork* fk = nullptr;
    if (seg_fork_for(&fk) != VLA_OK) return VLA_ERR_CUDA;
    bool ok = cudaEventRecord(fk->start, s) == cudaSuccess &&
              cudaStreamWaitEvent(fk->side[0], fk->start, 0) == cudaSuccess &&
              cudaMemsetAsync(ws + sp.vzero, 0, (size_t)sp.L1 * D * sizeof(TIn), s) == cudaSuccess;
    if (ok) {
        tk<<<BH, vla::tc::THREADS, LY::SMEM, fk->side[0]>>>(g0);
        ok = cudaGetLastError() == cudaSuccess;
    }
    // the side stream joins `s` below whatever happened, so that nothing of
    // this call is left running unordered with the caller's later work
    const bool side0 = ok;
    if (ok) {
        pk<<<BH * pp.nsplit, vla::seg::THREADS, p_smem, s>>>(pp);
        ik<<<BH, vla::seg::THREADS, i_smem, s>>>(ip);
        ok = cudaGetLastError() == cudaSuccess && cudaEventRecord(fk->cut, s) == cudaSuccess &&
             cudaStreamWaitEvent(fk->side[1], fk->cut, 0) == cudaSuccess;
    }
    const bool side1 = ok;
    if (ok) {
        tk<<<BH, vla::tc::THREADS, LY::SMEM, fk->side[1]>>>(g2);
        tk<<<BH, vla::tc::THREADS, LY::SMEM, s>>>(g1);
        ok = cudaGetLastError() == cudaSuccess;
    }
    if (side0) ok = cudaEventRecord(fk->done[0], fk->side[0]) == cudaSuccess &&
                    cudaStreamWaitEvent(s, fk->done[0], 0) == cudaSuccess && ok;
    if (side1) ok = cudaEventRecord(fk->done[1], fk->side[1]) == cudaSuccess &&
                    cudaStreamWaitEvent(s, fk->done[1], 0) == cudaSuccess && ok;
    if (!ok) return VLA_ERR_CUDA;
    ck<<<dim3(BH, ntile + 1), vla::seg::THREADS, c_smem, s>>>(cp);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

template <typename TIn>
vla_status launch_seg_d(int d, const vla::Params& p, int BH, unsigned char* ws, const SegPlan& sp, cudaStream_t s) {
    switch (d) {
        case 32: return launch_seg<32, TIn>(p, BH, ws, sp, s);
        case 64: return launch_seg<64, TIn>(p, BH, ws, sp, s);
        case 96: return launch_seg<96, TIn>(p, BH, ws, sp, s);
        default: return VLA_ERR_UNSUPPORTED;
    }
}

// algo: VLA_ALGO_AUTO picks the decode kernel for short sequences; for
// d = 96 and 128 the row-split cluster kernel (3 CTAs per head) when all of
// its clusters fit on the SMs at once, measured faster there; otherwise the
// single-CTA chunked tensor-core kernel for d <= 96 and the cluster-pair
// chunked kernel for d = 128.
template <typename TIn>
vla_status launch_d(int d, int algo, bool fixed_a, const vla::Params& p, int BH, cudaStream_t s) {
    if (algo == VLA_ALGO_DECODE || (algo == VLA_ALGO_AUTO && p.T <= kDecodeMaxT)) {
        switch (d) {
            case 32: return launch_dec<32, TIn>(p, BH, fixed_a, s);
            case 64: return launch_dec<64, TIn>(p, BH, fixed_a, s);
            case 96: return launch_dec<96, TIn>(p, BH, fixed_a, s);
            case 128: return launch_dec<128, TIn>(p, BH, fixed_a, s);
            default: return VLA_ERR_UNSUPPORTED;
        }
    }
    if (fixed_a && algo == VLA_ALGO_PER_TOKEN) return VLA_ERR_UNSUPPORTED;
    if (algo == VLA_ALGO_AUTO && d >= 96 && 3LL * BH <= (long long)sm_count()) algo = VLA_ALGO_CHUNKED_ROWS;
    if (algo == VLA_ALGO_CHUNKED_ROWS) {
        // S's rows on one CTA up to d = 64, on two CTAs above
        switch (d) {
            case 32: return launch_tc3<32, TIn, 1>(p, BH, s);
            case 64: return launch_tc3<64, TIn, 1>(p, BH, s);
            case 96: return launch_tc3<96, TIn, 2>(p, BH, s);
            case 128: return launch_tc3<128, TIn, 2>(p, BH, s);
            default: return VLA_ERR_UNSUPPORTED;
        }
    }
    if (algo == VLA_ALGO_CHUNKED_PAIR || (algo == VLA_ALGO_AUTO && d == 128)) {
        switch (d) {
            case 32: return launch_tc2<32, TIn>(p, BH, s);
            case 64: return launch_tc2<64, TIn>(p, BH, s);
            case 96: return launch_tc2<96, TIn>(p, BH, s);
            case 128: return launch_tc2<128, TIn>(p, BH, s);
            default: return VLA_ERR_UNSUPPORTED;
        }
    }
    const bool chunked = algo == VLA_ALGO_CHUNKED || (algo == VLA_ALGO_AUTO && d <= 96);
    if (chunked) {
        switch (d) {
            case 32: return launch_tc<32, TIn>(p, BH, s);
            case 64: return launch_tc<64, TIn>(p, BH, s);
            case 96: return launch_tc<96, TIn>(p, BH, s);
            default: return VLA_ERR_UNSUPPORTED;
        }
    }
    switch (d) {
        case 32: return launch_fused<32, TIn>(p, BH, s);
        case 64: return launch_fused<64, TIn>(p, BH, s);
        case 96: return launch_fused<96, TIn>(p, BH, s);
        case 128: return launch_fused<128, TIn>(p, BH, s);
        default: return VLA_ERR_UNSUPPORTED;
    }
}

template <typename TIn>
void launch_la(int d, const TIn* k, const TIn* v, int T, float* S, int BH, cudaStream_t s) {
    switch (d) {
        case 32: vla::la_state_kernel<32, TIn><<<BH, vla::LA_THREADS, 0, s>>>(k, v, T, S); break;
        case 64: vla::la_state_kernel<64, TIn><<<BH, vla::LA_THREADS, 0, s>>>(k, v, T, S); break;
        case 96: vla::la_state_kernel<96, TIn><<<BH, vla::LA_THREADS, 0, s>>>(k, v, T, S); break;
        default: vla::la_state_kernel<128, TIn><<<BH, vla::LA_THREADS, 0, s>>>(k, v, T, S); break;
    }
}

}  // namespace

extern "C" {

size_t vla_workspace_bytes(int B, int H, int T, int d) {
    if (B < 0 || H < 0 || T < 0) return 0;
    if (d != 32 && d != 64 && d != 96 && d != 128) return 0;
    const long long BH = (long long)B * H;
    if (BH > 2147483647LL) return 0;
    // the segmented path's buffers, where VLA_ALGO_AUTO would take it (the
    // current device's SM count; 152 when no device answers)
    int n_sm = sm_count();
    if (n_sm <= 0) n_sm = 152;
    SegPlan sp;
    if (seg_auto(BH, T, d, n_sm) && seg_plan(BH, T, d, &sp)) return sp.total;
    return kWorkspaceBytes;
}

size_t vla_workspace_bytes_ex(int B, int H, int T, int d, int algo) {
    if (algo == VLA_ALGO_AUTO) return vla_workspace_bytes(B, H, T, d);
    if (algo < VLA_ALGO_AUTO || algo > VLA_ALGO_SEGMENTED) return 0;
    if (vla_workspace_bytes(B, H, T, d) == 0) return 0;
    if (algo != VLA_ALGO_SEGMENTED) return kWorkspaceBytes;
    SegPlan sp;
    return seg_plan((long long)B * H, T, d, &sp) ? sp.total : 0;
}

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
    return vla_impl::forward(q, k, v, u, dtype, B, H, T, d, lambda0, eps, S0, A0, zk0, o, S_out, A_out, zk_out,
                             workspace, workspace_bytes, stream, opts, 0);
}

}  // extern "C"

size_t vla_impl::status_bytes() { return kWorkspaceBytes; }

vla_status vla_impl::forward(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B,
                             int H, int T, int d, float lambda0, float eps, const float* S0, const float* A0,
                             const float* zk0, float* o, float* S_out, float* A_out, float* zk_out, void* workspace,
                             size_t workspace_bytes, void* stream, const vla_options* opts, size_t o_head_stride) {
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
    if (o_head_stride == 0) o_head_stride = (size_t)T * d;
    if (o_head_stride < (size_t)T * d || (o_head_stride * sizeof(float)) % 16 != 0) return VLA_ERR_INVALID_ARG;
    if (BH == 0) return VLA_OK;
    const bool no_u = opts && opts->fixed_a;  // the fixed-A variant does not read u
    if (T > 0) {
        if (!q || !k || !v || (!u && !no_u) || !o) return VLA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (u && !aligned16(u)) || !aligned16(o))
            return VLA_ERR_INVALID_ARG;
    }
    if (!S_out || !A_out || !aligned16(S_out) || !aligned16(A_out)) return VLA_ERR_INVALID_ARG;
    if ((S0 && !aligned4(S0)) || (A0 && !aligned4(A0)) || (zk0 && !aligned4(zk0)) ||
        (zk_out && !aligned4(zk_out)))
        return VLA_ERR_INVALID_ARG;

    vla::Params p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.u = u;
    p.S0 = S0;
    p.A0 = A0;
    p.zk0 = zk0;
    p.o = o;
    p.o_stride = o_head_stride;
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
    p.fixed_a = (opts && opts->fixed_a) ? 1 : 0;
    if (p.fixed_a && !u) p.u = k;  // u is not used; staging reads a valid buffer of the same shape

    const int algo = opts ? opts->algo : VLA_ALGO_AUTO;
    const bool fixed_a = opts && opts->fixed_a;
    if (algo != VLA_ALGO_AUTO && algo != VLA_ALGO_PER_TOKEN && algo != VLA_ALGO_CHUNKED && algo != VLA_ALGO_DECODE &&
        algo != VLA_ALGO_CHUNKED_PAIR && algo != VLA_ALGO_CHUNKED_ROWS && algo != VLA_ALGO_SEGMENTED)
        return VLA_ERR_INVALID_ARG;
    if ((algo == VLA_ALGO_CHUNKED || algo == VLA_ALGO_SEGMENTED) && d > 96) return VLA_ERR_UNSUPPORTED;
    if (fixed_a && algo == VLA_ALGO_PER_TOKEN) return VLA_ERR_UNSUPPORTED;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the segmented path: asked for, or chosen for few heads of a long sequence
    // when its buffers fit (with the status record alone, VLA_ALGO_AUTO keeps
    // to the other kernels); they are the scratch of the options if given,
    // else the workspace past its status record
    const bool own = opts && opts->scratch;
    void* segbuf = own ? opts->scratch : workspace;
    const size_t segbytes = own ? opts->scratch_bytes : workspace_bytes;
    SegPlan sp;
    bool seg = false;
    if (algo == VLA_ALGO_SEGMENTED) {
        if (!seg_plan(BH, T, d, &sp) || segbytes < sp.total) return VLA_ERR_INVALID_ARG;
        seg = true;
    } else if (algo == VLA_ALGO_AUTO && T > kDecodeMaxT && seg_auto(BH, T, d, sm_count()) &&
               seg_plan(BH, T, d, &sp) && segbytes >= sp.total) {
        seg = true;
    }
    if (seg) {
        if (!aligned256(segbuf)) return VLA_ERR_INVALID_ARG;
        unsigned char* ws = static_cast<unsigned char*>(segbuf);
        return dtype == VLA_BF16 ? launch_seg_d<__nv_bfloat16>(d, p, (int)BH, ws, sp, s)
                                 : launch_seg_d<float>(d, p, (int)BH, ws, sp, s);
    }
    return dtype == VLA_BF16 ? launch_d<__nv_bfloat16>(d, algo, fixed_a, p, (int)BH, s)
                             : launch_d<float>(d, algo, fixed_a, p, (int)BH, s);
}

extern "C" {

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

}  // extern "C"

// ---------------------------------------------------------------------------
// No-allocation variant: the status record lives in a file-scope device array.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = 256;
static_assert(sizeof(vla::DeviceStatus) <= kNoAllocScratchBytes, "status record fits the static scratch");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once
// per device, with that device current).
vla_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return VLA_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return VLA_OK;
}

}  // namespace

extern "C" {

vla_status vla_forward_noalloc(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B,
                               int H, int T, int d, float lambda0, float eps, const float* S0, const float* A0,
                               const float* zk0, float* o, float* S_out, float* A_out, float* zk_out,
                               void* stream, int* device_status) {
    // a call that returns an error has no device-side status of its own: report the error there too
    auto fail = [device_status](vla_status e) {
        if (device_status) *device_status = e;
        return e;
    };
    // arguments that need no device are rejected before the one-time set-up
    if (B < 0 || H < 0 || T < 0) return fail(VLA_ERR_INVALID_ARG);
    if (dtype != VLA_F32 && dtype != VLA_BF16) return fail(VLA_ERR_INVALID_ARG);
    if (d != 32 && d != 64 && d != 96 && d != 128) return fail(VLA_ERR_UNSUPPORTED);
    // the status record, all the workspace this entry point gives the kernels,
    // must fit the static array (with no more than that, the automatic kernel
    // choice never takes the segmented path, which needs more)
    if (vla_impl::status_bytes() > kNoAllocScratchBytes) return fail(VLA_ERR_UNSUPPORTED);
    void* scratch = nullptr;
    vla_status st = noalloc_scratch(&scratch);
    if (st != VLA_OK) return fail(st);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the record must start at zero: the previous call's contents stay in the array
    if (cudaMemsetAsync(scratch, 0, sizeof(vla::DeviceStatus), s) != cudaSuccess) return fail(VLA_ERR_CUDA);
    st = vla_forward_ex(q, k, v, u, dtype, B, H, T, d, lambda0, eps, S0, A0, zk0, o, S_out, A_out, zk_out, scratch,
                        kNoAllocScratchBytes, stream, nullptr);
    if (st != VLA_OK) return fail(st);
    if (!device_status) return VLA_OK;
    vla::DeviceStatus h;
    if (cudaMemcpyAsync(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return fail(VLA_ERR_CUDA);
    if (cudaStreamSynchronize(s) != cudaSuccess) return fail(VLA_ERR_CUDA);
    *device_status = h.bits == 0 ? VLA_OK : ((h.bits & vla::BIT_TIMEOUT) ? VLA_ERR_TIMEOUT : VLA_ERR_NONFINITE);
    return VLA_OK;
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
        launch_la<__nv_bfloat16>(d, static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), T,
                                 S_out, (int)BH, s);
    else
        launch_la<float>(d, static_cast<const float*>(k), static_cast<const float*>(v), T, S_out, (int)BH, s);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// backward pass
// ---------------------------------------------------------------------------
namespace {

struct BwSizes {
    size_t tape, ckpt, fin, total;
};

bool bw_sizes(int B, int H, int T, int d, BwSizes* out) {
    if (B < 0 || H < 0 || T < 0 || d <= 0) return false;
    const unsigned long long BH = (unsigned long long)B * (unsigned long long)H;
    const unsigned long long nck = (unsigned long long)((T + vla::bw::CK - 1) / vla::bw::CK + 1);
    const unsigned long long tape = BH * (unsigned long long)T * (unsigned long long)(3 * d + 8) * 4ull;
    const unsigned long long ck =
        BH * nck * (2ull * (unsigned long long)d * (unsigned long long)d + (unsigned long long)d) * 4ull;
    if (BH > (1ull << 31) || tape > (1ull << 50) || ck > (1ull << 50)) return false;
    auto al = [](unsigned long long x) { return (x + 255ull) / 256ull * 256ull; };
    const unsigned long long fin = BH * (2ull * (unsigned long long)d * (unsigned long long)d + (unsigned long long)d) * 4ull;
    out->tape = (size_t)al(tape);
    out->ckpt = (size_t)al(ck);
    out->fin = (size_t)al(fin);
    out->total = kWorkspaceBytes + out->tape + out->ckpt + out->fin;
    return true;
}

// The forward pass that the reverse sweep replays, writing the tape, the
// checkpoints and the final state to `fin`: the chunked tensor-core kernel for
// d <= 96 (its o goes to dq, which the reverse sweep overwrites), the per-token
// phase of the backward kernel for d = 128.
template <int D, typename TIn>
vla_status launch_bw_forward(const vla::Params& p, int BH, float* dq, float* tape, float* ckpt, float* fin,
                             cudaStream_t s) {
    if constexpr (D <= 96) {
        using TL = vla::tc::Lay<D, TIn>;
        vla::Params pf = p;
        pf.o = dq;
        pf.o_stride = (size_t)p.T * D;
        pf.S_out = fin;
        pf.A_out = fin + (size_t)BH * D * D;
        pf.zk_out = fin + 2 * (size_t)BH * D * D;
        pf.tape = tape;
        pf.ckpt = ckpt;
        pf.stall_producer = 0;  // the test hook is for the reverse sweep's wait
        auto fk = vla::vla_tc_kernel<D, TIn, true>;
        if (cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TL::SMEM) != cudaSuccess)
            return VLA_ERR_CUDA;
        fk<<<BH, vla::tc::THREADS, TL::SMEM, s>>>(pf);
    } else {
        // d = 128: the cluster-pair chunked kernel (A-pass and S-pass on two SMs)
        using LY = vla::tc2::Lay2<D, TIn>;
        if ((long long)BH * 2 > 2147483647LL) return VLA_ERR_INVALID_ARG;
        vla::Params pf = p;
        pf.o = dq;
        pf.o_stride = (size_t)p.T * D;
        pf.S_out = fin;
        pf.A_out = fin + (size_t)BH * D * D;
        pf.zk_out = fin + 2 * (size_t)BH * D * D;
        pf.tape = tape;
        pf.ckpt = ckpt;
        pf.stall_producer = 0;  // the test hook is for the reverse sweep's wait
        auto fk = vla::vla_tc2_kernel<D, TIn, true>;
        if (cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::SMEM_LAUNCH) != cudaSuccess)
            return VLA_ERR_CUDA;
        fk<<<2 * BH, vla::tc2::THREADS, LY::SMEM_LAUNCH, s>>>(pf);
    }
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

template <int D, typename TIn>
vla_status launch_bw(const vla::Params& p, int BH, const float* dO, const float* dST, const float* dAT,
                     const float* dzkT, float* dq, float* dk, float* dv, float* du, float* dS0, float* dA0,
                     float* dzk0, float* tape, float* ckpt, float* fin, bool split, cudaStream_t s) {
    if (p.T > 0) {
        const vla_status st = launch_bw_forward<D, TIn>(p, BH, dq, tape, ckpt, fin, s);
        if (st != VLA_OK) return st;
    }
    if constexpr (D <= 96) {
        if (!split) {
            using BL = vla::bw::BLay<D, TIn>;
            auto kern = vla::bw::vla_backward_kernel<D, TIn>;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BL::SMEM) != cudaSuccess)
                return VLA_ERR_CUDA;
            kern<<<BH, BL::THREADS, BL::SMEM, s>>>(p, dO, dST, dAT, dzkT, dq, dk, dv, du, dS0, dA0, dzk0, tape, ckpt,
                                                   p.T > 0 ? fin : nullptr);
            return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
        }
    }
    // the split sweep: its S side and A side side by side, a cluster of two
    // CTAs per head (vla_backward_split.cuh)
    using PL = vla::bw::PairLay<D, TIn>;
    if (BH > (1 << 30)) return VLA_ERR_INVALID_ARG;  // grid 2 BH
    auto pk = vla::bw::vla_backward_pair_kernel<D, TIn>;
    if (cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PL::SMEM) != cudaSuccess)
        return VLA_ERR_CUDA;
    pk<<<2 * BH, vla::bw::SLay<D, TIn>::THREADS, PL::SMEM, s>>>(p, dO, dST, dAT, dzkT, dq, dk, dv, du, dS0, dA0, dzk0,
                                                               tape, ckpt, fin);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

template <typename TIn>
vla_status launch_bw_d(int d, const vla::Params& p, int BH, const float* dO, const float* dST, const float* dAT,
                       const float* dzkT, float* dq, float* dk, float* dv, float* du, float* dS0, float* dA0,
                       float* dzk0, float* tape, float* ckpt, float* fin, bool split, cudaStream_t s) {
    switch (d) {
        case 32:
            return launch_bw<32, TIn>(p, BH, dO, dST, dAT, dzkT, dq, dk, dv, du, dS0, dA0, dzk0, tape, ckpt, fin,
                                      split, s);
        case 64:
            return launch_bw<64, TIn>(p, BH, dO, dST, dAT, dzkT, dq, dk, dv, du, dS0, dA0, dzk0, tape, ckpt, fin,
                                      split, s);
        case 96:
            return launch_bw<96, TIn>(p, BH, dO, dST, dAT, dzkT, dq, dk, dv, du, dS0, dA0, dzk0, tape, ckpt, fin,
                                      split, s);
        case 128:
            return launch_bw<128, TIn>(p, BH, dO, dST, dAT, dzkT, dq, dk, dv, du, dS0, dA0, dzk0, tape, ckpt, fin,
                                       true, s);
        default: return VLA_ERR_UNSUPPORTED;
    }
}

vla_status backward_impl(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B, int H,
                         int T, int d, float lambda0, float eps, const float* S0, const float* A0, const float* zk0,
                         const float* dO, const float* dS_T, const float* dA_T, const float* dzk_T, float* dq,
                         float* dk, float* dv, float* du, float* dS0, float* dA0, float* dzk0, void* workspace,
                         size_t workspace_bytes, void* stream, bool split, const vla_options* opts) {
    if (B < 0 || H < 0 || T < 0) return VLA_ERR_INVALID_ARG;
    if (dtype != VLA_F32 && dtype != VLA_BF16) return VLA_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 96 && d != 128) return VLA_ERR_UNSUPPORTED;
    if (!(lambda0 > 0.f) || !std::isfinite(lambda0)) return VLA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || !std::isfinite(eps)) return VLA_ERR_INVALID_ARG;
    BwSizes z;
    if (!bw_sizes(B, H, T, d, &z)) return VLA_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < z.total) return VLA_ERR_INVALID_ARG;
    const long long BH = (long long)B * H;
    if (BH == 0) return VLA_OK;
    if (T > 0) {
        if (!q || !k || !v || !u || !dq || !dk || !dv || !du) return VLA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(u) || !aligned16(dq) ||
            !aligned16(dk) || !aligned16(dv) || !aligned16(du) || (dO && !aligned16(dO)))
            return VLA_ERR_INVALID_ARG;
    }
    const float* st[] = {S0, A0, zk0, dS_T, dA_T, dzk_T, dS0, dA0, dzk0};
    for (const float* x : st)
        if (x && !aligned4(x)) return VLA_ERR_INVALID_ARG;

    vla::Params p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.u = u;
    p.S0 = S0;
    p.A0 = A0;
    p.zk0 = zk0;
    p.status = static_cast<vla::DeviceStatus*>(workspace);
    p.T = T;
    p.inv_lambda0 = 1.0f / lambda0;
    p.eps = eps;
    p.wait_ns = 1000ull * ((opts && opts->wait_limit_us) ? opts->wait_limit_us : kDefaultWaitUs);
    p.stall_producer = (opts && opts->test_stall_producer) ? 1 : 0;
    unsigned char* w = static_cast<unsigned char*>(workspace);
    float* tape = reinterpret_cast<float*>(w + kWorkspaceBytes);
    float* ckpt = reinterpret_cast<float*>(w + kWorkspaceBytes + z.tape);
    float* fin = reinterpret_cast<float*>(w + kWorkspaceBytes + z.tape + z.ckpt);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == VLA_BF16 ? launch_bw_d<__nv_bfloat16>(d, p, (int)BH, dO, dS_T, dA_T, dzk_T, dq, dk, dv, du, dS0,
                                                          dA0, dzk0, tape, ckpt, fin, split, s)
                             : launch_bw_d<float>(d, p, (int)BH, dO, dS_T, dA_T, dzk_T, dq, dk, dv, du, dS0, dA0,
                                                  dzk0, tape, ckpt, fin, split, s);
}

}  // namespace

extern "C" {

size_t vla_backward_workspace_bytes(int B, int H, int T, int d) {
    BwSizes z;
    return bw_sizes(B, H, T, d, &z) ? z.total : 0;
}

vla_status vla_backward(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B,
                        int H, int T, int d, float lambda0, float eps, const float* S0, const float* A0,
                        const float* zk0, const float* dO, const float* dS_T, const float* dA_T,
                        const float* dzk_T, float* dq, float* dk, float* dv, float* du, float* dS0, float* dA0,
                        float* dzk0, void* workspace, size_t workspace_bytes, void* stream) {
    return backward_impl(q, k, v, u, dtype, B, H, T, d, lambda0, eps, S0, A0, zk0, dO, dS_T, dA_T, dzk_T, dq, dk, dv,
                         du, dS0, dA0, dzk0, workspace, workspace_bytes, stream, false, nullptr);
}

vla_status vla_backward_split(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B,
                              int H, int T, int d, float lambda0, float eps, const float* S0, const float* A0,
                              const float* zk0, const float* dO, const float* dS_T, const float* dA_T,
                              const float* dzk_T, float* dq, float* dk, float* dv, float* du, float* dS0,
                              float* dA0, float* dzk0, void* workspace, size_t workspace_bytes, void* stream) {
    return backward_impl(q, k, v, u, dtype, B, H, T, d, lambda0, eps, S0, A0, zk0, dO, dS_T, dA_T, dzk_T, dq, dk, dv,
                         du, dS0, dA0, dzk0, workspace, workspace_bytes, stream, true, nullptr);
}

vla_status vla_backward_ex(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B, int H,
                           int T, int d, float lambda0, float eps, const float* S0, const float* A0, const float* zk0,
                           const float* dO, const float* dS_T, const float* dA_T, const float* dzk_T, float* dq,
                           float* dk, float* dv, float* du, float* dS0, float* dA0, float* dzk0, void* workspace,
                           size_t workspace_bytes, void* stream, int split, const vla_options* opts) {
    return backward_impl(q, k, v, u, dtype, B, H, T, d, lambda0, eps, S0, A0, zk0, dO, dS_T, dA_T, dzk_T, dq, dk, dv,
                         du, dS0, dA0, dzk0, workspace, workspace_bytes, stream, split != 0, opts);
}

}  // extern "C"
