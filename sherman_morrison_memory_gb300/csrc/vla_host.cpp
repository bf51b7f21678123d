// vla_host.cpp -- vla_forward over HOST buffers, with the host<->device copies
// overlapped with the kernels ("Variational Linear Attention", §3.3 eq. 9-11).
//
// The recurrence is causal: the state (S, A, z^key) after token t is all that
// tokens > t need. So the sequence is cut into chunks of Tc tokens and each
// chunk is one vla_forward_ex() launch over every head, carrying the state in
// device memory from launch to launch. Four streams form a pipeline:
//
//   copy-in   H2D of chunk j+2's q, k, v, u (pitched copies: one row of Tc*d
//             elements per head) into input slot (j+2) mod 3, on two streams
//             (q, v on one, k, u on the other: one stream of pitched copies
//             alone moves about half of what the link carries for chunks of
//             a few hundred tokens, two reach the contiguous-copy rate)
//   caller's  the kernel of chunk j on input slot j mod 3 -> output slot j mod 3
//   copy-out  D2H of chunk j's o into the host array, then the final state
//
// When the host o is page-locked and mapped into the device's address space
// (cudaHostGetDevicePointer succeeds, e.g. cudaHostAlloc memory), the kernels
// write o straight into it (plain stores, rows of head h at h * T * d) and
// only the final state is copied out: o then crosses the link while the
// kernels run, in the direction the input copies do not use.
//
// Host code only (no kernels): compiled as its own translation unit.
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <mutex>

#include "vla.h"
#include "vla_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;
constexpr int kSlots = 3;  // chunks in flight: being copied in, computed, copied out

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Streams and events of the pipeline, created on a device's first call and
// kept until the process exits.
struct Pipe {
    bool ready = false;
    cudaStream_t in[2] = {}, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t h2d[kSlots][2] = {}, kern[kSlots] = {}, d2h[kSlots] = {};
};
std::mutex g_mutex;
Pipe g_pipe[kMaxDevices];

vla_status pipe_for(int dev, Pipe** out) {
    if (dev < 0 || dev >= kMaxDevices) return VLA_ERR_CUDA;
    Pipe& P = g_pipe[dev];
    if (!P.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&P.in[0], cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&P.in[1], cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&P.out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&P.start, ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&P.done, ef) != cudaSuccess)
            return VLA_ERR_CUDA;
        for (int i = 0; i < kSlots; ++i)
            if (cudaEventCreateWithFlags(&P.h2d[i][0], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&P.h2d[i][1], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&P.kern[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&P.d2h[i], ef) != cudaSuccess)
                return VLA_ERR_CUDA;
        P.ready = true;
    }
    *out = &P;
    return VLA_OK;
}

// Chunks: tc tokens each, or with the automatic choice a first and a last
// chunk of ra = tc / 4 tokens around chunks of tc: the copy of the first
// chunk, which nothing overlaps, and the launch of the last one, after the
// last copy, are then short. Workspace layout: status record | S | A | z^key |
// kSlots input slots (q, k, v, u of one chunk, compact [B*H, n, d]) | kSlots
// output slots (o, [B*H, n, d] fp32), sized for tc tokens.
struct Plan {
    int T = 0, tc = 0, ra = 0, nchunks = 0;
    size_t es = 0, status = 0, status_bytes = 0, S = 0, A = 0, zk = 0, in_arr = 0, in_slot[kSlots] = {},
           out_slot[kSlots] = {}, total = 0;
    // first token and length of chunk j
    long long start(int j) const {
        if (ra == 0 || j == 0) return (long long)j * tc;
        if (j == nchunks - 1) return (long long)T - ra;
        return ra + (long long)(j - 1) * tc;
    }
    int len(int j) const {
        if (T == 0) return 0;
        if (ra > 0 && (j == 0 || j == nchunks - 1)) return ra;
        const long long end = (ra > 0) ? (long long)T - ra : (long long)T;
        const long long n = end - start(j);
        return (int)(n < tc ? n : tc);
    }
};

bool make_plan(vla_dtype dtype, long long BH, int T, int d, int chunk_tokens, Plan* pl) {
    if (BH < 0 || T < 0 || chunk_tokens < 0) return false;
    pl->T = T;
    if (T == 0) {
        pl->tc = 0;
        pl->nchunks = 1;  // one launch with T = 0 writes the initial state out
    } else {
        int tc = chunk_tokens, ra = 0;
        if (tc == 0) {  // about T/4 tokens, a multiple of 16, at least 256; short first and last chunks
            long long c = ((long long)T + 3) / 4;
            c = (c + 15) / 16 * 16;
            tc = (int)(c < 256 ? 256 : c);
            ra = tc / 4 / 16 * 16;
            if ((long long)T < 2LL * ra + tc) ra = 0;  // too short to gain from the ramps
        }
        if (tc > T) tc = T;
        pl->tc = tc;
        pl->ra = ra;
        const long long mid = (long long)T - 2LL * ra;
        pl->nchunks = (int)((mid + tc - 1) / tc) + (ra > 0 ? 2 : 0);
    }
    pl->es = dtype == VLA_BF16 ? 2 : 4;
    const size_t bh = (size_t)BH, dd = (size_t)d;
    // the status record that every launch of the call shares (the launches
    // then keep to the kernels that need no more workspace than that)
    if (vla_workspace_bytes(1, 1, T, d) == 0) return false;
    pl->status_bytes = vla_impl::status_bytes();
    size_t off = round_up(pl->status_bytes);
    pl->status = 0;
    pl->S = off;
    off += round_up(bh * dd * dd * 4);
    pl->A = off;
    off += round_up(bh * dd * dd * 4);
    pl->zk = off;
    off += round_up(bh * dd * 4);
    pl->in_arr = round_up(bh * (size_t)pl->tc * dd * pl->es);
    for (int s = 0; s < kSlots; ++s) {
        pl->in_slot[s] = off;
        off += 4 * pl->in_arr;
    }
    for (int s = 0; s < kSlots; ++s) {
        pl->out_slot[s] = off;
        off += round_up(bh * (size_t)pl->tc * dd * 4);
    }
    pl->total = off;
    return true;
}

bool ok(cudaError_t e) { return e == cudaSuccess; }

}  // namespace

extern "C" {

size_t vla_forward_host_workspace_bytes(vla_dtype dtype, int B, int H, int T, int d, int chunk_tokens) {
    if (B < 0 || H < 0 || (dtype != VLA_F32 && dtype != VLA_BF16)) return 0;
    if (d != 32 && d != 64 && d != 96 && d != 128) return 0;
    Plan pl;
    if (!make_plan(dtype, (long long)B * H, T, d, chunk_tokens, &pl)) return 0;
    return pl.total;
}

vla_status vla_forward_host(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype, int B,
                            int H, int T, int d, float lambda0, float eps, const float* S0, const float* A0,
                            const float* zk0, float* o, float* S_out, float* A_out, float* zk_out,
                            int chunk_tokens, void* workspace, size_t workspace_bytes, void* stream,
                            const vla_options* opts) {
    if (B < 0 || H < 0 || T < 0 || chunk_tokens < 0) return VLA_ERR_INVALID_ARG;
    if (dtype != VLA_F32 && dtype != VLA_BF16) return VLA_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 96 && d != 128) return VLA_ERR_UNSUPPORTED;
    if (!(lambda0 > 0.f) || !std::isfinite(lambda0) || !(eps > 0.f) || !std::isfinite(eps))
        return VLA_ERR_INVALID_ARG;
    const long long BH = (long long)B * H;
    if (BH > 2147483647LL) return VLA_ERR_INVALID_ARG;
    if ((unsigned long long)BH * (unsigned long long)T * (unsigned long long)d > (1ULL << 60))
        return VLA_ERR_INVALID_ARG;
    Plan pl;
    if (!make_plan(dtype, BH, T, d, chunk_tokens, &pl)) return VLA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) || workspace_bytes < pl.total)
        return VLA_ERR_INVALID_ARG;
    if (BH == 0) return VLA_OK;
    const bool no_u = opts && opts->fixed_a;
    if (T > 0 && (!q || !k || !v || (!u && !no_u) || !o)) return VLA_ERR_INVALID_ARG;
    if (!S_out || !A_out) return VLA_ERR_INVALID_ARG;

    int dev = 0;
    if (!ok(cudaGetDevice(&dev))) return VLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    Pipe* P = nullptr;
    vla_status st = pipe_for(dev, &P);
    if (st != VLA_OK) return st;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* dS = reinterpret_cast<float*>(ws + pl.S);
    float* dA = reinterpret_cast<float*>(ws + pl.A);
    float* dZ = reinterpret_cast<float*>(ws + pl.zk);
    const size_t bh = (size_t)BH, dd = (size_t)d, es = pl.es;
    const size_t state_bytes = bh * dd * dd * 4;
    const void* hin[4] = {q, k, v, no_u ? nullptr : u};
    // device alias of the host o, if it is page-locked and mapped
    float* od = nullptr;
    if (T > 0) {
        void* dp = nullptr;
        if (cudaHostGetDevicePointer(&dp, o, 0) == cudaSuccess && dp && !(reinterpret_cast<uintptr_t>(dp) & 15u))
            od = static_cast<float*>(dp);
        else
            (void)cudaGetLastError();  // pageable memory: clear the error, copy o out instead
    }

    // Leave the internal streams drained on an error, so that no copy touches
    // the caller's buffers after the call has returned.
    auto fail = [&](vla_status s) {
        cudaStreamSynchronize(P->in[0]);
        cudaStreamSynchronize(P->in[1]);
        cudaStreamSynchronize(P->out);
        return s;
    };

    // every copy starts after the work already queued on the caller's stream
    if (!ok(cudaEventRecord(P->start, cs)) || !ok(cudaStreamWaitEvent(P->in[0], P->start, 0)) ||
        !ok(cudaStreamWaitEvent(P->in[1], P->start, 0)) || !ok(cudaStreamWaitEvent(P->out, P->start, 0)))
        return fail(VLA_ERR_CUDA);
    if ((S0 && !ok(cudaMemcpyAsync(dS, S0, state_bytes, cudaMemcpyHostToDevice, P->in[0]))) ||
        (A0 && !ok(cudaMemcpyAsync(dA, A0, state_bytes, cudaMemcpyHostToDevice, P->in[1]))) ||
        (zk0 && !ok(cudaMemcpyAsync(dZ, zk0, bh * dd * 4, cudaMemcpyHostToDevice, P->in[0]))))
        return fail(VLA_ERR_CUDA);

    auto chunk_len = [&](int j) { return pl.len(j); };
    // H2D of chunk j into input slot j mod kSlots, compact [B*H, n, d]; array a
    // on copy-in stream a mod 2
    auto h2d = [&](int j) -> bool {
        const int slot = j % kSlots, n = chunk_len(j);
        for (int c = 0; c < 2; ++c)
            if (j >= kSlots && !ok(cudaStreamWaitEvent(P->in[c], P->kern[slot], 0))) return false;
        const size_t row = (size_t)n * dd * es;
        for (int a = 0; a < 4; ++a) {
            if (!hin[a] || n == 0) continue;
            const char* src = static_cast<const char*>(hin[a]) + (size_t)pl.start(j) * dd * es;
            if (!ok(cudaMemcpy2DAsync(ws + pl.in_slot[slot] + a * pl.in_arr, row, src, (size_t)T * dd * es, row, bh,
                                      cudaMemcpyHostToDevice, P->in[a & 1])))
                return false;
        }
        return ok(cudaEventRecord(P->h2d[slot][0], P->in[0])) && ok(cudaEventRecord(P->h2d[slot][1], P->in[1]));
    };

    for (int j = 0; j < kSlots - 1 && j < pl.nchunks; ++j)
        if (!h2d(j)) return fail(VLA_ERR_CUDA);
    for (int j = 0; j < pl.nchunks; ++j) {
        if (j + kSlots - 1 < pl.nchunks && !h2d(j + kSlots - 1)) return fail(VLA_ERR_CUDA);
        const int slot = j % kSlots, n = chunk_len(j);
        if (!ok(cudaStreamWaitEvent(cs, P->h2d[slot][0], 0)) || !ok(cudaStreamWaitEvent(cs, P->h2d[slot][1], 0)))
            return fail(VLA_ERR_CUDA);
        if (!od && j >= kSlots && !ok(cudaStreamWaitEvent(cs, P->d2h[slot], 0))) return fail(VLA_ERR_CUDA);
        const bool first = j == 0;
        char* in = ws + pl.in_slot[slot];
        const bool has = n > 0;
        // o of the chunk: straight into the mapped host array (row pitch T * d), or an output slot
        float* dO = od ? od + (size_t)pl.start(j) * dd : reinterpret_cast<float*>(ws + pl.out_slot[slot]);
        st = vla_impl::forward(has ? in : nullptr, has ? in + pl.in_arr : nullptr,
                               has ? in + 2 * pl.in_arr : nullptr, (has && hin[3]) ? in + 3 * pl.in_arr : nullptr,
                               dtype, B, H, n, d, lambda0, eps, (first && !S0) ? nullptr : dS,
                               (first && !A0) ? nullptr : dA, (first && !zk0) ? nullptr : dZ, has ? dO : nullptr, dS,
                               dA, dZ, ws + pl.status, pl.status_bytes, stream, opts,
                               od ? (size_t)T * dd : 0);
        if (st != VLA_OK) return fail(st);
        if (!ok(cudaEventRecord(P->kern[slot], cs))) return fail(VLA_ERR_CUDA);
        if (has && !od) {
            const size_t row = (size_t)n * dd * 4;
            if (!ok(cudaStreamWaitEvent(P->out, P->kern[slot], 0)) ||
                !ok(cudaMemcpy2DAsync(o + (size_t)pl.start(j) * dd, (size_t)T * dd * 4, dO, row, row, bh,
                                      cudaMemcpyDeviceToHost, P->out)) ||
                !ok(cudaEventRecord(P->d2h[slot], P->out)))
                return fail(VLA_ERR_CUDA);
        }
    }
    const int last = (pl.nchunks - 1) % kSlots;
    if (!ok(cudaStreamWaitEvent(P->out, P->kern[last], 0)) ||
        !ok(cudaMemcpyAsync(S_out, dS, state_bytes, cudaMemcpyDeviceToHost, P->out)) ||
        !ok(cudaMemcpyAsync(A_out, dA, state_bytes, cudaMemcpyDeviceToHost, P->out)) ||
        (zk_out && !ok(cudaMemcpyAsync(zk_out, dZ, bh * dd * 4, cudaMemcpyDeviceToHost, P->out))) ||
        !ok(cudaEventRecord(P->done, P->out)) || !ok(cudaStreamWaitEvent(cs, P->done, 0)))
        return fail(VLA_ERR_CUDA);
    return VLA_OK;
}

}  // extern "C"
