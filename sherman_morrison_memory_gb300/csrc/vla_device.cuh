// vla_device.cuh -- PTX helpers shared by the VLA kernels (sm_103a).
//
// mbarrier waits are always bounded: a wait gives up after a time limit (read
// from %globaltimer) or when the CTA's abort flag is raised, and returns false
// so that the caller can record VLA_ERR_TIMEOUT and leave without hanging the
// GPU.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace vla {

// Status record kept in the caller's workspace.
struct DeviceStatus {
    int bits;         // VLA_BIT_* or'ed together
    int role;         // role of the first failure (0 staging, 1 gate, 2 A-pass, 3 S-pass)
    int head;         // head index (b * H + h) of the first failure
    int token;        // token index of the first failure
};

constexpr int BIT_TIMEOUT = 1;
constexpr int BIT_NONFINITE = 2;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread for up to `hint_ns`
// while the phase is incomplete (it resumes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Slow path of mbar_wait: suspend in hardware between checks (no polling
// loop that would take issue slots from working warps), give up after
// `limit_ns` or when the abort flag (if not null) is raised.
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                            uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Wait until the phase of `bar` with parity `parity` has completed. Returns
// false if `limit_ns` elapsed or the abort flag (if not null) was raised first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag, limit_ns);
}

// 1-D TMA bulk copy global -> shared, completing on `bar` (tx bytes).
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32) that also ORs a
// predicate across them, so that every participant takes the same decision.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1 : 0), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void record_failure(DeviceStatus* st, int bit, int role, int head, int token) {
    if (atomicOr(&st->bits, bit) == 0) {
        st->role = role;
        st->head = head;
        st->token = token;
    }
}

// ---------------------------------------------------------------------------
// Reduce-scatter of N per-lane floats across the aligned group of 2*H lanes
// that differ in lane bits H, H/2, ..., 1. At each level a lane keeps one half
// of its values (the upper half if its bit is set) and adds its partner's copy
// of that half. On return v[0 .. rs_count<N,H>()-1] hold fully reduced values;
// v[i] is original value number rs_index<N,H>(lane, i), or a padding zero
// when rs_index returns -1.
// ---------------------------------------------------------------------------
template <int N, int H>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
    if constexpr (H >= 1) {
        constexpr int M = (N + 1) / 2;
        const bool hi = (lane & H) != 0;
#pragma unroll
        for (int i = 0; i < M; ++i) {
            const float lo_v = v[i];
            const float hi_v = (i + M < N) ? v[(i + M < N) ? i + M : 0] : 0.f;
            const float send = hi ? lo_v : hi_v;
            const float keep = hi ? hi_v : lo_v;
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, H);
        }
        reduce_scatter<M, H / 2>(v, lane);
    }
}

template <int N, int H>
__host__ __device__ constexpr int rs_count() {
    if constexpr (H >= 1)
        return rs_count<(N + 1) / 2, H / 2>();
    else
        return N;
}

// Original value number of v[i] after reduce_scatter<N, H>, or -1 for a
// padding slot. A lane that keeps the lower half at a level keeps M real
// values; one that keeps the upper half keeps N - M real values followed by
// padding when N is odd.
template <int N, int H>
__device__ __forceinline__ int rs_index(int lane, int i) {
    if constexpr (H >= 1) {
        constexpr int M = (N + 1) / 2;
        const int r = rs_index<M, H / 2>(lane, i);
        if (lane & H) return (r < 0 || r >= N - M) ? -1 : M + r;
        return r;
    } else {
        return i < N ? i : -1;
    }
}

// Inverse of rs_index: the lane bits (within the group) and slot that hold
// original value number r after reduce_scatter<N, H>.
template <int N, int H>
__host__ __device__ constexpr int rs_owner_lane(int r) {
    if constexpr (H >= 1) {
        constexpr int M = (N + 1) / 2;
        return r < M ? rs_owner_lane<M, H / 2>(r) : (H | rs_owner_lane<M, H / 2>(r - M));
    } else {
        return 0;
    }
}
template <int N, int H>
__host__ __device__ constexpr int rs_owner_slot(int r) {
    if constexpr (H >= 1) {
        constexpr int M = (N + 1) / 2;
        return r < M ? rs_owner_slot<M, H / 2>(r) : rs_owner_slot<M, H / 2>(r - M);
    } else {
        return r;
    }
}

// Butterfly all-reduce (sum) across lane bits H, H/2, ..., 1.
template <int N, int H>
__device__ __forceinline__ void allreduce(float* v) {
#pragma unroll
    for (int h = H; h >= 1; h >>= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], h);
    }
}

}  // namespace vla
