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

// ---------------------------------------------------------------------------
// 5th-generation tensor cores (tcgen05) and tensor memory (TMEM), sm_100+.
// Operand tiles in shared memory use the K-major, no-swizzle canonical
// layout: "core matrices" of 8 rows x 16 bytes (4 tf32) stored as 128
// contiguous bytes; core matrices adjacent in K are 128 bytes apart (the
// leading byte offset) and 8-row groups are (K/4)*128 bytes apart (the
// stride byte offset). TMEM addresses are (lane << 16) | column.
// ---------------------------------------------------------------------------

// float offset of element (r, k) in a K-major no-swizzle tile of rows of kk elements
__host__ __device__ constexpr int cm_off(int r, int k, int kk) {
    return ((r >> 3) * (kk >> 2) + (k >> 2)) * 32 + ((r & 7) << 2) + (k & 3);
}

// shared-memory matrix descriptor: start address, leading byte offset (K
// direction), stride byte offset (8-row groups), descriptor version 1, no swizzle
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// instruction descriptor of kind::tf32: fp32 accumulator, tf32 A and B, both
// K-major, M x N tile
__host__ __device__ constexpr uint32_t tc_idesc_tf32(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]^T, one K step of 8 tf32
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.s32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, one K step of 8 tf32
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.s32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive (once) on `bar` when every tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// warp-wide: allocate / free `ncols` TMEM columns (a power of two >= 32); the
// base address is written to shared memory at `dst`
__device__ __forceinline__ void tc_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// warp-wide: lane l of the warp reads 16 consecutive 32-bit columns of TMEM
// lane (lane window of the warp) + l, starting at column taddr & 0xffff
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// tf32 operands are read by truncation of the fp32 bits: x = hi(x) + lo(x)
// with hi(x) = x with the low 13 mantissa bits cleared (what the tensor core
// sees of x) and lo(x) = x - hi(x) (exact).
__device__ __forceinline__ float tf32_lo(float x) {
    return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// plain named barrier over `nthreads` threads
__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace vla
