// vla_probe.cu -- FP32 fused multiply-add throughput probe (include/vla_probe.h).
//
// Every thread runs 8 independent FMA chains (4 packed pairs when `PACKED`),
// 32 fused multiply-adds per loop iteration either way, so a warp always has
// independent work to issue and the FMA pipes, not the chain latency, set the
// rate. The multiplier and addend come from kernel
// arguments, so the compiler cannot fold the chains.
#include <cuda_runtime.h>

#include "vla_probe.h"

namespace {

template <bool PACKED>
__global__ void vla_ffma_probe_kernel(int iters, float a, float b, float* sink) {
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = (float)(tid + j) * 1e-7f;
    if constexpr (PACKED) {
        float2 y[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) y[j] = make_float2(x[2 * j], x[2 * j + 1]);
        const float2 a2 = make_float2(a, a), b2 = make_float2(b, b);
#pragma unroll 1
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int j = 0; j < 4; ++j) y[j] = __ffma2_rn(y[j], a2, b2);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[2 * j] = y[j].x;
            x[2 * j + 1] = y[j].y;
        }
    } else {
#pragma unroll 1
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = fmaf(x[j], a, b);
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += x[j];
    sink[tid] = s;
}

bool sizes_ok(int blocks, int threads, int iters) {
    return blocks >= 1 && threads >= 32 && threads <= 1024 && threads % 32 == 0 && iters >= 1;
}

}  // namespace

extern "C" {

double vla_probe_ffma_flop(int blocks, int threads, int iters, int packed) {
    if (!sizes_ok(blocks, threads, iters)) return 0.0;
    // per thread and iteration: 4 rounds of 8 chains (scalar) or of 4 packed pairs
    (void)packed;
    return 2.0 * 32.0 * (double)iters * (double)blocks * (double)threads;
}

vla_status vla_probe_ffma(int blocks, int threads, int iters, int packed, float* sink, void* stream) {
    if (!sizes_ok(blocks, threads, iters)) return VLA_ERR_INVALID_ARG;
    if (!sink || (reinterpret_cast<unsigned long long>(sink) & 3u)) return VLA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the multiplier keeps the chains bounded (|x| stays below b / (1 - a))
    if (packed)
        vla_ffma_probe_kernel<true><<<blocks, threads, 0, s>>>(iters, 0.999f, 1e-3f, sink);
    else
        vla_ffma_probe_kernel<false><<<blocks, threads, 0, s>>>(iters, 0.999f, 1e-3f, sink);
    return cudaGetLastError() == cudaSuccess ? VLA_OK : VLA_ERR_CUDA;
}

}  // extern "C"
