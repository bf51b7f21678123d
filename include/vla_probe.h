/*
 * vla_probe.h -- measurement helper of libvla_gb300.so: the FP32 FMA peak of
 * the GPU it runs on, the denominator of the forward recurrence's roofline.
 *
 * The recurrence of "Variational Linear Attention" (arXiv 2605.11196, §3.3
 * eq. 9-11) costs about 12 d^2 FLOP per head and token (six d x d
 * matrix-vector products or rank-1 updates of 2 d^2 FLOP each), and its
 * roofline is stated against the FP32 fused multiply-add rate of the chip.
 * This probe measures that rate instead of deriving it from unit counts and
 * the maximum clock: it does nothing the recurrence needs.
 */
#ifndef VLA_GB300_PROBE_H
#define VLA_GB300_PROBE_H

#include "vla.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * vla_probe_ffma -- enqueue `blocks` CTAs of `threads` threads on `stream`;
 * every thread advances 8 independent fused multiply-add chains by 4 steps
 * per iteration, for `iters` iterations (as packed two-wide FMA instructions
 * when `packed` is nonzero, scalar fma.rn.f32 otherwise), and writes one
 * float per thread to `sink`.
 *
 *  blocks   >= 1;  threads: a multiple of 32 in [32, 1024];  iters >= 1.
 *  sink     device array of blocks * threads floats, 4-byte aligned, owned
 *           by the caller (its values are meaningless; they keep the chains
 *           from being optimised away).
 *  stream   cudaStream_t as void*.
 *
 * Each thread performs 32 * iters fused multiply-adds (in 32 scalar or 16
 * packed instructions per iteration); vla_probe_ffma_flop() gives the FLOP
 * of a call (2 per FMA). Time
 * the call with CUDA events on `stream`. Asynchronous; returns
 * VLA_ERR_INVALID_ARG for bad sizes or a NULL / misaligned sink and
 * VLA_ERR_CUDA if the launch fails.
 */
vla_status vla_probe_ffma(int blocks, int threads, int iters, int packed, float* sink, void* stream);

/* FLOP that one vla_probe_ffma() call with these arguments performs
 * (2 per fused multiply-add); 0 for invalid sizes. */
double vla_probe_ffma_flop(int blocks, int threads, int iters, int packed);

#ifdef __cplusplus
}
#endif

#endif /* VLA_GB300_PROBE_H */
