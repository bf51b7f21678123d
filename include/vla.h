/*
 * vla.h -- C ABI of the GB300 (sm_103a) Variational Linear Attention forward
 * recurrence library (libvla_gb300.so).
 *
 * The operation is the per-token recurrence of "Variational Linear
 * Attention: Stable Associative Memory for Long-Context Transformers"
 * (Pandey, Singh; arXiv 2605.11196), §3.3, for every (batch, head):
 *
 *   eq. 9   z_t = A_{t-1} u^_t,  delta_t = 1 + u^_t . z_t,
 *           A_t = A_{t-1} - z_t z_t^T / delta_t             (Sherman-Morrison)
 *   eq. 10  e_t = v_t - S_{t-1} k^_t,
 *           alpha^_t = A_t k^_t / ||A_t k^_t||,
 *           S_t = S_{t-1} + e_t alpha^_t^T
 *   eq. 11  z^key_t = z^key_{t-1} + phi(k_t),
 *           o_t = S_t phi(q_t) / max(phi(q_t) . z^key_t, eps),  phi = ELU + 1
 *
 * with u^ = u / max(||u||, 1e-12) and k^ = k / max(||k||, 1e-12) formed inside
 * the op (§3.2: unit penalty directions; §3.3: unit keys), the same guard on
 * ||A_t k^_t||, phi applied to the raw q and k, and, by default,
 * S_0 = 0, A_0 = I / lambda0 (§3.2), z^key_0 = 0.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or keeps them.
 *  - Sequences are [B, H, T, d] row-major (d fastest); states are
 *    S, A: [B, H, d, d] row-major with S[i][j] mapping key coordinate j to
 *    output coordinate i; z^key: [B, H, d].
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Calls are asynchronous on that stream: argument errors are
 *    returned at once, failures inside the kernel are recorded in the
 *    workspace and read back by vla_get_last_device_status().
 *  - Supported head dimensions d: 32, 64, 96, 128 (else VLA_ERR_UNSUPPORTED).
 *  - Arithmetic and state are fp32 on the device.
 */
#ifndef VLA_GB300_H
#define VLA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VLA_OK = 0,
    VLA_ERR_INVALID_ARG = 1,   /* NULL/misaligned pointer, bad size, dtype or scalar */
    VLA_ERR_UNSUPPORTED = 2,   /* head dimension not in {32, 64, 96, 128} */
    VLA_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
    VLA_ERR_TIMEOUT = 4,       /* a bounded in-kernel wait ran out; outputs are invalid */
    VLA_ERR_NONFINITE = 5      /* a NaN/Inf appeared in delta_t or the gate norm */
} vla_status;

typedef enum {
    VLA_F32 = 0,               /* q, k, v, u are float32 */
    VLA_BF16 = 1               /* q, k, v, u are bfloat16 (widened to fp32 on load) */
} vla_dtype;

/* Optional knobs of vla_forward_ex(). Zero-fill for the defaults. */
typedef struct {
    unsigned int wait_limit_us;  /* limit of every in-kernel wait, microseconds; 0 = 2,000,000 */
    int test_stall_producer;     /* TESTING ONLY: nonzero makes the input-staging warp publish
                                    nothing, so every consumer's bounded wait runs out and the
                                    call reports VLA_ERR_TIMEOUT without faulting the GPU */
    unsigned long long* trace;   /* PROFILING ONLY, builds compiled with -DVLA_TRACE: device buffer
                                    of 16*T u64 that receives per-token SM clock stamps of head 0
                                    (roles and sub-steps of the per-token kernel); else ignored */
    int algo;                    /* VLA_ALGO_*: which kernel runs the recurrence (0 = automatic) */
    int fixed_a;                 /* nonzero: the fixed-A variant ("Variational Linear Attention",
                                    §3.5 ablation): A is held at its initial value (A0, or I/lambda0)
                                    and eq. 9 is skipped, so alpha^_t = A0 k^_t / ||A0 k^_t||; u is
                                    not read and may be NULL. Runs on VLA_ALGO_CHUNKED (d <= 96;
                                    the A team only forms A0 k^), VLA_ALGO_CHUNKED_PAIR and
                                    VLA_ALGO_DECODE; VLA_ALGO_AUTO picks as for the full
                                    recurrence; VLA_ALGO_PER_TOKEN returns VLA_ERR_UNSUPPORTED */
    void* scratch;               /* the segmented path's buffers for this call, in place of the
                                    workspace past its status record (NULL: the workspace holds
                                    them). Device memory of scratch_bytes >=
                                    vla_workspace_bytes_ex(B, H, T, d, VLA_ALGO_SEGMENTED) bytes,
                                    256-byte aligned, laid out as that workspace (its first 256
                                    bytes unused), no zero-fill needed. With it, calls that may
                                    overlap on the GPU share one status record and each keeps
                                    buffers of its own; under VLA_ALGO_AUTO the segmented path is
                                    taken when either buffer holds them */
    size_t scratch_bytes;
} vla_options;

/* Kernels behind vla_forward_ex() (vla_options.algo). All compute eq. 9-11
 * exactly up to rounding order.
 *   VLA_ALGO_AUTO       decode kernel for T <= 4; with 3 * B * H at most the device's SM
 *                       count: VLA_ALGO_SEGMENTED for d <= 96 and T >= 1024 when the
 *                       workspace holds its buffers, else VLA_ALGO_CHUNKED_ROWS for d = 96
 *                       and 128; otherwise the chunked tensor-core kernel for d <= 96 and
 *                       the cluster-pair chunked kernel for d = 128
 *   VLA_ALGO_PER_TOKEN  one token at a time on the FMA pipes (any supported d)
 *   VLA_ALGO_CHUNKED    16 tokens at a time: the Sherman-Morrison steps of a chunk as an
 *                       LDL^T factorisation, the d x d products on the tcgen05 tensor cores
 *                       in 3-term tf32 (fp32 accuracy); d in {32, 64, 96}, else
 *                       VLA_ERR_UNSUPPORTED
 *   VLA_ALGO_DECODE     one token at a time with S and A in registers, laid out to stream
 *                       the carried state: for decode (T = 1) and short sequences (any d)
 *   VLA_ALGO_CHUNKED_PAIR  the chunked tensor-core recurrence on a cluster of two CTAs per
 *                       head: one SM runs the A-pass (eq. 9 and the gate of eq. 10) and
 *                       sends each chunk's gate to the other, which runs the S-pass
 *                       (eq. 10-11); each state has a whole SM's tensor memory, so d = 128
 *                       runs too (any supported d)
 *   VLA_ALGO_CHUNKED_ROWS  the chunked tensor-core recurrence on a cluster of 1 + NS CTAs
 *                       per head, the rows of S split over NS of them (the residual write
 *                       of eq. 10 acts on each row of S on its own): rank 0 runs the A-pass
 *                       and sends each chunk's gate to every S rank through distributed
 *                       shared memory; NS = 1 for d <= 64, 2 for d = 96 and 128 (any
 *                       supported d). Uses 1 + NS SMs per head, so that fewer heads than
 *                       SMs keep more of the chip busy
 *   VLA_ALGO_SEGMENTED  the sequence cut in two halves that run side by side (d <= 96,
 *                       T >= 32): A and z^key at the cut from the first half's prefix sums
 *                       of u^ u^^T (§3.2) and phi(k); the second half from S = 0 and, for the
 *                       transition, from S = I with v = 0 (eq. 12's composition); then
 *                       S_T = S_cut Pi_T + G_T and o_t += S_cut Pi_t phi_t / den_t. Three
 *                       chunked CTAs per head. Needs the larger workspace that
 *                       vla_workspace_bytes() reports (else VLA_ERR_INVALID_ARG)
 * Any other value: VLA_ERR_INVALID_ARG. */
enum { VLA_ALGO_AUTO = 0, VLA_ALGO_PER_TOKEN = 1, VLA_ALGO_CHUNKED = 2, VLA_ALGO_DECODE = 3,
       VLA_ALGO_CHUNKED_PAIR = 4, VLA_ALGO_CHUNKED_ROWS = 5, VLA_ALGO_SEGMENTED = 6 };

/* Bytes of device workspace vla_forward() needs for a call over B x H heads
 * of T tokens at head dimension d, with the kernel that VLA_ALGO_AUTO picks on
 * the current device (152 SMs assumed when no device answers). 256 bytes
 * (the status record: 16 bytes, the rest reserved) for every shape whose
 * kernel keeps all intermediates on chip. Where the segmented path serves the
 * shape (d <= 96, T >= 1024, 3 * B * H <= the SM count) it also holds that
 * path's buffers: per head a few d x d states and d-vectors plus T/2 x d
 * floats. A call given only 256 bytes keeps to the other kernels. 0 for
 * negative sizes or a d outside {32, 64, 96, 128}. The first 256 bytes must
 * be zero-filled before the first use (cudaMemset or vla_workspace_reset);
 * vla_get_last_device_status() clears them again. */
size_t vla_workspace_bytes(int B, int H, int T, int d);

/* The same for a given kernel choice `algo` (VLA_ALGO_*): what
 * vla_forward_ex() with that vla_options.algo needs. VLA_ALGO_AUTO gives
 * vla_workspace_bytes(); VLA_ALGO_SEGMENTED its buffers (0 where it does not
 * run: d = 128 or T < 32); every other kernel 256. 0 for invalid sizes or an
 * unknown algo. */
size_t vla_workspace_bytes_ex(int B, int H, int T, int d, int algo);

/* Zero the status record in `workspace` (asynchronous on `stream`). */
vla_status vla_workspace_reset(void* workspace, void* stream);

/*
 * vla_forward -- run eq. 9-11 over T tokens for all B*H heads (§3.3).
 *
 *  q, k, v, u   [B, H, T, d] device arrays of `dtype`, 16-byte aligned.
 *               May be NULL only when T == 0.
 *  B, H, T      sizes, >= 0 (B*H <= 2^31-1). T == 0 copies the initial
 *               state to the state outputs.
 *  d            head dimension, one of 32, 64, 96, 128.
 *  lambda0      > 0, finite: the default A_0 = I / lambda0 (the paper uses 0.1).
 *  eps          > 0, finite: the readout floor of eq. 11 (the paper uses 1e-4).
 *  S0, A0       [B, H, d, d] float32 carried-in state, or NULL for the defaults
 *               S_0 = 0 and A_0 = I / lambda0 (chunked or decode use passes the
 *               previous call's S_out / A_out here).
 *  zk0          [B, H, d] float32 carried-in z^key, or NULL for 0.
 *  o            [B, H, T, d] float32 output, 16-byte aligned (NULL only if T == 0).
 *  S_out, A_out [B, H, d, d] float32 final state, 16-byte aligned, required.
 *  zk_out       [B, H, d] float32 final z^key, or NULL to skip.
 *  workspace    device memory, its first 256 bytes zero-filled (the device status
 *               record), 16-byte aligned; 256 bytes suffice for every kernel but the
 *               segmented path, which needs vla_workspace_bytes(B, H, T, d) bytes and
 *               256-byte alignment (or its own buffers, vla_options.scratch). Those
 *               buffers are the call's scratch: calls that may overlap on the GPU
 *               (different streams, no ordering between them) need separate ones.
 *               The status record may be shared: the kernels OR their error bits
 *               into it atomically and keep the details of the first failure.
 *  stream       cudaStream_t as void*.
 *
 * Inputs and outputs must not overlap (S0/S_out, A0/A_out, zk0/zk_out may be
 * the same buffer: each head reads its initial state before it writes the
 * final one). Returns VLA_OK once the kernel is enqueued, or the first
 * argument / launch error.
 */
vla_status vla_forward(const void* q, const void* k, const void* v, const void* u,
                       vla_dtype dtype, int B, int H, int T, int d,
                       float lambda0, float eps,
                       const float* S0, const float* A0, const float* zk0,
                       float* o, float* S_out, float* A_out, float* zk_out,
                       void* workspace, size_t workspace_bytes, void* stream);

/* vla_forward with options (opts may be NULL = defaults). */
vla_status vla_forward_ex(const void* q, const void* k, const void* v, const void* u,
                          vla_dtype dtype, int B, int H, int T, int d,
                          float lambda0, float eps,
                          const float* S0, const float* A0, const float* zk0,
                          float* o, float* S_out, float* A_out, float* zk_out,
                          void* workspace, size_t workspace_bytes, void* stream,
                          const vla_options* opts);

/*
 * Synchronise `stream`, read and clear the status record that kernels on it
 * wrote into `workspace`. Returns VLA_OK, VLA_ERR_TIMEOUT (takes precedence)
 * or VLA_ERR_NONFINITE, or VLA_ERR_CUDA if the copy/sync itself failed.
 * If `detail` is not NULL it receives {role, head, token} of the first
 * recorded failure (role: 0 staging, 1 gate, 2 A-pass, 3 S-pass), or -1s.
 */
vla_status vla_get_last_device_status(void* workspace, void* stream, int* detail);

/*
 * vla_forward_noalloc -- the same operation as vla_forward, for callers that
 * cannot allocate device memory: code running under a fixed device-memory
 * budget that another runtime has already reserved in full (cudaMalloc would
 * fail), real-time or serving loops that must not call the allocator (it can
 * synchronise the device and fragment memory), and callers without any device
 * allocator of their own. The paper has no counterpart; this is an interface
 * convenience.
 *
 * Instead of a caller-provided workspace, the status record lives in a
 * file-scope __device__ array of the library (256 bytes, held by every device
 * that loads the library until the process exits). The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress) with the device
 * current and keeps it for the life of the process; make that first call
 * before any stream capture. cudaDeviceReset() (or anything else that tears
 * down the device's primary context) makes the kept address stale: this entry
 * point is not supported after such a reset. Every call clears the record
 * before its launch, so a call starts from a zero status. All calls share the
 * one record: calls that overlap on the GPU (different streams, no ordering)
 * race on it and their statuses are unreliable. The call allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine). It returns
 * VLA_ERR_UNSUPPORTED if the status record that vla_workspace_bytes(B, H, T, d)
 * asks for does not fit in the array. Arguments are as for vla_forward,
 * without workspace; if `device_status` is not NULL the call synchronises
 * `stream` after the launch and stores there the device-side status (VLA_OK,
 * VLA_ERR_TIMEOUT or VLA_ERR_NONFINITE); otherwise it returns as soon as the
 * work is enqueued. When the call itself returns an error, nothing was
 * launched and `device_status` (if not NULL) receives that same error.
 */
vla_status vla_forward_noalloc(const void* q, const void* k, const void* v, const void* u,
                               vla_dtype dtype, int B, int H, int T, int d,
                               float lambda0, float eps,
                               const float* S0, const float* A0, const float* zk0,
                               float* o, float* S_out, float* A_out, float* zk_out,
                               void* stream, int* device_status);

/*
 * vla_forward_host -- vla_forward (eq. 9-11 of §3.3, every head) over HOST
 * buffers, with the host<->device copies overlapped with the computation.
 *
 * The recurrence is causal: the state after token t is all that later tokens
 * need. The call therefore cuts the sequence into chunks of `chunk_tokens`
 * tokens (0 = automatic: about 4 chunks, multiples of 16 tokens, at least
 * 256) and runs one vla_forward_ex() launch per chunk over all heads, with
 * the state (S, A, z^key) carried in the workspace from launch to launch.
 * While chunk j computes on `stream`, the next chunks' q, k, v, u are copied
 * in and chunk j-1's o is copied out on streams of the library. The result
 * equals one vla_forward() over the whole sequence up to rounding order.
 *
 *  q, k, v, u   [B, H, T, d] HOST arrays of `dtype` (u may be NULL for the
 *               fixed-A variant). Page-locked memory (cudaHostAlloc,
 *               cudaHostRegister) gives the overlap; pageable memory works
 *               but each copy then waits for the host.
 *  S0, A0, zk0  HOST initial state as for vla_forward (NULL = defaults).
 *  o, S_out, A_out, zk_out   HOST outputs as for vla_forward (zk_out may be NULL).
 *               If o is page-locked and mapped into the device's address space
 *               (cudaHostGetDevicePointer succeeds, as for cudaHostAlloc memory)
 *               and 16-byte aligned, the kernels write o straight into it and
 *               only the final state is copied out; otherwise o is copied out
 *               chunk by chunk.
 *  chunk_tokens tokens per launch, >= 0 (0 = automatic; values above T mean T).
 *  workspace    device memory of vla_forward_host_workspace_bytes() bytes,
 *               256-byte aligned, its first 256 bytes zero-filled before the
 *               first use (the status record, read by
 *               vla_get_last_device_status(workspace, stream)). It holds the
 *               carried state and three input and three output slots of one chunk.
 *  stream, opts as for vla_forward_ex (the kernels run on `stream`).
 *
 * Asynchronous: returns once everything is enqueued. All work of the call,
 * copies included, is complete when `stream` reaches the point after the
 * call (e.g. cudaStreamSynchronize(stream)); until then the host buffers and
 * the workspace are in use. Copies start only after the work queued on
 * `stream` before the call. The first call on a device creates three streams
 * (two for copies in, one for copies out) and fourteen events that live until the
 * process exits; calls from several
 * host threads are serialised while they enqueue. Two calls that may overlap
 * on the GPU need separate workspaces. On an error return nothing the call
 * enqueued is still copying.
 */
size_t vla_forward_host_workspace_bytes(vla_dtype dtype, int B, int H, int T, int d, int chunk_tokens);

vla_status vla_forward_host(const void* q, const void* k, const void* v, const void* u,
                            vla_dtype dtype, int B, int H, int T, int d,
                            float lambda0, float eps,
                            const float* S0, const float* A0, const float* zk0,
                            float* o, float* S_out, float* A_out, float* zk_out,
                            int chunk_tokens, void* workspace, size_t workspace_bytes,
                            void* stream, const vla_options* opts);

/* Static text for a status code. */
const char* vla_status_string(vla_status s);

/*
 * Plain cumulative linear-attention state, the comparison of §4.1:
 * S_out[b, h] = sum_t v_t phi(k_t)^T ([B, H, d, d] float32, 16-byte aligned),
 * for k, v [B, H, T, d] of `dtype`. Used to report ||S_T||_F next to VLA's.
 */
vla_status vla_linear_attention_state(const void* k, const void* v, vla_dtype dtype,
                                      int B, int H, int T, int d,
                                      float* S_out, void* stream);

/* Bytes of device workspace vla_backward() needs for (B, H, T, d): one status
 * record, a per-token tape of the forward pass (z_t, alpha^_t, e_t, delta_t,
 * ||A_t k^_t||, den_t, ||u_t||^2, ||k_t||^2: 3d + 8 floats per head-token) and
 * S, A, z^key checkpoints every 64 tokens (2 d^2 + d floats each), and the
 * forward's final S, A, z^key (2 d^2 + d floats per head). 0 if the
 * sizes overflow. */
size_t vla_backward_workspace_bytes(int B, int H, int T, int d);

/* Reverse-mode gradient of vla_forward() (the backward pass of the recurrence
 * of "Variational Linear Attention", §3.3 eq. 9-11; §4.2 eq. 14 is the state
 * Jacobian it propagates, and Corollary 1 bounds the result).
 *
 * For a scalar loss L of the forward outputs, given the upstream gradients
 *   dO    [B,H,T,d] = dL/do                    (NULL: zero)
 *   dS_T, dA_T [B,H,d,d] = dL/dS_T, dL/dA_T     (NULL: zero)
 *   dzk_T [B,H,d]   = dL/dz^key_T               (NULL: zero)
 * it writes dq, dk, dv, du [B,H,T,d] = dL/dq_t ... (fp32) and, where not NULL,
 * dS0, dA0 [B,H,d,d] and dzk0 [B,H,d] = dL/d(initial state). q, k, v, u,
 * dtype, sizes, lambda0, eps and the optional initial state (S0, A0, zk0) are
 * those of the forward call; the forward pass is recomputed inside. A0, when
 * given, must be symmetric, as every state of the recurrence is (A_t is the
 * inverse of a symmetric matrix); the kernel uses A_t^T = A_t.
 *
 * Layout and ownership as for vla_forward(); every gradient is fp32,
 * row-major, caller-owned device memory, 16-byte aligned (state pointers
 * 4-byte). workspace: device memory of vla_backward_workspace_bytes() bytes,
 * 16-byte aligned, its first 16 bytes zero-filled (status record, read by
 * vla_get_last_device_status). Asynchronous on `stream`.
 * For d <= 96 the reverse sweep is one kernel per head holding S, A and their
 * adjoints; for d = 128, where those four d x d matrices do not fit one SM,
 * it is the split sweep of vla_backward_split().
 * Errors: VLA_ERR_INVALID_ARG as for vla_forward() (including a workspace
 * smaller than required); VLA_ERR_UNSUPPORTED for d outside
 * {32, 64, 96, 128}; VLA_ERR_NONFINITE is recorded on the device when a
 * gradient or an intermediate is NaN/Inf. */
vla_status vla_backward(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype,
                        int B, int H, int T, int d, float lambda0, float eps,
                        const float* S0, const float* A0, const float* zk0,
                        const float* dO, const float* dS_T, const float* dA_T, const float* dzk_T,
                        float* dq, float* dk, float* dv, float* du,
                        float* dS0, float* dA0, float* dzk0,
                        void* workspace, size_t workspace_bytes, void* stream);

/* vla_backward() with the reverse sweep split by state, for any supported d
 * (the path d = 128 always takes). The adjoint recursion of S (eq. 10, 11)
 * needs nothing from the A side, and the A side (eq. 9, 10) needs only the
 * gate's gradient g_a = (g_alpha - alpha^ (alpha^ . g_alpha)) / ||A_t k^_t||
 * per token from it. So one kernel runs a cluster of two CTAs per head: one
 * sweeps t = T-1 .. 0 with S and its adjoint, writing dq, dv, the S part of
 * dk and g_a (into the workspace's tape); the other sweeps with A and its
 * adjoint a few tokens behind, as the first publishes its progress, writing
 * du and adding the A part of dk. Same arguments, workspace size, results
 * (to rounding) and errors as vla_backward(), and VLA_ERR_TIMEOUT if the A
 * side's wait for the S side's progress (2 s) runs out. */
vla_status vla_backward_split(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype,
                              int B, int H, int T, int d, float lambda0, float eps,
                              const float* S0, const float* A0, const float* zk0,
                              const float* dO, const float* dS_T, const float* dA_T, const float* dzk_T,
                              float* dq, float* dk, float* dv, float* du,
                              float* dS0, float* dA0, float* dzk0,
                              void* workspace, size_t workspace_bytes, void* stream);

/* vla_backward() (split == 0) or vla_backward_split() (split != 0) with
 * options (opts may be NULL = defaults). Of vla_options only two fields apply:
 *   wait_limit_us        limit of the split sweep's one wait, where the A side
 *                        waits for the S side's progress (0 = 2,000,000). The
 *                        forward pass before the sweep takes the same limit.
 *   test_stall_producer  TESTING ONLY: nonzero makes the split sweep's S side
 *                        publish no progress. The A side's wait then runs out
 *                        and the call records VLA_ERR_TIMEOUT, without faulting
 *                        the GPU; the gradients are then not meaningful. The
 *                        single-kernel sweep (split == 0 at d <= 96) has no
 *                        wait, and the flag does nothing there.
 * The other fields are ignored. */
vla_status vla_backward_ex(const void* q, const void* k, const void* v, const void* u, vla_dtype dtype,
                           int B, int H, int T, int d, float lambda0, float eps,
                           const float* S0, const float* A0, const float* zk0,
                           const float* dO, const float* dS_T, const float* dA_T, const float* dzk_T,
                           float* dq, float* dk, float* dv, float* du,
                           float* dS0, float* dA0, float* dzk0,
                           void* workspace, size_t workspace_bytes, void* stream,
                           int split, const vla_options* opts);

#ifdef __cplusplus
}
#endif

#endif /* VLA_GB300_H */
