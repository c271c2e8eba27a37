/*
 * m3scan.h -- C ABI of libm3scan.so, the B300 (sm_103a) Mamba-3 selective
 * SSM scan: a chunked prefill (m3_scan_fwd; m3_scan_fwd_from continues a
 * sequence from a state; m3_scan_fwd_bcnorm fuses the block's B / C
 * normalisation; m3_scan_fwd_host takes host buffers and overlaps the copies
 * with the scan), its backward pass (m3_scan_bwd), a single-token decode step
 * (m3_step) and a k-token decode step (m3_step_k).
 *
 * The operation (Mamba-3 summary page, "Mamba-3: Expressive SSM with MIMO"):
 * for every batch row b and head h independently, with scalar A_h < 0 and
 *
 *   alpha_t = exp(dt_t A_h), beta_t = (1 - lambda_t) dt_t alpha_t,
 *   gamma_t = lambda_t dt_t                       (§3.1.1, eq. (5)-(6))
 *   u_t     = sum_r B_t[r] x_t[r]^T   (N x P)     (§3.3, MIMO rank R)
 *   h'_t    = Rot(theta_t) (alpha_t h'_{t-1} + beta_t u_{t-1}) + gamma_t u_t
 *   y_t[r]  = C_t[r]^T h'_t
 *
 * where Rot(theta_t) rotates every state row pair (2k, 2k+1), k < N/2, by the
 * angle theta_t[k]:  (a, b) -> (a cos - b sin, a sin + b cos)  -- the complex
 * state of §3.2 (Proposition 3.2.1) written as real 2x2 blocks.  theta_t is the
 * per-step angle and already includes dt.  The prefill computes it in the
 * rotated (data-dependent RoPE) frame of Propositions 3.2.2 / 3.2.3, with the
 * trapezoid mask of eq. (7); the state it returns is in the complex frame
 * above, the same frame m3_step reads and writes, so decode continues a
 * prefill directly.  lambda = 1 and theta = 0 give the Mamba-2 (SSD) update.
 *
 * Conventions for every entry point:
 *  - Pointers are CUDA device pointers (device memory or managed memory the
 *    device can read; m3_scan_fwd_host's tensors are host memory) owned by
 *    the caller, C-contiguous and aligned to their element size; the fp32 state / final_state must be 16-byte aligned, and
 *    the tensor-core prefill (M3_ALGO_CHUNKED_TC) also needs x, B, C, theta
 *    and y 16-byte aligned (it returns M3_ERR_ALIGN otherwise).
 *    The library never allocates device memory and never frees a pointer;
 *    scratch (m3_scan_bwd) is a caller-owned workspace.
 *  - Arguments are validated on the host before any launch; on error nothing
 *    is launched and a negative status is returned.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns before it completes.
 *  - Device-side errors (a bounded wait that ran out) are recorded in a
 *    per-device status word; m3_device_status() reads and clears it.
 *  - Not thread-safe per device for concurrent calls only in that the status
 *    word is shared; outputs never overlap inputs.
 */
#ifndef M3SCAN_H
#define M3SCAN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define M3_API __attribute__((visibility("default")))
#else
#define M3_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of x, B, C, theta, y (and of x_t, B_t, C_t, theta_t, prev_B,
 * prev_x, y_t for m3_step).  dt, lambda, A and the state are always fp32. */
typedef enum { M3_F32 = 0, M3_BF16 = 1 } m3_dtype;

/* Problem sizes.  batch b >= 0, seqlen T >= 0 (ignored by m3_step),
 * heads h >= 1, headdim P in [4, 256] with P % 4 == 0, dstate N in [2, 256]
 * even, rank R in [1, 8], chunk Q in {16, 32, 64, 128} (tokens per chunk of
 * the prefill, executed as given by the chunked kernels; the result does not
 * depend on it beyond rounding). */
typedef struct {
    int64_t batch;
    int64_t seqlen;
    int64_t heads;
    int64_t headdim;  /* P */
    int64_t dstate;   /* N */
    int64_t rank;     /* R, 1 = SISO */
    int64_t chunk;    /* Q */
    int32_t dtype;    /* m3_dtype */
    int32_t reserved; /* must be 0 */
} m3_dims;

/* Status codes. */
#define M3_OK 0
#define M3_ERR_NULL (-1)        /* a required pointer is NULL */
#define M3_ERR_SHAPE (-2)       /* a size is out of range */
#define M3_ERR_DTYPE (-3)       /* unknown dtype */
#define M3_ERR_ALIGN (-4)       /* a pointer is not aligned as required */
#define M3_ERR_CUDA (-5)        /* a CUDA call or launch failed (no device, ...) */
#define M3_ERR_UNSUPPORTED (-6) /* valid sizes no kernel of the library takes */
#define M3_ERR_DEVICE (-7)      /* the device status word was set */
#define M3_ERR_WORKSPACE (-8)   /* workspace too small */
#define M3_ERR_VALUE (-9)       /* a scalar argument is out of range (e.g. a negative epsilon) */

/* Prefill algorithms (what m3_scan_fwd would run for given dims).  Both
 * chunked kernels execute exactly d->chunk tokens per chunk. */
#define M3_ALGO_NONE (-1)         /* no kernel for these dims */
#define M3_ALGO_SEQUENTIAL 0      /* CUDA-core kernel, one token at a time (no chunks) */
#define M3_ALGO_CHUNKED_TC 1      /* chunked tcgen05 (tensor core) kernel */
#define M3_ALGO_CHUNKED_SIMT 2    /* chunked kernel on CUDA cores, fp32 arithmetic */

/* Bytes of device workspace m3_scan_fwd needs for `d` (0 for every forward
 * kernel of the library).  Returns 0 for invalid dims as well. */
M3_API size_t m3_scan_workspace_size(const m3_dims* d);

/* Which prefill kernel m3_scan_fwd runs for `d` (M3_ALGO_NONE for invalid
 * dims):
 *   M3_ALGO_CHUNKED_TC    bf16 inputs, P == 64, N in {64, 128}, R in {1, 2, 4}
 *                         and chunk * R == 64 (one 64-row tile per chunk:
 *                         Q = 64, 32, 16 tokens for R = 1, 2, 4);
 *   M3_ALGO_CHUNKED_SIMT  every other shape and chunk, fp32 or bf16, whose
 *                         chunk fits in shared memory (inputs staged in their
 *                         dtype: about (2 N + P) chunk R elements, the fp32
 *                         N x P state and a 64-row block of the chunk's mask);
 *   M3_ALGO_SEQUENTIAL    the rest (one token at a time).
 * The result does not depend on the algorithm or the chunk beyond rounding. */
M3_API int m3_scan_algorithm(const m3_dims* d);

/* Chunked prefill from the zero state (Mamba-3 summary page §3.1-§3.3; the
 * chunked evaluation is the SSD intra-chunk / inter-chunk split of the
 * Mamba-2 chapter page, "Foundation Model Engineering" ch. 20.2 §2).
 *   x      [b, T, h, R, P]  dtype
 *   dt     [b, T, h]        fp32, > 0
 *   A      [h]              fp32, <= 0
 *   B, C   [b, T, h, R, N]  dtype
 *   lambda [b, T, h]        fp32 in [0, 1], or NULL for lambda = 1
 *   theta  [b, T, h, N/2]   dtype, or NULL for theta = 0
 *   y      [b, T, h, R, P]  dtype, written
 *   final_state [b, h, N, P] fp32, written (complex frame), or NULL
 *   workspace / workspace_bytes: device scratch of at least
 *          m3_scan_workspace_size(d) bytes (may be NULL when that is 0).
 * Returns M3_OK or a negative status; T == 0 writes only final_state (zero). */
M3_API int m3_scan_fwd(const m3_dims* d, const void* x, const float* dt, const float* A,
                const void* B, const void* C, const float* lambda, const void* theta,
                void* y, float* final_state, void* workspace, size_t workspace_bytes,
                void* stream);

/* Prefill with inputs and outputs in HOST memory: the scan of m3_scan_fwd for
 * a caller whose data lives on the host.  The pages have no counterpart; this
 * is the runtime around the scan: the batch is processed in slices of `slice`
 * batch rows (every (b, h) sequence is independent, so a slice is a smaller
 * call of the same kernel and its results are bit-identical to one call over
 * the whole batch).  Each slice's inputs are copied into one of two device
 * staging sets in `workspace`, scanned on `stream`, and its y and final_state
 * copied back; the copies of one slice overlap the scans and copies of the
 * others (host-to-device and device-to-host run on two streams of the
 * library's own, forked from and joined back to `stream` with events).
 *   x, dt, A, B, C, lambda, theta   host memory, layouts and NULL rules as in
 *                                   m3_scan_fwd (A [h] included)
 *   y, final_state                  host memory, written (final_state may be NULL)
 *   Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 *   the copies to overlap; pageable memory works without the overlap.  They
 *   must stay valid until `stream` completes.
 *   slice      batch rows per slice, >= 0 (0: ceil(batch / 8); M3_ERR_VALUE if < 0)
 *   workspace  device memory, 256-byte aligned (M3_ERR_ALIGN), of at least
 *              m3_scan_fwd_host_workspace_size(d, slice) bytes (M3_ERR_WORKSPACE);
 *              in use until `stream` completes.
 * Returns once everything is enqueued; `stream` completes when y and
 * final_state are in host memory.  The copy streams and their events are made on
 * a device's first call and kept (handles only: the library still allocates no
 * device memory; made again after a device reset); calls from several host
 * threads are serialised while they enqueue.  T == 0 writes only final_state (zero). */
M3_API size_t m3_scan_fwd_host_workspace_size(const m3_dims* d, int64_t slice);
M3_API int m3_scan_fwd_host(const m3_dims* d, const void* x, const float* dt, const float* A,
                     const void* B, const void* C, const float* lambda, const void* theta,
                     void* y, float* final_state, int64_t slice, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Prefill that continues a sequence: the same computation as m3_scan_fwd,
 * started from a given state instead of zero (the chunked-prefill continuation
 * of a serving loop: prefill -> decode -> prefill ...).  With h_{-1} the state
 * before x's first token and u_{-1} = sum_r prev_B[r] prev_x[r]^T the input of
 * the token before it, the first token's update is
 *   h'_0 = Rot(theta_0)(alpha_0 h_{-1} + beta_0 u_{-1}) + gamma_0 u_0
 * (Mamba-3 summary page §3.1 eq. (5): the previous-token term), and the rest
 * as in m3_scan_fwd.
 *   initial_state [b, h, N, P] fp32, complex frame (the frame final_state and
 *                 m3_step use), 16-byte aligned, or NULL for zero
 *   prev_B [b, h, R, N], prev_x [b, h, R, P]  dtype: the previous token's B and
 *                 x, or both NULL (no previous token)
 * Every other argument as in m3_scan_fwd.  T == 0 copies initial_state (or
 * zero) to final_state. */
M3_API int m3_scan_fwd_from(const m3_dims* d, const void* x, const float* dt, const float* A,
                     const void* B, const void* C, const float* lambda, const void* theta,
                     const float* initial_state, const void* prev_B, const void* prev_x,
                     void* y, float* final_state, void* workspace, size_t workspace_bytes,
                     void* stream);

/* Prefill with the B / C normalisation and biases of the Mamba-3 block fused
 * into the prologue (Mamba-3 summary page, §3.4: an RMS normalisation of the B
 * and C projections, then a learnable bias per head and per channel, then the
 * data-dependent rotation).  The pages fix neither the norm's scale nor its
 * epsilon; this entry point takes a scale per channel shared by the heads and
 * ranks and a bias per head and channel shared by the ranks:
 *   B^[b,t,h,r,n] = B[b,t,h,r,n] / sqrt(mean_n' B[b,t,h,r,n']^2 + eps) * norm_B[n]
 *                   + bias_B[h,n]             (C likewise with norm_C, bias_C)
 * and runs the scan of m3_scan_fwd on the raw B, C with B^, C^ in their place.
 * The arithmetic is fp32.  With theta, B^ is rounded to bf16 after the
 * normalisation and again after the rotation, C^ once after its rotation;
 * without theta each is rounded once.  With eps == 0 an all-zero row of B or C
 * has no defined normalisation (0 / 0); the kernel maps it to the bias.
 *   norm_B, norm_C [N]     fp32   bias_B, bias_C [h, N] fp32   (all required)
 *   eps                    finite, >= 0 (M3_ERR_VALUE otherwise)
 * Every other argument as in m3_scan_fwd.  Only the tensor-core kernel's shapes
 * take it (bf16, P = 64, N in {64, 128}, R in {1, 2, 4}); other shapes return
 * M3_ERR_UNSUPPORTED.  The decode step takes B_t, C_t already normalised (a few
 * hundred bytes per token next to the state).  T == 0 writes only final_state
 * (zero). */
M3_API int m3_scan_fwd_bcnorm(const m3_dims* d, const void* x, const float* dt, const float* A,
                       const void* B, const void* C, const float* lambda, const void* theta,
                       const float* norm_B, const float* norm_C, const float* bias_B,
                       const float* bias_C, float eps, void* y, float* final_state,
                       void* workspace, size_t workspace_bytes, void* stream);

/* One decode step for every (b, h) (same recurrence, one token):
 *   state   [b, h, N, P]  fp32, read and overwritten with h'_t (complex frame)
 *   x_t     [b, h, R, P]  dtype      dt_t, lambda_t [b, h] fp32 (lambda_t may
 *   B_t,C_t [b, h, R, N]  dtype      be NULL for 1)       A [h] fp32
 *   theta_t [b, h, N/2]   dtype, the angle of this step (NULL for 0)
 *   prev_B  [b, h, R, N], prev_x [b, h, R, P]  dtype: the previous token's B
 *           and x (the beta term's B_{t-1} x_{t-1}^T); both NULL for none.
 *   y_t     [b, h, R, P]  dtype, written.
 * d->seqlen and d->chunk are ignored.  The caller keeps (B_t, x_t) as the next
 * call's (prev_B, prev_x). */
M3_API int m3_step(const m3_dims* d, float* state, const void* x_t, const float* dt_t,
            const float* A, const void* B_t, const void* C_t, const float* lambda_t,
            const void* theta_t, const void* prev_B, const void* prev_x, void* y_t,
            void* stream);

/* Bytes of device workspace m3_scan_bwd needs for `d` (0 when m3_scan_bwd does
 * not take these dims): the chunk states of every (b, h), (ceil(T / chunk) + 1)
 * N P fp32 each, the angles at every chunk start and one float per (b, h). */
M3_API size_t m3_scan_bwd_workspace_size(const m3_dims* d);

/* Backward pass of the prefill from the zero state (m3_scan_fwd): given the
 * upstream gradients dy of y and dfinal of final_state, the gradients of
 *   L = <dy, y> + <dfinal, final_state>
 * with respect to every input, for training (the recompute-in-backward of the
 * Mamba-1 review page, "hardware-aware algorithm" step 4; the chunked training
 * path of "Foundation Model Engineering" ch. 20.2).  A first pass recomputes
 * the chunk states into the workspace; a second pass walks the chunks in
 * reverse and differentiates the chunked form (the intra-chunk mask, the
 * inter-chunk term, the state update, the trapezoid weights, the cumulative
 * rotation); a third sums dA over the batch.  bf16 with N = P = 64, R in
 * {1, 2, 4}, chunk R = 64 and x, B, C, theta, dy, dx, dB, dC, dtheta 16-byte
 * aligned runs the chunk products on the tensor cores (bf16 operands, fp32
 * accumulators and epilogues); every other case in fp32 on CUDA cores.  Both
 * are deterministic (fixed-order sums).
 *   x, dt, A, B, C, lambda, theta   the forward's inputs (as in m3_scan_fwd)
 *   dy      [b, T, h, R, P]  dtype        dfinal [b, h, N, P] fp32 or NULL (0)
 *   dx      [b, T, h, R, P]  dtype        ddt    [b, T, h]    fp32
 *   dA      [h]              fp32 (summed over the batch and time)
 *   dB, dC  [b, T, h, R, N]  dtype
 *   dlambda [b, T, h] fp32 (required when lambda is given, else ignored)
 *   dtheta  [b, T, h, N/2] dtype (required when theta is given, else ignored)
 *   workspace: >= m3_scan_bwd_workspace_size(d) bytes, 256-byte aligned
 *           (M3_ERR_WORKSPACE if smaller).
 * Takes chunk * R <= 64 rows per chunk (M3_ERR_UNSUPPORTED otherwise, or when
 * a chunk does not fit in shared memory: N = P = 64 takes chunk 64 at R = 1).
 * The chunk changes only the rounding.  T == 0 writes dA = 0 only. */
M3_API int m3_scan_bwd(const m3_dims* d, const void* x, const float* dt, const float* A,
                       const void* B, const void* C, const float* lambda, const void* theta,
                       const void* dy, const float* dfinal, void* dx, float* ddt, float* dA,
                       void* dB, void* dC, float* dlambda, void* dtheta, void* workspace,
                       size_t workspace_bytes, void* stream);

/* m3_scan_bwd for callers that cannot allocate device memory -- a host whose
 * allocator belongs to another runtime or framework, a process held to a fixed
 * memory budget, or code that must not call the allocator inside a serving
 * loop.  The pages have no counterpart: this is an interface choice.  Same
 * arguments and result as m3_scan_bwd, without the workspace: the scratch is a
 * fixed 32 MiB array inside the library's device image, present on every GPU
 * that loads the library until the process exits.
 *   - Sizes whose workspace (m3_scan_bwd_workspace_size) exceeds 32 MiB are
 *     rejected with M3_ERR_WORKSPACE before anything runs.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it, per context (after a device reset
 *     it is looked up again); make that first call before any stream capture.
 *   - Every call on a device shares the one array.  Calls whose work overlaps
 *     on the GPU (other streams, other host threads) race on it and corrupt
 *     each other's result: order them on one stream or synchronise.  No part of
 *     the array needs to start at zero (every byte a call reads it wrote
 *     first), so the previous call's contents do no harm.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine. */
M3_API int m3_scan_bwd_noalloc(const m3_dims* d, const void* x, const float* dt, const float* A,
                               const void* B, const void* C, const float* lambda, const void* theta,
                               const void* dy, const float* dfinal, void* dx, float* ddt, float* dA,
                               void* dB, void* dC, float* dlambda, void* dtheta, void* stream);

/* k decode steps in one launch (multi-token / speculative decode): the same
 * recurrence over k = d->seqlen consecutive tokens of every (b, h), reading
 * and writing the state once instead of k times (Mamba-3 summary page §3.3:
 * decode is bound by the state's bytes, so k tokens per pass over the state
 * raise the arithmetic intensity about k-fold).  The result equals k m3_step
 * calls, and m3_scan_fwd_from over the same k tokens.
 *   state   [b, h, N, P]    fp32, read and overwritten with the state after
 *                           the k-th token (complex frame), 16-byte aligned
 *   x [b, k, h, R, P], B / C [b, k, h, R, N], theta [b, k, h, N/2] (or NULL)
 *           dtype, token-major as in m3_scan_fwd
 *   dt, lambda [b, k, h]    fp32 (lambda may be NULL for 1)   A [h] fp32
 *   prev_B [b, h, R, N], prev_x [b, h, R, P]  dtype: the token before the
 *           first one (both NULL for none)
 *   y       [b, k, h, R, P] dtype, written
 * d->chunk is ignored; k == 0 does nothing.  For P in {32, 64, 128}, N % 8 == 0,
 * R in {1, 2, 4} with 16-byte aligned state, x, B, C, theta, prev_B and prev_x
 * one kernel keeps the state in registers across the k tokens; other shapes
 * run the continued prefill on the state in place. */
M3_API int m3_step_k(const m3_dims* d, float* state, const void* x, const float* dt, const float* A,
                     const void* B, const void* C, const float* lambda, const void* theta,
                     const void* prev_B, const void* prev_x, void* y, void* stream);

/* Reads and clears the device status word of the current device after
 * synchronising `stream`: M3_OK, M3_ERR_DEVICE if a kernel reported a
 * device-side error since the last call, or M3_ERR_CUDA. */
M3_API int m3_device_status(void* stream);

/* Self-test of the failure detection (no counterpart on the pages): launches
 * one CTA whose first thread waits, with a budget of budget_cycles clock
 * cycles, on an mbarrier that nothing completes -- the bounded wait every
 * kernel of this library uses.  When the budget runs out the thread records a
 * wait timeout in the device status word and the kernel returns, leaving the
 * context usable; m3_device_status() then returns M3_ERR_DEVICE and clears it.
 *   budget_cycles  in [1, 4e9] (M3_ERR_VALUE otherwise)
 * Returns M3_OK once the launch is enqueued, or M3_ERR_CUDA. */
M3_API int m3_selftest_wait_timeout(long long budget_cycles, void* stream);

/* Static text for a status code. */
M3_API const char* m3_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* M3SCAN_H */
