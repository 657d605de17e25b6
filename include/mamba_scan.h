/*
 * mamba_scan.h: C ABI of the GB300 (sm_103a) selective-scan library, libmambascan.so.
 *
 * The operation is the selective state-space scan of a Mamba layer and its reverse-time
 * backward (BPTT). With A = -exp(A_log), it runs independently for every row (b, d) and every
 * state n:
 *
 *   h_t[d,n] = exp(delta_t[d] * A[d,n]) * h_{t-1}[d,n] + delta_t[d] * u_t[d] * B_t[n],  h_{-1} = 0
 *   y_t[d]   = sum_n C_t[n] * h_t[d,n] + D[d] * u_t[d]
 *   out_t[d] = y_t[d] * SiLU(gate_t[d])
 *
 * The backward follows mamba-rs src/mamba_ssm/cpu/backward.rs. Phase B2 is the gating
 * backward: d_y = dy * SiLU(gate), d_gate = dy * y * sigmoid(g) * (1 + g * (1 - sigmoid(g))).
 * Phase B3 is the sequential SSM BPTT. Running t from T-1 down to 0 with d_h = 0 at t = T, it
 * does d_h += d_y*C, then accumulates d_delta, d_u, d_B, d_C, d_A_log and d_D, and finally
 * sets d_h = exp(delta*A) * d_h. The pre-computation a_neg = -exp(A_log), which saves
 * d_inner*d_state transcendentals per step, is that file's "O3" optimisation. Here it runs
 * once per call, inside the kernels.
 *
 * Conventions for every entry point below.
 *  - Tensors are float32, row-major, dense, in DEVICE memory owned by the caller:
 *      delta, u, gate, dy, out, y, d_delta, d_u, d_gate : [batch, T, d_inner]  (d fastest)
 *      B, C, d_B, d_C                                   : [batch, T, d_state]  (n fastest)
 *      A_log, d_A_log                                   : [d_inner, d_state]
 *      D, d_D                                           : [d_inner]
 *    Every pointer must be 16-byte aligned. Inputs are read-only. Outputs must not alias any
 *    input or one another.
 *  - The library never allocates or frees memory. The checkpoint buffer and the scratch
 *    buffer are sized by the *_bytes functions and owned by the caller.
 *  - Calls are asynchronous on `stream`. `stream` is a cudaStream_t passed as void*; NULL
 *    means the legacy default stream. The call returns after enqueueing the work, and errors
 *    that surface only on the device appear at the next synchronisation
 *    (see mamba_scan_status).
 *  - Gradients are OVERWRITTEN, not accumulated. This deviates from the page's `+=` into
 *    weight gradients. d_A_log and d_D are summed over batch and time, d_B and d_C over
 *    d_inner.
 *  - dy is the gradient of the loss with respect to `out`. d_delta is taken with respect to
 *    the post-softplus delta that is passed in, and d_gate with respect to the pre-SiLU gate.
 *  - Sizes: batch >= 1, T >= 1, d_inner >= 1, 1 <= d_state <= 64, batch <= 65535,
 *    batch*T*d_inner < 2^31 and batch*T*d_state < 2^31.
 *  - Results are deterministic: the same inputs give bitwise-identical outputs on every call.
 *
 * Return codes (int): MAMBA_OK or one of the errors below. On any error nothing is launched,
 * except for MAMBA_ERR_CUDA, which reports a launch failure.
 */
#ifndef MAMBA_SCAN_H
#define MAMBA_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MAMBA_OK 0
#define MAMBA_ERR_INVALID_ARG 1 /* null pointer, size out of range, or aliasing outputs      */
#define MAMBA_ERR_MISALIGNED 2  /* a pointer is not 16-byte aligned                          */
#define MAMBA_ERR_WORKSPACE 3   /* checkpoint or scratch buffer smaller than required        */
#define MAMBA_ERR_CUDA 4        /* a CUDA runtime call or kernel launch failed               */
#define MAMBA_ERR_UNSUPPORTED 5 /* d_state outside 1..64, or sizes a variant does not take
                                   (mamba_scan_fwd_bwd_bf16, mamba_conv_*)                   */
#define MAMBA_ERR_NOALLOC_LIMIT 6 /* mamba_scan_bwd_noalloc: the sizes need more scratch than
                                     MAMBA_SCAN_NOALLOC_SCRATCH_BYTES                        */
#define MAMBA_ERR_TIMEOUT 7     /* reported by mamba_scan_status: a kernel gave up waiting
                                   (1 s) for one of its own asynchronous copies; the outputs
                                   of the calls since the last status check are invalid     */
#define MAMBA_ERR_BOUNDS 8      /* reported by mamba_scan_status of a bounds-checked build
                                   (libmambascan_checked.so): a kernel computed an offset
                                   outside its buffer; the access was not made, and the
                                   outputs since the last status check are invalid          */

/* Bytes of the checkpoint buffer that mamba_scan_fwd writes and mamba_scan_bwd reads. The
 * forward stores the state h at every 16-step chunk boundary of the time axis, so that the
 * backward recomputes h inside one chunk at a time instead of storing it for every t. It also
 * stores the per-segment aggregates of its time-parallel scan, and y = sum_n C*h + D*u, which
 * the gating backward needs. The layout is internal to the library. Returns 0 for invalid
 * sizes; mamba_scan_fwd then reports the error. */
size_t mamba_scan_ckpt_bytes(int64_t batch, int64_t T, int64_t d_inner, int64_t d_state);

/* Bytes of the scratch buffer mamba_scan_bwd needs for its deterministic two-level reductions
 * (per-CTA partial sums of d_B, d_C, d_A_log, d_D, summed in a fixed order by a second kernel).
 * The contents need no initialisation and are meaningless after the call. */
size_t mamba_scan_scratch_bytes(int64_t batch, int64_t T, int64_t d_inner, int64_t d_state);

/* Forward scan. Writes out and, when y is non-NULL, y = sum_n C*h + D*u (the pre-gate
 * output). Writes the checkpoint buffer (ckpt_bytes >= mamba_scan_ckpt_bytes(...)).
 * Mamba-rs keeps h_prev, h_curr and exp(delta*A) for every t (the "MambaLayerFlat"
 * activations); this library keeps only the chunk-boundary states. */
int mamba_scan_fwd(const float* delta, const float* u, const float* B, const float* C,
                   const float* gate, const float* A_log, const float* D, float* out, float* y,
                   void* ckpt, size_t ckpt_bytes, int64_t batch, int64_t T, int64_t d_inner,
                   int64_t d_state, void* stream);

/* Backward scan (Phases B2 and B3 of the page). Needs the inputs of the matching forward call
 * and the checkpoint buffer it wrote. Writes all seven gradients. The scratch buffer must hold
 * mamba_scan_scratch_bytes(...) bytes. Scratch and ckpt must not overlap each other or any
 * other argument. */
int mamba_scan_bwd(const float* delta, const float* u, const float* B, const float* C,
                   const float* gate, const float* A_log, const float* D, const float* dy,
                   const void* ckpt, size_t ckpt_bytes, void* scratch, size_t scratch_bytes,
                   float* d_delta, float* d_u, float* d_B, float* d_C, float* d_A_log,
                   float* d_D, float* d_gate, int64_t batch, int64_t T, int64_t d_inner,
                   int64_t d_state, void* stream);

/* The same two passes with the softplus in front of the scan fused into the kernels (the
 * Softplus backward step of the page, with its threshold 20; the forward applies
 * delta = raw > 20 ? raw : log(1 + exp(raw)), the function whose derivative that step takes).
 * `delta_raw` replaces `delta`, with the same layout, in both calls. The backward writes
 * d_delta_raw = d_delta * (raw > 20 ? 1 : sigmoid(raw)) in place of d_delta. Everything else,
 * including the checkpoint and scratch sizes and the error codes, is as for mamba_scan_fwd
 * and mamba_scan_bwd. */
int mamba_scan_fwd_softplus(const float* delta_raw, const float* u, const float* B,
                            const float* C, const float* gate, const float* A_log,
                            const float* D, float* out, float* y, void* ckpt,
                            size_t ckpt_bytes, int64_t batch, int64_t T, int64_t d_inner,
                            int64_t d_state, void* stream);
int mamba_scan_bwd_softplus(const float* delta_raw, const float* u, const float* B,
                            const float* C, const float* gate, const float* A_log,
                            const float* D, const float* dy, const void* ckpt,
                            size_t ckpt_bytes, void* scratch, size_t scratch_bytes,
                            float* d_delta_raw, float* d_u, float* d_B, float* d_C,
                            float* d_A_log, float* d_D, float* d_gate, int64_t batch, int64_t T,
                            int64_t d_inner, int64_t d_state, void* stream);

/* Forward and backward in one call, for a training step in which dy is known before the
 * forward runs (the page's layer forward followed by its Phases B2 and B3). Writes out and the
 * seven gradients, exactly what mamba_scan_fwd followed by mamba_scan_bwd writes (y is not
 * returned). Same inputs, layouts, checkpoint and scratch buffers (mamba_scan_ckpt_bytes,
 * mamba_scan_scratch_bytes) and error codes; out must not overlap any other argument, and
 * every check runs before the first launch. For d_state 9..16 the forward pass keeps only the
 * chunk-boundary states (it reads neither C nor gate and writes neither out nor y) and the
 * backward forms y = sum_n C*h + D*u from the states it recomputes anyway, so out, y and the
 * gate are not carried through device memory between the passes. For d_state 17..64, where
 * that reduction costs the backward more than it saves, and for d_state <= 8, the call runs
 * the two passes as the separate entry points do. The checkpoint buffer's contents
 * afterwards are unspecified. Asynchronous on `stream`; device pointers, owned by the caller.
 * When T spans several backward segments, the backward's segment pre-pass and the composition
 * of its carries (which read only inputs) run on a library-owned side stream beside the
 * forward: the call records an event on `stream`, the side stream waits for it, and `stream`
 * waits for the side stream before the rest of the backward. The side stream and its events are created on the first such call of
 * each host thread on each device and kept for the thread's lifetime; stream capture sees a
 * fork and a join. */
int mamba_scan_fwd_bwd(const float* delta, const float* u, const float* B, const float* C,
                       const float* gate, const float* A_log, const float* D, const float* dy,
                       float* out, void* ckpt, size_t ckpt_bytes, void* scratch,
                       size_t scratch_bytes, float* d_delta, float* d_u, float* d_B, float* d_C,
                       float* d_A_log, float* d_D, float* d_gate, int64_t batch, int64_t T,
                       int64_t d_inner, int64_t d_state, void* stream);

/* mamba_scan_fwd_bwd with bf16 I/O: delta, u, B, C, gate, dy and the outputs out, d_delta, d_u,
 * d_B, d_C, d_gate are bfloat16 (2 bytes per element, same layouts); A_log, D, d_A_log and d_D
 * stay fp32, and so do the checkpoint and scratch buffers (same sizes as for fp32). The
 * kernels widen the inputs to fp32 in shared memory, compute everything in fp32 exactly as the
 * fp32 call does (forming y in the backward at every d_state), and round each bf16 output
 * once, to nearest even. Takes 9 <= d_state <= 64,
 * d_inner and d_state multiples of 8 and T > 16 (bf16 rows then start on 16-byte boundaries,
 * which the tensor-memory copies need); other sizes return MAMBA_ERR_UNSUPPORTED before
 * anything is launched. Pointers must be 16-byte aligned. */
int mamba_scan_fwd_bwd_bf16(const void* delta, const void* u, const void* B, const void* C,
                            const void* gate, const float* A_log, const float* D,
                            const void* dy, void* out, void* ckpt, size_t ckpt_bytes,
                            void* scratch, size_t scratch_bytes, void* d_delta, void* d_u,
                            void* d_B, void* d_C, float* d_A_log, float* d_D, void* d_gate,
                            int64_t batch, int64_t T, int64_t d_inner, int64_t d_state,
                            void* stream);

/* Causal depthwise conv1d + SiLU, the step that feeds u to the scan (the page's Phase B6 is
 * its backward):
 *   pre[b,t,d] = bias[d] + sum_{j<d_conv} w[d,j] * x[b, t-(d_conv-1)+j, d]  (x = 0 before t=0)
 *   u[b,t,d]   = pre * sigmoid(pre)
 * x, u, d_u, d_x: [batch, T, d_inner]; w, d_w: [d_inner, d_conv]; bias, d_bias: [d_inner];
 * device pointers, 16-byte aligned; 1 <= d_conv <= 8 (else MAMBA_ERR_UNSUPPORTED). The
 * backward recomputes pre from x and OVERWRITES d_x, d_w and d_bias (d_w and d_bias summed over
 * batch and time in a fixed order: deterministic). Its scratch holds
 * mamba_conv_scratch_bytes(...) bytes of per-run partials. Asynchronous on `stream`; the return
 * codes are those above. */
size_t mamba_conv_scratch_bytes(int64_t batch, int64_t T, int64_t d_inner, int64_t d_conv);
int mamba_conv_fwd(const float* x, const float* w, const float* bias, float* u, int64_t batch,
                   int64_t T, int64_t d_inner, int64_t d_conv, void* stream);
int mamba_conv_bwd(const float* x, const float* w, const float* bias, const float* d_u,
                   void* scratch, size_t scratch_bytes, float* d_x, float* d_w, float* d_bias,
                   int64_t batch, int64_t T, int64_t d_inner, int64_t d_conv, void* stream);

/* End-to-end call for callers that hold their data in HOST memory (pinned memory lets the
 * copies overlap; pageable memory works too, but more slowly). The call copies the eight
 * inputs host->device into `workspace`, runs the forward and the backward there, copies out
 * and the seven gradients device->host, and synchronises `stream` before it returns. All
 * tensor pointers here are HOST pointers, with the same layouts as above. `workspace` is DEVICE
 * memory of at least mamba_scan_host_workspace_bytes(...) bytes, owned by the caller.
 * The work is cut into slices. The first runs on `stream`, the others on streams of the
 * library, so that copies in both directions overlap the kernels of other slices. A batch of 4
 * rows or more is cut into up to 4 slices of batch rows (when a batch row of T*d_inner and of
 * T*d_state floats is a multiple of 4); d_A_log and d_D are then the slices' sums added in
 * slice order. A smaller batch with d_inner a multiple of 4 and at least 128 is cut into up to
 * 6 blocks of channels (at least 64 each; the first and the last about half as wide as the
 * others): each slice is the whole batch over its channels, moved with 2-D copies, and d_B and
 * d_C are the slices' sums added in slice order. Either way
 * the result is
 * deterministic, but rounded differently from one mamba_scan_bwd call over the whole problem.
 * Calls on the same device share the library's streams and events: calls from different host
 * threads run one at a time (each holds a per-device lock from its first enqueue to its
 * return). */
size_t mamba_scan_host_workspace_bytes(int64_t batch, int64_t T, int64_t d_inner, int64_t d_state);
int mamba_scan_fwd_bwd_host(const float* delta, const float* u, const float* B, const float* C,
                            const float* gate, const float* A_log, const float* D,
                            const float* dy, float* out, float* d_delta, float* d_u, float* d_B,
                            float* d_C, float* d_A_log, float* d_D, float* d_gate,
                            void* workspace, size_t workspace_bytes, int64_t batch, int64_t T,
                            int64_t d_inner, int64_t d_state, void* stream);

/* Backward scan that allocates nothing: the same computation and arguments as mamba_scan_bwd
 * minus the scratch buffer. The paper has no counterpart to this entry point.
 *
 * It is for callers that are handed only their input and output buffers and may not allocate
 * device memory: a plugin inside a host framework that owns all device memory, or a
 * latency-critical loop that forbids cudaMalloc (which can synchronise the device). The scratch
 * comes from a static device array of MAMBA_SCAN_NOALLOC_SCRATCH_BYTES that the library holds
 * on every GPU that loads it, until the process exits. Sizes whose
 * mamba_scan_scratch_bytes(...) exceeds that limit are rejected with MAMBA_ERR_NOALLOC_LIMIT
 * before anything is launched. The first call on each device looks up the array's device
 * address (with that device current) and caches it with the identity of the current CUDA
 * context; a call in another context (after cudaDeviceReset, or under a context the caller made
 * current) looks it up again. So the first call in a context should come before any stream
 * capture. A failed look-up returns MAMBA_ERR_CUDA, and mamba_scan_strerror names the CUDA
 * error. All calls on a device share the array, and it keeps the last call's contents.
 * Nothing needs clearing, because the backward rewrites all the scratch it reads. Calls that
 * overlap on the GPU race on the array: order them (one stream, or explicit events). No
 * cudaMalloc, cudaFree or allocating library routine is called. */
#define MAMBA_SCAN_NOALLOC_SCRATCH_BYTES (64u << 20) /* 64 MiB */
int mamba_scan_bwd_noalloc(const float* delta, const float* u, const float* B, const float* C,
                           const float* gate, const float* A_log, const float* D,
                           const float* dy, const void* ckpt, size_t ckpt_bytes, float* d_delta,
                           float* d_u, float* d_B, float* d_C, float* d_A_log, float* d_D,
                           float* d_gate, int64_t batch, int64_t T, int64_t d_inner,
                           int64_t d_state, void* stream);

/* Failure-path test of the bounded copy waits (for tests only; the paper has no counterpart).
 * The same arguments and buffers as mamba_scan_bwd, which it runs with one fault planted on the
 * host side: the tensor-memory backward issues no copy for the last chunk that each of its
 * CTAs walks, and every copy wait of the call gives up after 1 ms instead of 1 s. So the wait
 * for that chunk runs out: the kernel sets its fault word, goes on with the stale stage (no
 * address depends on the data), and exits with no copy in flight, since every copy it did
 * issue was waited for before use. The next mamba_scan_status then returns MAMBA_ERR_TIMEOUT
 * and clears the word; the call's outputs are invalid, while later calls are unaffected.
 * Only sizes that run that kernel with tensor copies are taken (9 <= d_state <= 64, d_inner
 * and d_state multiples of 4, T > 16); others return MAMBA_ERR_UNSUPPORTED before anything is
 * launched. */
int mamba_scan_bwd_test_timeout(const float* delta, const float* u, const float* B,
                                const float* C, const float* gate, const float* A_log,
                                const float* D, const float* dy, const void* ckpt,
                                size_t ckpt_bytes, void* scratch, size_t scratch_bytes,
                                float* d_delta, float* d_u, float* d_B, float* d_C,
                                float* d_A_log, float* d_D, float* d_gate, int64_t batch,
                                int64_t T, int64_t d_inner, int64_t d_state, void* stream);

/* Failure-path test of the forward's bounded copy waits: mamba_scan_fwd, except that the
 * forward kernel leaves the tensor copies of the last chunk each CTA walks unissued and gives
 * up waiting for them after 1 ms. The next mamba_scan_status then returns MAMBA_ERR_TIMEOUT
 * (and clears it); out, y and the checkpoints of that call are invalid. Every copy that was
 * issued is waited for before use, so none is in flight when a CTA exits. Only sizes that run
 * the forward with tensor copies are taken (33 <= d_state <= 64, d_inner and d_state multiples
 * of 4, T > 16); others return MAMBA_ERR_UNSUPPORTED before anything is launched. */
int mamba_scan_fwd_test_timeout(const float* delta, const float* u, const float* B,
                                const float* C, const float* gate, const float* A_log,
                                const float* D, float* out, float* y, void* ckpt,
                                size_t ckpt_bytes, int64_t batch, int64_t T, int64_t d_inner,
                                int64_t d_state, void* stream);

/* Synchronises `stream` and reports any asynchronous CUDA error (MAMBA_ERR_CUDA), a
 * kernel that gave up waiting for its own copies (MAMBA_ERR_TIMEOUT), or, in a bounds-checked
 * build, an access a kernel computed outside its buffer (MAMBA_ERR_BOUNDS). Each flag is
 * cleared once reported. MAMBA_OK otherwise. */
int mamba_scan_status(void* stream);

/* Bounds-checked build. The library compiled with -DMAMBA_BOUNDS_CHECK
 * (libmambascan_checked.so, the same source) checks every global access whose offset a kernel
 * computes against the length of its buffer, taken from the call's sizes. An access outside
 * is not made (a load reads zero, a store is dropped) and is recorded for mamba_scan_status.
 * No check traps. TMA copies are bounded by their tensor maps and are not checked again.
 * mamba_scan_bounds_checked returns 1 in that build and 0 in the default one.
 * mamba_scan_test_bounds_shrink (test hook) makes every kernel take each buffer `elements`
 * elements shorter than it is, so a test can see the check fire while every access it blocks
 * is inside the real buffer; 0 restores the real lengths. It returns MAMBA_ERR_UNSUPPORTED in
 * the default build and MAMBA_ERR_INVALID_ARG for a negative count. It applies to the
 * device current at the call. */
int mamba_scan_bounds_checked(void);
int mamba_scan_test_bounds_shrink(int64_t elements);

/* Static, human-readable text of a return code. When the code is MAMBA_ERR_CUDA it names the
 * last CUDA error this library saw. Never NULL. */
const char* mamba_scan_strerror(int code);

/* Number of kernel launches the last successful mamba_scan_fwd / mamba_scan_bwd call on this
 * host thread enqueued. The bench's launch count relies on it. */
int mamba_scan_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MAMBA_SCAN_H */
