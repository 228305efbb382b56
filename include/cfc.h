/*
 * cfc.h -- C ABI of the GB300 (sm_103a) CfC K-loop library: forward recurrence, reverse-time
 * backpropagation through time, and deterministic weight / bias / input / initial-state
 * gradients for a batch of B sequences over K steps.
 *
 * Source of the operations.  The K-loop parallelization spec (page "K-loop Parallelization --
 * Block-per-Batch Kernel Refactor") names the per-step forward kernel cfc_step_batched and
 * backward kernel cfc_step_backward_batched (section "Problem"), the per-(batch row, channel)
 * gradient scratch and the reducer reduce_axis0 with overwrite semantics (section
 * "Architecture Choice", item 3), and the rule that a final gradient buffer holds meaningful
 * data only after its reducer ran (section "AdamW-after-reducer invariant").  The pages do not
 * print the cell's equations; this library computes the four-gate closed-form continuous-time
 * cell
 *
 *     z_t  = [u_t ; h_{t-1}]            (n_in = n_x + C, h_{-1} = h0)
 *     P_g  = W_g z_t + b_g              for the gates g = ff1, ff2, ta, tb, in that order
 *     h_t  = tanh(P_ff1) * (1 - s) + s * tanh(P_ff2),   s = sigmoid(P_ta * ts[t][b] + P_tb)
 *
 * and, for an upstream gradient dH = dL/dH, the exact gradients dW, db, du, dh0 of
 * L = sum dH * H.
 *
 * Conventions shared by every entry point.
 *   - Every tensor pointer is a DEVICE pointer to fp32 data, row-major with the last index
 *     fastest, 16-byte aligned (CFC_ERR_MISALIGNED otherwise).  The caller allocates and owns
 *     every buffer; the library never allocates, frees or synchronises.
 *   - Every output is OVERWRITTEN in full (nothing accumulates across calls) and is valid only
 *     after the work queued on `stream` has completed.
 *   - `stream` is a cudaStream_t (0 = the legacy default stream).  Calls only enqueue work, so
 *     they may be captured into a CUDA graph once an eager call with the same sizes has run
 *     on the device (the first call per device and size class sets kernel attributes).
 *   - Status: 0 on success, a negative CFC_ERR_* code otherwise; argument errors are detected
 *     on the host before any work is enqueued.  Nothing aborts or throws.
 *   - Size envelope: 1 <= C <= 256, 1 <= n_x <= 512, B >= 1, K >= 1, K * B * 4 * C < 2^31.
 */
#ifndef CFC_H
#define CFC_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CFC_OK 0
#define CFC_ERR_INVALID_DIM (-1)        /* a size is <= 0 or outside the envelope above      */
#define CFC_ERR_NULL_PTR (-2)           /* a required pointer is NULL                        */
#define CFC_ERR_MISALIGNED (-3)         /* a tensor pointer is not 16-byte aligned           */
#define CFC_ERR_WS_TOO_SMALL (-4)       /* workspace shorter than cfc_workspace_bytes()      */
#define CFC_ERR_UNSUPPORTED_DEVICE (-5) /* current device is not compute capability 10.3     */
#define CFC_ERR_LAUNCH_FAILED (-6)      /* a kernel launch returned an error                 */
#define CFC_ERR_DEVICE_TIMEOUT (-7)     /* a kernel abandoned a wait (see cfc_device_status) */
#define CFC_ERR_INVALID_ARG (-8)        /* an enumerated argument is out of range            */
#define CFC_ERR_CUDA (-9)               /* another CUDA runtime call failed                  */
#define CFC_ERR_SCRATCH_LIMIT (-10)     /* problem needs more than the built-in scratch holds */

/*
 * Weight-gradient contraction modes for cfc_backward (argument dw_mode): how dW, db and du are
 * computed from d_pre.  The recurrences (H, d_pre, dh0) are the same in every mode.
 *   CFC_DW_ACCURATE   tensor cores, each fp32 operand as two bf16 terms (hi + lo, 16
 *                     significand bits) and three products per step; measured error against
 *                     the fp64 oracle ~5e-6 of max|dW| (up to 5e-5 on the 2048 x 128 x 256
 *                     workload, whose gradient cancels heavily).
 *   CFC_DW_BF16       tensor cores, one bf16 product per step: each operand rounded to bf16
 *                     (relative error at most 2^-8, so at most 2^-7 per product), measured
 *                     2e-3 to 3e-3 of max|dW|.  For throughput, not for the 1e-4 tolerance.
 *   CFC_DW_TF32       tensor cores, one tf32 product per step (10 explicit mantissa bits).
 *                     For throughput, not for the 1e-4 tolerance.
 *   CFC_DW_SIMT_FP32  CUDA-core fp32 FMA contraction (the reference path).
 */
#define CFC_DW_ACCURATE 0
#define CFC_DW_BF16 1
#define CFC_DW_TF32 2
#define CFC_DW_SIMT_FP32 3

typedef void* cfc_stream_t; /* a cudaStream_t */

/*
 * cfc_workspace_bytes -- bytes of device workspace cfc_backward (and cfc_forward_backward,
 * whose forward uses its tail) needs for these sizes and dw_mode.  Writes *bwd_ws_bytes; the
 * forward cache is always K*B*3*C floats and needs no query.  Returns CFC_OK,
 * CFC_ERR_INVALID_DIM, CFC_ERR_NULL_PTR or CFC_ERR_INVALID_ARG.
 * The workspace starts with the pre-activation gradients dL/dP of every step and row, readable
 * after cfc_backward completes, in the form the mode's contraction reads:
 *   CFC_DW_TF32, CFC_DW_SIMT_FP32: fp32 d_pre [K][B][4][C];
 *   CFC_DW_ACCURATE, CFC_DW_BF16:  K*B rows of 4*MP bytes, MP = 4C rounded up to a multiple of
 *     8; row (t, b) holds MP bf16 values hi[g*C + c] = bf16(d_pre) and then MP bf16 values
 *     lo[g*C + c] = bf16(d_pre - hi) (CFC_DW_BF16 leaves lo unwritten).  hi + lo is d_pre to
 *     16 significand bits.
 * The rest is internal (contraction operands and split partial sums).
 */
int cfc_workspace_bytes(int B, int K, int C, int n_x, int dw_mode, size_t* bwd_ws_bytes);

/*
 * cfc_forward_workspace_bytes -- bytes of device workspace cfc_forward and
 * cfc_forward_recurrence need: 0 below the batch sizes that take the tensor-core recurrence
 * (B >= 384 at C = 256, B >= 768 at C = 128), otherwise its exchange buffer, 8*C bytes per
 * batch row rounded up to a whole row tile (about 4.4 MB at B = 2048, C = 256).  Writes
 * *bytes; returns CFC_OK, CFC_ERR_INVALID_DIM or CFC_ERR_NULL_PTR.
 */
int cfc_forward_workspace_bytes(int B, int K, int C, int n_x, size_t* bytes);

/*
 * cfc_forward -- the K-step forward recurrence (successor of cfc_step_batched, which ran one
 * step per launch; page "K-loop Parallelization -- Block-per-Batch Kernel Refactor", section
 * "Problem").  One persistent launch runs all K steps.
 *   u     [K][B][n_x]  inputs u_t
 *   h0    [B][C]       initial state
 *   W     [4][C][n_x+C] gate weights (ff1, ff2, ta, tb); columns follow z = [u_t ; h_{t-1}]
 *   b     [4][C]       gate biases
 *   ts    [K][B]       time-scale per step and row (multiplies P_ta only)
 *   H     [K][B][C]    OUTPUT: h_t for every step
 *   cache [K][B][3][C] OUTPUT: ff1, ff2 and the gate s for every step (read by cfc_backward)
 *   ws, ws_bytes       device workspace of at least cfc_forward_workspace_bytes() bytes,
 *                      16-byte aligned; may be NULL when that is 0.  Transient: free for other
 *                      use once the call's work on the stream is done.
 * Exactly cfc_input_projection followed by cfc_forward_recurrence (two launches).  Returns
 * CFC_ERR_NULL_PTR / CFC_ERR_WS_TOO_SMALL for a missing or short workspace.
 */
int cfc_forward(const float* u, const float* h0, const float* W, const float* b,
                const float* ts, int B, int K, int C, int n_x, float* H, float* cache, void* ws,
                size_t ws_bytes, cfc_stream_t stream);

/*
 * cfc_input_projection -- the first stage of cfc_forward alone: X = W_u u_t + b for every step
 * at once (it does not depend on h), one parallel contraction over the B*K rows.  X is handed
 * to the recurrence in place: gate ff1 in H[t][b][:], gates ff2 / ta / tb in cache[t][b][0..2][:]
 * (together exactly 4C values per row).  u, W, b, H, cache as for cfc_forward.
 */
int cfc_input_projection(const float* u, const float* W, const float* b, int B, int K, int C,
                         int n_x, float* H, float* cache, cfc_stream_t stream);

/*
 * cfc_forward_recurrence -- the second stage of cfc_forward alone: the K-step recurrence,
 * adding W_h h_{t-1} to the X that cfc_input_projection left in H / cache and overwriting
 * H / cache with the outputs.  h0, W, ts, H, cache, ws, ws_bytes as for cfc_forward.
 */
int cfc_forward_recurrence(const float* h0, const float* W, const float* ts, int B, int K,
                           int C, int n_x, float* H, float* cache, void* ws, size_t ws_bytes,
                           cfc_stream_t stream);

/*
 * cfc_step_launches -- number of kernel launches one cfc_forward plus one cfc_backward enqueue
 * for these sizes (with_du = 0 when du is NULL).  Writes *launches; returns CFC_OK or the
 * argument error codes of cfc_workspace_bytes.
 */
int cfc_step_launches(int B, int K, int C, int n_x, int dw_mode, int with_du, int* launches);

/*
 * cfc_backward -- reverse-time BPTT over the K steps (successor of cfc_step_backward_batched;
 * same page, sections "Problem" and "Per-Kernel Breakdown"), then the weight gradient as one
 * dense contraction over the B*K rows and the bias gradient through reduce_axis0: exactly
 * cfc_backward_recurrence into the head of ws followed by cfc_weight_grad.
 *   dH    [K][B][C]     upstream gradient dL/dh_t (the loss is L = sum dH * H)
 *   u, h0, W, ts        the forward's inputs;  H, cache: the forward's outputs
 *   dW    [4][C][n_x+C] OUTPUT: dL/dW
 *   db    [4][C]        OUTPUT: dL/db
 *   du    [K][B][n_x]   OUTPUT: dL/du (may be NULL to skip it)
 *   dh0   [B][C]        OUTPUT: dL/dh0
 *   ws, ws_bytes        device workspace of at least cfc_workspace_bytes() bytes, 16-byte
 *                       aligned; its head receives d_pre (see cfc_workspace_bytes)
 *   dw_mode             one of the CFC_DW_* modes
 */
int cfc_backward(const float* dH, const float* u, const float* h0, const float* W,
                 const float* ts, const float* H, const float* cache, int B, int K, int C,
                 int n_x, float* dW, float* db, float* du, float* dh0, void* ws,
                 size_t ws_bytes, int dw_mode, cfc_stream_t stream);

/*
 * cfc_forward_backward -- one training step: exactly cfc_forward followed by cfc_backward,
 * with the same arguments and outputs, and bitwise the same results.  One workspace of
 * cfc_workspace_bytes() bytes serves both (the forward's part is its tail).  Because the
 * forward writes nothing the backward recurrence reads before its dependency wait (W, dH),
 * the recurrence is launched as a programmatic dependent of the forward: its clusters are
 * scheduled and stage W_h^T while the forward's last steps run.  Returns the error codes of
 * cfc_forward and cfc_backward; all arguments are checked before anything is launched.
 */
int cfc_forward_backward(const float* u, const float* h0, const float* W, const float* b,
                         const float* ts, const float* dH, int B, int K, int C, int n_x,
                         float* H, float* cache, float* dW, float* db, float* du, float* dh0,
                         void* ws, size_t ws_bytes, int dw_mode, cfc_stream_t stream);

/*
 * BF16 state.  The pages defer mixed precision to a future spec (page "K-loop
 * Parallelization -- Block-per-Batch Kernel Refactor", section "Non-goals", and section
 * "Post-refactor bottleneck analysis": "BF16 trunk").  Here it is the storage of the per-step
 * activations in bf16 with all arithmetic and accumulation in fp32: H and the cache are
 * written as bf16 (round to nearest even of exactly the fp32 values cfc_forward computes; the
 * recurrence itself carries h in fp32), the backward reads them as bf16, keeps d_pre in one
 * bf16 plane and computes dW, db and du with single-pass bf16 contractions (as CFC_DW_BF16).
 * The persistent activation memory (H and cache, kept from forward to backward) is halved.
 * Accuracy: H and the cache are cfc_forward's rounded to bf16 (relative error at most 2^-8,
 * the bf16 unit roundoff); the gradients carry the bf16 rounding of the cache, d_pre and z
 * (measured 2e-3 to 4e-3 of the largest entry, max-normalised, against the fp64 definition;
 * bound 2^-6).  C must be even.  H and cache point to uint16 storage of
 * bf16 values in the layouts of cfc_forward ([K][B][C], [K][B][3][C]).
 */

/*
 * cfc_forward_bf16_workspace_bytes -- device workspace cfc_forward_bf16 needs: the input
 * projection X = W_u u + b of every step in fp32 (4 C floats per batch row and step, plus
 * alignment), then the recurrence's own (cfc_forward_workspace_bytes).  Returns CFC_OK,
 * CFC_ERR_INVALID_DIM (also for odd C) or CFC_ERR_NULL_PTR.
 */
int cfc_forward_bf16_workspace_bytes(int B, int K, int C, int n_x, size_t* bytes);

/*
 * cfc_forward_bf16 -- cfc_forward with H and the cache stored as bf16.
 *   u, h0, W, b, ts     as for cfc_forward (fp32)
 *   H     [K][B][C]     OUTPUT, bf16
 *   cache [K][B][3][C]  OUTPUT, bf16 (ff1, ff2, gate)
 *   ws, ws_bytes        16-byte aligned device workspace of at least
 *                       cfc_forward_bf16_workspace_bytes() bytes (transient: it may be reused
 *                       once the call's work on the stream is done)
 * Returns the error codes of cfc_forward, CFC_ERR_INVALID_DIM for odd C and
 * CFC_ERR_WS_TOO_SMALL.
 */
int cfc_forward_bf16(const float* u, const float* h0, const float* W, const float* b,
                     const float* ts, int B, int K, int C, int n_x, void* H, void* cache,
                     void* ws, size_t ws_bytes, cfc_stream_t stream);

/*
 * cfc_backward_bf16 -- cfc_backward for the bf16 H and cache of cfc_forward_bf16.  The
 * workspace is that of cfc_workspace_bytes(B, K, C, n_x, CFC_DW_BF16, ...); its head receives
 * d_pre as bf16 operand rows.  Outputs dW, db, du (may be NULL), dh0 are fp32, as for
 * cfc_backward.  Returns the error codes of cfc_backward and CFC_ERR_INVALID_DIM for odd C.
 */
int cfc_backward_bf16(const float* dH, const float* u, const float* h0, const float* W,
                      const float* ts, const void* H, const void* cache, int B, int K, int C,
                      int n_x, float* dW, float* db, float* du, float* dh0, void* ws,
                      size_t ws_bytes, cfc_stream_t stream);

/*
 * The pages' own leaky (tau-decay) cell.  Page "K-loop Parallelization -- Block-per-Batch
 * Kernel Refactor" names its backward's gradients grad_w_in, grad_w_rec, grad_b and grad_tau
 * (section "Per-Kernel Breakdown") and a per-block decay vector sdecay (section "Large
 * shared-mem note"), without equations.  The cell computed (a reading of those names):
 *
 *     a_t = W [x_t ; h_{t-1}] + b,  e_t = tanh(a_t),  d_t = exp(-ts[t][b] / tau),
 *     h_t = d_t * h_{t-1} + (1 - d_t) * e_t            (per hidden unit; h_{-1} = h0)
 *
 * with the exact gradients dW (= [dW_in | dW_rec]), db, dtau, dx and dh0 of L = sum dH * H.
 * Sizes: 1 <= C <= 128 hidden units, 1 <= n_x <= 512 inputs; every tau must be positive.
 * Layouts: x [K][B][n_x], h0 [B][C], W [C][n_x + C], b [C], tau [C], ts [K][B],
 * H and E [K][B][C] (E = tanh(a_t), read by the backward), dH [K][B][C], dW [C][n_x + C],
 * db [C], dtau [C], dx [K][B][n_x], dh0 [B][C].
 */

/*
 * cfc_decay_forward -- the K-step forward of the tau-decay cell: the input projection
 * W_in x_t + b for every step at once (written into E), then one persistent launch of the
 * recurrence, which overwrites E with tanh(a_t) and writes H.  Returns the argument codes of
 * cfc_forward (CFC_ERR_INVALID_DIM also for C > 128).
 */
int cfc_decay_forward(const float* x, const float* h0, const float* W, const float* b,
                      const float* tau, const float* ts, int B, int K, int C, int n_x, float* H,
                      float* E, cfc_stream_t stream);

/*
 * cfc_decay_workspace_bytes -- device workspace cfc_decay_backward needs (the gradients of
 * the pre-activations as contraction operand rows, the contraction's other operands and split
 * partial sums, and per-row dtau sums).  Returns CFC_OK, CFC_ERR_INVALID_DIM or CFC_ERR_NULL_PTR.
 */
int cfc_decay_workspace_bytes(int B, int K, int C, int n_x, size_t* bytes);

/*
 * cfc_decay_backward -- BPTT of the tau-decay cell, then dW and db as one dense contraction
 * over the B*K rows on the tensor cores (two bf16 terms per operand, three products, as
 * CFC_DW_ACCURATE), dx as a second one, and dtau as a fixed-order sum over the batch rows.
 * dx may be NULL.  Outputs are overwritten.  Returns the codes of cfc_backward.
 */
int cfc_decay_backward(const float* dH, const float* x, const float* h0, const float* W,
                       const float* tau, const float* ts, const float* H, const float* E, int B,
                       int K, int C, int n_x, float* dW, float* db, float* dtau, float* dx,
                       float* dh0, void* ws, size_t ws_bytes, cfc_stream_t stream);

/*
 * cfc_backward_recurrence -- the first stage of cfc_backward alone: the reverse-time
 * recurrence, writing the pre-activation gradients and dh0.
 *   dH, W, ts, cache   as for cfc_backward
 *   d_pre [K][B][4][C] OUTPUT: dL/dP for every step, row, gate and channel
 *   dh0   [B][C]       OUTPUT: dL/dh0
 */
int cfc_backward_recurrence(const float* dH, const float* W, const float* ts,
                            const float* cache, int B, int K, int C, int n_x, float* d_pre,
                            float* dh0, cfc_stream_t stream);

/*
 * cfc_bptt_workspace_bytes -- bytes of device workspace cfc_backward_recurrence_ws takes for
 * these sizes: for C = 256 with B >= 1024, or C = 128 with B >= 1185, the recurrence runs each step's contraction
 * delta = d_pre W_h on the tensor cores and first writes W_h^T there as three bf16 terms
 * (24 C^2 bytes); otherwise 0.  Writes *bytes; returns the argument codes of
 * cfc_workspace_bytes.
 */
int cfc_bptt_workspace_bytes(int B, int K, int C, int n_x, size_t* bytes);

/*
 * cfc_backward_recurrence_ws -- cfc_backward_recurrence with a workspace, so that it takes
 * the tensor-core recurrence where cfc_backward would (the same kernels, bitwise the same
 * d_pre and dh0 as cfc_backward writes).  That path also needs dH, cache and d_pre 32-byte
 * aligned; otherwise the CUDA-core recurrence runs.
 *   ws, ws_bytes  device workspace of at least cfc_bptt_workspace_bytes() bytes, 16-byte
 *                 aligned, owned by the caller (contents are scratch); may be NULL when that
 *                 size is 0.  Too small: CFC_ERR_WS_TOO_SMALL before any launch.
 * Other arguments and errors as for cfc_backward_recurrence.
 */
int cfc_backward_recurrence_ws(const float* dH, const float* W, const float* ts,
                               const float* cache, int B, int K, int C, int n_x, float* d_pre,
                               float* dh0, void* ws, size_t ws_bytes, cfc_stream_t stream);

/*
 * cfc_weight_grad -- the second stage of cfc_backward alone: dW = sum_{t,b} d_pre z^T as one
 * contraction over the B*K rows (z = [u_t ; h_{t-1}], h_{-1} = h0), db = sum_{t,b} d_pre
 * through reduce_axis0, and du = W_u^T d_pre (skipped when du is NULL).  The weight gradient
 * as a dense contraction over the batch replaces the per-sample atomicAdd accumulation, as
 * the DQN plan on page "H100 Epoch Optimization Phase 2" (Task 2) does for its layers.
 *   d_pre [K][B][4][C]  fp32 input (e.g. from cfc_backward_recurrence)
 *   u, h0, W, H         the forward's inputs and output
 *   dW, db, du          OUTPUTS as for cfc_backward
 *   ws, ws_bytes        workspace as for cfc_backward.  d_pre may lie outside it, or, when C
 *                       is even, start exactly at its head: for CFC_DW_ACCURATE / CFC_DW_BF16
 *                       the stage first rewrites d_pre into the head's bf16 form, in place
 *                       in that case.  Any other overlap returns CFC_ERR_INVALID_ARG.
 */
int cfc_weight_grad(const float* d_pre, const float* u, const float* h0, const float* W,
                    const float* H, int B, int K, int C, int n_x, float* dW, float* db,
                    float* du, void* ws, size_t ws_bytes, int dw_mode, cfc_stream_t stream);

/*
 * reduce_axis0 -- out[n] = sum_{r < n_batch} per_batch[r][n] for n < n_tail, OVERWRITING out
 * (page "K-loop Parallelization -- Block-per-Batch Kernel Refactor", section "Architecture
 * Choice", item 3: block tree-reduce over the batch index, no atomicAdd, grid over the tail).
 * The summation order depends only on (n_batch, n_tail): results are bitwise reproducible.
 *   per_batch [n_batch][n_tail] device fp32, 4-byte aligned (16-byte alignment with n_tail a
 *             multiple of 4 selects the vectorised path; both give identical sums)
 *   out       [n_tail] device fp32
 * Returns CFC_OK, CFC_ERR_INVALID_DIM (n_batch or n_tail <= 0), CFC_ERR_NULL_PTR,
 * CFC_ERR_MISALIGNED, CFC_ERR_UNSUPPORTED_DEVICE or CFC_ERR_LAUNCH_FAILED.
 */
int reduce_axis0(const float* per_batch, int n_batch, int n_tail, float* out,
                 cfc_stream_t stream);

/*
 * cfc_backward_noalloc -- cfc_backward for callers that cannot allocate device memory.  (The
 * pages have no counterpart of this entry point.)
 *
 * Who needs it: a plugin or callback hosted by a framework that owns the GPU's memory and gives
 * the plugin no allocator, or a program that fixes its device memory footprint at start-up and
 * may not grow it later.  Such callers cannot provide cfc_backward's workspace.
 *
 * What it does: the same computation and outputs as cfc_backward with the same arguments
 * (minus ws / ws_bytes), using as workspace a device array built into the library.  Every GPU
 * that loads the library holds that array, CFC_NOALLOC_SCRATCH_BYTES bytes, until the process
 * exits.  The call allocates and frees nothing.
 *   - Limit: problems whose cfc_workspace_bytes() exceeds CFC_NOALLOC_SCRATCH_BYTES are
 *     rejected with CFC_ERR_SCRATCH_LIMIT before any work is enqueued.  (The 32 x 64 x 128 and
 *     32 x 64 x 256 workloads fit; 256 x 64 x 128 does not.)
 *   - Set-up: the first call on each device looks up the array's device address on the current
 *     device; make that first call before any stream capture begins.  The address is kept for
 *     the life of the process, so do not call cudaDeviceReset between calls (the library's
 *     other per-device set-up, done by the first call of any entry point, is kept the same
 *     way).
 *   - Sharing: all calls share the one array.  Nothing in it needs to start at zero (every
 *     entry a call reads, the same call wrote first), but calls whose work overlaps on the GPU
 *     -- concurrent streams, or several host threads -- race on it.  Serialise them (one
 *     stream, or events between streams).
 * Returns the codes of cfc_backward and cfc_workspace_bytes, plus CFC_ERR_SCRATCH_LIMIT.
 */
#define CFC_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int cfc_backward_noalloc(const float* dH, const float* u, const float* h0, const float* W,
                         const float* ts, const float* H, const float* cache, int B, int K, int C,
                         int n_x, float* dW, float* db, float* du, float* dh0, int dw_mode,
                         cfc_stream_t stream);

/*
 * Measurement aids.  (The pages have no counterpart: they set the roofline denominators of the
 * CUDA-core kernels on the device at hand.)  Each enqueues one throughput kernel on `stream`
 * and writes, on the host, the work it does; the caller times the call with CUDA events.
 *
 * cfc_probe_fma -- `blocks` CTAs of 256 threads, each running 8 independent chains of `iters`
 * packed fp32 FMAs; `out` (device, blocks * 256 floats) receives one sum per thread; *flop the
 * floating-point operations performed (4 per packed FMA).
 *
 * cfc_probe_l2_read -- `blocks` CTAs of 256 threads read the n_floats floats at `buf` (device,
 * 16-byte aligned) `passes` times with 16-byte loads cached in L2 only; `out` (device, blocks *
 * 256 floats) receives one sum per thread; *bytes the bytes read.  With `buf` smaller than the
 * L2 cache, this measures L2 read bandwidth.
 *
 * Both return CFC_OK, CFC_ERR_NULL_PTR, CFC_ERR_INVALID_DIM, CFC_ERR_MISALIGNED or
 * CFC_ERR_LAUNCH_FAILED.
 */
int cfc_probe_fma(float* out, int blocks, int iters, double* flop, cfc_stream_t stream);
int cfc_probe_l2_read(const float* buf, size_t n_floats, int passes, float* out, int blocks,
                      double* bytes, cfc_stream_t stream);

/*
 * cfc_copy -- dst[0 .. bytes) <- src[0 .. bytes), enqueued on `stream` as one kernel of the
 * library (the SMs move the data; no copy engine).  For bringing a step's inputs in from the
 * host and its gradients back: each of src and dst is device memory, managed memory, or host
 * memory that is pinned or registered with CUDA and so mapped into the device's address space
 * (read and written directly over the host link).  Both pointers and `bytes` must be multiples
 * of 16 (CFC_ERR_MISALIGNED); the ranges must not overlap, and memory the device cannot reach
 * is refused (CFC_ERR_INVALID_ARG).  bytes == 0 enqueues nothing.  The caller owns both buffers
 * and keeps them alive until the copy has run.  Returns CFC_OK, CFC_ERR_NULL_PTR,
 * CFC_ERR_MISALIGNED, CFC_ERR_INVALID_ARG or CFC_ERR_LAUNCH_FAILED.
 */
int cfc_copy(const void* src, void* dst, size_t bytes, cfc_stream_t stream);

/* cfc_error_string -- static English text for a status code (never NULL). */
const char* cfc_error_string(int code);

/*
 * cfc_device_status -- synchronises the current device, then reads and clears the library's
 * device status word (set by a kernel that abandoned a bounded wait).  *status receives 0 when
 * no kernel reported a problem since the last read.  A nonzero value means that some call
 * enqueued since then left its outputs incomplete: treat the outputs of every such call as
 * invalid.  Kernels only write the word, never read it, so a value left unread does not
 * affect later calls.  Returns CFC_OK, CFC_ERR_NULL_PTR or CFC_ERR_CUDA.  This is the only
 * entry point that synchronises.
 */
int cfc_device_status(int* status);

/*
 * cfc_wait_self_test -- checks, on the device, that an abandoned wait is reported rather than
 * hung: enqueues on `stream` one single-thread kernel that waits, with the bounded wait every
 * kernel of the library uses, on an mbarrier that nothing completes.  After the wait limit
 * (2 s) the kernel records a timeout in the device status word and returns; cfc_device_status
 * then reports 1 (and clears it).  No fault is raised and the context stays usable, and
 * other work of this library, before or after it, is not affected.  Returns CFC_OK,
 * CFC_ERR_UNSUPPORTED_DEVICE, CFC_ERR_CUDA or CFC_ERR_LAUNCH_FAILED.
 */
int cfc_wait_self_test(cfc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CFC_H */
