/*
 * ttm.h — C ABI of libttm.so, the GB300 (sm_103a) chunked test-time-training
 * memory scan.
 *
 * What one call computes (per batch row b and head h, independently):
 *
 *   a fast-weight memory M takes one gradient step per token on the inner
 *   loss  l(M; k_t, v_t) = || f(k_t; M) - v_t ||^2
 *     ("TTT layers 与 fast weights", eqs (1)-(2); "论文速览 | Titans" §3.6);
 *   mini-batch rule: every gradient inside a chunk of `chunk` tokens is taken
 *   at the state left by the previous chunk; chunk c covers tokens
 *   [c*chunk, min((c+1)*chunk, T)) and the last chunk may be shorter
 *     ("TTT layers 与 fast weights", eq (6); "论文速览 | Titans" §4.2);
 *   Titans momentum and forgetting:
 *     S_t = eta_t S_{t-1} - theta_t grad_t,   M_t = (1 - alpha_t) M_{t-1} + S_t
 *     ("论文速览 | Titans" §3.4, §3.7);
 *   read after the token's own write: z_t = f(q_t; M_t)
 *     ("TTT layers 与 fast weights", eq (3)).
 *
 * Conventions shared by every entry point
 *   - Column vectors: linear memory f(k; W) = W k with W stored [dv][dk]
 *     row-major; the deep memory is f(k) = W2 GELU(W1 k), GELU exact (erf).
 *   - q, k: [B][H][T][dk], v and z: [B][H][T][dv] (deep memory: dk = dv = d),
 *     contiguous, element type `dtype` (TTM_F32 or TTM_BF16); z is written in
 *     `dtype`, rounded to nearest even.  All arithmetic accumulates in fp32.
 *   - Gates eta (momentum), theta (step), alpha (forgetting): fp32 [B][H][T],
 *     contiguous, used as given (no clamping).
 *   - Initial state: fp32 [B][H][...], or [1][H][...] shared by every batch
 *     row when w0_shared_over_batch != 0 (the same flag applies to S0).
 *     NULL S0 (and S1_0/S2_0) means a zero momentum state.
 *   - Final state: fp32 [B][H][...]; S_out (S1_out/S2_out) may be NULL to skip.
 *     Continuing a sequence by passing a call's final state as the next call's
 *     initial state is exact when the first call's T is a multiple of chunk.
 *   - Pointers are device pointers owned by the caller.  The library
 *     allocates no memory and keeps no state between calls, except the
 *     process-wide kernel policy and the device status word below.
 *     Every pointer must be 16-byte aligned.  Outputs must not overlap inputs,
 *     except that W_out may be W0 (and S_out S0; W1_out/W2_out likewise) when
 *     w0_shared_over_batch == 0.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  The call is
 *     asynchronous: it validates on the host, enqueues kernels and returns.
 *   - Workspace: the tensor-core path of the linear / Titans scan first
 *     computes every chunk's coefficients (they depend only on the gates) into
 *     device scratch that the caller provides: `workspace` (16-byte aligned,
 *     not overlapping any other argument) of at least
 *     ttm_linear_workspace_size(...) bytes.  Its contents on entry are
 *     ignored and on return are unspecified.  Kernels that need none accept
 *     NULL / 0.
 *
 * Errors
 *   Argument validation happens on the host before anything is enqueued; a
 *   failure returns TTM_ERR_INVALID_ARG (malformed) or TTM_ERR_UNSUPPORTED (a
 *   well-formed shape no kernel of the current policy handles) and launches
 *   nothing.  A CUDA launch failure returns TTM_ERR_CUDA.  A device-side wait
 *   that gave up (tensor-core kernels bound every wait) is reported later
 *   through ttm_device_status().
 */
#ifndef TTM_H
#define TTM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TTM_OK = 0,
    TTM_ERR_INVALID_ARG = 1,
    TTM_ERR_UNSUPPORTED = 2,
    TTM_ERR_CUDA = 3,
    TTM_ERR_TIMEOUT = 4
} ttm_status;

typedef enum { TTM_F32 = 0, TTM_BF16 = 1 } ttm_dtype;

/* Kernel selection policy (process-wide; default TTM_KERNEL_AUTO).
 *   AUTO: tensor-core kernel where the shape and dtype allow it, else the
 *         fp32 CUDA-core kernel.
 *   SIMT: always the fp32 CUDA-core kernel.
 *   TC:   the tensor-core kernel or TTM_ERR_UNSUPPORTED, never a substitute. */
typedef enum { TTM_KERNEL_AUTO = 0, TTM_KERNEL_SIMT = 1, TTM_KERNEL_TC = 2 } ttm_kernel_policy;

/* Kernel ids reported by ttm_last_kernel(). */
typedef enum {
    TTM_KID_NONE = 0,
    TTM_KID_LINEAR_SIMT = 1,   /* fp32 CUDA-core chunked scan, linear memory */
    TTM_KID_MLP_SIMT = 2,      /* fp32 CUDA-core chunked scan, 2-layer memory */
    TTM_KID_LINEAR_TC = 3,     /* tcgen05 + TMA chunked scan, linear memory */
    TTM_KID_MLP_TC = 4,        /* tcgen05 chunked scan, 2-layer memory */
    TTM_KID_LINEAR_SEQ = 5,    /* tcgen05 + TMA scan, one CTA per sequence, d = 64,
                                  gradient points every 16 or 32 tokens */
    TTM_KID_DGD_STEP = 6,      /* fp32 CUDA-core token loop, DGD memory */
    TTM_KID_DGD_TC = 7,        /* tcgen05 + TMA chunk form, DGD memory (pre-pass + scan) */
    TTM_KID_BWD_SIMT = 8,      /* gradient: every pass on the fp32 CUDA cores */
    TTM_KID_BWD_TC = 9         /* gradient: chain and local pass on tcgen05 */
} ttm_kernel_id;

/*
 * TTT-Linear: linear memory, plain mini-batch gradient descent
 * ("TTT layers 与 fast weights", eqs (4)-(9): W_t = W_{t'} - theta sum of
 * 2 (W_{t'} k_s - v_s) k_s^T over the chunk so far).
 *   eta and alpha must be NULL (this form has no momentum or forgetting).
 *   theta: required.  W0: [B|1][H][dv][dk].  W_out: [B][H][dv][dk].
 *   z: [B][H][T][dv] in dtype.
 * Shapes: B, H >= 1; T >= 0; dk, dv >= 1 (multiples of 8 for TTM_BF16,
 * of 4 for TTM_F32); chunk >= 1.
 * Kernels (policy AUTO): bf16 with dk = dv in {64, 128} and chunk 64 run the
 * tcgen05 row-slice scan (workspace below); bf16 with dk = dv = 64 and chunk
 * 16 or 32 run the tcgen05 scan with one CTA per sequence, whose 64-token
 * tiles solve the tile's unit block-lower-triangular error system in the key
 * products (no workspace); everything else runs the fp32 CUDA-core scan.
 */
int ttm_linear_fwd(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                   const void* q, const void* k, const void* v,
                   const float* eta, const float* theta, const float* alpha,
                   const float* W0, int w0_shared_over_batch,
                   void* z, float* W_out, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * Titans neural memory with linear memory: momentum ("past surprise") and
 * forgetting ("论文速览 | Titans" §3.4-§3.7, chunked as in §4.2-§4.5).
 *   eta, alpha: may be NULL (treated as all zero).  theta: required.
 *   S0: momentum state [B|1][H][dv][dk] or NULL (zero).
 *   S_out: [B][H][dv][dk] or NULL (not written).
 * Other arguments and shape rules as ttm_linear_fwd.
 */
int ttm_titans_fwd(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                   const void* q, const void* k, const void* v,
                   const float* eta, const float* theta, const float* alpha,
                   const float* W0, const float* S0, int w0_shared_over_batch,
                   void* z, float* W_out, float* S_out, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace ttm_linear_fwd / ttm_titans_fwd need for these sizes
 * under the current kernel policy: 0 when the selected kernel needs none (or
 * the shape is rejected), else B*H*ceil(T/64) * 17424 for the tensor-core
 * path: one record per (sequence, 64-token chunk) of the chunk coefficients
 * of the matrix form ("TTT layers 与 fast weights" §1.1 eq (9) with the decay
 * and momentum unrolling of "论文速览 | Titans" §4.3-§4.5): the matrix C,
 * beta_t, c_t and the last rows of C and of the momentum weights.
 */
size_t ttm_linear_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype);

/* The Titans scan with chunk-level gates ("论文速览 | Titans" §4.6): theta, eta
 * and alpha are shared by all tokens of a chunk rather than given per token,
 * which makes the recurrence inside each chunk time-invariant.  Identical to
 * ttm_titans_fwd except that eta, theta, alpha are [B][H][ceil(T / chunk)] fp32
 * (one value per sequence and chunk; eta / alpha may be NULL = 0), and that
 * the kernels read them directly.  Same shapes, workspace
 * (ttm_linear_workspace_size), errors and aliasing rules as ttm_titans_fwd. */
int ttm_titans_fwd_chunk_gates(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                               const void* q, const void* k, const void* v,
                               const float* eta, const float* theta, const float* alpha,
                               const float* W0, const float* S0, int w0_shared_over_batch,
                               void* z, float* W_out, float* S_out,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * The Titans / linear scan with every tensor in HOST memory: the sequence is
 * streamed through the device in segments of `seg_tokens` tokens (a positive
 * multiple of `chunk`).  While segment i is scanned on `stream`, an internal
 * stream copies segment i + 1's q, k, v and gates in and another copies
 * segment i - 1's z out.  The state crosses segment boundaries in fp32 on the
 * device; a boundary falls between two chunks, where the chunk form restarts
 * from whatever state the previous chunk left ("TTT layers 与 fast weights" eq
 * (6): every gradient of a chunk is taken at the chunk-start state), so the
 * result is that of ttm_titans_fwd up to rounding order.
 *   q, k, v, eta, theta, alpha, W0, S0: host, layouts as ttm_titans_fwd (page-
 *     locked memory gives full copy bandwidth; pageable memory works, slower).
 *   z, W_out, S_out: host, written asynchronously: synchronise `stream` before
 *     reading them.  S_out may be NULL.
 *   workspace: device memory, 256-byte aligned, at least
 *     ttm_titans_fwd_host_workspace_size(...) bytes (two segments of inputs and
 *     outputs, four state buffers and the scan's own workspace); the caller
 *     owns it and must not touch it until `stream` has passed the call.
 * `stream` (the caller's) runs the scans; on return it has been made to wait
 * for every copy of the call.  The internal streams and events are created
 * once per device on first use and reused; calls are serialised on the host.
 * Errors: TTM_ERR_INVALID_ARG for malformed arguments or a short workspace
 * (nothing enqueued), anything ttm_titans_fwd returns for a segment, and
 * TTM_ERR_CUDA for a failed copy or event operation.
 */
size_t ttm_titans_fwd_host_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                          int dtype, int seg_tokens);
int ttm_titans_fwd_host(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                        const void* q, const void* k, const void* v,
                        const float* eta, const float* theta, const float* alpha,
                        const float* W0, const float* S0, int w0_shared_over_batch,
                        void* z, float* W_out, float* S_out, int seg_tokens,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Deep memory: f(x) = W2 GELU(W1 x), hidden units `hidden`, analytic inner
 * gradients e = 2 (y - v), dW2 = e a^T, dW1 = ((W2^T e) * GELU'(h)) k^T
 * ("论文速览 | Titans" §3.9 with L_M = 2; "Continual Learning: From Attention
 * to Neural Memory" §4.2), with the same momentum/forgetting and chunk rule.
 *   q, k, v, z: [B][H][T][d].  W1_0, S1_0: [B|1][H][hidden][d].
 *   W2_0, S2_0: [B|1][H][d][hidden].  Outputs likewise with B rows.
 *   eta, alpha, S1_0, S2_0: may be NULL.  S1_out and S2_out are both NULL or
 *   both given, and must be given whenever eta is (they double as the running
 *   momentum state).
 * Shapes: d a multiple of 8, hidden a multiple of 8 (kernel limits reported
 * as TTM_ERR_UNSUPPORTED).
 * Kernels: fp32 arithmetic by default (a two-CTA cluster per sequence with the
 * state in shared memory for (d, hidden) in {(32, 128), (64, 256), (128, 128)}
 * and chunk <= 16; one CTA per sequence otherwise).  Under the tensor-core
 * policy (ttm_set_kernel_policy) bf16 inputs with d = 64, hidden = 256,
 * chunk 16 run a tcgen05 kernel whose recurrent operands are rounded to bf16.
 */
int ttm_mlp_fwd(int B, int H, int T, int d, int hidden, int chunk, int dtype,
                const void* q, const void* k, const void* v,
                const float* eta, const float* theta, const float* alpha,
                const float* W1_0, const float* W2_0, const float* S1_0, const float* S2_0,
                int w0_shared_over_batch,
                void* z, float* W1_out, float* W2_out, float* S1_out, float* S2_out,
                void* stream);

/*
 * ttm_titans_fwd_noalloc — ttm_titans_fwd for callers that cannot allocate
 * device memory.  (No counterpart on the pages: this is a deployment variant
 * of the same scan, not part of the method.)
 *
 * Who needs it: callers that are handed only their input and output buffers
 * and may not call cudaMalloc or any allocating routine themselves, so they
 * cannot provide the workspace ttm_titans_fwd needs for its tensor-core path
 * (for example a plug-in inside a host framework that plans all device memory
 * in advance, or code that must stay allocation-free).
 *
 * Arguments, results and errors are those of ttm_titans_fwd without the
 * workspace arguments.  The scratch comes from one block of
 * TTM_NOALLOC_SCRATCH_BYTES (16 MiB) compiled into the library: every GPU that
 * loads the library holds that block until the process exits.
 *   - Limit: a call whose workspace requirement (ttm_linear_workspace_size)
 *     exceeds TTM_NOALLOC_SCRATCH_BYTES returns TTM_ERR_UNSUPPORTED before
 *     touching the GPU; with the tensor-core path that is
 *     B*H*ceil(T/64) * 17424 bytes, i.e. at most 962 (sequence, 64-token
 *     chunk) pairs.
 *   - Set-up: the first call on each device looks up the block's device
 *     address (with that device current); make that first call before any
 *     stream capture.
 *   - Sharing: all calls on a device use the same block and it keeps the
 *     last call's contents (nothing in it needs to start at zero).  Calls
 *     that overlap on the GPU (e.g. on two streams) race on it: serialise them.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define TTM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int ttm_titans_fwd_noalloc(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                           const void* q, const void* k, const void* v,
                           const float* eta, const float* theta, const float* alpha,
                           const float* W0, const float* S0, int w0_shared_over_batch,
                           void* z, float* W_out, float* S_out, void* stream);

/*
 * Streaming decode step of the Titans / linear memory: continues every
 * sequence by n tokens in the primal, token-by-token form, as the pages
 * prescribe for decoding after a chunked (dual-form) prefill ("TTT layers 与
 * fast weights" §1.1 and eq (6): the gradient of every token of a chunk is
 * taken at the chunk-start state; momentum and forgetting as in
 * "论文速览 | Titans" §3.4-§3.7).  Per token t, with Wc the memory at the start
 * of the current chunk:
 *     e = Wc k_t - v_t;  S = eta_t S - theta_t 2 e k_t^T;
 *     W = (1 - alpha_t) W + S;  z_t = W q_t  (read after the token's own write);
 * a token that opens a chunk first sets Wc = W.
 *   pos: tokens of the current chunk processed before this call, 0 <= pos <
 *     chunk, the same for every sequence of the call (sequences decoded in
 *     lockstep).  After the call the position is (pos + n) % chunk; the caller
 *     keeps it.  A prefill by ttm_titans_fwd over a multiple of `chunk` tokens
 *     continues with W = W_out, S = S_out, pos = 0 (Wc is then set by the first
 *     token).
 *   q, k: [B][H][n][dk], v: [B][H][n][dv] in dtype; eta, theta, alpha: [B][H][n]
 *     fp32 (eta, alpha may be NULL = 0; theta required); z: [B][H][n][dv] in
 *     dtype, written.
 *   W, S, Wc: [B][H][dv][dk] fp32, read and updated in place (S may be NULL
 *     only when eta is NULL; Wc is written when a chunk opens during the call).
 *   All pointers are device memory owned by the caller, 16-byte aligned; the
 *   outputs must not overlap each other or the inputs.
 * Shapes: B, H, n >= 1; chunk >= 1; dk, dv as for ttm_titans_fwd, dk <= 512
 * (else TTM_ERR_UNSUPPORTED).  Asynchronous on `stream`; TTM_ERR_INVALID_ARG
 * for malformed arguments, TTM_ERR_CUDA if the launch fails.
 */
int ttm_titans_step(int B, int H, int n, int dk, int dv, int chunk, int pos, int dtype,
                    const void* q, const void* k, const void* v,
                    const float* eta, const float* theta, const float* alpha,
                    float* W, float* S, float* Wc, void* z, void* stream);

/* The decode step of TTT-Linear (no momentum, no forgetting): ttm_titans_step
 * with eta = alpha = S = NULL, i.e. W = W - theta_t 2 (Wc k_t - v_t) k_t^T. */
int ttm_linear_step(int B, int H, int n, int dk, int dv, int chunk, int pos, int dtype,
                    const void* q, const void* k, const void* v, const float* theta,
                    float* W, float* Wc, void* z, void* stream);

/* Gradient of the linear / Titans scan (the outer, "meta" gradient): the
 * derivative of a scalar outer loss L with respect to every input of
 * ttm_titans_fwd, given the adjoints of its outputs.  The outer loss trains
 * the projections, the rates and W0 through the inner updates, so the
 * gradient follows the chain of state transitions backward, through every
 * write ("Continual Learning: From Attention to Neural Memory" §4.5 and its
 * expanded note; "TTT layers 与 fast weights" §1.2, which also prescribes the
 * finite-difference and primal / dual gradient checks).
 *   Inputs: exactly those of the ttm_titans_fwd call whose outputs the
 *     adjoints belong to (same shapes, dtype, layouts, shared flag).
 *   dz: [B][H][T][dv] in dtype, dL/dz.  dW, dS: [B][H][dv][dk] fp32, dL/dW_out
 *     and dL/dS_out (NULL = 0).
 *   Outputs (written, fp32 unless stated): dq_out, dk_out [B][H][T][dk] and
 *     dv_out [B][H][T][dv] in dtype (dL/dq, dL/dk, dL/dv); dtheta [B][H][T]; deta, dalpha [B][H][T] (NULL to
 *     skip; must be NULL when eta / alpha are); dW0, dS0 shaped like W0 / S0
 *     ([1][H][dv][dk] summed over the batch when W0 is shared; dS0 NULL to skip).
 *   workspace: device scratch of ttm_titans_bwd_workspace_size() bytes (may be
 *     NULL when T = 0): the state and its adjoint at every chunk boundary plus
 *     per-chunk coefficient records (and score tiles on the tensor-core path).
 *     Contents on return are unspecified.
 *   All pointers are device memory owned by the caller, 16-byte aligned; no
 *   output may overlap an input, another output or the workspace.
 * Shapes: as for ttm_titans_fwd, with chunk <= 64 and dk <= 128
 * (TTM_ERR_UNSUPPORTED otherwise).  Computation follows the chunk form: the
 * forward scan writes the state at every chunk start, a reverse pass over the
 * chunks carries the adjoint of the state, and a chunk-parallel pass forms the
 * token gradients.  For bf16 with dk = dv in {64, 128} and chunk 64 (unless the
 * policy is TTM_KERNEL_SIMT) those passes run on the tensor cores: bf16
 * operands with fp32 accumulation, the state and its adjoint kept in bf16 at the
 * chunk boundaries, the adjoint carried in fp32 between them
 * (ttm_last_kernel() reports TTM_KID_BWD_TC); otherwise in fp32 on the CUDA
 * cores (TTM_KID_BWD_SIMT).  Asynchronous on `stream`; TTM_ERR_INVALID_ARG for
 * malformed arguments or a short workspace, TTM_ERR_CUDA if a launch fails; a
 * bounded wait of the tensor-core passes that gives up sets the device status
 * word to TTM_ERR_TIMEOUT (ttm_device_status). */
size_t ttm_titans_bwd_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                                     int w0_shared_over_batch);
int ttm_titans_bwd(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                   const void* q, const void* k, const void* v,
                   const float* eta, const float* theta, const float* alpha,
                   const float* W0, const float* S0, int w0_shared_over_batch,
                   const void* dz, const float* dW, const float* dS,
                   void* dq_out, void* dk_out, void* dv_out,
                   float* deta, float* dtheta, float* dalpha,
                   float* dW0, float* dS0,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Gradient of TTT-Linear (no momentum, no forgetting): ttm_titans_bwd with
 * eta = alpha = S0 = dS = NULL and no deta / dalpha / dS0; the workspace size
 * is ttm_titans_bwd_workspace_size() of the same shape. */
int ttm_linear_bwd(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                   const void* q, const void* k, const void* v, const float* theta,
                   const float* W0, int w0_shared_over_batch,
                   const void* dz, const float* dW,
                   void* dq_out, void* dk_out, void* dv_out, float* dtheta, float* dW0,
                   void* workspace, size_t workspace_bytes, void* stream);

/* DGD memory scan: the update of "Nested Learning" §8.1 eq (88) with a matrix
 * memory and the L2 objective of eq (93), taken chunk-wise as in §8.2 (every
 * gradient of a chunk at the state left by the previous chunk, Mc):
 *     z_t = M_{t-1} q_t   (read before the token's write, as eq (86) prints
 *                          y_t = M_{memory,t-1}(q_t))
 *     M_t = M_{t-1} (alpha_t I - eta_t k_t k_t^T) - eta_t (Mc k_t - v_t) k_t^T
 * eta_t is the step and alpha_t a retention factor (alpha = 1 keeps the
 * memory), both as the page prints them: note that alpha here multiplies the
 * memory, unlike the forgetting rate of ttm_titans_fwd (which keeps 1 - alpha),
 * and the gradient carries no factor 2.  Unlike the Titans memory, the
 * k k^T term acts on the running state, so the tokens of a chunk are coupled
 * through the key products k_s . k_t.
 *   q, k: [B][H][T][dk], v: [B][H][T][dv] in dtype; eta, alpha: [B][H][T] fp32
 *     (both required when T > 0); W0: [B or 1][H][dv][dk] fp32 (1 when
 *     w0_shared_over_batch); z: [B][H][T][dv] in dtype and W_out: [B][H][dv][dk]
 *     fp32, written.  W_out may be W0 (in place) when W0 is not shared.
 *   workspace: device scratch of ttm_dgd_workspace_size() bytes for these sizes
 *     (NULL when that is 0), owned by the caller, no overlap with any other
 *     argument.
 *   All pointers are device memory owned by the caller, 16-byte aligned; no
 *   other overlap is allowed.
 * Shapes: B, H >= 1; T >= 0; chunk >= 1; dk, dv as for ttm_titans_fwd, dk <= 512
 * (else TTM_ERR_UNSUPPORTED).  Kernels (under the ttm_set_kernel_policy policy):
 *   - bf16, dk = dv in {64, 128}, chunk 64: the chunk form on the tensor cores.
 *     With a_t the product of the chunk's alpha up to t and R[t][s] the product
 *     of alpha over s < tau < t, the chunk's gradients g solve the unit
 *     lower-triangular system (I + L) g = R0, L[t][s] = eta_t R[t][s] (k_s.k_t),
 *     R0_t = eta_t ((a_{t-1} + 1) Mc k_t - v_t); a pre-pass computes, for every
 *     chunk at once, N = (I + L)^-1 in fp32 and the chunk operators
 *     A~N (A~[t][s] = R[t][s] (q_t.k_s), s < t) and K^T diag(R[n-1][.]) N in
 *     bf16 into the workspace (8192 + 128 dk + 1024 bytes per (sequence,
 *     64-token chunk)); the scan then applies them with two tensor-core
 *     products per chunk.  Operands bf16, accumulation fp32.
 *   - otherwise (or under TTM_KERNEL_SIMT): fp32, token by token per row of M
 *     (every row evolves on its own), one warp per (sequence, row); no
 *     workspace.
 * Asynchronous on `stream`; TTM_ERR_INVALID_ARG for malformed arguments or a
 * short workspace, TTM_ERR_CUDA if the launch fails. */
int ttm_dgd_fwd(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                const void* q, const void* k, const void* v,
                const float* eta, const float* alpha,
                const float* W0, int w0_shared_over_batch,
                void* z, float* W_out, void* workspace, size_t workspace_bytes,
                void* stream);

/* Bytes of workspace ttm_dgd_fwd needs for these sizes under the current
 * kernel policy: B*H*ceil(T/64) * (8192 + 128 dk + 1024) on the tensor-core
 * path, else 0 (also for shapes no kernel takes). */
size_t ttm_dgd_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype);

/* Decode step of the DGD memory: continues every sequence by n tokens from the
 * state W at in-chunk position pos, exactly as ttm_titans_step does for the
 * Titans memory (same meaning of pos, Wc, shapes and errors), with the DGD
 * update of ttm_dgd_fwd.  eta, alpha: [B][H][n] fp32, both required. */
int ttm_dgd_step(int B, int H, int n, int dk, int dv, int chunk, int pos, int dtype,
                 const void* q, const void* k, const void* v,
                 const float* eta, const float* alpha,
                 float* W, float* Wc, void* z, void* stream);

/* LMM layer: the neural memory used on its own as a sequence layer
 * ("论文速览 | Titans" §6.4) with the projection details of §7.1-§7.3, for
 * x [B][T][D] (D = H d) in bf16:
 *   p = x W_in                          W_in [D][4D + 3H] bf16: columns q | k | v | g (D
 *                                       each), then the theta, eta, alpha logits (H each)
 *   q, k, v = SiLU(causal depthwise conv of width conv_k of p's q, k, v columns);
 *     conv_w [3][D][conv_k] fp32, tap j weighting token t - (conv_k - 1) + j
 *     (tokens before the sequence start read zero); q and k l2-normalised per head
 *   theta = theta_scale sigmoid, eta = sigmoid, alpha = sigmoid of the logits
 *   z = the Titans memory scan of ttm_titans_fwd per head, from W0 ([B or 1][H][d][d]
 *     fp32, 1 when w0_shared_over_batch; S0 = 0)
 *   o = z / sqrt(mean_d(z^2) + 1e-6) * rms_w * g   (per head; rms_w [d] fp32; g the
 *     linear gate from p)
 *   y = x + o W_o                       W_o [D][D] bf16; y [B][T][D] bf16, written
 * W_out and S_out ([B][H][d][d] fp32; S_out may be NULL) receive the final memory.
 * The pages leave the wiring open; this is the plainest reading: the
 * projection, conv, SiLU order of the modern recurrent layers the page cites,
 * and a linear (un-squashed) output gate.
 * The two projections are plain bf16 GEMMs through cuBLAS (fp32 accumulation);
 * p, q, k, v, z and o are stored in bf16.  workspace: device scratch of
 * ttm_lmm_layer_workspace_size() bytes, owned by the caller (it also serves as
 * cuBLAS's workspace).  All pointers are device memory, 16-byte aligned; no
 * output may overlap an input, another output or the workspace.
 * Shapes: B, T, H >= 1; d in {32, 64, 128, 256}; 1 <= conv_k <= 8; chunk >= 1
 * (TTM_ERR_UNSUPPORTED otherwise).  Asynchronous on `stream`;
 * TTM_ERR_INVALID_ARG for malformed arguments or a short workspace,
 * TTM_ERR_CUDA if a launch or a GEMM fails. */
size_t ttm_lmm_layer_workspace_size(int B, int T, int H, int d, int chunk, int w0_shared);
int ttm_lmm_layer_fwd(int B, int T, int H, int d, int chunk, int conv_k,
                      const void* x, const void* W_in, const float* conv_w,
                      const float* rms_w, const void* W_o, float theta_scale,
                      const float* W0, int w0_shared_over_batch,
                      void* y, float* W_out, float* S_out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* The activation of the 2-layer memory and its derivative, evaluated on the
 * device exactly as the tensor-core 2-layer kernel evaluates them: for the n
 * values x[i], y[i] = GELU(x) = x Phi(x) and, if dy is not NULL,
 * dy[i] = GELU'(x) = Phi(x) + x phi(x).  The pages name no activation for the
 * memory MLP; the library reads it as the erf-based GELU (Phi the standard
 * normal CDF, phi its density).  x, y, dy: device fp32 arrays of n elements,
 * owned by the caller; y may be x (in place), dy must not overlap x or y.
 * Asynchronous on `stream`.  Returns TTM_ERR_INVALID_ARG for n < 0 or bad
 * pointers, TTM_ERR_CUDA if the launch fails. */
int ttm_mlp_gelu(const float* x, float* y, float* dy, int n, void* stream);

/* Static English text for a ttm_status value (never NULL). */
const char* ttm_status_str(int status);

/* Sets the process-wide kernel policy (ttm_kernel_policy); returns the previous
 * one, or -1 for an unknown value (policy unchanged).  Not thread-safe with
 * concurrent ttm_*_fwd calls. */
int ttm_set_kernel_policy(int policy);

/* ttm_kernel_id of the main kernel enqueued by this thread's last successful
 * ttm_*_fwd call (TTM_KID_NONE before any). */
int ttm_last_kernel(void);

/* Number of kernels this process has enqueued through ttm_*_fwd so far
 * (monotonic; successful calls only; the tensor-core linear path enqueues two:
 * the coefficient pre-pass and the scan). */
unsigned long long ttm_launch_count(void);

/* Failure-detection hooks for tests (no counterpart on the pages: they exist
 * so that the error paths can be exercised without faulting a GPU).
 *   TTM_DBG_WAIT_CYCLES, n >= 0: every bounded device wait of the tensor-core
 *     kernels gives up after n SM clock cycles (0 restores the default, about
 *     2 s).  Applies to calls made from now on.
 *   TTM_DBG_STALL_CHUNK, c >= 0: the next call that runs the tensor-core
 *     linear / Titans scan announces 16 bytes more for chunk c's input tiles
 *     than it copies, so that chunk's barrier never completes: every wait on it
 *     runs out, the kernel sets the device status word to TTM_ERR_TIMEOUT,
 *     drains its copies and MMAs, frees its tensor memory and returns (its
 *     outputs are then invalid).  A ttm_titans_bwd / ttm_linear_bwd call on
 *     the tensor-core path takes the setting for its chain pass instead, with
 *     c counted in the chain's order (c = 0 is the last chunk).  The setting
 *     is used up by that one call; -1 clears it.  Nothing faults, traps or
 *     hangs.
 *   TTM_DBG_FAIL_CALLS, n >= 0: the next n calls of ttm_linear_fwd,
 *     ttm_titans_fwd (and the variants built on them) and ttm_mlp_fwd return
 *     TTM_ERR_CUDA after validating their arguments, without enqueueing
 *     anything (host-side injection of a failed launch).
 * Returns TTM_OK, or TTM_ERR_INVALID_ARG for an unknown option or a value out
 * of range.  The settings are process-wide. */
enum { TTM_DBG_WAIT_CYCLES = 1, TTM_DBG_STALL_CHUNK = 2, TTM_DBG_FAIL_CALLS = 3 };
int ttm_debug_set(int option, long long value);

/* Number of CUDA devices this library's own runtime can reach (0 when there
 * is no GPU or no usable driver).  Touches no device memory; host-side test
 * suites use it to decide whether a GPU is reachable. */
int ttm_cuda_device_count(void);

/* Synchronises the current device, then returns and clears its status word:
 * TTM_OK, or TTM_ERR_TIMEOUT if a tensor-core kernel abandoned a bounded wait
 * since the last query (its outputs are then invalid).  TTM_ERR_CUDA if the
 * synchronisation itself failed. */
int ttm_device_status(void);

#ifdef __cplusplus
}
#endif

#endif /* TTM_H */
