// Internal interface between the C-ABI layer (ttm_api.cu) and the kernel
// translation units.  Host-side only; no torch types anywhere.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

namespace ttm {

// One call of the linear / Titans scan.  Pointers are device pointers that the
// API layer has already validated (non-NULL where required, 16-byte aligned).
struct LinearArgs {
    int B, H, T, dk, dv, chunk;
    int bf16;                 // 1: q, k, v, z are bf16; 0: fp32
    const void *q, *k, *v;
    const float *eta, *theta, *alpha;   // eta / alpha may be NULL (= 0)
    const float *W0, *S0;               // S0 may be NULL (= 0)
    int shared;                         // W0/S0 have a leading dim of 1
    void* z;
    float *W_out, *S_out;               // S_out may be NULL
    void* workspace;                    // caller-provided device scratch (may be NULL)
    size_t workspace_bytes;
    int* status;                        // device status word (bounded waits)
    // When set, the state at every chunk start is written to
    // ckpt[seq][chunk][W | S][dv][dk] (fp32), and z / W_out may be NULL.  The
    // gradient passes read these checkpoints.
    float* ckpt;
    int ckpt_bf16;            // tensor-core scan only: ckpt holds bf16 values
    // Tensor-core scan with ckpt only (may be NULL): the masked score tile
    // A~[t][s] = C[t][s] (q_t . k_s) (zero for s > t and outside the chunk) of
    // every chunk in bf16, score_tiles[seq][chunk] = 64 rows t of 128 bytes,
    // the 16-byte group g of row t stored at position g ^ (t % 8).
    void* score_tiles;
    // Chunk-shared gates: theta / eta / alpha hold one value per (sequence,
    // chunk), [B][H][ceil(T / chunk)], instead of one per token.
    int gates_per_chunk;
    // Limit of every bounded wait of the tensor-core kernels, in SM clock
    // cycles (0: the default, about 2 s).
    long long wait_cycles;
    // Failure-detection test hook of the tensor-core scan (0: off).  With
    // c + 1 the producer announces 16 bytes more for chunk c's tiles than it
    // copies, so that chunk's barrier never completes and every wait on it
    // runs out: the kernel then reports TTM_ERR_TIMEOUT and unwinds.
    int debug_stall;
};

// Per-chunk coefficient record that the tensor-core scan's pre-pass writes
// into its workspace (record seq * nchunks + chunk, kCoefRecBytes each): the
// table C[t][s] (64 x 64 fp32, row t at 256 t bytes, its 16-byte groups
// XOR-permuted by t % 16), then at kCoefVec the vectors beta_t, c_t, C[n-1][s],
// theta_s m(s, n-1) (64 floats each, offsets below) and the scalars
// beta_{n-1}, c_{n-1}, P_{n-1}, n.
constexpr uint32_t kCoefRecBytes = 17424;
constexpr uint32_t kCoefVec = 16384;
constexpr uint32_t kCoefBeta = 0, kCoefC = 256, kCoefCend = 512, kCoefPend = 768,
                   kCoefScal = 1024, kCoefVecBytes = 1040;   // relative to kCoefVec

// Index of token t's gate of sequence seq (per token, or per chunk).
__host__ __device__ inline size_t gate_index(const LinearArgs& a, size_t seq, int t) {
    if (!a.gates_per_chunk) return seq * a.T + t;
    const int nch = (a.T + a.chunk - 1) / a.chunk;
    return seq * nch + t / a.chunk;
}

struct MlpArgs {
    int B, H, T, d, hidden, chunk;
    int bf16;
    const void *q, *k, *v;
    const float *eta, *theta, *alpha;
    const float *W1_0, *W2_0, *S1_0, *S2_0;
    int shared;
    void* z;
    float *W1_out, *W2_out, *S1_out, *S2_out;
    int* status;
};

// One call of the decode step (step.cu): n tokens per sequence in the primal
// form.  W, S, Wc are updated in place; pos is the shared position within the
// chunk at the call's start.
struct StepArgs {
    int B, H, n, dk, dv, chunk, pos;
    int bf16;
    const void *q, *k, *v;
    const float *eta, *theta, *alpha;   // eta / alpha may be NULL (= 0)
    float *W, *S, *Wc;                  // S may be NULL when eta is NULL; Wc NULL: not kept
    void* z;
    // mode 0: linear / Titans memory.  mode 1: DGD memory, with theta the step
    // eta_t and alpha the retention factor alpha_t (required); eta, S unused.
    int mode;
    // When W_in is set the state starts from W_in ([B or 1][H][dv][dk], 1 when
    // w_shared) instead of W, and W only receives the result (a whole scan).
    const float* W_in;
    int w_shared;
};

// One call of the DGD memory scan in chunk form (scan_dgd_tc.cu): eta is the
// step and alpha the retention factor, [B][H][T] fp32, both required.
struct DgdArgs {
    int B, H, T, dk, dv, chunk;
    int bf16;
    const void *q, *k, *v;
    const float *eta, *alpha;
    const float* W0;          // [B or 1][H][dv][dk]
    int shared;
    void* z;
    float* W_out;
    void* workspace;          // caller-provided device scratch
    size_t workspace_bytes;
    int* status;              // device status word (bounded waits)
    long long wait_cycles;    // bounded-wait limit in SM clock cycles (0: default)
};

// One call of the gradient of the linear / Titans scan (scan_bwd.cu).  Inputs
// as in LinearArgs plus the adjoints of the outputs; every output is a
// gradient of the same shape as its input (dq / dk / dv in the input dtype,
// the rest fp32).  dW / dS (adjoints of the final state), deta, dalpha and dS0
// may be NULL.
struct BwdArgs {
    int B, H, T, dk, dv, chunk;
    int bf16;
    const void *q, *k, *v;
    const float *eta, *theta, *alpha;
    const float *W0, *S0;
    int shared;
    const void* dz;
    const float *dW, *dS;
    void *dq, *dk_, *dv_;
    float *deta, *dtheta, *dalpha;
    float *dW0, *dS0;
    void* workspace;
    size_t workspace_bytes;
    int fwd_tc;     // 1: the tensor-core scan writes the checkpoints (bf16, d 64 / 128, chunk 64)
    int local_tc;   // 1: the local pass runs on the tensor cores (bf16, d 64 / 128, chunk 64)
    // Failure-detection test hook of the tensor-core chain (0: off): with k + 1
    // the chain's loader announces 16 bytes more than it copies for its k-th
    // chunk (in reverse order), so that stage's waits run out.
    int debug_stall;
    int* status;    // device status word of the tensor-core kernels' bounded waits
    long long wait_cycles;   // their wait limit in SM clock cycles (0: the default)
};

// One call of the LMM layer (lmm_layer.cu + the scan); bf16 activations.
struct LmmArgs {
    int B, T, H, d, chunk, conv_k;
    const void* x;          // [B][T][D] bf16, D = H d
    const void* W_in;       // [D][4D + 3H] bf16: q | k | v | g | theta, eta, alpha logits
    const float* conv_w;    // [3][D][conv_k]: causal depthwise taps of q, k, v
    const float* rms_w;     // [d]: per-channel scale of the per-head RMS norm
    const void* W_o;        // [D][D] bf16
    float theta_scale;      // theta = theta_scale * sigmoid(logit)
    const float* W0;        // [B or 1][H][d][d] initial memory
    int w0_shared;
};

// fp32 CUDA-core kernels (scan_simt.cu).  The *_supported functions decide
// on the host whether a shape fits the kernel's on-chip budget.
bool linear_simt_supported(const LinearArgs& a);
cudaError_t linear_simt_launch(const LinearArgs& a, cudaStream_t s);
bool mlp_simt_supported(const MlpArgs& a);
cudaError_t mlp_simt_launch(const MlpArgs& a, cudaStream_t s);
// Register-blocked CUDA-core MLP kernel (scan_mlp_simt.cu): d in {16, 32, 64,
// 128}, hidden a multiple of 4, chunk <= 32, 16-byte aligned state buffers.
// mlp_simt_launch uses it whenever it applies.
bool mlp_simt2_supported(const MlpArgs& a);
cudaError_t mlp_simt2_launch(const MlpArgs& a, cudaStream_t s);
// Two-CTA cluster variant (scan_mlp_cluster.cu): each CTA keeps half of the
// state in shared memory.  (d, hidden) in {(32, 128), (64, 256), (128, 128)},
// chunk <= 16.  mlp_simt_launch prefers it whenever it applies.
bool mlp_cluster_supported(const MlpArgs& a);
cudaError_t mlp_cluster_launch(const MlpArgs& a, cudaStream_t s);

// tcgen05 + TMA kernel for the linear / Titans scan (scan_linear_tc.cu).  It
// needs linear_tc_workspace_bytes() of workspace for the per-chunk
// coefficients computed by its pre-pass.
bool linear_tc_supported(const LinearArgs& a);
size_t linear_tc_workspace_bytes(const LinearArgs& a);
cudaError_t linear_tc_launch(const LinearArgs& a, cudaStream_t s);

// 3-D TMA map (a CUtensorMap, passed as void*) of a bf16 tensor viewed as
// [BH sequences][T tokens][D], tile box {bx, 64 tokens, 1}, optionally with the
// 128-byte swizzle (scan_linear_tc.cu).
bool make_token_tile_map(void* map, const void* ptr, int BH, int T, int D, int bx, bool swz);

// tcgen05 + TMA kernel with one CTA per sequence for d_k = d_v = 64
// (scan_linear_seq.cu): 64-token tiles whose gradient points fall every
// `chunk` in {16, 32} tokens; no workspace.
bool linear_seq_supported(const LinearArgs& a);
cudaError_t linear_seq_launch(const LinearArgs& a, cudaStream_t s);

// tcgen05 + TMA kernel for the 2-layer MLP memory (scan_mlp_tc.cu): bf16,
// d = 64, hidden = 256, chunk 16; one cluster of two CTAs per sequence.
bool mlp_tc_supported(const MlpArgs& a);
cudaError_t mlp_tc_launch(const MlpArgs& a, cudaStream_t s);
// tcgen05 + TMA kernels of the DGD memory in chunk form (scan_dgd_tc.cu):
// bf16, d_k = d_v in {64, 128}, chunk 64.  A pre-pass writes per chunk the
// operators A~N and K^T diag(r) N (dgd_tc_workspace_bytes() of workspace), then
// the scan runs one CTA per (sequence, 16 rows of the memory).
bool dgd_tc_supported(const DgdArgs& a);
size_t dgd_tc_workspace_bytes(const DgdArgs& a);
cudaError_t dgd_tc_launch(const DgdArgs& a, cudaStream_t s);

// Decode step (step.cu): one warp per row of W; dk <= 512.
bool linear_step_supported(const StepArgs& a);
cudaError_t linear_step_launch(const StepArgs& a, cudaStream_t s);

// Tensor-core local pass of the gradient (scan_bwd_tc.cu): bf16, dk = dv in
// {64, 128}, chunk 64; reads the chunk-start checkpoints and chunk-end adjoints
// (fp32, [seq][chunk][W | S][dv][dk]) that the other passes leave in the workspace.
bool bwd_local_tc_supported(const BwdArgs& a);
// Its chain pass on the tensor cores (same shapes): the adjoint at every chunk
// end from the records pass's records; offsets in floats into the workspace.
// The tensor-core scan that wrote the checkpoints also wrote its coefficient
// records (coef, kCoefRecBytes per chunk) and the masked score tiles (tiles).
cudaError_t bwd_chain_tc_launch(const BwdArgs& a, float* ws, size_t off_adj, const void* coef,
                                const void* tiles, size_t off_part, cudaStream_t s);
// Checkpoints (ckpt) and adjoints (adj) are bf16 [seq][chunk][W | S][d][d]:
// the tensor-core scan writes them with ckpt_bf16, the tensor-core chain the
// adjoints.
cudaError_t bwd_local_tc_launch(const BwdArgs& a, const void* ckpt, const void* adj,
                                const void* coef, cudaStream_t s);

// Gradient of the linear / Titans scan (scan_bwd.cu): chunk <= 64, dk <= 128.
// The workspace holds the state and its adjoint at every chunk boundary.
bool linear_bwd_supported(const BwdArgs& a);
size_t linear_bwd_workspace_bytes(const BwdArgs& a);
cudaError_t linear_bwd_launch(const BwdArgs& a, cudaStream_t s, int* launches);

// LMM layer pieces (lmm_layer.cu): d a multiple of 32 up to 256, conv width 1..8.
bool lmm_supported(const LmmArgs& a);
cudaError_t lmm_prep_launch(const LmmArgs& a, const void* proj, void* qkv, float* gates,
                            cudaStream_t s);
cudaError_t lmm_post_launch(const LmmArgs& a, const void* proj, const void* z, void* o,
                            cudaStream_t s);
bool gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, float beta,
               void* scratch, size_t scratch_bytes, cudaStream_t s);

// The activation of that kernel on n values: y = GELU(x), dy = GELU'(x) (dy may be NULL).
cudaError_t mlp_gelu_launch(const float* x, float* y, float* dy, int n, cudaStream_t s);

}  // namespace ttm
