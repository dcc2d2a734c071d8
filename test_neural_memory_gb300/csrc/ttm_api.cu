// C ABI of libttm.so: host-side argument validation, kernel selection and
// launch.  Declarations and the full contract are in include/ttm.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/ttm.h"
#include "kernels.h"

namespace {

// Device status word: tensor-core kernels set it when a bounded wait gives up.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];  // per-device address of g_status_word
std::mutex g_status_mu;          // guards the first lookup on each device

int g_policy = TTM_KERNEL_AUTO;

// Failure-detection test hooks (ttm_debug_set).
std::atomic<long long> g_wait_cycles{0};   // bounded-wait limit of the tensor-core kernels
std::atomic<int> g_stall_chunk{-1};        // next tensor-core linear scan: chunk that stalls
std::atomic<int> g_fail_calls{0};          // scan calls still to fail before their launch

// Host-side fault injection: true when this call must report a failed launch
// (the hook counts down one call each time).
bool injected_failure() {
    int n = g_fail_calls.load();
    while (n > 0)
        if (g_fail_calls.compare_exchange_weak(n, n - 1)) return true;
    return false;
}
unsigned long long g_launches = 0;
thread_local int t_last_kernel = TTM_KID_NONE;

int* status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
    const void* p;
    size_t bytes;
};

bool overlap(Span a, Span b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Output `o` may coincide exactly with input `in` only when `exact_ok`.
bool bad_alias(Span o, Span in, bool exact_ok) {
    if (!overlap(o, in)) return false;
    return !(exact_ok && o.p == in.p && o.bytes == in.bytes);
}

bool dims_ok(int x, int dtype) { return x >= 1 && x % (dtype == TTM_BF16 ? 8 : 4) == 0; }

// Kernel the current policy would pick for these arguments (host decision).
// The two tensor-core kernels never compete: the sequence-per-CTA kernel
// takes d = 64 with gradient points every 16 or 32 tokens, the row-slice
// kernel chunk 64.
int select_linear(const ttm::LinearArgs& a) {
    const bool seq_ok = ttm::linear_seq_supported(a);
    const bool tc_ok = ttm::linear_tc_supported(a);
    const bool simt_ok = ttm::linear_simt_supported(a);
    const int tc_kid = seq_ok ? TTM_KID_LINEAR_SEQ : (tc_ok ? TTM_KID_LINEAR_TC : TTM_KID_NONE);
    if (g_policy == TTM_KERNEL_TC) return tc_kid;
    if (g_policy == TTM_KERNEL_SIMT) return simt_ok ? TTM_KID_LINEAR_SIMT : TTM_KID_NONE;
    return tc_kid != TTM_KID_NONE ? tc_kid : (simt_ok ? TTM_KID_LINEAR_SIMT : TTM_KID_NONE);
}

cudaError_t launch_linear(int kid, const ttm::LinearArgs& a, cudaStream_t s) {
    if (kid == TTM_KID_LINEAR_TC) return ttm::linear_tc_launch(a, s);
    if (kid == TTM_KID_LINEAR_SEQ) return ttm::linear_seq_launch(a, s);
    return ttm::linear_simt_launch(a, s);
}

// The tensor-core 2-layer kernel rounds its recurrent operands to bf16.  Over
// long sequences whose memory decays towards zero the relative error of the
// final state then grows with the number of chunks (4e-2 after 1024 chunks of
// 16), so the automatic choice stays on the fp32 CUDA-core kernel; the
// tensor-core kernel runs when the policy asks for it.
int select_mlp(const ttm::MlpArgs& a) {
    const bool tc_ok = ttm::mlp_tc_supported(a);
    const bool simt_ok = ttm::mlp_simt_supported(a);
    if (g_policy == TTM_KERNEL_TC) return tc_ok ? TTM_KID_MLP_TC : TTM_KID_NONE;
    return simt_ok ? TTM_KID_MLP_SIMT : TTM_KID_NONE;
}

// The gradient's checkpoint pass runs the forward scan the policy would pick
// for the same shape (the tensor-core scan when it applies).
int bwd_forward_tc(const ttm::BwdArgs& b) {
    ttm::LinearArgs f{};
    f.B = b.B; f.H = b.H; f.T = b.T; f.dk = b.dk; f.dv = b.dv; f.chunk = b.chunk;
    f.bf16 = b.bf16;
    return select_linear(f) == TTM_KID_LINEAR_TC ? 1 : 0;
}

int linear_common(int B, int H, int T, int dk, int dv, int chunk, int dtype, const void* q,
                  const void* k, const void* v, const float* eta, const float* theta,
                  const float* alpha, const float* W0, const float* S0, int shared, void* z,
                  float* W_out, float* S_out, void* workspace, size_t workspace_bytes,
                  void* stream, int gates_per_chunk = 0) {
    if (B < 1 || H < 1 || T < 0 || chunk < 1) return TTM_ERR_INVALID_ARG;
    if (dtype != TTM_F32 && dtype != TTM_BF16) return TTM_ERR_INVALID_ARG;
    if (!dims_ok(dk, dtype) || !dims_ok(dv, dtype)) return TTM_ERR_INVALID_ARG;
    if ((long long)B * H > (1LL << 31) - 1 || (long long)dv > 65535LL * 16)
        return TTM_ERR_UNSUPPORTED;
    if (!W0 || !W_out) return TTM_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !theta || !z)) return TTM_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, eta, theta, alpha, W0, S0, z, W_out, S_out, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return TTM_ERR_INVALID_ARG;

    const size_t es = dtype == TTM_BF16 ? 2 : 4;
    const size_t tok = (size_t)B * H * T;
    const size_t nb0 = shared ? 1 : (size_t)B;
    const size_t st = (size_t)H * dv * dk * sizeof(float);
    const Span sq{q, tok * dk * es}, sk{k, tok * dk * es}, sv{v, tok * dv * es};
    const size_t ngate = gates_per_chunk ? (size_t)B * H * ((T + chunk - 1) / chunk) : tok;
    const Span sg[] = {{eta, ngate * 4}, {theta, ngate * 4}, {alpha, ngate * 4}};
    const Span sW0{W0, nb0 * st}, sS0{S0, nb0 * st};
    const Span sz{z, tok * dv * es}, sW{W_out, (size_t)B * st}, sS{S_out, (size_t)B * st};
    const Span outs[] = {sz, sW, sS};
    for (const Span& o : outs) {
        if (bad_alias(o, sq, false) || bad_alias(o, sk, false) || bad_alias(o, sv, false))
            return TTM_ERR_INVALID_ARG;
        for (const Span& g : sg)
            if (bad_alias(o, g, false)) return TTM_ERR_INVALID_ARG;
    }
    // W_out may be W0 (S_out may be S0) in place when W0 is not shared.
    if (bad_alias(sW, sW0, !shared) || bad_alias(sW, sS0, false)) return TTM_ERR_INVALID_ARG;
    if (bad_alias(sS, sS0, !shared) || bad_alias(sS, sW0, false)) return TTM_ERR_INVALID_ARG;
    if (overlap(sz, sW) || overlap(sz, sS) || overlap(sW, sS)) return TTM_ERR_INVALID_ARG;
    if (bad_alias(sz, sW0, false) || bad_alias(sz, sS0, false)) return TTM_ERR_INVALID_ARG;
    const Span swk{workspace, workspace_bytes};
    {
        const Span all[] = {sq, sk, sv, sg[0], sg[1], sg[2], sW0, sS0, sz, sW, sS};
        for (const Span& x : all)
            if (overlap(swk, x)) return TTM_ERR_INVALID_ARG;
    }

    ttm::LinearArgs a{};
    a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.chunk = chunk;
    a.bf16 = dtype == TTM_BF16;
    a.q = q; a.k = k; a.v = v;
    a.eta = eta; a.theta = theta; a.alpha = alpha;
    a.W0 = W0; a.S0 = S0; a.shared = shared ? 1 : 0;
    a.z = z; a.W_out = W_out; a.S_out = S_out;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.gates_per_chunk = gates_per_chunk ? 1 : 0;

    const int kid = select_linear(a);
    if (kid == TTM_KID_NONE) return TTM_ERR_UNSUPPORTED;
    if (kid == TTM_KID_LINEAR_TC &&
        (!workspace || workspace_bytes < ttm::linear_tc_workspace_bytes(a)))
        return TTM_ERR_INVALID_ARG;

    if (injected_failure()) return TTM_ERR_CUDA;
    a.status = status_ptr();
    if (!a.status) return TTM_ERR_CUDA;
    a.wait_cycles = g_wait_cycles.load();
    if (kid == TTM_KID_LINEAR_TC || kid == TTM_KID_LINEAR_SEQ)
        a.debug_stall = g_stall_chunk.exchange(-1) + 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = launch_linear(kid, a, s);
    if (e != cudaSuccess) return TTM_ERR_CUDA;
    t_last_kernel = kid;
    // the tensor-core path enqueues the coefficient pre-pass and the scan
    __atomic_add_fetch(&g_launches, kid == TTM_KID_LINEAR_TC ? 2ULL : 1ULL, __ATOMIC_RELAXED);
    return TTM_OK;
}

// Decode step of the linear / Titans (mode 0) or DGD (mode 1) memory.
int step_common(int mode, int B, int H, int n, int dk, int dv, int chunk, int pos, int dtype,
                const void* q, const void* k, const void* v, const float* eta,
                const float* theta, const float* alpha, float* W, float* S, float* Wc, void* z,
                void* stream) {
    if (B < 1 || H < 1 || n < 1 || chunk < 1 || pos < 0 || pos >= chunk) return TTM_ERR_INVALID_ARG;
    if (dtype != TTM_F32 && dtype != TTM_BF16) return TTM_ERR_INVALID_ARG;
    if (!dims_ok(dk, dtype) || !dims_ok(dv, dtype)) return TTM_ERR_INVALID_ARG;
    if (!q || !k || !v || !theta || !W || !Wc || !z) return TTM_ERR_INVALID_ARG;
    if (mode == 1 && !alpha) return TTM_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, eta, theta, alpha, W, S, Wc, z};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return TTM_ERR_INVALID_ARG;
    const size_t es = dtype == TTM_BF16 ? 2 : 4;
    const size_t tok = (size_t)B * H * n;
    const size_t st = (size_t)B * H * dv * dk * sizeof(float);
    const Span ins[] = {{q, tok * dk * es}, {k, tok * dk * es}, {v, tok * dv * es},
                        {eta, tok * 4}, {theta, tok * 4}, {alpha, tok * 4}};
    const Span outs[] = {{W, st}, {S, st}, {Wc, st}, {z, tok * dv * es}};
    for (int o = 0; o < 4; ++o) {
        for (const Span& i : ins)
            if (overlap(outs[o], i)) return TTM_ERR_INVALID_ARG;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlap(outs[o], outs[o2])) return TTM_ERR_INVALID_ARG;
    }
    ttm::StepArgs a{};
    a.B = B; a.H = H; a.n = n; a.dk = dk; a.dv = dv; a.chunk = chunk; a.pos = pos;
    a.bf16 = dtype == TTM_BF16;
    a.q = q; a.k = k; a.v = v;
    a.eta = eta; a.theta = theta; a.alpha = alpha;
    a.W = W; a.S = S; a.Wc = Wc; a.z = z;
    a.mode = mode;
    if (!ttm::linear_step_supported(a)) return TTM_ERR_UNSUPPORTED;
    if (ttm::linear_step_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TTM_ERR_CUDA;
    __atomic_add_fetch(&g_launches, 1ULL, __ATOMIC_RELAXED);
    return TTM_OK;
}

// Workspace of the LMM layer (bytes, each piece 256-byte aligned): projection
// output, q / k / v, gates, z, o, the scan's own workspace and cuBLAS scratch.
struct LmmLayout {
    size_t proj, qkv, gates, z, o, scan, blas, total, scan_bytes;
};

constexpr size_t kBlasScratch = 32u << 20;

LmmLayout lmm_layout(const ttm::LmmArgs& a, const ttm::LinearArgs& scan) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t BT = (size_t)a.B * a.T, D = (size_t)a.H * a.d, P = 4 * D + 3 * a.H;
    const size_t tok = (size_t)a.B * a.H * a.T;
    LmmLayout L;
    L.proj = 0;
    L.qkv = L.proj + up(BT * P * 2);
    L.gates = L.qkv + up(3 * tok * a.d * 2);
    L.z = L.gates + up(3 * tok * 4);
    L.o = L.z + up(tok * a.d * 2);
    L.scan = L.o + up(BT * D * 2);
    L.scan_bytes = select_linear(scan) == TTM_KID_LINEAR_TC ? ttm::linear_tc_workspace_bytes(scan) : 0;
    L.blas = L.scan + up(L.scan_bytes);
    L.total = L.blas + kBlasScratch;
    return L;
}

ttm::LinearArgs lmm_scan_args(const ttm::LmmArgs& a) {
    ttm::LinearArgs s{};
    s.B = a.B; s.H = a.H; s.T = a.T; s.dk = a.d; s.dv = a.d; s.chunk = a.chunk;
    s.bf16 = 1;
    s.shared = a.w0_shared;
    return s;
}

}  // namespace

extern "C" {

int ttm_linear_fwd(int B, int H, int T, int dk, int dv, int chunk, int dtype, const void* q,
                   const void* k, const void* v, const float* eta, const float* theta,
                   const float* alpha, const float* W0, int w0_shared_over_batch, void* z,
                   float* W_out, void* workspace, size_t workspace_bytes, void* stream) {
    if (eta || alpha) return TTM_ERR_INVALID_ARG;
    return linear_common(B, H, T, dk, dv, chunk, dtype, q, k, v, nullptr, theta, nullptr, W0,
                         nullptr, w0_shared_over_batch, z, W_out, nullptr, workspace,
                         workspace_bytes, stream);
}

int ttm_titans_fwd(int B, int H, int T, int dk, int dv, int chunk, int dtype, const void* q,
                   const void* k, const void* v, const float* eta, const float* theta,
                   const float* alpha, const float* W0, const float* S0,
                   int w0_shared_over_batch, void* z, float* W_out, float* S_out,
                   void* workspace, size_t workspace_bytes, void* stream) {
    return linear_common(B, H, T, dk, dv, chunk, dtype, q, k, v, eta, theta, alpha, W0, S0,
                         w0_shared_over_batch, z, W_out, S_out, workspace, workspace_bytes,
                         stream);
}

int ttm_titans_fwd_chunk_gates(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                               const void* q, const void* k, const void* v, const float* eta,
                               const float* theta, const float* alpha, const float* W0,
                               const float* S0, int w0_shared_over_batch, void* z,
                               float* W_out, float* S_out, void* workspace,
                               size_t workspace_bytes, void* stream) {
    return linear_common(B, H, T, dk, dv, chunk, dtype, q, k, v, eta, theta, alpha, W0, S0,
                         w0_shared_over_batch, z, W_out, S_out, workspace, workspace_bytes,
                         stream, 1);
}

size_t ttm_linear_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype) {
    if (B < 1 || H < 1 || T < 0 || chunk < 1 || (dtype != TTM_F32 && dtype != TTM_BF16) ||
        !dims_ok(dk, dtype) || !dims_ok(dv, dtype))
        return 0;
    ttm::LinearArgs a{};
    a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.chunk = chunk;
    a.bf16 = dtype == TTM_BF16;
    return select_linear(a) == TTM_KID_LINEAR_TC ? ttm::linear_tc_workspace_bytes(a) : 0;
}

int ttm_mlp_fwd(int B, int H, int T, int d, int hidden, int chunk, int dtype, const void* q,
                const void* k, const void* v, const float* eta, const float* theta,
                const float* alpha, const float* W1_0, const float* W2_0, const float* S1_0,
                const float* S2_0, int w0_shared_over_batch, void* z, float* W1_out,
                float* W2_out, float* S1_out, float* S2_out, void* stream) {
    if (B < 1 || H < 1 || T < 0 || chunk < 1) return TTM_ERR_INVALID_ARG;
    if (dtype != TTM_F32 && dtype != TTM_BF16) return TTM_ERR_INVALID_ARG;
    if (d < 1 || hidden < 1 || d % 8 || hidden % 8) return TTM_ERR_INVALID_ARG;
    if ((long long)B * H > (1LL << 31) - 1) return TTM_ERR_UNSUPPORTED;
    if (!W1_0 || !W2_0 || !W1_out || !W2_out) return TTM_ERR_INVALID_ARG;
    if ((S1_out == nullptr) != (S2_out == nullptr)) return TTM_ERR_INVALID_ARG;
    if (eta && !S1_out) return TTM_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !theta || !z)) return TTM_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, eta, theta, alpha, W1_0, W2_0, S1_0, S2_0,
                          z, W1_out, W2_out, S1_out, S2_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return TTM_ERR_INVALID_ARG;

    const size_t es = dtype == TTM_BF16 ? 2 : 4;
    const size_t tok = (size_t)B * H * T;
    const size_t nb0 = w0_shared_over_batch ? 1 : (size_t)B;
    const size_t st = (size_t)H * hidden * d * sizeof(float);
    const Span ins[] = {{q, tok * d * es}, {k, tok * d * es}, {v, tok * d * es},
                        {eta, tok * 4}, {theta, tok * 4}, {alpha, tok * 4}};
    const Span init[] = {{W1_0, nb0 * st}, {W2_0, nb0 * st}, {S1_0, nb0 * st}, {S2_0, nb0 * st}};
    const Span outs[] = {{W1_out, (size_t)B * st}, {W2_out, (size_t)B * st},
                         {S1_out, (size_t)B * st}, {S2_out, (size_t)B * st}};
    const Span sz{z, tok * d * es};
    for (const Span& i : ins) {
        if (overlap(sz, i)) return TTM_ERR_INVALID_ARG;
        for (const Span& o : outs)
            if (overlap(o, i)) return TTM_ERR_INVALID_ARG;
    }
    for (int o = 0; o < 4; ++o) {
        if (overlap(outs[o], sz)) return TTM_ERR_INVALID_ARG;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlap(outs[o], outs[o2])) return TTM_ERR_INVALID_ARG;
        for (int i = 0; i < 4; ++i)
            if (bad_alias(outs[o], init[i], i == o && !w0_shared_over_batch))
                return TTM_ERR_INVALID_ARG;
    }
    for (const Span& i : init)
        if (overlap(sz, i)) return TTM_ERR_INVALID_ARG;

    ttm::MlpArgs a{};
    a.B = B; a.H = H; a.T = T; a.d = d; a.hidden = hidden; a.chunk = chunk;
    a.bf16 = dtype == TTM_BF16;
    a.q = q; a.k = k; a.v = v;
    a.eta = eta; a.theta = theta; a.alpha = alpha;
    a.W1_0 = W1_0; a.W2_0 = W2_0; a.S1_0 = S1_0; a.S2_0 = S2_0;
    a.shared = w0_shared_over_batch ? 1 : 0;
    a.z = z; a.W1_out = W1_out; a.W2_out = W2_out; a.S1_out = S1_out; a.S2_out = S2_out;

    const int kid = select_mlp(a);
    if (kid == TTM_KID_NONE) return TTM_ERR_UNSUPPORTED;
    if (injected_failure()) return TTM_ERR_CUDA;
    a.status = status_ptr();
    if (!a.status) return TTM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        kid == TTM_KID_MLP_TC ? ttm::mlp_tc_launch(a, s) : ttm::mlp_simt_launch(a, s);
    if (e != cudaSuccess) return TTM_ERR_CUDA;
    t_last_kernel = kid;
    __atomic_add_fetch(&g_launches, 1ULL, __ATOMIC_RELAXED);
    return TTM_OK;
}

int ttm_titans_step(int B, int H, int n, int dk, int dv, int chunk, int pos, int dtype,
                    const void* q, const void* k, const void* v, const float* eta,
                    const float* theta, const float* alpha, float* W, float* S, float* Wc,
                    void* z, void* stream) {
    if (eta && !S) return TTM_ERR_INVALID_ARG;   // momentum needs its state
    return step_common(0, B, H, n, dk, dv, chunk, pos, dtype, q, k, v, eta, theta, alpha, W, S,
                       Wc, z, stream);
}

int ttm_linear_step(int B, int H, int n, int dk, int dv, int chunk, int pos, int dtype,
                    const void* q, const void* k, const void* v, const float* theta, float* W,
                    float* Wc, void* z, void* stream) {
    return ttm_titans_step(B, H, n, dk, dv, chunk, pos, dtype, q, k, v, nullptr, theta, nullptr,
                           W, nullptr, Wc, z, stream);
}

size_t ttm_titans_bwd_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype,
                                     int w0_shared_over_batch) {
    if (B < 1 || H < 1 || T < 0 || chunk < 1 || (dtype != TTM_F32 && dtype != TTM_BF16) ||
        !dims_ok(dk, dtype) || !dims_ok(dv, dtype))
        return 0;
    ttm::BwdArgs a{};
    a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.chunk = chunk;
    a.bf16 = dtype == TTM_BF16;
    a.shared = w0_shared_over_batch ? 1 : 0;
    a.fwd_tc = bwd_forward_tc(a);
    if (!ttm::linear_bwd_supported(a)) return 0;
    return ttm::linear_bwd_workspace_bytes(a);
}

int ttm_titans_bwd(int B, int H, int T, int dk, int dv, int chunk, int dtype, const void* q,
                   const void* k, const void* v, const float* eta, const float* theta,
                   const float* alpha, const float* W0, const float* S0,
                   int w0_shared_over_batch, const void* dz, const float* dW, const float* dS,
                   void* dq, void* dk_, void* dv_, float* deta, float* dtheta, float* dalpha,
                   float* dW0, float* dS0, void* workspace, size_t workspace_bytes,
                   void* stream) {
    if (B < 1 || H < 1 || T < 0 || chunk < 1) return TTM_ERR_INVALID_ARG;
    if (dtype != TTM_F32 && dtype != TTM_BF16) return TTM_ERR_INVALID_ARG;
    if (!dims_ok(dk, dtype) || !dims_ok(dv, dtype)) return TTM_ERR_INVALID_ARG;
    if (!W0 || !dW0) return TTM_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !theta || !dz || !dq || !dk_ || !dv_ || !dtheta))
        return TTM_ERR_INVALID_ARG;
    if ((deta && !eta) || (dalpha && !alpha)) return TTM_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, eta, theta, alpha, W0, S0, dz, dW, dS, dq, dk_, dv_,
                          deta, dtheta, dalpha, dW0, dS0, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return TTM_ERR_INVALID_ARG;
    const int shared = w0_shared_over_batch ? 1 : 0;
    ttm::BwdArgs a{};
    a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.chunk = chunk;
    a.bf16 = dtype == TTM_BF16;
    a.q = q; a.k = k; a.v = v; a.eta = eta; a.theta = theta; a.alpha = alpha;
    a.W0 = W0; a.S0 = S0; a.shared = shared;
    a.dz = dz; a.dW = dW; a.dS = dS;
    a.dq = dq; a.dk_ = dk_; a.dv_ = dv_;
    a.deta = deta; a.dtheta = dtheta; a.dalpha = dalpha; a.dW0 = dW0; a.dS0 = dS0;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.fwd_tc = bwd_forward_tc(a);
    if (!ttm::linear_bwd_supported(a)) return TTM_ERR_UNSUPPORTED;
    if ((long long)B * H > (1LL << 31) - 1 || (T + chunk - 1) / chunk > 65535)
        return TTM_ERR_UNSUPPORTED;

    const size_t es = dtype == TTM_BF16 ? 2 : 4;
    const size_t tok = (size_t)B * H * T;
    const size_t st = (size_t)H * dv * dk * sizeof(float);
    const size_t nb0 = shared ? 1 : (size_t)B;
    const Span ins[] = {{q, tok * dk * es}, {k, tok * dk * es}, {v, tok * dv * es},
                        {eta, tok * 4}, {theta, tok * 4}, {alpha, tok * 4},
                        {W0, nb0 * st}, {S0, nb0 * st}, {dz, tok * dv * es},
                        {dW, (size_t)B * st}, {dS, (size_t)B * st}};
    const Span outs[] = {{dq, tok * dk * es}, {dk_, tok * dk * es}, {dv_, tok * dv * es},
                         {deta, tok * 4}, {dtheta, tok * 4}, {dalpha, tok * 4},
                         {dW0, nb0 * st}, {dS0, nb0 * st}};
    const size_t need = ttm::linear_bwd_workspace_bytes(a);
    if (T > 0 && (!workspace || workspace_bytes < need)) return TTM_ERR_INVALID_ARG;
    const Span swk{workspace, T > 0 ? workspace_bytes : 0};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
        for (const Span& in : ins)
            if (overlap(outs[i], in)) return TTM_ERR_INVALID_ARG;
        for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
            if (overlap(outs[i], outs[j])) return TTM_ERR_INVALID_ARG;
        if (overlap(outs[i], swk)) return TTM_ERR_INVALID_ARG;
    }
    for (const Span& in : ins)
        if (overlap(in, swk)) return TTM_ERR_INVALID_ARG;

    a.status = status_ptr();
    if (!a.status) return TTM_ERR_CUDA;
    a.wait_cycles = g_wait_cycles.load();
    // the tensor-core passes read what the tensor-core scan leaves in the workspace
    a.local_tc = g_policy != TTM_KERNEL_SIMT && a.fwd_tc && ttm::bwd_local_tc_supported(a) ? 1 : 0;
    if (a.local_tc) a.debug_stall = g_stall_chunk.exchange(-1) + 1;   // the chain takes the hook
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    const cudaError_t e = ttm::linear_bwd_launch(a, s, &launches);
    if (e != cudaSuccess) return TTM_ERR_CUDA;
    __atomic_add_fetch(&g_launches, (unsigned long long)launches, __ATOMIC_RELAXED);
    t_last_kernel = a.local_tc ? TTM_KID_BWD_TC : TTM_KID_BWD_SIMT;
    return TTM_OK;
}

int ttm_linear_bwd(int B, int H, int T, int dk, int dv, int chunk, int dtype, const void* q,
                   const void* k, const void* v, const float* theta, const float* W0,
                   int w0_shared_over_batch, const void* dz, const float* dW, void* dq,
                   void* dk_, void* dv_, float* dtheta, float* dW0, void* workspace,
                   size_t workspace_bytes, void* stream) {
    return ttm_titans_bwd(B, H, T, dk, dv, chunk, dtype, q, k, v, nullptr, theta, nullptr, W0,
                          nullptr, w0_shared_over_batch, dz, dW, nullptr, dq, dk_, dv_, nullptr,
                          dtheta, nullptr, dW0, nullptr, workspace, workspace_bytes, stream);
}

namespace {

ttm::DgdArgs dgd_args(int B, int H, int T, int dk, int dv, int chunk, int dtype) {
    ttm::DgdArgs a{};
    a.B = B; a.H = H; a.T = T; a.dk = dk; a.dv = dv; a.chunk = chunk;
    a.bf16 = dtype == TTM_BF16;
    return a;
}

// The chunk form on the tensor cores where it applies, else the fp32 token
// loop of the decode kernel (which takes every shape up to dk = 512).
int select_dgd(const ttm::DgdArgs& a) {
    ttm::StepArgs s{};
    s.B = a.B; s.H = a.H; s.n = a.T; s.dk = a.dk; s.dv = a.dv; s.chunk = a.chunk;
    s.bf16 = a.bf16; s.mode = 1;
    const bool tc_ok = ttm::dgd_tc_supported(a);
    const bool simt_ok = ttm::linear_step_supported(s);
    if (g_policy == TTM_KERNEL_TC) return tc_ok ? TTM_KID_DGD_TC : TTM_KID_NONE;
    if (g_policy == TTM_KERNEL_SIMT) return simt_ok ? TTM_KID_DGD_STEP : TTM_KID_NONE;
    return tc_ok ? TTM_KID_DGD_TC : (simt_ok ? TTM_KID_DGD_STEP : TTM_KID_NONE);
}

}  // namespace

size_t ttm_dgd_workspace_size(int B, int H, int T, int dk, int dv, int chunk, int dtype) {
    if (B < 1 || H < 1 || T < 1 || chunk < 1) return 0;
    if (dtype != TTM_F32 && dtype != TTM_BF16) return 0;
    if (!dims_ok(dk, dtype) || !dims_ok(dv, dtype)) return 0;
    const ttm::DgdArgs a = dgd_args(B, H, T, dk, dv, chunk, dtype);
    return select_dgd(a) == TTM_KID_DGD_TC ? ttm::dgd_tc_workspace_bytes(a) : 0;
}

int ttm_dgd_fwd(int B, int H, int T, int dk, int dv, int chunk, int dtype, const void* q,
                const void* k, const void* v, const float* eta, const float* alpha,
                const float* W0, int w0_shared_over_batch, void* z, float* W_out,
                void* workspace, size_t workspace_bytes, void* stream) {
    if (B < 1 || H < 1 || T < 0 || chunk < 1) return TTM_ERR_INVALID_ARG;
    if (dtype != TTM_F32 && dtype != TTM_BF16) return TTM_ERR_INVALID_ARG;
    if (!dims_ok(dk, dtype) || !dims_ok(dv, dtype)) return TTM_ERR_INVALID_ARG;
    if (!W0 || !W_out) return TTM_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !eta || !alpha || !z)) return TTM_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, eta, alpha, W0, z, W_out, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return TTM_ERR_INVALID_ARG;
    const int shared = w0_shared_over_batch ? 1 : 0;
    const size_t es = dtype == TTM_BF16 ? 2 : 4;
    const size_t tok = (size_t)B * H * T;
    const size_t st = (size_t)H * dv * dk * sizeof(float);
    const Span ins[] = {{q, tok * dk * es}, {k, tok * dk * es}, {v, tok * dv * es},
                        {eta, tok * 4}, {alpha, tok * 4}};
    const Span sW0{W0, (shared ? 1 : (size_t)B) * st};
    const Span sz{z, tok * dv * es}, sW{W_out, (size_t)B * st};
    for (const Span& i : ins)
        if (overlap(sz, i) || overlap(sW, i)) return TTM_ERR_INVALID_ARG;
    if (overlap(sz, sW) || overlap(sz, sW0)) return TTM_ERR_INVALID_ARG;
    if (bad_alias(sW, sW0, !shared)) return TTM_ERR_INVALID_ARG;   // in place when not shared
    const Span swk{workspace, workspace_bytes};
    for (const Span& i : ins)
        if (overlap(swk, i)) return TTM_ERR_INVALID_ARG;
    if (overlap(swk, sz) || overlap(swk, sW) || overlap(swk, sW0)) return TTM_ERR_INVALID_ARG;
    ttm::DgdArgs g = dgd_args(B, H, T, dk, dv, chunk, dtype);
    const int kid = select_dgd(g);
    if (kid == TTM_KID_NONE) return TTM_ERR_UNSUPPORTED;
    if (kid == TTM_KID_DGD_TC) {
        if (!workspace || workspace_bytes < ttm::dgd_tc_workspace_bytes(g)) return TTM_ERR_INVALID_ARG;
        int* status = status_ptr();
        if (!status) return TTM_ERR_CUDA;
        g.q = q; g.k = k; g.v = v; g.eta = eta; g.alpha = alpha;
        g.W0 = W0; g.shared = shared; g.z = z; g.W_out = W_out;
        g.workspace = workspace; g.workspace_bytes = workspace_bytes;
        g.status = status; g.wait_cycles = g_wait_cycles.load();
        if (injected_failure()) return TTM_ERR_CUDA;
        if (ttm::dgd_tc_launch(g, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return TTM_ERR_CUDA;
        __atomic_add_fetch(&g_launches, 2ULL, __ATOMIC_RELAXED);
        t_last_kernel = kid;
        return TTM_OK;
    }
    ttm::StepArgs a{};
    a.B = B; a.H = H; a.n = T; a.dk = dk; a.dv = dv; a.chunk = chunk; a.pos = 0;
    a.bf16 = dtype == TTM_BF16;
    a.q = q; a.k = k; a.v = v;
    a.theta = eta; a.alpha = alpha;
    a.W = W_out; a.z = z;
    a.mode = 1;
    a.W_in = W0; a.w_shared = shared;
    if (!ttm::linear_step_supported(a)) return TTM_ERR_UNSUPPORTED;
    if (injected_failure()) return TTM_ERR_CUDA;
    if (ttm::linear_step_launch(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TTM_ERR_CUDA;
    __atomic_add_fetch(&g_launches, 1ULL, __ATOMIC_RELAXED);
    t_last_kernel = kid;
    return TTM_OK;
}

int ttm_dgd_step(int B, int H, int n, int dk, int dv, int chunk, int pos, int dtype,
                 const void* q, const void* k, const void* v, const float* eta,
                 const float* alpha, float* W, float* Wc, void* z, void* stream) {
    return step_common(1, B, H, n, dk, dv, chunk, pos, dtype, q, k, v, nullptr, eta, alpha, W,
                       nullptr, Wc, z, stream);
}

size_t ttm_lmm_layer_workspace_size(int B, int T, int H, int d, int chunk, int w0_shared) {
    if (B < 1 || T < 1 || H < 1 || chunk < 1) return 0;
    ttm::LmmArgs a{};
    a.B = B; a.T = T; a.H = H; a.d = d; a.chunk = chunk; a.conv_k = 1;
    a.w0_shared = w0_shared ? 1 : 0;
    if (!ttm::lmm_supported(a)) return 0;
    return lmm_layout(a, lmm_scan_args(a)).total;
}

int ttm_lmm_layer_fwd(int B, int T, int H, int d, int chunk, int conv_k, const void* x,
                      const void* W_in, const float* conv_w, const float* rms_w,
                      const void* W_o, float theta_scale, const float* W0,
                      int w0_shared_over_batch, void* y, float* W_out, float* S_out,
                      void* workspace, size_t workspace_bytes, void* stream) {
    if (B < 1 || T < 1 || H < 1 || chunk < 1) return TTM_ERR_INVALID_ARG;
    if (!x || !W_in || !conv_w || !rms_w || !W_o || !W0 || !y || !W_out || !workspace)
        return TTM_ERR_INVALID_ARG;
    const void* ptrs[] = {x, W_in, conv_w, rms_w, W_o, W0, y, W_out, S_out, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return TTM_ERR_INVALID_ARG;
    ttm::LmmArgs a{};
    a.B = B; a.T = T; a.H = H; a.d = d; a.chunk = chunk; a.conv_k = conv_k;
    a.x = x; a.W_in = W_in; a.conv_w = conv_w; a.rms_w = rms_w; a.W_o = W_o;
    a.theta_scale = theta_scale; a.W0 = W0; a.w0_shared = w0_shared_over_batch ? 1 : 0;
    if (!ttm::lmm_supported(a) || (long long)B * T > (1LL << 31) - 1) return TTM_ERR_UNSUPPORTED;
    ttm::LinearArgs sc = lmm_scan_args(a);
    if (select_linear(sc) == TTM_KID_NONE) return TTM_ERR_UNSUPPORTED;
    const LmmLayout L = lmm_layout(a, sc);
    if (workspace_bytes < L.total) return TTM_ERR_INVALID_ARG;
    const size_t BT = (size_t)B * T, D = (size_t)H * d, P = 4 * D + 3 * H;
    const size_t st = (size_t)H * d * d * 4;
    const Span ins[] = {{x, BT * D * 2}, {W_in, D * P * 2}, {conv_w, 3 * D * conv_k * 4},
                        {rms_w, (size_t)d * 4}, {W_o, D * D * 2},
                        {W0, (a.w0_shared ? 1 : (size_t)B) * st}};
    const Span outs[] = {{y, BT * D * 2}, {W_out, (size_t)B * st}, {S_out, (size_t)B * st},
                         {workspace, workspace_bytes}};
    for (int o = 0; o < 4; ++o) {
        for (const Span& i : ins)
            if (overlap(outs[o], i)) return TTM_ERR_INVALID_ARG;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlap(outs[o], outs[o2])) return TTM_ERR_INVALID_ARG;
    }
    int* status = status_ptr();
    if (!status) return TTM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* proj = ws + L.proj;
    uint8_t* qkv = ws + L.qkv;
    float* gates = reinterpret_cast<float*>(ws + L.gates);
    void* z = ws + L.z;
    void* o = ws + L.o;
    const size_t tok = (size_t)B * H * T;
    // p = x W_in
    if (!ttm::gemm_bf16(x, W_in, proj, (int)BT, (int)P, (int)D, 0.f, ws + L.blas, kBlasScratch, s))
        return TTM_ERR_CUDA;
    if (ttm::lmm_prep_launch(a, proj, qkv, gates, s) != cudaSuccess) return TTM_ERR_CUDA;
    // the memory scan over the prepared q, k, v and gates
    sc.q = qkv; sc.k = qkv + tok * d * 2; sc.v = qkv + 2 * tok * d * 2;
    sc.theta = gates; sc.eta = gates + tok; sc.alpha = gates + 2 * tok;
    sc.W0 = W0; sc.z = z; sc.W_out = W_out; sc.S_out = S_out;
    sc.workspace = L.scan_bytes ? ws + L.scan : nullptr;
    sc.workspace_bytes = L.scan_bytes;
    sc.status = status;
    const int kid = select_linear(sc);
    const cudaError_t e = launch_linear(kid, sc, s);
    if (e != cudaSuccess) return TTM_ERR_CUDA;
    if (ttm::lmm_post_launch(a, proj, z, o, s) != cudaSuccess) return TTM_ERR_CUDA;
    // y = x + o W_o
    if (cudaMemcpyAsync(y, x, BT * D * 2, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return TTM_ERR_CUDA;
    if (!ttm::gemm_bf16(o, W_o, y, (int)BT, (int)D, (int)D, 1.f, ws + L.blas, kBlasScratch, s))
        return TTM_ERR_CUDA;
    t_last_kernel = kid;
    __atomic_add_fetch(&g_launches, kid == TTM_KID_LINEAR_TC ? 4ULL : 3ULL, __ATOMIC_RELAXED);
    return TTM_OK;
}

int ttm_mlp_gelu(const float* x, float* y, float* dy, int n, void* stream) {
    if (n < 0 || (n > 0 && (!x || !y))) return TTM_ERR_INVALID_ARG;
    if (overlap({y, (size_t)n * 4}, {x, (size_t)n * 4}) && y != x) return TTM_ERR_INVALID_ARG;
    if (dy && (overlap({dy, (size_t)n * 4}, {x, (size_t)n * 4}) ||
               overlap({dy, (size_t)n * 4}, {y, (size_t)n * 4})))
        return TTM_ERR_INVALID_ARG;
    const cudaError_t e = ttm::mlp_gelu_launch(x, y, dy, n, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TTM_OK : TTM_ERR_CUDA;
}

const char* ttm_status_str(int status) {
    switch (status) {
        case TTM_OK: return "ok";
        case TTM_ERR_INVALID_ARG: return "invalid argument";
        case TTM_ERR_UNSUPPORTED: return "shape or dtype not supported by the selected kernels";
        case TTM_ERR_CUDA: return "CUDA error";
        case TTM_ERR_TIMEOUT: return "a device-side wait timed out";
        default: return "unknown status";
    }
}

int ttm_set_kernel_policy(int policy) {
    if (policy != TTM_KERNEL_AUTO && policy != TTM_KERNEL_SIMT && policy != TTM_KERNEL_TC)
        return -1;
    const int old = g_policy;
    g_policy = policy;
    return old;
}

int ttm_last_kernel(void) { return t_last_kernel; }

unsigned long long ttm_launch_count(void) { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

int ttm_debug_set(int option, long long value) {
    switch (option) {
        case TTM_DBG_WAIT_CYCLES:
            if (value < 0) return TTM_ERR_INVALID_ARG;
            g_wait_cycles = value;
            return TTM_OK;
        case TTM_DBG_STALL_CHUNK:
            if (value < -1 || value > (1LL << 30)) return TTM_ERR_INVALID_ARG;
            g_stall_chunk = (int)value;
            return TTM_OK;
        case TTM_DBG_FAIL_CALLS:
            if (value < 0 || value > (1LL << 30)) return TTM_ERR_INVALID_ARG;
            g_fail_calls = (int)value;
            return TTM_OK;
        default: return TTM_ERR_INVALID_ARG;
    }
}

int ttm_cuda_device_count(void) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess) return 0;
    return n;
}

int ttm_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return TTM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return TTM_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return TTM_ERR_CUDA;
    return v == 0 ? TTM_OK : v;
}

}  // extern "C"
