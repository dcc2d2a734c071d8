// Host-buffer entry point of the Titans / linear scan: inputs and outputs in
// host memory, the sequence streamed through the device in segments of whole
// chunks.  Three streams overlap the work of consecutive segments:
//   copy-in  (internal): q, k, v and gates of segment i + 1, host -> device
//   compute  (caller's): the scan of segment i, its state carried in fp32 from
//                        segment i - 1 (the chunk form restarts exactly at a
//                        chunk boundary: "TTT layers 与 fast weights" eq (6) takes
//                        each chunk's gradients at the state the previous chunk
//                        left, whatever produced it)
//   copy-out (internal): z of segment i - 1, device -> host
// Every segment's buffers are double-buffered in the caller's device workspace.
// The caller's stream waits for every copy before the call's last operation,
// so synchronising that stream is enough to read the outputs.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/ttm.h"

namespace {

constexpr int kMaxDev = 64;

struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_ready[2] = {}, comp_done[2] = {}, out_done[2] = {};
    bool ready = false;
};
HostPipe g_pipe[kMaxDev];
std::mutex g_pipe_mutex;

// Streams and events of this device, created once and reused by every call.
HostPipe* pipe_for_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    HostPipe& p = g_pipe[dev];
    if (p.ready) return &p;
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess)
        return nullptr;
    for (int b = 0; b < 2; ++b)
        if (cudaEventCreateWithFlags(&p.in_ready[b], ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.comp_done[b], ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.out_done[b], ef) != cudaSuccess)
            return nullptr;
    p.ready = true;
    return &p;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Byte layout of the workspace for segments of `seg` tokens.
struct HostLayout {
    size_t q, k, v, g, z, slot;   // sizes of one slot's buffers; slot = their sum
    size_t state;                 // one W (or S) buffer, B x H x dv x dk floats
    size_t scan;                  // scan workspace for one segment
    size_t total;
};

HostLayout host_layout(int B, int H, int seg, int dk, int dv, int chunk, int dtype) {
    HostLayout L{};
    const size_t es = dtype == TTM_BF16 ? 2 : 4, bh = (size_t)B * H;
    L.q = up256(bh * seg * dk * es);
    L.k = L.q;
    L.v = up256(bh * seg * dv * es);
    L.g = up256(bh * seg * sizeof(float));
    L.z = L.v;
    L.slot = L.q + L.k + L.v + 3 * L.g + L.z;
    L.state = up256(bh * dv * dk * sizeof(float));
    L.scan = up256(ttm_linear_workspace_size(B, H, seg, dk, dv, chunk, dtype));
    L.total = 2 * L.slot + 4 * L.state + L.scan;
    return L;
}

int segment_tokens(int T, int chunk, int seg_tokens) {
    const int whole = (T + chunk - 1) / chunk * chunk;
    return whole < seg_tokens ? (whole > 0 ? whole : chunk) : seg_tokens;
}

// H2D / D2H copy of a [rows][len] block out of [rows][ld] (element bytes es).
cudaError_t copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                      size_t rows, cudaMemcpyKind kind, cudaStream_t s) {
    if (width == 0 || rows == 0) return cudaSuccess;
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
}

}  // namespace

extern "C" {

size_t ttm_titans_fwd_host_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                          int dtype, int seg_tokens) {
    if (B < 1 || H < 1 || T < 0 || chunk < 1 || seg_tokens < chunk || seg_tokens % chunk)
        return 0;
    if (dtype != TTM_F32 && dtype != TTM_BF16) return 0;
    return host_layout(B, H, segment_tokens(T, chunk, seg_tokens), dk, dv, chunk, dtype).total;
}

int ttm_titans_fwd_host(int B, int H, int T, int dk, int dv, int chunk, int dtype, const void* q,
                        const void* k, const void* v, const float* eta, const float* theta,
                        const float* alpha, const float* W0, const float* S0,
                        int w0_shared_over_batch, void* z, float* W_out, float* S_out,
                        int seg_tokens, void* workspace, size_t workspace_bytes, void* stream) {
    if (B < 1 || H < 1 || T < 0 || chunk < 1 || seg_tokens < chunk || seg_tokens % chunk)
        return TTM_ERR_INVALID_ARG;
    if (dtype != TTM_F32 && dtype != TTM_BF16) return TTM_ERR_INVALID_ARG;
    if (dk < 1 || dv < 1 || !W0 || !W_out || !workspace) return TTM_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !theta || !z)) return TTM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return TTM_ERR_INVALID_ARG;
    const int seg = segment_tokens(T, chunk, seg_tokens);
    const HostLayout L = host_layout(B, H, seg, dk, dv, chunk, dtype);
    if (workspace_bytes < L.total) return TTM_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe* P = pipe_for_device();
    if (!P) return TTM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t es = dtype == TTM_BF16 ? 2 : 4, bh = (size_t)B * H;
    const size_t nb0 = w0_shared_over_batch ? 1 : (size_t)B;
    const size_t st = (size_t)H * dv * dk * sizeof(float);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto slot = [&](int b) { return ws + (size_t)b * L.slot; };
    float* Wb[2] = {reinterpret_cast<float*>(ws + 2 * L.slot),
                    reinterpret_cast<float*>(ws + 2 * L.slot + L.state)};
    float* Sb[2] = {reinterpret_cast<float*>(ws + 2 * L.slot + 2 * L.state),
                    reinterpret_cast<float*>(ws + 2 * L.slot + 3 * L.state)};
    void* scan_ws = ws + 2 * L.slot + 4 * L.state;
    const float* gates[3] = {eta, theta, alpha};

#define TTM_CK(x) do { if ((x) != cudaSuccess) return TTM_ERR_CUDA; } while (0)
    // the previous call on this stream may still use the workspace
    TTM_CK(cudaEventRecord(P->start, s));
    TTM_CK(cudaStreamWaitEvent(P->in, P->start, 0));
    TTM_CK(cudaStreamWaitEvent(P->out, P->start, 0));
    // initial state into the buffers the first segment reads
    TTM_CK(cudaMemcpyAsync(Wb[1], W0, nb0 * st, cudaMemcpyHostToDevice, s));
    if (S0) TTM_CK(cudaMemcpyAsync(Sb[1], S0, nb0 * st, cudaMemcpyHostToDevice, s));

    const int nseg = T > 0 ? (T + seg - 1) / seg : 1;
    for (int i = 0; i < nseg; ++i) {
        const int b = i & 1;
        const int t0 = i * seg, n = T > 0 ? (T - t0 < seg ? T - t0 : seg) : 0;
        uint8_t* sq = slot(b);
        uint8_t* sk = sq + L.q;
        uint8_t* sv = sk + L.k;
        uint8_t* sg = sv + L.v;
        uint8_t* sz = sg + 3 * L.g;
        const float* dg[3] = {nullptr, nullptr, nullptr};
        // copy-in: after the scan of segment i - 2 has read this slot
        if (i >= 2) TTM_CK(cudaStreamWaitEvent(P->in, P->comp_done[b], 0));
        if (n > 0) {
            const size_t rk = (size_t)n * dk * es, rv = (size_t)n * dv * es;
            TTM_CK(copy_rows(sq, rk, static_cast<const uint8_t*>(q) + (size_t)t0 * dk * es,
                             (size_t)T * dk * es, rk, bh, cudaMemcpyHostToDevice, P->in));
            TTM_CK(copy_rows(sk, rk, static_cast<const uint8_t*>(k) + (size_t)t0 * dk * es,
                             (size_t)T * dk * es, rk, bh, cudaMemcpyHostToDevice, P->in));
            TTM_CK(copy_rows(sv, rv, static_cast<const uint8_t*>(v) + (size_t)t0 * dv * es,
                             (size_t)T * dv * es, rv, bh, cudaMemcpyHostToDevice, P->in));
            for (int g = 0; g < 3; ++g) {
                if (!gates[g]) continue;
                dg[g] = reinterpret_cast<const float*>(sg + g * L.g);
                TTM_CK(copy_rows(sg + g * L.g, (size_t)n * 4, gates[g] + t0, (size_t)T * 4,
                                 (size_t)n * 4, bh, cudaMemcpyHostToDevice, P->in));
            }
        }
        TTM_CK(cudaEventRecord(P->in_ready[b], P->in));
        // scan of segment i on the caller's stream, after its inputs landed
        // and after z of segment i - 2 left this slot
        TTM_CK(cudaStreamWaitEvent(s, P->in_ready[b], 0));
        if (i >= 2) TTM_CK(cudaStreamWaitEvent(s, P->out_done[b], 0));
        const int first = i == 0;
        const int r = ttm_titans_fwd(
            B, H, n, dk, dv, chunk, dtype, sq, sk, sv, dg[0], dg[1], dg[2], Wb[(i + 1) & 1],
            (first && !S0) ? nullptr : Sb[(i + 1) & 1], first ? w0_shared_over_batch : 0, sz,
            Wb[b], Sb[b], scan_ws, L.scan, s);
        if (r != TTM_OK) return r;
        TTM_CK(cudaEventRecord(P->comp_done[b], s));
        // copy-out of z
        TTM_CK(cudaStreamWaitEvent(P->out, P->comp_done[b], 0));
        if (n > 0) {
            const size_t rv = (size_t)n * dv * es;
            TTM_CK(copy_rows(static_cast<uint8_t*>(z) + (size_t)t0 * dv * es, (size_t)T * dv * es,
                             sz, rv, rv, bh, cudaMemcpyDeviceToHost, P->out));
        }
        TTM_CK(cudaEventRecord(P->out_done[b], P->out));
    }
    // final state, then the caller's stream waits for the outstanding copies
    const int last = (nseg - 1) & 1;
    TTM_CK(cudaMemcpyAsync(W_out, Wb[last], (size_t)B * st, cudaMemcpyDeviceToHost, s));
    if (S_out) TTM_CK(cudaMemcpyAsync(S_out, Sb[last], (size_t)B * st, cudaMemcpyDeviceToHost, s));
    TTM_CK(cudaStreamWaitEvent(s, P->out_done[last], 0));
    if (nseg > 1) TTM_CK(cudaStreamWaitEvent(s, P->out_done[last ^ 1], 0));
#undef TTM_CK
    return TTM_OK;
}

}  // extern "C"
