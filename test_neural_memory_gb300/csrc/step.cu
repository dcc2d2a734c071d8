// Streaming decode step of the linear / Titans memory: continues every
// sequence by n tokens in the primal, token-by-token form ("TTT layers 与 fast
// weights" §1.1: decoding runs the primal form after a chunked prefill; the
// gradient of every token of a chunk is taken at the chunk-start state, eq (6);
// momentum and forgetting as in "论文速览 | Titans" §3.4-§3.7).
//
// Per token t, with W_c the memory at the start of the current chunk:
//   e   = W_c k_t - v_t
//   S   = eta_t S - theta_t 2 e k_t^T
//   W   = (1 - alpha_t) W + S
//   z_t = W q_t
// and W_c is re-taken (W_c = W) whenever a token opens a chunk.
//
// The DGD memory ("Nested Learning" §8.1 eq (88) with the matrix memory and
// L2 objective of eq (93), chunk-wise per §8.2) uses the same row structure:
//   z_t = W q_t                       (read before the write, eq (86))
//   W = W (alpha_t I - eta_t k k^T) - eta_t (W_c k - v) k^T
// so row r takes W_r = alpha_t W_r - eta_t ((W_c + W)_r . k - v_r) k^T: one dot
// product per token and row, like the Titans step.  Run over a whole sequence
// from W0 (W_in) it is the DGD scan.
//
// Every row of W, S and W_c evolves on its own (row r only needs e_r), so one
// warp owns one row of one sequence for the whole call: lane l holds the
// columns l, l + 32, ... of the three rows in registers, the two dot products
// per token are warp reductions, and the state is read and written once per
// call whatever n is.  A one-token call is bound by HBM (it moves the state
// W, S, W_c once in each direction plus one token's q, k, v, z) and issues
// all its loads up front; a longer call is bound by the per-token chain and
// stages its tokens through shared memory in groups, one memory round trip
// per group instead of one per token.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace ttm {
namespace {

constexpr int kStepThreads = 256;   // 8 rows per block

template <typename TIn>
__device__ __forceinline__ float ld_in(const TIn* p);
template <>
__device__ __forceinline__ float ld_in<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename TIn>
__device__ __forceinline__ void st_out(TIn* p, float x);
template <>
__device__ __forceinline__ void st_out<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// One token per call (the streaming case): the call is bound by reading and
// writing the state, so every load is issued as early as possible and nothing
// is staged.  NJ = columns per lane (dk <= 32 NJ).
// Initial row of the state: W_in (a whole scan; possibly shared over the
// batch) or the caller's running state W.
__device__ __forceinline__ const float* initial_row(const StepArgs& a, long long seq, int r) {
    if (!a.W_in) return a.W + ((size_t)seq * a.dv + r) * a.dk;
    const long long src = a.w_shared ? seq % a.H : seq;
    return a.W_in + ((size_t)src * a.dv + r) * a.dk;
}

template <typename TIn, int NJ, int kMode>
__global__ void __launch_bounds__(kStepThreads) linear_step_direct(const StepArgs a) {
    const long long gw = ((long long)blockIdx.x * kStepThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long nrows = (long long)a.B * a.H * a.dv;
    if (gw >= nrows) return;
    const int r = (int)(gw % a.dv);
    const long long seq = gw / a.dv;
    const int dk = a.dk;
    const size_t row = ((size_t)seq * a.dv + r) * dk;
    const size_t tok = (size_t)seq;   // n == 1: token index = sequence index
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);

    const float* w0 = initial_row(a, seq, r);
    const bool opens = a.pos == 0;   // the token opens a chunk: its gradient point is now
    float w[NJ], s[NJ], wc[NJ], kv[NJ], qv[NJ];
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
        const int j = lane + 32 * i;
        const bool in = j < dk;
        w[i] = in ? w0[j] : 0.f;
        s[i] = (in && a.S) ? a.S[row + j] : 0.f;
        wc[i] = (in && !opens) ? a.Wc[row + j] : 0.f;
        kv[i] = in ? ld_in<TIn>(k + tok * dk + j) : 0.f;
        qv[i] = in ? ld_in<TIn>(q + tok * dk + j) : 0.f;
    }
    const float th = __ldg(a.theta + tok);
    const float et = a.eta ? __ldg(a.eta + tok) : 0.f;
    const float al = a.alpha ? __ldg(a.alpha + tok) : 0.f;
    const float vr = ld_in<TIn>(static_cast<const TIn*>(a.v) + tok * a.dv + r);
    if (opens) {
#pragma unroll
        for (int i = 0; i < NJ; ++i) wc[i] = w[i];
    }
    float acc = 0.f;
    float zq = 0.f;
    if constexpr (kMode == 0) {
#pragma unroll
        for (int i = 0; i < NJ; ++i) acc = fmaf(wc[i], kv[i], acc);
        const float ge = 2.f * th * (warp_sum(acc) - vr);   // theta times the gradient's row factor
        const float keep = 1.f - al;
#pragma unroll
        for (int i = 0; i < NJ; ++i) {
            s[i] = fmaf(et, s[i], -ge * kv[i]);
            w[i] = fmaf(keep, w[i], s[i]);
            zq = fmaf(w[i], qv[i], zq);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NJ; ++i) {
            acc = fmaf(wc[i] + w[i], kv[i], acc);
            zq = fmaf(w[i], qv[i], zq);              // the read sees the memory before the write
        }
        const float g = th * (warp_sum(acc) - vr);   // eta_t ((W_c + W) k - v)_r
#pragma unroll
        for (int i = 0; i < NJ; ++i) w[i] = fmaf(al, w[i], -g * kv[i]);
    }
    zq = warp_sum(zq);
    if (lane == 0) st_out<TIn>(static_cast<TIn*>(a.z) + tok * a.dv + r, zq);
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
        const int j = lane + 32 * i;
        if (j >= dk) continue;
        a.W[row + j] = w[i];
        if (a.S) a.S[row + j] = s[i];
        if (opens && a.Wc) a.Wc[row + j] = wc[i];
    }
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// Copies the keys and queries of tokens [t0, t0 + len) of one sequence into
// the warp's staging area (k rows then q rows, G rows each) as 16-byte pieces;
// rows are contiguous in memory and dk * sizeof(TIn) is a multiple of 16.
template <typename TIn>
__device__ __forceinline__ void stage_tokens(TIn* ks, int G, const TIn* k, const TIn* q,
                                             size_t first, int len, int dk, int lane) {
    const int nvec = (int)((size_t)len * dk * sizeof(TIn) / 16);
    const char* kg = reinterpret_cast<const char*>(k + first * dk);
    const char* qg = reinterpret_cast<const char*>(q + first * dk);
    char* kd = reinterpret_cast<char*>(ks);
    char* qd = kd + (size_t)G * dk * sizeof(TIn);
    for (int i = lane; i < nvec; i += 32) {
        cp_async16(kd + 16 * i, kg + 16 * i);
        cp_async16(qd + 16 * i, qg + 16 * i);
    }
}

template <typename TIn>
__device__ __forceinline__ float to_f(TIn x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// One token of one row (one row per warp, NJ columns per lane): the error at
// the chunk-start point, the row's update and the read of the updated row,
// summed over the warp.  ks / qs: the token's staged key and query; vr, th,
// et, keep: its value on this row and its gates (mode 0: theta, eta and
// 1 - alpha; mode 1: the DGD step eta and retention alpha).
template <typename TIn, int NJ, int kMode>
__device__ __forceinline__ float row_token(float (&w)[NJ], float (&s)[NJ], const float (&wc)[NJ],
                                           const TIn* ks, const TIn* qs, int dk, int lane,
                                           float vr, float th, float et, float keep) {
    float kv[NJ], qv[NJ];
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
        const int j = lane + 32 * i;
        kv[i] = j < dk ? to_f<TIn>(ks[j]) : 0.f;
        qv[i] = j < dk ? to_f<TIn>(qs[j]) : 0.f;
    }
    float acc = 0.f, zq = 0.f;
    if constexpr (kMode == 0) {
#pragma unroll
        for (int i = 0; i < NJ; ++i) acc = fmaf(wc[i], kv[i], acc);
        const float ge = 2.f * th * (warp_sum(acc) - vr);   // theta times the gradient's row factor
#pragma unroll
        for (int i = 0; i < NJ; ++i) {
            s[i] = fmaf(et, s[i], -ge * kv[i]);
            w[i] = fmaf(keep, w[i], s[i]);
            zq = fmaf(w[i], qv[i], zq);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NJ; ++i) {
            acc = fmaf(wc[i] + w[i], kv[i], acc);
            zq = fmaf(w[i], qv[i], zq);              // the read sees the memory before the write
        }
        // eta_t ((W_c + W) k - v)_r; the retention factor rides in `keep`
        const float g = th * (warp_sum(acc) - vr);
#pragma unroll
        for (int i = 0; i < NJ; ++i) w[i] = fmaf(keep, w[i], -g * kv[i]);
    }
    return warp_sum(zq);
}

// Several tokens per call.  NJ = columns per lane (dk <= 32 NJ).  Tokens are
// taken in groups of G: one
// round trip brings a group's keys and queries into the warp's shared-memory
// staging area (the first group's copy is issued before the state is read,
// so the two overlap) and lanes 0..G-1 fetch the group's per-token scalars,
// which are broadcast by shuffles as each token is processed.  Without the
// grouping every token would wait for its own loads, a full memory latency
// per token.
template <typename TIn, int NJ, int kMode>
__global__ void __launch_bounds__(kStepThreads, NJ <= 4 ? 5 : 1)
    linear_step_staged(const StepArgs a, int G) {
    extern __shared__ __align__(16) unsigned char step_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * (kStepThreads / 32) + warp;
    const long long nrows = (long long)a.B * a.H * a.dv;
    if (gw >= nrows) return;
    const int r = (int)(gw % a.dv);
    const long long seq = gw / a.dv;
    const int dk = a.dk, n = a.n;
    const size_t row = ((size_t)seq * a.dv + r) * dk;
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* v = static_cast<const TIn*>(a.v);
    TIn* z = static_cast<TIn*>(a.z);
    TIn* ks = reinterpret_cast<TIn*>(step_smem) + (size_t)warp * 2 * G * dk;
    const TIn* qs = ks + (size_t)G * dk;

    stage_tokens<TIn>(ks, G, k, q, (size_t)seq * n, min(G, n), dk, lane);
    const float* w0 = initial_row(a, seq, r);
    float w[NJ], s[NJ], wc[NJ];
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
        const int j = lane + 32 * i;
        const bool in = j < dk;
        w[i] = in ? w0[j] : 0.f;
        s[i] = (in && a.S) ? a.S[row + j] : 0.f;
        wc[i] = (in && a.pos != 0) ? a.Wc[row + j] : 0.f;
    }
    int p = a.pos;
    bool wc_changed = false;
    for (int t0 = 0; t0 < n; t0 += G) {
        const int len = min(G, n - t0);
        if (t0 > 0) {
            __syncwarp();   // every lane is done reading the previous group
            stage_tokens<TIn>(ks, G, k, q, (size_t)seq * n + t0, len, dk, lane);
        }
        float vr = 0.f, th = 0.f, et = 0.f, keep = 1.f;
        if (lane < len) {
            const size_t tok = (size_t)seq * n + t0 + lane;
            vr = ld_in<TIn>(v + tok * a.dv + r);
            th = __ldg(a.theta + tok);
            et = a.eta ? __ldg(a.eta + tok) : 0.f;
            const float al = a.alpha ? __ldg(a.alpha + tok) : 0.f;
            keep = kMode == 0 ? 1.f - al : al;
        }
        cp_async_wait_all();
        __syncwarp();
        for (int u = 0; u < len; ++u) {
            if (p == 0) {   // this token opens a chunk: its gradient point is now
#pragma unroll
                for (int i = 0; i < NJ; ++i) wc[i] = w[i];
                wc_changed = true;
            }
            const float zq = row_token<TIn, NJ, kMode>(w, s, wc, ks + u * dk, qs + u * dk, dk, lane,
                                                       __shfl_sync(0xffffffffu, vr, u),
                                                       __shfl_sync(0xffffffffu, th, u),
                                                       kMode == 0 ? __shfl_sync(0xffffffffu, et, u) : 0.f,
                                                       __shfl_sync(0xffffffffu, keep, u));
            if (lane == 0) st_out<TIn>(z + ((size_t)seq * n + t0 + u) * a.dv + r, zq);
            p = p + 1 == a.chunk ? 0 : p + 1;
        }
    }
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
        const int j = lane + 32 * i;
        if (j >= dk) continue;
        a.W[row + j] = w[i];
        if (a.S) a.S[row + j] = s[i];
        if (wc_changed && a.Wc) a.Wc[row + j] = wc[i];
    }
}

// Several tokens per call when the 8 warps of a block share one sequence
// (dv a multiple of 8): the block stages each group of G tokens' keys and
// queries once for all its rows, into one of two buffers, while it processes
// the previous group from the other; lanes 0..G-1 of every warp load the
// group's per-token scalars for that warp's row into registers one group
// ahead.  One block barrier per group both publishes the group's copies and
// frees the other buffer.
template <typename TIn>
__device__ __forceinline__ void stage_block(TIn* ks, int G, const TIn* k, const TIn* q,
                                            size_t first, int len, int dk) {
    const int nvec = (int)((size_t)len * dk * sizeof(TIn) / 16);
    const char* kg = reinterpret_cast<const char*>(k + first * dk);
    const char* qg = reinterpret_cast<const char*>(q + first * dk);
    char* kd = reinterpret_cast<char*>(ks);
    char* qd = kd + (size_t)G * dk * sizeof(TIn);
    for (int i = threadIdx.x; i < nvec; i += kStepThreads) {
        cp_async16(kd + 16 * i, kg + 16 * i);
        cp_async16(qd + 16 * i, qg + 16 * i);
    }
}

template <typename TIn, int NJ, int kMode>
__global__ void __launch_bounds__(kStepThreads, NJ <= 4 ? 5 : 1)
    linear_step_block(const StepArgs a, int G) {
    extern __shared__ __align__(16) unsigned char step_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * (kStepThreads / 32) + warp;
    const int r = (int)(gw % a.dv);         // every warp of the block is a row of `seq`
    const long long seq = gw / a.dv;
    const int dk = a.dk, n = a.n;
    const size_t row = ((size_t)seq * a.dv + r) * dk;
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* v = static_cast<const TIn*>(a.v);
    TIn* z = static_cast<TIn*>(a.z);
    TIn* const buf0 = reinterpret_cast<TIn*>(step_smem);
    TIn* const buf1 = buf0 + (size_t)2 * G * dk;

    stage_block<TIn>(buf0, G, k, q, (size_t)seq * n, min(G, n), dk);
    auto scalars = [&](int t0, int len, float& vr, float& th, float& et, float& keep) {
        vr = 0.f; th = 0.f; et = 0.f; keep = 1.f;
        if (lane < len) {
            const size_t tok = (size_t)seq * n + t0 + lane;
            vr = ld_in<TIn>(v + tok * a.dv + r);
            th = __ldg(a.theta + tok);
            et = a.eta ? __ldg(a.eta + tok) : 0.f;
            const float al = a.alpha ? __ldg(a.alpha + tok) : 0.f;
            keep = kMode == 0 ? 1.f - al : al;
        }
    };
    float vr, th, et, keep;
    scalars(0, min(G, n), vr, th, et, keep);
    const float* w0 = initial_row(a, seq, r);
    float w[NJ], s[NJ], wc[NJ];
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
        const int j = lane + 32 * i;
        const bool in = j < dk;
        w[i] = in ? w0[j] : 0.f;
        s[i] = (in && a.S) ? a.S[row + j] : 0.f;
        wc[i] = (in && a.pos != 0) ? a.Wc[row + j] : 0.f;
    }
    int p = a.pos;
    bool wc_changed = false;
    for (int t0 = 0; t0 < n; t0 += G) {
        const int len = min(G, n - t0);
        const bool odd = ((t0 / G) & 1) != 0;
        const TIn* ks = odd ? buf1 : buf0;
        const TIn* qs = ks + (size_t)G * dk;
        cp_async_wait_all();   // this thread's copies of the group
        __syncthreads();       // everyone's; and every warp is done with the other buffer
        float vn = 0.f, thn = 0.f, etn = 0.f, keepn = 1.f;
        if (t0 + G < n) {
            const int ln = min(G, n - t0 - G);
            stage_block<TIn>(odd ? buf0 : buf1, G, k, q, (size_t)seq * n + t0 + G, ln, dk);
            scalars(t0 + G, ln, vn, thn, etn, keepn);
        }
        for (int u = 0; u < len; ++u) {
            if (p == 0) {   // this token opens a chunk: its gradient point is now
#pragma unroll
                for (int i = 0; i < NJ; ++i) wc[i] = w[i];
                wc_changed = true;
            }
            const float zq = row_token<TIn, NJ, kMode>(w, s, wc, ks + u * dk, qs + u * dk, dk, lane,
                                                       __shfl_sync(0xffffffffu, vr, u),
                                                       __shfl_sync(0xffffffffu, th, u),
                                                       kMode == 0 ? __shfl_sync(0xffffffffu, et, u) : 0.f,
                                                       __shfl_sync(0xffffffffu, keep, u));
            if (lane == 0) st_out<TIn>(z + ((size_t)seq * n + t0 + u) * a.dv + r, zq);
            p = p + 1 == a.chunk ? 0 : p + 1;
        }
        vr = vn; th = thn; et = etn; keep = keepn;
    }
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
        const int j = lane + 32 * i;
        if (j >= dk) continue;
        a.W[row + j] = w[i];
        if (a.S) a.S[row + j] = s[i];
        if (wc_changed && a.Wc) a.Wc[row + j] = wc[i];
    }
}

// Several tokens per call, four rows per warp: lanes 8g ... 8g + 7 hold row
// 4 (warp) + g of the block's rows, lane 8g + c its DK/8 consecutive columns
// c DK/8 ..., so a row's two dot products per token reduce over 8 lanes (three
// shuffles each) and every staged key / query load feeds four rows.  The block
// stages each group of G tokens' keys, queries and its rows' values once,
// double-buffered, with one block barrier per group (as linear_step_block).
template <typename TIn, int DK, int kMode>
__global__ void __launch_bounds__(kStepThreads, 2) linear_step_quad(const StepArgs a, int G) {
    constexpr int CPL = DK / 8;                  // columns per lane
    constexpr int kEl = 16 / (int)sizeof(TIn);   // elements per 16-byte piece
    static_assert(CPL % kEl == 0, "whole pieces per lane");
    extern __shared__ __align__(16) unsigned char step_smem[];
    const int wpb = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 3, c = lane & 7;
    const int rows_pb = 4 * wpb;
    const long long row0 = (long long)blockIdx.x * rows_pb;   // the block's first row overall
    const long long seq = row0 / a.dv;
    const int rb = (int)(row0 % a.dv);
    const int lr = 4 * warp + grp;                            // row within the block
    const int r = rb + lr;
    const int n = a.n;
    const size_t row = ((size_t)seq * a.dv + r) * DK;
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* v = static_cast<const TIn*>(a.v);
    TIn* z = static_cast<TIn*>(a.z);
    // buffer b: [G][DK] keys, [G][DK] queries, [G][rows_pb] values
    const size_t kq = (size_t)G * DK, bufsz = 2 * kq + (size_t)G * rows_pb;
    TIn* const buf = reinterpret_cast<TIn*>(step_smem);
    auto stage = [&](int b, int t0, int len) {
        TIn* kd = buf + b * bufsz;
        TIn* qd = kd + kq;
        TIn* vd = qd + kq;
        const size_t first = (size_t)seq * n + t0;
        const int nkq = len * DK / kEl;
        for (int i = threadIdx.x; i < nkq; i += blockDim.x) {
            cp_async16(kd + i * kEl, k + first * DK + (size_t)i * kEl);
            cp_async16(qd + i * kEl, q + first * DK + (size_t)i * kEl);
        }
        const int vpt = rows_pb / kEl;                       // pieces per token
        for (int i = threadIdx.x; i < len * vpt; i += blockDim.x) {
            const int t = i / vpt, pc = i % vpt;
            cp_async16(vd + t * rows_pb + pc * kEl, v + (first + t) * a.dv + rb + pc * kEl);
        }
    };
    stage(0, 0, min(G, n));
    auto gates = [&](int t0, int len, float& th, float& et, float& keep) {
        th = 0.f; et = 0.f; keep = 1.f;
        if (lane < len) {
            const size_t tok = (size_t)seq * n + t0 + lane;
            th = __ldg(a.theta + tok);
            et = a.eta ? __ldg(a.eta + tok) : 0.f;
            const float al = a.alpha ? __ldg(a.alpha + tok) : 0.f;
            keep = kMode == 0 ? 1.f - al : al;
        }
    };
    float th, et, keep;
    gates(0, min(G, n), th, et, keep);
    const float* w0 = initial_row(a, seq, r);
    float w[CPL], sm_[CPL], wc[CPL];
#pragma unroll
    for (int i4 = 0; i4 < CPL / 4; ++i4) {
        const int j = c * CPL + 4 * i4;
        const float4 x = *reinterpret_cast<const float4*>(w0 + j);
        const float4 y = (kMode == 0 && a.S) ? *reinterpret_cast<const float4*>(a.S + row + j)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 u = a.pos != 0 ? *reinterpret_cast<const float4*>(a.Wc + row + j)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        w[4 * i4] = x.x; w[4 * i4 + 1] = x.y; w[4 * i4 + 2] = x.z; w[4 * i4 + 3] = x.w;
        sm_[4 * i4] = y.x; sm_[4 * i4 + 1] = y.y; sm_[4 * i4 + 2] = y.z; sm_[4 * i4 + 3] = y.w;
        wc[4 * i4] = u.x; wc[4 * i4 + 1] = u.y; wc[4 * i4 + 2] = u.z; wc[4 * i4 + 3] = u.w;
    }
    int p = a.pos;
    bool wc_changed = false;
    for (int t0 = 0; t0 < n; t0 += G) {
        const int len = min(G, n - t0);
        const int b = (t0 / G) & 1;
        const TIn* ks = buf + b * bufsz;
        const TIn* qs = ks + kq;
        const TIn* vs = qs + kq;
        cp_async_wait_all();
        __syncthreads();
        float thn = 0.f, etn = 0.f, keepn = 1.f;
        if (t0 + G < n) {
            const int ln = min(G, n - t0 - G);
            stage(b ^ 1, t0 + G, ln);
            gates(t0 + G, ln, thn, etn, keepn);
        }
        // The read of token u - 1 is summed over its 8 lanes together with token
        // u's error (two independent shuffle chains issued side by side), so
        // only the error's chain is on the state's dependency path.
        float zprev = 0.f;
        for (int u = 0; u < len; ++u) {
            if (p == 0) {   // this token opens a chunk: its gradient point is now
#pragma unroll
                for (int i = 0; i < CPL; ++i) wc[i] = w[i];
                wc_changed = true;
            }
            float kv[CPL], qv[CPL];
#pragma unroll
            for (int i = 0; i < CPL; i += kEl) {
                const uint4 kk = *reinterpret_cast<const uint4*>(ks + u * DK + c * CPL + i);
                const uint4 qq = *reinterpret_cast<const uint4*>(qs + u * DK + c * CPL + i);
                if constexpr (sizeof(TIn) == 2) {
                    const uint32_t kw[4] = {kk.x, kk.y, kk.z, kk.w}, qw[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kv[i + 2 * e] = __uint_as_float(kw[e] << 16);
                        kv[i + 2 * e + 1] = __uint_as_float(kw[e] & 0xffff0000u);
                        qv[i + 2 * e] = __uint_as_float(qw[e] << 16);
                        qv[i + 2 * e + 1] = __uint_as_float(qw[e] & 0xffff0000u);
                    }
                } else {
                    kv[i] = __uint_as_float(kk.x); kv[i + 1] = __uint_as_float(kk.y);
                    kv[i + 2] = __uint_as_float(kk.z); kv[i + 3] = __uint_as_float(kk.w);
                    qv[i] = __uint_as_float(qq.x); qv[i + 1] = __uint_as_float(qq.y);
                    qv[i + 2] = __uint_as_float(qq.z); qv[i + 3] = __uint_as_float(qq.w);
                }
            }
            const float vr = to_f<TIn>(vs[u * rows_pb + lr]);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; i += 2) {
                if constexpr (kMode == 0) {
                    a0 = fmaf(wc[i], kv[i], a0);
                    a1 = fmaf(wc[i + 1], kv[i + 1], a1);
                } else {
                    a0 = fmaf(wc[i] + w[i], kv[i], a0);
                    a1 = fmaf(wc[i + 1] + w[i + 1], kv[i + 1], a1);
                }
            }
            float acc = a0 + a1, zp = zprev;
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            zp += __shfl_xor_sync(0xffffffffu, zp, 4);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            zp += __shfl_xor_sync(0xffffffffu, zp, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            zp += __shfl_xor_sync(0xffffffffu, zp, 1);
            if (u > 0 && c == 0) st_out<TIn>(z + ((size_t)seq * n + t0 + u - 1) * a.dv + r, zp);
            const float thu = __shfl_sync(0xffffffffu, th, u);
            const float keepu = __shfl_sync(0xffffffffu, keep, u);
            float z0 = 0.f, z1 = 0.f;
            if constexpr (kMode == 0) {
                const float ge = 2.f * thu * (acc - vr);   // theta times the gradient's row factor
                const float etu = __shfl_sync(0xffffffffu, et, u);
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    sm_[i] = fmaf(etu, sm_[i], -ge * kv[i]);
                    w[i] = fmaf(keepu, w[i], sm_[i]);
                    if (i & 1) z1 = fmaf(w[i], qv[i], z1);
                    else z0 = fmaf(w[i], qv[i], z0);
                }
            } else {
                const float gg = thu * (acc - vr);         // eta_t ((W_c + W) k - v)_r
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    // the read sees the memory before the write
                    if (i & 1) z1 = fmaf(w[i], qv[i], z1);
                    else z0 = fmaf(w[i], qv[i], z0);
                    w[i] = fmaf(keepu, w[i], -gg * kv[i]);
                }
            }
            zprev = z0 + z1;
            p = p + 1 == a.chunk ? 0 : p + 1;
        }
        // the group's last read
        zprev += __shfl_xor_sync(0xffffffffu, zprev, 4);
        zprev += __shfl_xor_sync(0xffffffffu, zprev, 2);
        zprev += __shfl_xor_sync(0xffffffffu, zprev, 1);
        if (len > 0 && c == 0) st_out<TIn>(z + ((size_t)seq * n + t0 + len - 1) * a.dv + r, zprev);
        th = thn; et = etn; keep = keepn;
    }
#pragma unroll
    for (int i4 = 0; i4 < CPL / 4; ++i4) {
        const int j = c * CPL + 4 * i4;
        *reinterpret_cast<float4*>(a.W + row + j) =
            make_float4(w[4 * i4], w[4 * i4 + 1], w[4 * i4 + 2], w[4 * i4 + 3]);
        if (kMode == 0 && a.S)
            *reinterpret_cast<float4*>(a.S + row + j) =
                make_float4(sm_[4 * i4], sm_[4 * i4 + 1], sm_[4 * i4 + 2], sm_[4 * i4 + 3]);
        if (wc_changed && a.Wc)
            *reinterpret_cast<float4*>(a.Wc + row + j) =
                make_float4(wc[4 * i4], wc[4 * i4 + 1], wc[4 * i4 + 2], wc[4 * i4 + 3]);
    }
}

// Tokens per staged group: the keys and queries of a group take at most
// 4 KB per warp (32 KB per block), and a group never exceeds 32 tokens (one
// per lane for the per-token scalars).
int group_of(const StepArgs& a) {
    const int es = a.bf16 ? 2 : 4;
    const int per_token = 2 * a.dk * es;
    int G = 4096 / per_token;
    if (G < 1) G = 1;
    if (G > 32) G = 32;
    if (G > a.n && a.n > 0) G = a.n;
    return G;
}

template <typename TIn, int NJ, int kMode>
void launch_mode(const StepArgs& a, unsigned blocks, cudaStream_t s) {
    if (a.n == 1) {
        linear_step_direct<TIn, NJ, kMode><<<blocks, kStepThreads, 0, s>>>(a);
    } else if ((NJ == 2 || NJ == 4) && a.dk == 32 * NJ && a.dv % 8 == 0) {
        // four rows per warp; blocks of 8, 4 or 2 warps (the largest that still
        // gives two blocks per SM, since a long sequence has few rows)
        static int sms = 0;
        if (sms == 0) {
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                sms = 152;
        }
        const long long rows = (long long)a.B * a.H * a.dv;
        int wpb = 2;
        for (int cand = 8; cand >= 2; cand /= 2)
            if (a.dv % (4 * cand) == 0 && rows / (4 * cand) >= 2LL * sms) { wpb = cand; break; }
        const int rows_pb = 4 * wpb;
        const int per_token = (2 * a.dk + rows_pb) * (int)sizeof(TIn);
        int G = 8192 / per_token;
        G = G < 1 ? 1 : (G > 32 ? 32 : G);
        if (G > a.n) G = a.n;
        const size_t smem = (size_t)2 * G * (2 * a.dk + rows_pb) * sizeof(TIn);
        const unsigned qblocks = (unsigned)(rows / rows_pb);
        linear_step_quad<TIn, 32 * (NJ == 2 ? 2 : 4), kMode>
            <<<qblocks, 32 * wpb, smem, s>>>(a, G);
    } else if (a.dv % (kStepThreads / 32) == 0) {
        // whole blocks of one sequence: block-shared staging, groups of up to
        // 32 tokens within 8 KB per buffer
        const int per_token = 2 * a.dk * (int)sizeof(TIn);
        int G = 8192 / per_token;
        G = G < 1 ? 1 : (G > 32 ? 32 : G);
        if (G > a.n) G = a.n;
        const size_t smem = (size_t)4 * G * a.dk * sizeof(TIn);
        linear_step_block<TIn, NJ, kMode><<<blocks, kStepThreads, smem, s>>>(a, G);
    } else {
        const int G = group_of(a);
        const size_t smem = (size_t)(kStepThreads / 32) * 2 * G * a.dk * sizeof(TIn);
        linear_step_staged<TIn, NJ, kMode><<<blocks, kStepThreads, smem, s>>>(a, G);
    }
}

template <typename TIn, int NJ>
void launch_nj(const StepArgs& a, unsigned blocks, cudaStream_t s) {
    if (a.mode == 1) launch_mode<TIn, NJ, 1>(a, blocks, s);
    else launch_mode<TIn, NJ, 0>(a, blocks, s);
}

template <typename TIn>
cudaError_t launch_typed(const StepArgs& a, cudaStream_t s) {
    const long long warps = (long long)a.B * a.H * a.dv;
    const unsigned blocks = (unsigned)((warps * 32 + kStepThreads - 1) / kStepThreads);
    const int nj = (a.dk + 31) / 32;
    if (nj <= 1) launch_nj<TIn, 1>(a, blocks, s);
    else if (nj <= 2) launch_nj<TIn, 2>(a, blocks, s);
    else if (nj <= 4) launch_nj<TIn, 4>(a, blocks, s);
    else if (nj <= 8) launch_nj<TIn, 8>(a, blocks, s);
    else launch_nj<TIn, 16>(a, blocks, s);
    return cudaGetLastError();
}

}  // namespace

bool linear_step_supported(const StepArgs& a) { return a.dk >= 1 && a.dk <= 512; }

cudaError_t linear_step_launch(const StepArgs& a, cudaStream_t s) {
    return a.bf16 ? launch_typed<__nv_bfloat16>(a, s) : launch_typed<float>(a, s);
}

}  // namespace ttm
