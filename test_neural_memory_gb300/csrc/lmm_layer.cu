// LMM layer around the scan: the neural memory used on its own as a sequence
// layer ("论文速览 | Titans" §6.4), with the projection details of §7.1-§7.3
// (SiLU after the q, k, v projections, l2-normalised q and k, a short causal
// depthwise convolution after the projections, residual connection,
// normalisation and linear gating before the output projection).
//
//   p = x W_in                      one bf16 GEMM (cuBLAS): q | k | v | g | 3H gate logits
//   prep: q, k, v = SiLU(causal depthwise conv of width K of p's q / k / v columns),
//         q, k l2-normalised per head, stored head-major [B][H][T][d] in bf16;
//         theta = s sigmoid, eta = sigmoid, alpha = sigmoid of the logits, [B][H][T]
//   z = Titans memory scan (the library's scan kernels)
//   post: o = RMSNorm_head(z) * rms_w * g, [B][T][D] in bf16
//   y = x + o W_o                   one bf16 GEMM (cuBLAS), residual as beta = 1
//
// The prep and post kernels are HBM-bound elementwise / per-head reductions
// with a warp per (tile of tokens, head, stream) or (token, head), lanes over
// the head's d channels.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace ttm {
namespace {

constexpr int kLayerThreads = 256;

__device__ __forceinline__ float lwarp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }

// VW consecutive bf16 values at p (p aligned to VW elements when kVec).
template <int VW, bool kVec>
__device__ __forceinline__ void load_vw(const __nv_bfloat16* p, float* out) {
    if constexpr (kVec && VW == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            out[2 * e] = __uint_as_float(w[e] << 16);
            out[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    } else if constexpr (kVec && VW == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        out[0] = __uint_as_float(u.x << 16); out[1] = __uint_as_float(u.x & 0xffff0000u);
        out[2] = __uint_as_float(u.y << 16); out[3] = __uint_as_float(u.y & 0xffff0000u);
    } else if constexpr (kVec && VW == 2) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        out[0] = __uint_as_float(u << 16); out[1] = __uint_as_float(u & 0xffff0000u);
    } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) out[e] = __bfloat162float(p[e]);
    }
}

template <int VW>
__device__ __forceinline__ void store_vw(__nv_bfloat16* p, const float* x) {
#pragma unroll
    for (int e = 0; e < VW; e += 2)
        *reinterpret_cast<__nv_bfloat162*>(p + e) = __floats2bfloat162_rn(x[e], x[e + 1]);
}

constexpr int kTile = 4;    // tokens per prep warp

// NJ consecutive bf16 values at p (NJ-aligned), one store.
template <int NJ>
__device__ __forceinline__ void store_nj(__nv_bfloat16* p, const float* x) {
    if constexpr (NJ == 1) {
        p[0] = __float2bfloat16_rn(x[0]);
    } else if constexpr (NJ == 2) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x[0], x[1]);
    } else {
        uint32_t w[NJ / 2];
#pragma unroll
        for (int e = 0; e < NJ / 2; ++e) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&v);
        }
        if constexpr (NJ == 4) *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
        else *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

constexpr int kPrepWarps = kLayerThreads / 32;   // tiles per block

// A block owns one (b, stream, head) and kPrepWarps consecutive tiles of kTile
// tokens; the head's conv taps are staged once per block in shared memory,
// transposed to [window slot][channel]; lane l holds the NJ consecutive
// channels l NJ ... of the head, so each input row and each output row is one
// vector access per lane (kVec: the projection's row length keeps NJ-element
// alignment, else element-wise loads).
template <int NJ, int NW, bool kVec>
__global__ void __launch_bounds__(kLayerThreads, NJ <= 4 ? 4 : 2)
    lmm_prep_kernel(const LmmArgs a, const __nv_bfloat16* proj, __nv_bfloat16* qkv,
                     float* gates) {
    __shared__ __align__(16) float taps[NW][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, d = a.d, T = a.T, K = a.conv_k;
    const int ntile = (T + kTile - 1) / kTile;
    const int ngroup = (ntile + kPrepWarps - 1) / kPrepWarps;
    long long bid = blockIdx.x;
    const int grp = (int)(bid % ngroup);
    bid /= ngroup;
    const int h = (int)(bid % H);
    bid /= H;
    const int s = (int)(bid % 3);
    const int b = (int)(bid / 3);
    const int D = H * d, P = 4 * D + 3 * H;
    const int c0 = s * D + h * d;                     // first channel of the head
    // window slot j of token t0 + i is row i + j; its weight is tap j - (NW - K)
    for (int x = threadIdx.x; x < NW * d; x += kLayerThreads) {
        const int j = x / d, c = x % d;
        const int tap = j - (NW - K);
        taps[j][c] = tap >= 0 ? a.conv_w[(size_t)(c0 + c) * K + tap] : 0.f;
    }
    __syncthreads();
    const int tile = grp * kPrepWarps + warp;
    if (tile >= ntile) return;
    const int t0 = tile * kTile, t1 = min(T, t0 + kTile);
    const int cl = lane * NJ;                         // this lane's first channel
    float wwin[NW][NJ];
#pragma unroll
    for (int j = 0; j < NW; ++j)
#pragma unroll
        for (int i = 0; i < NJ; ++i) wwin[j][i] = taps[j][cl + i];
    constexpr int kRowsT = kTile + NW - 1;
    float xr[kRowsT][NJ];
#pragma unroll
    for (int r = 0; r < kRowsT; ++r) {
        const int ts = t0 - (NW - 1) + r;
        const bool live = ts >= 0 && ts < t1 && r >= NW - K;
        if (live) {
            load_vw<NJ, kVec>(proj + ((size_t)b * T + ts) * P + c0 + cl, xr[r]);
        } else {
#pragma unroll
            for (int i = 0; i < NJ; ++i) xr[r][i] = 0.f;
        }
    }
    const size_t plane = (size_t)a.B * H * T;
    if (s == 0) {   // lanes 0..kTile-1: the three gates of token t0 + lane of head h
        const int t = t0 + lane;
        if (lane < kTile && t < t1) {
            const __nv_bfloat16* lg = proj + ((size_t)b * T + t) * P + 4 * D + h;
            const size_t gi = ((size_t)b * H + h) * T + t;
            gates[gi] = a.theta_scale * sigm(__bfloat162float(lg[0]));
            gates[plane + gi] = sigm(__bfloat162float(lg[H]));
            gates[2 * plane + gi] = sigm(__bfloat162float(lg[2 * H]));
        }
    }
    const size_t stream_stride = (size_t)a.B * H * T * d;
#pragma unroll
    for (int tt = 0; tt < kTile; ++tt) {
        const int t = t0 + tt;
        if (t >= t1) break;
        float u[NJ];
#pragma unroll
        for (int i = 0; i < NJ; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < NW; ++j) acc = fmaf(wwin[j][i], xr[tt + j][i], acc);
            // SiLU; the fast intrinsics' error is far below the bf16 rounding of the output
            u[i] = __fdividef(acc, 1.f + __expf(-acc));
        }
        if (s < 2) {   // l2-normalise q and k per head
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < NJ; ++i) ss += u[i] * u[i];
            const float inv = 1.f / fmaxf(sqrtf(lwarp_sum(ss)), 1e-6f);
#pragma unroll
            for (int i = 0; i < NJ; ++i) u[i] *= inv;
        }
        store_nj<NJ>(qkv + s * stream_stride + (((size_t)b * H + h) * T + t) * d + cl, u);
    }
}

constexpr int kStrip = 64;   // tokens per warp of the strip kernel
constexpr int kGrp = 4;      // tokens per unrolled group

// Strip variant of the prep kernel for d <= 128 and conv width <= 4: a warp walks
// kStrip consecutive tokens of one (b, stream, head) with the conv window in
// registers, so every projection row is loaded once (one vector load per lane),
// the next group's rows are in flight while a group is computed, and the l2 norms
// of a group's kGrp tokens share their shuffle rounds.
template <int NJ, bool kVec>
__global__ void __launch_bounds__(kLayerThreads, 3)
    lmm_prep_strip_kernel(const LmmArgs a, const __nv_bfloat16* proj, __nv_bfloat16* qkv,
                          float* gates) {
    constexpr int NW = 4;                             // window: taps of a width-4 conv
    __shared__ __align__(16) float taps[NW][32 * NJ];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, d = a.d, T = a.T, K = a.conv_k;
    const int nstrip = (T + kStrip - 1) / kStrip;
    const int ngroup = (nstrip + kPrepWarps - 1) / kPrepWarps;
    long long bid = blockIdx.x;
    const int grp = (int)(bid % ngroup);
    bid /= ngroup;
    const int h = (int)(bid % H);
    bid /= H;
    const int s = (int)(bid % 3);
    const int b = (int)(bid / 3);
    const int D = H * d, P = 4 * D + 3 * H;
    const int c0 = s * D + h * d;                     // first channel of the head
    // window slot j of token t is row t - (NW - 1) + j; its weight is tap j - (NW - K)
    for (int x = threadIdx.x; x < NW * d; x += kLayerThreads) {
        const int j = x / d, c = x % d;
        const int tap = j - (NW - K);
        taps[j][c] = tap >= 0 ? a.conv_w[(size_t)(c0 + c) * K + tap] : 0.f;
    }
    __syncthreads();
    const int strip = grp * kPrepWarps + warp;
    if (strip >= nstrip) return;
    const int t0 = strip * kStrip, t1 = min(T, t0 + kStrip);
    const int cl = lane * NJ;
    float wt[NW][NJ];
#pragma unroll
    for (int j = 0; j < NW; ++j)
#pragma unroll
        for (int i = 0; i < NJ; ++i) wt[j][i] = taps[j][cl + i];
    const __nv_bfloat16* src = proj + (size_t)b * T * P + c0 + cl;
    auto load_row = [&](int t, bool live, float* out) {
        if (live && t >= 0) {
            load_vw<NJ, kVec>(src + (size_t)t * P, out);
        } else {
#pragma unroll
            for (int i = 0; i < NJ; ++i) out[i] = 0.f;
        }
    };
    const size_t plane = (size_t)a.B * H * T;
    if (s == 0) {   // the three gates of the strip's tokens of head h (lanes: t0 + lane, + 32)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int t = t0 + lane + 32 * r;
            if (t < t1) {
                const __nv_bfloat16* lg = proj + ((size_t)b * T + t) * P + 4 * D + h;
                const size_t gi = ((size_t)b * H + h) * T + t;
                gates[gi] = a.theta_scale * sigm(__bfloat162float(lg[0]));
                gates[plane + gi] = sigm(__bfloat162float(lg[H]));
                gates[2 * plane + gi] = sigm(__bfloat162float(lg[2 * H]));
            }
        }
    }
    float win[NW - 1][NJ], cur[kGrp][NJ], nxt[kGrp][NJ];
#pragma unroll
    for (int j = 0; j < NW - 1; ++j) load_row(t0 - (NW - 1) + j, true, win[j]);
#pragma unroll
    for (int i = 0; i < kGrp; ++i) load_row(t0 + i, t0 + i < t1, cur[i]);
    const size_t stream_stride = (size_t)a.B * H * T * d;
    __nv_bfloat16* dst = qkv + s * stream_stride + ((size_t)b * H + h) * T * d + cl;
    for (int tg = t0; tg < t1; tg += kGrp) {
#pragma unroll
        for (int i = 0; i < kGrp; ++i) load_row(tg + kGrp + i, tg + kGrp + i < t1, nxt[i]);
        float u[kGrp][NJ], ss[kGrp];
#pragma unroll
        for (int i = 0; i < kGrp; ++i) {
            ss[i] = 0.f;
#pragma unroll
            for (int e = 0; e < NJ; ++e) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const int r = i + j;              // row of [win; cur]
                    const float xv = r < NW - 1 ? win[r][e] : cur[r - (NW - 1)][e];
                    acc = fmaf(wt[j][e], xv, acc);
                }
                // SiLU; the fast intrinsics' error is far below the bf16 rounding of the output
                u[i][e] = __fdividef(acc, 1.f + __expf(-acc));
                ss[i] = fmaf(u[i][e], u[i][e], ss[i]);
            }
        }
        if (s < 2) {   // l2-normalise q and k per head, the group's four sums together
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int i = 0; i < kGrp; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], off);
#pragma unroll
            for (int i = 0; i < kGrp; ++i) {
                const float inv = 1.f / fmaxf(sqrtf(ss[i]), 1e-6f);
#pragma unroll
                for (int e = 0; e < NJ; ++e) u[i][e] *= inv;
            }
        }
#pragma unroll
        for (int i = 0; i < kGrp; ++i)
            if (tg + i < t1) store_nj<NJ>(dst + (size_t)(tg + i) * d, u[i]);
        // slide: the last NW - 1 rows of [win; cur] become the window
#pragma unroll
        for (int j = 0; j < NW - 1; ++j)
#pragma unroll
            for (int e = 0; e < NJ; ++e) win[j][e] = cur[kGrp - (NW - 1) + j][e];
#pragma unroll
        for (int i = 0; i < kGrp; ++i)
#pragma unroll
            for (int e = 0; e < NJ; ++e) cur[i][e] = nxt[i][e];
    }
}

// One warp per (b, t, h): o = z / sqrt(mean(z^2) + eps) * rms_w * g; lane l
// holds channels l VW ... of the head.
template <int VW, bool kVec>
__global__ void __launch_bounds__(kLayerThreads) lmm_post_kernel(const LmmArgs a,
                                                                 const __nv_bfloat16* proj,
                                                                 const __nv_bfloat16* z,
                                                                 __nv_bfloat16* o) {
    const long long gw = ((long long)blockIdx.x * kLayerThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int H = a.H, d = a.d, T = a.T;
    if (gw >= (long long)a.B * T * H) return;
    const int h = (int)(gw % H);
    const long long bt = gw / H;
    const int t = (int)(bt % T);
    const int b = (int)(bt / T);
    const int D = H * d, P = 4 * D + 3 * H;
    float zz[VW], gg[VW];
    load_vw<VW, true>(z + (((size_t)b * H + h) * T + t) * d + lane * VW, zz);
    load_vw<VW, kVec>(proj + ((size_t)b * T + t) * P + 3 * D + h * d + lane * VW, gg);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < VW; ++e) ss += zz[e] * zz[e];
    const float r = 1.f / sqrtf(lwarp_sum(ss) / d + 1e-6f);
    float out[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) out[e] = zz[e] * r * a.rms_w[lane * VW + e] * gg[e];
    __nv_bfloat16* orow = o + ((size_t)b * T + t) * D + h * d + lane * VW;
    if constexpr (VW == 1) orow[0] = __float2bfloat16_rn(out[0]);
    else store_vw<VW>(orow, out);
}

std::mutex g_blas_lock;
cublasHandle_t g_blas[64];

cublasHandle_t blas_handle() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_blas_lock);
    if (!g_blas[dev] && cublasCreate(&g_blas[dev]) != CUBLAS_STATUS_SUCCESS) g_blas[dev] = nullptr;
    return g_blas[dev];
}

}  // namespace

bool lmm_supported(const LmmArgs& a) {
    return (a.d == 32 || a.d == 64 || a.d == 128 || a.d == 256) && a.conv_k >= 1 &&
           a.conv_k <= 8;
}

template <int NJ>
void prep_nj(const LmmArgs& a, unsigned blocks, cudaStream_t s, const __nv_bfloat16* p,
             __nv_bfloat16* q, float* g) {
    const bool vec = (4 * a.H * a.d + 3 * a.H) % NJ == 0;
    if (a.conv_k <= 4) {
        if (vec) lmm_prep_kernel<NJ, 4, true><<<blocks, kLayerThreads, 0, s>>>(a, p, q, g);
        else lmm_prep_kernel<NJ, 4, false><<<blocks, kLayerThreads, 0, s>>>(a, p, q, g);
    } else {
        if (vec) lmm_prep_kernel<NJ, 8, true><<<blocks, kLayerThreads, 0, s>>>(a, p, q, g);
        else lmm_prep_kernel<NJ, 8, false><<<blocks, kLayerThreads, 0, s>>>(a, p, q, g);
    }
}

template <int VW>
void post_vw(const LmmArgs& a, unsigned blocks, cudaStream_t s, const __nv_bfloat16* p,
             const __nv_bfloat16* z, __nv_bfloat16* o) {
    const int P = 4 * a.H * a.d + 3 * a.H;
    if (P % VW == 0) lmm_post_kernel<VW, true><<<blocks, kLayerThreads, 0, s>>>(a, p, z, o);
    else lmm_post_kernel<VW, false><<<blocks, kLayerThreads, 0, s>>>(a, p, z, o);
}

cudaError_t lmm_prep_launch(const LmmArgs& a, const void* proj, void* qkv, float* gates,
                            cudaStream_t s) {
    auto p = static_cast<const __nv_bfloat16*>(proj);
    auto q = static_cast<__nv_bfloat16*>(qkv);
    if (a.d <= 128 && a.conv_k <= 4) {
        // one block per (b, stream, head, kPrepWarps strips of kStrip tokens)
        const long long nstrip = (a.T + kStrip - 1) / kStrip;
        const unsigned blocks =
            (unsigned)((long long)a.B * 3 * a.H * ((nstrip + kPrepWarps - 1) / kPrepWarps));
        const bool vec = (4 * a.H * a.d + 3 * a.H) % (a.d / 32) == 0;
        switch (a.d / 32) {
            case 1: lmm_prep_strip_kernel<1, true><<<blocks, kLayerThreads, 0, s>>>(a, p, q, gates); break;
            case 2:
                if (vec) lmm_prep_strip_kernel<2, true><<<blocks, kLayerThreads, 0, s>>>(a, p, q, gates);
                else lmm_prep_strip_kernel<2, false><<<blocks, kLayerThreads, 0, s>>>(a, p, q, gates);
                break;
            case 4:
                if (vec) lmm_prep_strip_kernel<4, true><<<blocks, kLayerThreads, 0, s>>>(a, p, q, gates);
                else lmm_prep_strip_kernel<4, false><<<blocks, kLayerThreads, 0, s>>>(a, p, q, gates);
                break;
            default: return cudaErrorInvalidValue;
        }
        return cudaGetLastError();
    }
    // one block per (b, stream, head, kPrepWarps tiles)
    const long long ntile = (a.T + kTile - 1) / kTile;
    const unsigned blocks =
        (unsigned)((long long)a.B * 3 * a.H * ((ntile + kPrepWarps - 1) / kPrepWarps));
    switch (a.d / 32) {
        case 1: prep_nj<1>(a, blocks, s, p, q, gates); break;
        case 2: prep_nj<2>(a, blocks, s, p, q, gates); break;
        case 4: prep_nj<4>(a, blocks, s, p, q, gates); break;
        case 8: prep_nj<8>(a, blocks, s, p, q, gates); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t lmm_post_launch(const LmmArgs& a, const void* proj, const void* z, void* o,
                            cudaStream_t s) {
    const long long warps = (long long)a.B * a.T * a.H;
    const unsigned blocks = (unsigned)((warps * 32 + kLayerThreads - 1) / kLayerThreads);
    auto p = static_cast<const __nv_bfloat16*>(proj);
    auto zz = static_cast<const __nv_bfloat16*>(z);
    auto oo = static_cast<__nv_bfloat16*>(o);
    switch (a.d / 32) {
        case 1: post_vw<1>(a, blocks, s, p, zz, oo); break;
        case 2: post_vw<2>(a, blocks, s, p, zz, oo); break;
        case 4: post_vw<4>(a, blocks, s, p, zz, oo); break;
        case 8: post_vw<8>(a, blocks, s, p, zz, oo); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// Row-major C[M x N] = alpha A[M x K] B[K x N] + beta C, bf16 operands, fp32
// accumulation (cuBLAS, column-major: C^T = B^T A^T).  `scratch` is handed to
// cuBLAS as its workspace so that the library allocates nothing.
bool gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, float beta,
               void* scratch, size_t scratch_bytes, cudaStream_t s) {
    cublasHandle_t h = blas_handle();
    if (!h) return false;
    if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return false;
    if (cublasSetWorkspace(h, scratch, scratch_bytes) != CUBLAS_STATUS_SUCCESS) return false;
    const float one = 1.f;
    return cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_N, N, M, K, &one, B, CUDA_R_16BF, N, A,
                        CUDA_R_16BF, K, &beta, C, CUDA_R_16BF, N, CUBLAS_COMPUTE_32F,
                        CUBLAS_GEMM_DEFAULT) == CUBLAS_STATUS_SUCCESS;
}

}  // namespace ttm
