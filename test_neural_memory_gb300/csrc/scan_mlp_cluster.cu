// fp32 CUDA-core kernel of the 2-layer memory scan, f(x) = W2 GELU(W1 x)
// ("论文速览 | Titans" §3.9; "Continual Learning: From Attention to Neural
// Memory" §4.2), chunk form with every gradient taken at the chunk-start state
// ("TTT layers 与 fast weights" eq (6)) and momentum / decay unrolled per chunk
// ("论文速览 | Titans" §4.3, §4.5).  Per chunk of n tokens, state (W1, W2, S1, S2):
//
//   H = W1 K,  A = GELU(H),  E = 2 (W2 A - V),  D1 = (W2^T E) * GELU'(H)
//   Hq_t = beta_t W1 q_t + c_t S1 q_t - sum_{s<=t} C[t][s] (q_t . k_s) D1_s
//   Aq = GELU(Hq),  z_t = beta_t W2 aq_t + c_t S2 aq_t - sum_{s<=t} C[t][s] (aq_t . a_s) e_s
//   W1 = beta_n W1 + c_n S1 - sum_s C[n][s] D1_s k_s^T,  S1 = P_n S1 - sum_s pm[s] D1_s k_s^T
//   W2 = beta_n W2 + c_n S2 - sum_s C[n][s] e_s a_s^T,   S2 = P_n S2 - sum_s pm[s] e_s a_s^T
//
// A cluster of two CTAs runs one sequence.  CTA r owns the hidden units
// r HH ... r HH + HH - 1: its rows of W1 / S1 and columns of W2 / S2 stay in
// its shared memory for the whole sequence.  Everything indexed by a hidden
// unit is local; three sums over the hidden units cross the cluster once per
// chunk through distributed shared memory:
//   W2 A (for E), aq_t . a_s (for the second score table), W2 aq_t (for z).
// Each CTA writes its partial sums into its own buffer, the cluster barrier
// publishes them, and both CTAs add the two partials (addition commutes, so
// both hold bit-identical E and score tables).  CTA r writes the outputs
// z[., i] of its half of the rows i.  The next chunk's inputs are loaded into
// registers while the current chunk computes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "simt_common.cuh"

namespace ttm {
namespace {

using simt::block_coefficients;
using simt::store_out;
using simt::dot4;
using simt::gelu;
using simt::gelu_grad;

constexpr int kCT = 512;   // threads per CTA

__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// Loads from the peer's shared memory.  Volatile keeps them after the cluster
// barrier (itself a compiler memory barrier); without a memory clobber the
// loads of one phase can all be in flight at once.
__device__ __forceinline__ float ld_cluster(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float4 ld_cluster4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}
// Every thread of both CTAs arrives; shared-memory writes before it are
// visible to the peer's reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory carve-up in floats.  Row strides: D + 4 for token rows and W1
// rows (16-byte rows that land on distinct bank groups for 8 consecutive rows);
// HH + 16 for W2 rows (two rows read by one quarter-warp fall on opposite
// halves of the banks); HH + 4 for token x hidden rows.
template <int NB, int D, int HH>
struct ClLayout {
    static constexpr int ld = D + 4, l1 = D + 4, l2 = HH + 16, lh = HH + 4, lc = NB + 1;
    static constexpr int up4(int x) { return (x + 3) / 4 * 4; }
    static constexpr int W1 = 0;
    static constexpr int S1 = W1 + HH * l1;
    static constexpr int W2 = S1 + HH * l1;
    static constexpr int S2 = W2 + D * l2;
    static constexpr int Ks = S2 + D * l2;
    static constexpr int Qs = Ks + NB * ld;
    static constexpr int Vs = Qs + NB * ld;
    static constexpr int E = Vs + NB * ld;
    static constexpr int Ak = E + NB * ld;
    static constexpr int Gp = Ak + NB * lh;
    static constexpr int D1 = Gp + NB * lh;
    static constexpr int Aq = D1 + NB * lh;
    static constexpr int C = Aq + NB * lh;
    static constexpr int SK = C + up4(NB * lc);
    static constexpr int SA = SK + up4(NB * lc);
    static constexpr int vec = SA + up4(NB * lc);
    static constexpr int Xe = vec + up4(7 * NB);   // [NB][D] partial W2 A
    static constexpr int Xs = Xe + NB * D;         // [NB][NB] partial aq . a
    static constexpr int Xz = Xs + NB * NB;        // [NB][D] partial beta W2 aq + c S2 aq
    static constexpr int total = Xz + NB * D;
    static constexpr size_t bytes = (size_t)total * sizeof(float);
};

template <typename Tin, int NB, int D, int HH>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kCT, 1) mlp_cl_kernel(MlpArgs p) {
    using L = ClLayout<NB, D, HH>;
    constexpr int ld = L::ld, l1 = L::l1, l2 = L::l2, lh = L::lh, lc = L::lc;
    constexpr int TG = kCT / HH;           // token groups of the hidden-unit phases
    constexpr int TPG = NB / TG;           // tokens per group
    constexpr int G = kCT / D;             // lanes per output row
    static_assert(kCT % HH == 0 && NB % TG == 0 && kCT % D == 0 && G <= 32, "shape");
    static_assert(HH % 16 == 0 && D % 16 == 0, "16-byte pieces, four per update thread");
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const uint32_t rank = cta_rank(), peer = rank ^ 1u;
    const int hid = 2 * HH, T = p.T;
    const int seq = blockIdx.x >> 1;
    const int b = seq / p.H, h = seq % p.H;
    const bool mom = p.eta != nullptr;
    const bool trackS = p.S1_out != nullptr;
    float* W1 = sm + L::W1;   // [HH][l1]  own rows of W1
    float* S1 = sm + L::S1;
    float* W2 = sm + L::W2;   // [D][l2]   own columns of W2
    float* S2 = sm + L::S2;
    float* Ks = sm + L::Ks;   // [NB][ld]
    float* Qs = sm + L::Qs;
    float* Vs = sm + L::Vs;
    float* E = sm + L::E;     // [NB][ld]  2 (W2 a_s - v_s), all rows
    float* Ak = sm + L::Ak;   // [NB][lh]  GELU(W1 k_s), own units
    float* Gp = sm + L::Gp;   //           GELU'(W1 k_s)
    float* D1 = sm + L::D1;   //           hidden-side error
    float* Aq = sm + L::Aq;   //           GELU of the query pre-activation
    float* C = sm + L::C;     // [NB][lc]
    float* SK = sm + L::SK;   //           C (q_t . k_s)
    float* SA = sm + L::SA;   //           C (aq_t . a_s)
    float* th = sm + L::vec;
    float* et = th + NB;
    float* al = et + NB;
    float* beta = al + NB;
    float* P = beta + NB;
    float* cc = P + NB;
    float* pm = cc + NB;
    float* Xe = sm + L::Xe;
    float* Xs = sm + L::Xs;
    float* Xz = sm + L::Xz;
    const uint32_t Xe_peer = cluster_addr(Xe, peer);
    const uint32_t Xs_peer = cluster_addr(Xs, peer);
    const uint32_t Xz_peer = cluster_addr(Xz, peer);

    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    Tin* z = static_cast<Tin*>(p.z);
    const size_t nst = (size_t)hid * D;
    const size_t init = ((size_t)(p.shared ? 0 : b) * p.H + h) * nst;
    const int u0 = (int)rank * HH;         // first own hidden unit
    for (int x = tid; x < HH * D; x += kCT) {
        const int u = x / D, j = x % D;
        const size_t g = init + (size_t)(u0 + u) * D + j;
        W1[u * l1 + j] = p.W1_0[g];
        S1[u * l1 + j] = (trackS && p.S1_0) ? p.S1_0[g] : 0.f;
    }
    for (int x = tid; x < D * HH; x += kCT) {
        const int i = x / HH, u = x % HH;
        const size_t g = init + (size_t)i * hid + u0 + u;
        W2[i * l2 + u] = p.W2_0[g];
        S2[i * l2 + u] = (trackS && p.S2_0) ? p.S2_0[g] : 0.f;
    }
    __syncthreads();
    const int hu = tid % HH, tg = tid / HH, t0 = tg * TPG;   // hidden-unit phases
    const int oi = tid / G, og = tid % G;                    // output phases

    // The next chunk's K, Q, V (16-byte pieces) and gates are loaded into
    // registers while the current chunk computes.
    constexpr int kEl = 16 / (int)sizeof(Tin);             // elements per piece
    constexpr int kRowP = D / kEl, kArrP = NB * kRowP;     // pieces per row / per array
    constexpr int RP = (3 * kArrP + kCT - 1) / kCT;        // pieces per thread
    static_assert(D % kEl == 0, "rows of whole pieces");
    uint4 pre[RP];
    float pth = 0.f, pet = 0.f, pal = 0.f;
    auto fetch = [&](int c0) {
        const int n = min(p.chunk, T - c0);
        const size_t tok0 = (size_t)seq * T + c0;
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const int x = tid + r * kCT;
            pre[r] = make_uint4(0u, 0u, 0u, 0u);
            const int arr = x / kArrP, s = (x % kArrP) / kRowP, j = (x % kRowP) * kEl;
            if (x < 3 * kArrP && s < n) {
                const Tin* src = arr == 0 ? k : (arr == 1 ? q : v);
                pre[r] = *reinterpret_cast<const uint4*>(src + (tok0 + s) * D + j);
            }
        }
        if (tid < NB) {
            const bool live = tid < n;
            pth = live ? p.theta[tok0 + tid] : 0.f;
            pet = (live && mom) ? p.eta[tok0 + tid] : 0.f;
            pal = (live && p.alpha) ? p.alpha[tok0 + tid] : 0.f;
        }
    };
    auto stage = [&]() {
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const int x = tid + r * kCT;
            if (x < 3 * kArrP) {
                const int arr = x / kArrP, s = (x % kArrP) / kRowP, j = (x % kRowP) * kEl;
                float* dst = (arr == 0 ? Ks : (arr == 1 ? Qs : Vs)) + s * ld + j;
                if constexpr (sizeof(Tin) == 2) {
                    const uint32_t w[4] = {pre[r].x, pre[r].y, pre[r].z, pre[r].w};
                    float f[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 t2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
                        f[2 * i] = t2.x;
                        f[2 * i + 1] = t2.y;
                    }
                    reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
                    reinterpret_cast<float4*>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
                } else {
                    *reinterpret_cast<float4*>(dst) = make_float4(
                        __uint_as_float(pre[r].x), __uint_as_float(pre[r].y),
                        __uint_as_float(pre[r].z), __uint_as_float(pre[r].w));
                }
            }
        }
        if (tid < NB) {
            th[tid] = pth;
            et[tid] = pet;
            al[tid] = pal;
        }
    };
    if (T > 0) fetch(0);

    for (int c0 = 0; c0 < T; c0 += p.chunk) {
        const int n = min(p.chunk, T - c0);
        const size_t tok0 = (size_t)seq * T + c0;
        stage();
        if (c0 + p.chunk < T) fetch(c0 + p.chunk);
        __syncthreads();
        block_coefficients(n, NB, th, et, al, beta, P, cc, C, lc, pm);

        // H = W1 K (own units), A = GELU(H), GELU'(H)
        {
            float acc[TPG];
#pragma unroll
            for (int s = 0; s < TPG; ++s) acc[s] = 0.f;
            const float4* w = reinterpret_cast<const float4*>(W1 + hu * l1);
#pragma unroll 4
            for (int j4 = 0; j4 < D / 4; ++j4) {
                const float4 w4 = w[j4];
#pragma unroll
                for (int s = 0; s < TPG; ++s)
                    acc[s] += dot4(w4, *reinterpret_cast<const float4*>(Ks + (t0 + s) * ld + 4 * j4));
            }
#pragma unroll
            for (int s = 0; s < TPG; ++s) {
                const bool live = t0 + s < n;
                Ak[(t0 + s) * lh + hu] = live ? gelu(acc[s]) : 0.f;
                Gp[(t0 + s) * lh + hu] = live ? gelu_grad(acc[s]) : 0.f;
            }
        }
        // scores C[t][s] (q_t . k_s), s <= t (both CTAs)
        for (int x = tid; x < NB * NB; x += kCT) {
            const int t = x / NB, s = x % NB;
            float acc = 0.f;
            if (s <= t && t < n) {
#pragma unroll 4
                for (int j = 0; j < D; j += 4)
                    acc += dot4(*reinterpret_cast<const float4*>(Qs + t * ld + j),
                                 *reinterpret_cast<const float4*>(Ks + s * ld + j));
                acc *= C[t * lc + s];
            }
            SK[t * lc + s] = acc;
        }
        __syncthreads();
        // partial W2 A over the own units: G lanes per row, 4-unit pieces og, og + G, ...
        {
            float acc[NB];
#pragma unroll
            for (int s = 0; s < NB; ++s) acc[s] = 0.f;
            const float4* w = reinterpret_cast<const float4*>(W2 + oi * l2);
#pragma unroll 2
            for (int u4 = og; u4 < HH / 4; u4 += G) {
                const float4 w4 = w[u4];
#pragma unroll
                for (int s = 0; s < NB; ++s)
                    acc[s] += dot4(w4, *reinterpret_cast<const float4*>(Ak + s * lh + 4 * u4));
            }
#pragma unroll
            for (int s = 0; s < NB; ++s) {
#pragma unroll
                for (int off = 1; off < G; off <<= 1) acc[s] += __shfl_xor_sync(0xffffffffu, acc[s], off);
            }
            if (og == 0) {
#pragma unroll
                for (int s = 0; s < NB; ++s) Xe[s * D + oi] = acc[s];
            }
        }
        cluster_sync();
        // E = 2 (W2 A - V) from the two partials
        for (int x4 = tid; x4 < NB * D / 4; x4 += kCT) {
            const int x = 4 * x4, s = x / D, i = x % D;
            const float4 mine = *reinterpret_cast<const float4*>(Xe + x);
            const float4 other = ld_cluster4(Xe_peer + 4u * (uint32_t)x);
            const float4 vv = *reinterpret_cast<const float4*>(Vs + s * ld + i);
            const bool live = s < n;
            *reinterpret_cast<float4*>(E + s * ld + i) =
                make_float4(live ? 2.f * (mine.x + other.x - vv.x) : 0.f,
                            live ? 2.f * (mine.y + other.y - vv.y) : 0.f,
                            live ? 2.f * (mine.z + other.z - vv.z) : 0.f,
                            live ? 2.f * (mine.w + other.w - vv.w) : 0.f);
        }
        __syncthreads();
        // D1 = (W2^T E) * GELU'(H), own units
        {
            float acc[TPG];
#pragma unroll
            for (int s = 0; s < TPG; ++s) acc[s] = 0.f;
#pragma unroll 2
            for (int i4 = 0; i4 < D / 4; ++i4) {
                const float4 w4 = make_float4(W2[(4 * i4) * l2 + hu], W2[(4 * i4 + 1) * l2 + hu],
                                              W2[(4 * i4 + 2) * l2 + hu], W2[(4 * i4 + 3) * l2 + hu]);
#pragma unroll
                for (int s = 0; s < TPG; ++s)
                    acc[s] += dot4(w4, *reinterpret_cast<const float4*>(E + (t0 + s) * ld + 4 * i4));
            }
#pragma unroll
            for (int s = 0; s < TPG; ++s)
                D1[(t0 + s) * lh + hu] = acc[s] * Gp[(t0 + s) * lh + hu];
        }
        __syncthreads();
        // Hq_t = beta_t W1 q_t + c_t S1 q_t - sum_{s<=t} SK[t][s] D1_s, Aq = GELU(Hq)
        {
            float aw[TPG], as[TPG];
#pragma unroll
            for (int t = 0; t < TPG; ++t) aw[t] = as[t] = 0.f;
            const float4* w = reinterpret_cast<const float4*>(W1 + hu * l1);
            const float4* sv = reinterpret_cast<const float4*>(S1 + hu * l1);
#pragma unroll 2
            for (int j4 = 0; j4 < D / 4; ++j4) {
                const float4 w4 = w[j4];
                const float4 s4 = mom ? sv[j4] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int t = 0; t < TPG; ++t) {
                    const float4 q4 = *reinterpret_cast<const float4*>(Qs + (t0 + t) * ld + 4 * j4);
                    aw[t] += dot4(w4, q4);
                    as[t] += dot4(s4, q4);
                }
            }
            float dcol[NB];
#pragma unroll
            for (int s = 0; s < NB; ++s) dcol[s] = D1[s * lh + hu];
#pragma unroll
            for (int t = 0; t < TPG; ++t) {
                const int tt = t0 + t;
                float corr = 0.f;
#pragma unroll
                for (int s = 0; s < NB; ++s)
                    if (s <= tt) corr += SK[tt * lc + s] * dcol[s];
                Aq[tt * lh + hu] = tt < n ? gelu(beta[tt] * aw[t] + cc[tt] * as[t] - corr) : 0.f;
            }
        }
        __syncthreads();
        // partial aq_t . a_s over the own units
        for (int x = tid; x < NB * NB; x += kCT) {
            const int t = x / NB, s = x % NB;
            float acc = 0.f;
            if (s <= t && t < n) {
#pragma unroll 4
                for (int u = 0; u < HH; u += 4)
                    acc += dot4(*reinterpret_cast<const float4*>(Aq + t * lh + u),
                                 *reinterpret_cast<const float4*>(Ak + s * lh + u));
            }
            Xs[x] = acc;
        }
        cluster_sync();
        // SA = C (aq . a) from the two partials; partial reads over the own units
        for (int x = tid; x < NB * NB; x += kCT) {
            const int t = x / NB, s = x % NB;
            SA[t * lc + s] = C[t * lc + s] * (Xs[x] + ld_cluster(Xs_peer + 4u * (uint32_t)x));
        }
        {
            float aw[NB], as[NB];
#pragma unroll
            for (int t = 0; t < NB; ++t) aw[t] = as[t] = 0.f;
            const float4* w = reinterpret_cast<const float4*>(W2 + oi * l2);
            const float4* sv = reinterpret_cast<const float4*>(S2 + oi * l2);
#pragma unroll 2
            for (int u4 = og; u4 < HH / 4; u4 += G) {
                const float4 w4 = w[u4];
                const float4 s4 = mom ? sv[u4] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int t = 0; t < NB; ++t) {
                    const float4 a4 = *reinterpret_cast<const float4*>(Aq + t * lh + 4 * u4);
                    aw[t] += dot4(w4, a4);
                    as[t] += dot4(s4, a4);
                }
            }
#pragma unroll
            for (int t = 0; t < NB; ++t) {
#pragma unroll
                for (int off = 1; off < G; off <<= 1) {
                    aw[t] += __shfl_xor_sync(0xffffffffu, aw[t], off);
                    as[t] += __shfl_xor_sync(0xffffffffu, as[t], off);
                }
            }
            if (og == 0) {
#pragma unroll
                for (int t = 0; t < NB; ++t)
                    Xz[t * D + oi] = t < n ? beta[t] * aw[t] + cc[t] * as[t] : 0.f;
            }
        }
        cluster_sync();
        // z for this CTA's half of the rows, four rows i per thread
        for (int x4 = tid; x4 < NB * (D / 8); x4 += kCT) {
            const int t = x4 / (D / 8), i = (int)rank * (D / 2) + 4 * (x4 % (D / 8));
            if (t < n) {
                const float4 mine = *reinterpret_cast<const float4*>(Xz + t * D + i);
                const float4 other = ld_cluster4(Xz_peer + 4u * (uint32_t)(t * D + i));
                float4 acc = make_float4(mine.x + other.x, mine.y + other.y, mine.z + other.z,
                                         mine.w + other.w);
                for (int s = 0; s <= t; ++s) {
                    const float a = SA[t * lc + s];
                    const float4 e4 = *reinterpret_cast<const float4*>(E + s * ld + i);
                    acc.x -= a * e4.x; acc.y -= a * e4.y; acc.z -= a * e4.z; acc.w -= a * e4.w;
                }
                const size_t o = (tok0 + t) * D + i;
                store_out(z, o, acc.x);
                store_out(z, o + 1, acc.y);
                store_out(z, o + 2, acc.z);
                store_out(z, o + 3, acc.w);
            }
        }
        // chunk-end state of the own units (rows of D1 / E past n are zero)
        {
            const float bn = beta[n - 1], cn = cc[n - 1], Pn = P[n - 1];
            const float* Cn = C + (n - 1) * lc;
            // W1 / S1: thread (u, jq) takes the pieces jq, jq + D/16, ... of row u
            // (consecutive lanes: consecutive rows, distinct bank groups)
            for (int x = tid; x < HH * (D / 16); x += kCT) {
                const int u = x % HH, jq = x / HH;
                float4 uw[4], us[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) uw[r] = us[r] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int s = 0; s < NB; ++s) {
                    const float g = D1[s * lh + u];
                    const float gw = Cn[s] * g, gs = pm[s] * g;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float4 k4 = *reinterpret_cast<const float4*>(Ks + s * ld + 4 * (jq + r * (D / 16)));
                        uw[r].x += gw * k4.x; uw[r].y += gw * k4.y; uw[r].z += gw * k4.z; uw[r].w += gw * k4.w;
                        us[r].x += gs * k4.x; us[r].y += gs * k4.y; us[r].z += gs * k4.z; us[r].w += gs * k4.w;
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int j4 = jq + r * (D / 16);
                    float4* wp = reinterpret_cast<float4*>(W1 + u * l1) + j4;
                    float4* sp = reinterpret_cast<float4*>(S1 + u * l1) + j4;
                    const float4 w = *wp, s1 = *sp;
                    *wp = make_float4(bn * w.x + cn * s1.x - uw[r].x, bn * w.y + cn * s1.y - uw[r].y,
                                      bn * w.z + cn * s1.z - uw[r].z, bn * w.w + cn * s1.w - uw[r].w);
                    if (trackS)
                        *sp = make_float4(Pn * s1.x - us[r].x, Pn * s1.y - us[r].y,
                                          Pn * s1.z - us[r].z, Pn * s1.w - us[r].w);
                }
            }
            // W2 / S2: thread (i, pq) takes the pieces pq, pq + HH/16, ... of row i
            for (int x = tid; x < D * (HH / 16); x += kCT) {
                const int pq = x % (HH / 16), i = x / (HH / 16);
                float4 uw[4], us[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) uw[r] = us[r] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int s = 0; s < NB; ++s) {
                    const float g = E[s * ld + i];
                    const float gw = Cn[s] * g, gs = pm[s] * g;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float4 a4 = *reinterpret_cast<const float4*>(Ak + s * lh + 4 * (pq + r * (HH / 16)));
                        uw[r].x += gw * a4.x; uw[r].y += gw * a4.y; uw[r].z += gw * a4.z; uw[r].w += gw * a4.w;
                        us[r].x += gs * a4.x; us[r].y += gs * a4.y; us[r].z += gs * a4.z; us[r].w += gs * a4.w;
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int u4 = pq + r * (HH / 16);
                    float4* wp = reinterpret_cast<float4*>(W2 + i * l2) + u4;
                    float4* sp = reinterpret_cast<float4*>(S2 + i * l2) + u4;
                    const float4 w = *wp, s2 = *sp;
                    *wp = make_float4(bn * w.x + cn * s2.x - uw[r].x, bn * w.y + cn * s2.y - uw[r].y,
                                      bn * w.z + cn * s2.z - uw[r].z, bn * w.w + cn * s2.w - uw[r].w);
                    if (trackS)
                        *sp = make_float4(Pn * s2.x - us[r].x, Pn * s2.y - us[r].y,
                                          Pn * s2.z - us[r].z, Pn * s2.w - us[r].w);
                }
            }
        }
        __syncthreads();
    }
    // final state of the own units
    const size_t dst = (size_t)seq * nst;
    for (int x = tid; x < HH * D; x += kCT) {
        const int u = x / D, j = x % D;
        const size_t g = dst + (size_t)(u0 + u) * D + j;
        p.W1_out[g] = W1[u * l1 + j];
        if (trackS) p.S1_out[g] = S1[u * l1 + j];
    }
    for (int x = tid; x < D * HH; x += kCT) {
        const int i = x / HH, u = x % HH;
        const size_t g = dst + (size_t)i * hid + u0 + u;
        p.W2_out[g] = W2[i * l2 + u];
        if (trackS) p.S2_out[g] = S2[i * l2 + u];
    }
    // the peer may still read this CTA's exchange buffers
    cluster_sync();
}

template <typename Tin, int NB, int D, int HH>
cudaError_t launch_cl(const MlpArgs& a, cudaStream_t s) {
    constexpr size_t smem = ClLayout<NB, D, HH>::bytes;
    static_assert(smem <= 227 * 1024, "shared memory");
    cudaError_t e = cudaFuncSetAttribute(mlp_cl_kernel<Tin, NB, D, HH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mlp_cl_kernel<Tin, NB, D, HH><<<2 * a.B * a.H, kCT, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_cl_shape(const MlpArgs& a, cudaStream_t s) {
    if (a.d == 64 && a.hidden == 256) return launch_cl<Tin, 16, 64, 128>(a, s);
    if (a.d == 32 && a.hidden == 128) return launch_cl<Tin, 16, 32, 64>(a, s);
    if (a.d == 128 && a.hidden == 128) return launch_cl<Tin, 16, 128, 64>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace

bool mlp_cluster_supported(const MlpArgs& a) {
    const bool shape = (a.d == 64 && a.hidden == 256) || (a.d == 32 && a.hidden == 128) ||
                       (a.d == 128 && a.hidden == 128);
    return shape && a.chunk >= 1 && a.chunk <= 16;
}

cudaError_t mlp_cluster_launch(const MlpArgs& a, cudaStream_t s) {
    return a.bf16 ? launch_cl_shape<__nv_bfloat16>(a, s) : launch_cl_shape<float>(a, s);
}

}  // namespace ttm
