// fp32 CUDA-core kernel of the 2-layer memory scan, f(x) = W2 GELU(W1 x)
// ("论文速览 | Titans" §3.9; "Continual Learning: From Attention to Neural
// Memory" §4.2), in the chunk form: every gradient of a chunk is taken at the
// chunk-start state ("TTT layers 与 fast weights" eq (6)), momentum and decay
// unrolled per chunk as for the linear memory ("论文速览 | Titans" §4.3, §4.5).
// Per chunk of n tokens, with state (W1, W2, S1, S2) at the chunk start:
//
//   H = W1 K,  A = GELU(H),  E = 2 (W2 A - V),  D1 = (W2^T E) * GELU'(H)
//   Hq_t = beta_t W1 q_t + c_t S1 q_t - sum_{s<=t} C[t][s] (q_t . k_s) D1_s
//   Aq = GELU(Hq),  z_t = beta_t W2 aq_t + c_t S2 aq_t - sum_{s<=t} C[t][s] (aq_t . a_s) e_s
//   W1 = beta_n W1 + c_n S1 - sum_s C[n][s] D1_s k_s^T,  S1 = P_n S1 - sum_s pm[s] D1_s k_s^T
//   W2 = beta_n W2 + c_n S2 - sum_s C[n][s] e_s a_s^T,   S2 = P_n S2 - sum_s pm[s] e_s a_s^T
//
// One CTA per sequence; the fp32 state stays in the caller's output buffers
// (4 x hidden x d floats: larger than shared memory) and is read through L2.
// Mappings that keep every thread busy and every state read 16 bytes wide:
//   hidden-unit phases (H, D1, Hq): thread u, all NB tokens of the chunk in
//     registers; the token rows are broadcast reads of shared memory;
//   output phases (E, z): G = 256 / d lanes per output row i, lane g taking the
//     4-unit pieces g, g + G, ... of the hidden dimension, summed by shuffles;
//   update phase: 16-byte pieces of the state, one thread each.
// NB (a power of two >= the chunk) sizes the register arrays.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "simt_common.cuh"

namespace ttm {
namespace {

using simt::block_coefficients;
using simt::load_in;
using simt::store_out;
using simt::dot4;
using simt::gelu;
using simt::gelu_grad;

constexpr int kMT = 256;   // threads per CTA



// Shared-memory carve-up (floats; rows of d + 4 / hidden + 4 keep 16-byte alignment).
struct MlpSmem {
    int ld, lh, lc;
    size_t Ks, Qs, Vs, E, Ak, Hk, D1, Aq, C, SK, SA, vec, total;
};

__host__ __device__ inline MlpSmem mlp_smem(int nb, int d, int hid) {
    MlpSmem m;
    m.ld = d + 4;
    m.lh = hid + 4;
    m.lc = nb + 1;
    auto up = [](size_t x) { return (x + 3) / 4 * 4; };
    size_t o = 0;
    m.Ks = o; o += (size_t)nb * m.ld;
    m.Qs = o; o += (size_t)nb * m.ld;
    m.Vs = o; o += (size_t)nb * m.ld;
    m.E = o; o += (size_t)nb * m.ld;
    m.Ak = o; o += (size_t)nb * m.lh;
    m.Hk = o; o += (size_t)nb * m.lh;
    m.D1 = o; o += (size_t)nb * m.lh;
    m.Aq = o; o += (size_t)nb * m.lh;
    m.C = o; o += up((size_t)nb * m.lc);
    m.SK = o; o += up((size_t)nb * m.lc);
    m.SA = o; o += up((size_t)nb * m.lc);
    m.vec = o; o += up(7 * (size_t)nb);
    m.total = o;
    return m;
}

template <typename Tin, int NB, int G>
__global__ void __launch_bounds__(kMT, 1) mlp_simt2_kernel(MlpArgs p) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const int d = p.d, hid = p.hidden, T = p.T;
    const MlpSmem M = mlp_smem(NB, d, hid);
    const int ld = M.ld, lh = M.lh, lc = M.lc;
    const int seq = blockIdx.x;
    const int b = seq / p.H, h = seq % p.H;
    const bool mom = p.eta != nullptr;
    float* Ks = sm + M.Ks;      // [NB][ld]
    float* Qs = sm + M.Qs;
    float* Vs = sm + M.Vs;
    float* E = sm + M.E;        // [NB][ld]  output-side error 2 (y - v)
    float* Ak = sm + M.Ak;      // [NB][lh]  GELU(W1 k)
    float* Hk = sm + M.Hk;      // [NB][lh]  W1 k
    float* D1 = sm + M.D1;      // [NB][lh]  hidden-side error
    float* Aq = sm + M.Aq;      // [NB][lh]  GELU of the query pre-activation
    float* C = sm + M.C;        // [NB][lc]
    float* SK = sm + M.SK;      // [NB][lc]  C * (q_t . k_s)
    float* SA = sm + M.SA;      // [NB][lc]  C * (aq_t . a_s)
    float* th = sm + M.vec;
    float* et = th + NB;
    float* al = et + NB;
    float* beta = al + NB;
    float* P = beta + NB;
    float* cc = P + NB;
    float* pm = cc + NB;

    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    Tin* z = static_cast<Tin*>(p.z);
    const bool trackS = p.S1_out != nullptr;
    const size_t nst = (size_t)hid * d;
    const size_t init = ((size_t)(p.shared ? 0 : b) * p.H + h) * nst;
    float* W1 = p.W1_out + (size_t)seq * nst;   // [hid][d]
    float* W2 = p.W2_out + (size_t)seq * nst;   // [d][hid]
    float* S1 = trackS ? p.S1_out + (size_t)seq * nst : nullptr;
    float* S2 = trackS ? p.S2_out + (size_t)seq * nst : nullptr;
    for (size_t x = tid; x < nst; x += kMT) {
        W1[x] = p.W1_0[init + x];
        W2[x] = p.W2_0[init + x];
        if (trackS) {
            S1[x] = p.S1_0 ? p.S1_0[init + x] : 0.f;
            S2[x] = p.S2_0 ? p.S2_0[init + x] : 0.f;
        }
    }
    __syncthreads();
    const int oi = tid / G, og = tid % G;          // output phases: row, lane in the group

    for (int c0 = 0; c0 < T; c0 += p.chunk) {
        const int n = min(p.chunk, T - c0);
        const size_t tok0 = (size_t)seq * T + c0;
        for (int x = tid; x < NB * d; x += kMT) {
            const int s = x / d, j = x % d;
            Ks[s * ld + j] = s < n ? load_in(k, (tok0 + s) * d + j) : 0.f;
            Qs[s * ld + j] = s < n ? load_in(q, (tok0 + s) * d + j) : 0.f;
            Vs[s * ld + j] = s < n ? load_in(v, (tok0 + s) * d + j) : 0.f;
        }
        for (int s = tid; s < NB; s += kMT) {
            th[s] = s < n ? p.theta[tok0 + s] : 0.f;
            et[s] = (s < n && mom) ? p.eta[tok0 + s] : 0.f;
            al[s] = (s < n && p.alpha) ? p.alpha[tok0 + s] : 0.f;
        }
        __syncthreads();
        block_coefficients(n, NB, th, et, al, beta, P, cc, C, lc, pm);

        // H = W1 K, A = GELU(H): thread u, every token
        for (int u = tid; u < hid; u += kMT) {
            float acc[NB];
#pragma unroll
            for (int s = 0; s < NB; ++s) acc[s] = 0.f;
            const float4* w = reinterpret_cast<const float4*>(W1 + (size_t)u * d);
            for (int j4 = 0; j4 < d / 4; ++j4) {
                const float4 w4 = w[j4];
#pragma unroll
                for (int s = 0; s < NB; ++s)
                    acc[s] += dot4(w4, *reinterpret_cast<const float4*>(Ks + s * ld + 4 * j4));
            }
#pragma unroll
            for (int s = 0; s < NB; ++s) {
                Hk[s * lh + u] = acc[s];
                Ak[s * lh + u] = s < n ? gelu(acc[s]) : 0.f;
            }
        }
        // scores C[t][s] (q_t . k_s), s <= t
        for (int x = tid; x < NB * NB; x += kMT) {
            const int t = x / NB, s = x % NB;
            float acc = 0.f;
            if (s <= t && t < n) {
                for (int j = 0; j < d; j += 4)
                    acc += dot4(*reinterpret_cast<const float4*>(Qs + t * ld + j),
                                *reinterpret_cast<const float4*>(Ks + s * ld + j));
                acc *= C[t * lc + s];
            }
            SK[t * lc + s] = acc;
        }
        __syncthreads();
        // E = 2 (W2 A - V): G lanes per output row i, 4-unit pieces og, og + G, ...
        {
            float acc[NB];
#pragma unroll
            for (int s = 0; s < NB; ++s) acc[s] = 0.f;
            if (oi < d) {
                const float4* w = reinterpret_cast<const float4*>(W2 + (size_t)oi * hid);
                for (int u4 = og; u4 < hid / 4; u4 += G) {
                    const float4 w4 = w[u4];
#pragma unroll
                    for (int s = 0; s < NB; ++s)
                        acc[s] += dot4(w4, *reinterpret_cast<const float4*>(Ak + s * lh + 4 * u4));
                }
            }
#pragma unroll
            for (int s = 0; s < NB; ++s) {
#pragma unroll
                for (int off = 1; off < G; off <<= 1) acc[s] += __shfl_xor_sync(0xffffffffu, acc[s], off);
            }
            if (oi < d && og == 0) {
#pragma unroll
                for (int s = 0; s < NB; ++s)
                    E[s * ld + oi] = s < n ? 2.f * (acc[s] - Vs[s * ld + oi]) : 0.f;
            }
        }
        __syncthreads();
        // D1 = (W2^T E) * GELU'(H): thread u, every token
        for (int u = tid; u < hid; u += kMT) {
            float acc[NB];
#pragma unroll
            for (int s = 0; s < NB; ++s) acc[s] = 0.f;
            for (int i4 = 0; i4 < d / 4; ++i4) {
                const float w0 = W2[(size_t)(4 * i4 + 0) * hid + u];
                const float w1 = W2[(size_t)(4 * i4 + 1) * hid + u];
                const float w2 = W2[(size_t)(4 * i4 + 2) * hid + u];
                const float w3 = W2[(size_t)(4 * i4 + 3) * hid + u];
                const float4 w4 = make_float4(w0, w1, w2, w3);
#pragma unroll
                for (int s = 0; s < NB; ++s)
                    acc[s] += dot4(w4, *reinterpret_cast<const float4*>(E + s * ld + 4 * i4));
            }
#pragma unroll
            for (int s = 0; s < NB; ++s)
                D1[s * lh + u] = s < n ? acc[s] * gelu_grad(Hk[s * lh + u]) : 0.f;
        }
        __syncthreads();
        // Hq_t = beta_t W1 q_t + c_t S1 q_t - sum_{s<=t} SK[t][s] D1_s, Aq = GELU(Hq)
        for (int u = tid; u < hid; u += kMT) {
            float aw[NB], as[NB];
#pragma unroll
            for (int t = 0; t < NB; ++t) aw[t] = as[t] = 0.f;
            const float4* w = reinterpret_cast<const float4*>(W1 + (size_t)u * d);
            const float4* sv = mom ? reinterpret_cast<const float4*>(S1 + (size_t)u * d) : nullptr;
            for (int j4 = 0; j4 < d / 4; ++j4) {
                const float4 w4 = w[j4];
                const float4 s4 = mom ? sv[j4] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int t = 0; t < NB; ++t) {
                    const float4 q4 = *reinterpret_cast<const float4*>(Qs + t * ld + 4 * j4);
                    aw[t] += dot4(w4, q4);
                    as[t] += dot4(s4, q4);
                }
            }
            float dcol[NB];
#pragma unroll
            for (int s = 0; s < NB; ++s) dcol[s] = D1[s * lh + u];
#pragma unroll
            for (int t = 0; t < NB; ++t) {
                float corr = 0.f;
#pragma unroll
                for (int s = 0; s <= t; ++s) corr += SK[t * lc + s] * dcol[s];
                Aq[t * lh + u] = t < n ? gelu(beta[t] * aw[t] + cc[t] * as[t] - corr) : 0.f;
            }
        }
        __syncthreads();
        // SA[t][s] = C[t][s] (aq_t . a_s), s <= t
        for (int x = tid; x < NB * NB; x += kMT) {
            const int t = x / NB, s = x % NB;
            float acc = 0.f;
            if (s <= t && t < n) {
                for (int u = 0; u < hid; u += 4)
                    acc += dot4(*reinterpret_cast<const float4*>(Aq + t * lh + u),
                                *reinterpret_cast<const float4*>(Ak + s * lh + u));
                acc *= C[t * lc + s];
            }
            SA[t * lc + s] = acc;
        }
        __syncthreads();
        // z_t = beta_t W2 aq_t + c_t S2 aq_t - sum_{s<=t} SA[t][s] e_s: G lanes per row i
        {
            float aw[NB], as[NB];
#pragma unroll
            for (int t = 0; t < NB; ++t) aw[t] = as[t] = 0.f;
            if (oi < d) {
                const float4* w = reinterpret_cast<const float4*>(W2 + (size_t)oi * hid);
                const float4* sv = mom ? reinterpret_cast<const float4*>(S2 + (size_t)oi * hid) : nullptr;
                for (int u4 = og; u4 < hid / 4; u4 += G) {
                    const float4 w4 = w[u4];
                    const float4 s4 = mom ? sv[u4] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int t = 0; t < NB; ++t) {
                        const float4 a4 = *reinterpret_cast<const float4*>(Aq + t * lh + 4 * u4);
                        aw[t] += dot4(w4, a4);
                        as[t] += dot4(s4, a4);
                    }
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
            if (oi < d && og == 0) {
#pragma unroll
                for (int t = 0; t < NB; ++t) {
                    if (t < n) {
                        float corr = 0.f;
                        for (int s = 0; s <= t; ++s) corr += SA[t * lc + s] * E[s * ld + oi];
                        store_out(z, (tok0 + t) * d + oi, beta[t] * aw[t] + cc[t] * as[t] - corr);
                    }
                }
            }
        }
        __syncthreads();
        // chunk-end state, one 16-byte piece per thread (rows of D1 / E past n are zero)
        {
            const float bn = beta[n - 1], cn = cc[n - 1], Pn = P[n - 1];
            const float* Cn = C + (n - 1) * lc;
            const int pr1 = d / 4, pr2 = hid / 4;
            for (int x = tid; x < hid * pr1; x += kMT) {
                const int u = x / pr1, j4 = x % pr1;
                float4 uw = make_float4(0.f, 0.f, 0.f, 0.f), us = uw;
#pragma unroll
                for (int s = 0; s < NB; ++s) {
                    const float4 k4 = *reinterpret_cast<const float4*>(Ks + s * ld + 4 * j4);
                    const float g = D1[s * lh + u];
                    const float gw = Cn[s] * g, gs = pm[s] * g;
                    uw.x += gw * k4.x; uw.y += gw * k4.y; uw.z += gw * k4.z; uw.w += gw * k4.w;
                    us.x += gs * k4.x; us.y += gs * k4.y; us.z += gs * k4.z; us.w += gs * k4.w;
                }
                float4* wp = reinterpret_cast<float4*>(W1) + x;
                float4 w = *wp;
                if (trackS) {
                    float4* sp = reinterpret_cast<float4*>(S1) + x;
                    const float4 s1 = *sp;
                    w.x = bn * w.x + cn * s1.x - uw.x; w.y = bn * w.y + cn * s1.y - uw.y;
                    w.z = bn * w.z + cn * s1.z - uw.z; w.w = bn * w.w + cn * s1.w - uw.w;
                    *sp = make_float4(Pn * s1.x - us.x, Pn * s1.y - us.y, Pn * s1.z - us.z,
                                      Pn * s1.w - us.w);
                } else {
                    w.x = bn * w.x - uw.x; w.y = bn * w.y - uw.y;
                    w.z = bn * w.z - uw.z; w.w = bn * w.w - uw.w;
                }
                *wp = w;
            }
            for (int x = tid; x < d * pr2; x += kMT) {
                const int i = x / pr2, u4 = x % pr2;
                float4 uw = make_float4(0.f, 0.f, 0.f, 0.f), us = uw;
#pragma unroll
                for (int s = 0; s < NB; ++s) {
                    const float4 a4 = *reinterpret_cast<const float4*>(Ak + s * lh + 4 * u4);
                    const float g = E[s * ld + i];
                    const float gw = Cn[s] * g, gs = pm[s] * g;
                    uw.x += gw * a4.x; uw.y += gw * a4.y; uw.z += gw * a4.z; uw.w += gw * a4.w;
                    us.x += gs * a4.x; us.y += gs * a4.y; us.z += gs * a4.z; us.w += gs * a4.w;
                }
                float4* wp = reinterpret_cast<float4*>(W2) + x;
                float4 w = *wp;
                if (trackS) {
                    float4* sp = reinterpret_cast<float4*>(S2) + x;
                    const float4 s2 = *sp;
                    w.x = bn * w.x + cn * s2.x - uw.x; w.y = bn * w.y + cn * s2.y - uw.y;
                    w.z = bn * w.z + cn * s2.z - uw.z; w.w = bn * w.w + cn * s2.w - uw.w;
                    *sp = make_float4(Pn * s2.x - us.x, Pn * s2.y - us.y, Pn * s2.z - us.z,
                                      Pn * s2.w - us.w);
                } else {
                    w.x = bn * w.x - uw.x; w.y = bn * w.y - uw.y;
                    w.z = bn * w.z - uw.z; w.w = bn * w.w - uw.w;
                }
                *wp = w;
            }
        }
        __syncthreads();
    }
}

template <typename Tin, int NB, int G>
cudaError_t launch_one(const MlpArgs& a, cudaStream_t s) {
    const size_t smem = mlp_smem(NB, a.d, a.hidden).total * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(mlp_simt2_kernel<Tin, NB, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mlp_simt2_kernel<Tin, NB, G><<<a.B * a.H, kMT, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, int NB>
cudaError_t launch_g(const MlpArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 16: return launch_one<Tin, NB, 16>(a, s);
        case 32: return launch_one<Tin, NB, 8>(a, s);
        case 64: return launch_one<Tin, NB, 4>(a, s);
        case 128: return launch_one<Tin, NB, 2>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename Tin>
cudaError_t launch_nb(const MlpArgs& a, cudaStream_t s, int nb) {
    switch (nb) {
        case 4: return launch_g<Tin, 4>(a, s);
        case 8: return launch_g<Tin, 8>(a, s);
        case 16: return launch_g<Tin, 16>(a, s);
        case 32: return launch_g<Tin, 32>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

int block_tokens(int chunk) {
    int nb = 4;
    while (nb < chunk) nb *= 2;
    return nb;
}

}  // namespace

bool mlp_simt2_supported(const MlpArgs& a) {
    if (a.d != 16 && a.d != 32 && a.d != 64 && a.d != 128) return false;
    if (a.hidden < 4 || a.hidden % 4 != 0 || a.chunk < 1 || a.chunk > 32) return false;
    const uintptr_t al = (uintptr_t)a.W1_out | (uintptr_t)a.W2_out | (uintptr_t)a.S1_out |
                         (uintptr_t)a.S2_out;
    if (al % 16 != 0) return false;
    return mlp_smem(block_tokens(a.chunk), a.d, a.hidden).total * sizeof(float) <= 227 * 1024;
}

cudaError_t mlp_simt2_launch(const MlpArgs& a, cudaStream_t s) {
    const int nb = block_tokens(a.chunk);
    return a.bf16 ? launch_nb<__nv_bfloat16>(a, s, nb) : launch_nb<float>(a, s, nb);
}

}  // namespace ttm
