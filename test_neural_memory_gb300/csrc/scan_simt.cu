// fp32 CUDA-core kernels of the chunked memory scan (linear / Titans memory
// and the 2-layer MLP memory).
//
// Both kernels evaluate one chunk at a time in the matrix ("dual") form: the
// gradients of every token in a chunk are taken at the chunk-start state, so
// the chunk's outputs and its end state follow from that state by a few dense
// contractions and a lower-triangular coefficient matrix, without forming a
// state per token ("TTT layers 与 fast weights", §1.1 eqs (7)-(9)).
// Momentum and forgetting enter through the unrolled recurrences of
// "论文速览 | Titans" §4.3 (decay products beta_t) and §4.5 (momentum as a
// linear recurrence): inside a block of n tokens that starts from state (W, S),
//
//   W_t = beta_t W + c_t S - sum_{s<=t} C[t][s] grad_s
//   S_t = P_t S - sum_{s<=t} theta_s m(s,t) grad_s
//
// with beta_t = prod (1 - alpha_j), P_t = prod eta_j, c_t = (1-alpha_t) c_{t-1}
// + P_t, C[t][s] = theta_s w(s,t), and per source column s the division-free
// recurrences m(s,s) = w(s,s) = 1, m(s,t) = eta_t m(s,t-1),
// w(s,t) = (1 - alpha_t) w(s,t-1) + m(s,t).
//
// Chunks longer than the on-chip token block are processed as several
// blocks: the errors of every block are still taken at the snapshot made at
// the chunk start, while the (W, S) carried between blocks is the running one.
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
using simt::gelu;
using simt::gelu_grad;

constexpr int kThreads = 256;

// ------------------------------------------------------------------------
// linear / Titans memory: one CTA per (sequence, slice of kRows rows of W)
// ------------------------------------------------------------------------

constexpr int kNB = 32;    // tokens per on-chip block
constexpr int kRows = 16;  // rows of W (d_v index) per CTA

size_t linear_smem_floats(int dk, bool snap) {
    const size_t ldk = dk + 1;
    return 2 * kNB * ldk + kNB * kRows + (snap ? 3 : 2) * (size_t)kRows * dk +
           kRows * (kNB + 1) + 2 * kNB * (kNB + 1) + 7 * kNB + kNB * (kRows + 1);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) linear_simt_kernel(LinearArgs p) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x;
    const int dk = p.dk, dv = p.dv, T = p.T, ldk = dk + 1;
    const int seq = blockIdx.x;
    const int b = seq / p.H, h = seq % p.H;
    const int r0 = blockIdx.y * kRows;
    const int nr = min(kRows, dv - r0);
    const bool snap = p.chunk > kNB;
    const bool mom = p.eta != nullptr;

    float* Ks = sm;                       // [kNB][ldk]
    float* Qs = Ks + kNB * ldk;           // [kNB][ldk]
    float* Vs = Qs + kNB * ldk;           // [kNB][kRows]
    float* W = Vs + kNB * kRows;          // [kRows][dk] running state
    float* S = W + kRows * dk;            // [kRows][dk]
    float* Wc = snap ? S + kRows * dk : W;  // chunk-start snapshot (errors)
    float* E = S + (snap ? 2 : 1) * kRows * dk;  // [kRows][kNB+1]
    float* A = E + kRows * (kNB + 1);     // [kNB][kNB+1] masked scores * C
    float* C = A + kNB * (kNB + 1);       // [kNB][kNB+1]
    float* th = C + kNB * (kNB + 1);
    float* et = th + kNB;
    float* al = et + kNB;
    float* beta = al + kNB;
    float* P = beta + kNB;
    float* cc = P + kNB;
    float* pm = cc + kNB;
    float* zs = pm + kNB;                 // [kNB][kRows+1]

    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    Tin* z = static_cast<Tin*>(p.z);

    const size_t init = (size_t)(p.shared ? 0 : b) * p.H + h;
    for (int x = tid; x < kRows * dk; x += kThreads) {
        const int i = x / dk, j = x % dk;
        const size_t src = (init * dv + r0 + i) * (size_t)dk + j;
        W[x] = i < nr ? p.W0[src] : 0.f;
        S[x] = (i < nr && p.S0) ? p.S0[src] : 0.f;
    }
    __syncthreads();

    const int nch = (T + p.chunk - 1) / p.chunk;
    for (int c0 = 0; c0 < T; c0 += p.chunk) {
        const int cend = min(c0 + p.chunk, T);
        if (p.ckpt) {   // state at this chunk's start, for the gradient passes
            float* dst = p.ckpt + ((size_t)seq * nch + c0 / p.chunk) * 2 * (size_t)dv * dk;
            for (int x = tid; x < nr * dk; x += kThreads) {
                const int i = x / dk, j = x % dk;
                dst[(size_t)(r0 + i) * dk + j] = W[x];
                dst[(size_t)dv * dk + (size_t)(r0 + i) * dk + j] = S[x];
            }
        }
        if (snap) {
            for (int x = tid; x < kRows * dk; x += kThreads) Wc[x] = W[x];
            __syncthreads();
        }
        for (int s0 = c0; s0 < cend; s0 += kNB) {
            const int n = min(kNB, cend - s0);
            const size_t tok0 = (size_t)seq * T + s0;
            for (int x = tid; x < kNB * dk; x += kThreads) {
                const int s = x / dk, j = x % dk;
                Ks[s * ldk + j] = s < n ? load_in(k, (tok0 + s) * dk + j) : 0.f;
                Qs[s * ldk + j] = s < n ? load_in(q, (tok0 + s) * dk + j) : 0.f;
            }
            for (int x = tid; x < kNB * kRows; x += kThreads) {
                const int s = x / kRows, i = x % kRows;
                Vs[x] = (s < n && i < nr) ? load_in(v, (tok0 + s) * dv + r0 + i) : 0.f;
            }
            for (int s = tid; s < kNB; s += kThreads) {
                const size_t g = gate_index(p, (size_t)seq, s0 + s);
                th[s] = s < n ? p.theta[g] : 0.f;
                et[s] = (s < n && mom) ? p.eta[g] : 0.f;
                al[s] = (s < n && p.alpha) ? p.alpha[g] : 0.f;
            }
            __syncthreads();
            block_coefficients(n, kNB, th, et, al, beta, P, cc, C, kNB + 1, pm);

            // scores A[t][s] = C[t][s] (q_t . k_s) for s <= t; errors E = Wc K^T - V^T
            for (int x = tid; x < kNB * kNB; x += kThreads) {
                const int t = x / kNB, s = x % kNB;
                float acc = 0.f;
                if (s <= t && t < n) {
                    for (int j = 0; j < dk; ++j) acc += Qs[t * ldk + j] * Ks[s * ldk + j];
                    acc *= C[t * (kNB + 1) + s];
                }
                A[t * (kNB + 1) + s] = acc;
            }
            for (int x = tid; x < kRows * kNB; x += kThreads) {
                const int i = x / kNB, s = x % kNB;
                float acc = 0.f;
                for (int j = 0; j < dk; ++j) acc += Wc[i * dk + j] * Ks[s * ldk + j];
                E[i * (kNB + 1) + s] = s < n ? acc - Vs[s * kRows + i] : 0.f;
            }
            __syncthreads();

            // reads z_t = beta_t W q_t + c_t S q_t - 2 sum_{s<=t} A[t][s] e_s
            for (int x = tid; x < kRows * kNB; x += kThreads) {
                const int i = x / kNB, t = x % kNB;
                float wq = 0.f, sq = 0.f;
                for (int j = 0; j < dk; ++j) {
                    const float qj = Qs[t * ldk + j];
                    wq += W[i * dk + j] * qj;
                    sq += S[i * dk + j] * qj;
                }
                float corr = 0.f;
                for (int s = 0; s <= t; ++s) corr += A[t * (kNB + 1) + s] * E[i * (kNB + 1) + s];
                zs[t * (kRows + 1) + i] = beta[t] * wq + cc[t] * sq - 2.f * corr;
            }
            __syncthreads();
            for (int x = tid; x < n * kRows; x += kThreads) {
                const int t = x / kRows, i = x % kRows;
                if (i < nr && z) store_out(z, (tok0 + t) * dv + r0 + i, zs[t * (kRows + 1) + i]);
            }
            // block-end state
            const float bn = beta[n - 1], cn = cc[n - 1], Pn = P[n - 1];
            const float* Cn = C + (n - 1) * (kNB + 1);
            for (int x = tid; x < kRows * dk; x += kThreads) {
                const int i = x / dk, j = x % dk;
                float uw = 0.f, us = 0.f;
                for (int s = 0; s < n; ++s) {
                    const float ek = E[i * (kNB + 1) + s] * Ks[s * ldk + j];
                    uw += Cn[s] * ek;
                    us += pm[s] * ek;
                }
                const float w = W[x], sv = S[x];
                W[x] = bn * w + cn * sv - 2.f * uw;
                S[x] = Pn * sv - 2.f * us;
            }
            __syncthreads();
        }
    }
    const size_t dst = (size_t)seq * dv * dk;
    for (int x = tid; x < nr * dk && p.W_out; x += kThreads) {
        const int i = x / dk, j = x % dk;
        p.W_out[dst + (size_t)(r0 + i) * dk + j] = W[x];
        if (p.S_out) p.S_out[dst + (size_t)(r0 + i) * dk + j] = S[x];
    }
}

// ------------------------------------------------------------------------
// 2-layer MLP memory: one CTA per sequence; the running state lives in the
// caller's output buffers (read at each chunk start, rewritten at its end).
// ------------------------------------------------------------------------

int mlp_block_tokens(int d, int hidden) {
    // largest power-of-two token block (<= 32) whose buffers fit in 200 KB
    for (int nb = 32; nb >= 1; nb /= 2) {
        const size_t fl = 4 * (size_t)nb * (d + 1) + 4 * (size_t)nb * (hidden + 1) +
                          3 * (size_t)nb * (nb + 1) + 7 * (size_t)nb;
        if (fl * 4 <= 200 * 1024) return nb;
    }
    return 0;
}

size_t mlp_smem_floats(int d, int hidden, int nb) {
    return 4 * (size_t)nb * (d + 1) + 4 * (size_t)nb * (hidden + 1) + 3 * (size_t)nb * (nb + 1) +
           7 * (size_t)nb;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) mlp_simt_kernel(MlpArgs p, int nb) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = kThreads / 32;
    const int d = p.d, hid = p.hidden, T = p.T, ld = d + 1, lh = hid + 1, lc = nb + 1;
    const int seq = blockIdx.x;
    const int b = seq / p.H, h = seq % p.H;
    const bool mom = p.eta != nullptr;

    float* Ks = sm;                 // [nb][ld]
    float* Qs = Ks + nb * ld;
    float* Vs = Qs + nb * ld;
    float* E = Vs + nb * ld;        // [nb][ld]   output-side error 2 (y - v)
    float* Ak = E + nb * ld;        // [nb][lh]   GELU(W1 k)
    float* Gp = Ak + nb * lh;       // [nb][lh]   GELU'(W1 k)
    float* D1 = Gp + nb * lh;       // [nb][lh]   hidden-side error
    float* Aq = D1 + nb * lh;       // [nb][lh]   GELU of the query pre-activation
    float* C = Aq + nb * lh;        // [nb][lc]
    float* SK = C + nb * lc;        // [nb][lc]   C * (q_t . k_s)
    float* SA = SK + nb * lc;       // [nb][lc]   C * (aq_t . ak_s)
    float* th = SA + nb * lc;
    float* et = th + nb;
    float* al = et + nb;
    float* beta = al + nb;
    float* P = beta + nb;
    float* cc = P + nb;
    float* pm = cc + nb;

    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    Tin* z = static_cast<Tin*>(p.z);

    // The momentum state is tracked whenever the caller asks for it (the API
    // requires S1_out/S2_out whenever eta is given): with eta = 0 it still ends
    // as the last token's step -theta_T grad_T.
    const bool trackS = p.S1_out != nullptr;
    const size_t nst = (size_t)hid * d;
    const size_t init = ((size_t)(p.shared ? 0 : b) * p.H + h) * nst;
    float* W1 = p.W1_out + (size_t)seq * nst;
    float* W2 = p.W2_out + (size_t)seq * nst;
    float* S1 = trackS ? p.S1_out + (size_t)seq * nst : nullptr;
    float* S2 = trackS ? p.S2_out + (size_t)seq * nst : nullptr;
    for (size_t x = tid; x < nst; x += kThreads) {
        const float w1 = p.W1_0[init + x], w2 = p.W2_0[init + x];
        float s1 = 0.f, s2 = 0.f;
        if (trackS) {
            s1 = p.S1_0 ? p.S1_0[init + x] : 0.f;
            s2 = p.S2_0 ? p.S2_0[init + x] : 0.f;
        }
        W1[x] = w1;
        W2[x] = w2;
        if (trackS) {
            S1[x] = s1;
            S2[x] = s2;
        }
    }
    __syncthreads();

    for (int c0 = 0; c0 < T; c0 += p.chunk) {
        const int n = min(p.chunk, T - c0);
        const size_t tok0 = (size_t)seq * T + c0;
        for (int x = tid; x < nb * d; x += kThreads) {
            const int s = x / d, j = x % d;
            Ks[s * ld + j] = s < n ? load_in(k, (tok0 + s) * d + j) : 0.f;
            Qs[s * ld + j] = s < n ? load_in(q, (tok0 + s) * d + j) : 0.f;
            Vs[s * ld + j] = s < n ? load_in(v, (tok0 + s) * d + j) : 0.f;
        }
        for (int s = tid; s < nb; s += kThreads) {
            th[s] = s < n ? p.theta[tok0 + s] : 0.f;
            et[s] = (s < n && mom) ? p.eta[tok0 + s] : 0.f;
            al[s] = (s < n && p.alpha) ? p.alpha[tok0 + s] : 0.f;
        }
        __syncthreads();
        block_coefficients(n, nb, th, et, al, beta, P, cc, C, lc, pm);

        // key pre-activations (lane = token, warp = hidden unit)
        for (int u = warp; u < hid; u += nwarps) {
            for (int s = lane; s < nb; s += 32) {
                float acc = 0.f;
                for (int j = 0; j < d; ++j) acc += W1[(size_t)u * d + j] * Ks[s * ld + j];
                Ak[s * lh + u] = s < n ? gelu(acc) : 0.f;
                Gp[s * lh + u] = s < n ? gelu_grad(acc) : 0.f;
            }
        }
        __syncthreads();
        // output-side error e_s = 2 (W2 a_s - v_s)
        for (int i = warp; i < d; i += nwarps) {
            for (int s = lane; s < nb; s += 32) {
                float acc = 0.f;
                for (int u = 0; u < hid; ++u) acc += W2[(size_t)i * hid + u] * Ak[s * lh + u];
                E[s * ld + i] = s < n ? 2.f * (acc - Vs[s * ld + i]) : 0.f;
            }
        }
        // scores q_t . k_s times the coefficients
        for (int x = tid; x < nb * nb; x += kThreads) {
            const int t = x / nb, s = x % nb;
            float acc = 0.f;
            if (s <= t && t < n) {
                for (int j = 0; j < d; ++j) acc += Qs[t * ld + j] * Ks[s * ld + j];
                acc *= C[t * lc + s];
            }
            SK[t * lc + s] = acc;
        }
        __syncthreads();
        // hidden-side error delta_s = (W2^T e_s) * GELU'(h_s)
        for (int u = warp; u < hid; u += nwarps) {
            for (int s = lane; s < nb; s += 32) {
                float acc = 0.f;
                for (int i = 0; i < d; ++i) acc += W2[(size_t)i * hid + u] * E[s * ld + i];
                D1[s * lh + u] = acc * Gp[s * lh + u];
            }
        }
        __syncthreads();
        // query pre-activation at the token's own state, then GELU
        for (int u = warp; u < hid; u += nwarps) {
            for (int t = lane; t < nb; t += 32) {
                float wq = 0.f, sq = 0.f;
                for (int j = 0; j < d; ++j) {
                    const float qj = Qs[t * ld + j];
                    wq += W1[(size_t)u * d + j] * qj;
                    if (mom) sq += S1[(size_t)u * d + j] * qj;
                }
                float corr = 0.f;
                for (int s = 0; s <= t && s < n; ++s) corr += SK[t * lc + s] * D1[s * lh + u];
                Aq[t * lh + u] = t < n ? gelu(beta[t] * wq + cc[t] * sq - corr) : 0.f;
            }
        }
        __syncthreads();
        for (int x = tid; x < nb * nb; x += kThreads) {
            const int t = x / nb, s = x % nb;
            float acc = 0.f;
            if (s <= t && t < n) {
                for (int u = 0; u < hid; ++u) acc += Aq[t * lh + u] * Ak[s * lh + u];
                acc *= C[t * lc + s];
            }
            SA[t * lc + s] = acc;
        }
        __syncthreads();
        // reads z_t = beta_t W2 aq_t + c_t S2 aq_t - sum_s SA[t][s] e_s
        for (int i = warp; i < d; i += nwarps) {
            for (int t = lane; t < n; t += 32) {
                float wa = 0.f, sa = 0.f;
                for (int u = 0; u < hid; ++u) {
                    const float a = Aq[t * lh + u];
                    wa += W2[(size_t)i * hid + u] * a;
                    if (mom) sa += S2[(size_t)i * hid + u] * a;
                }
                float corr = 0.f;
                for (int s = 0; s <= t; ++s) corr += SA[t * lc + s] * E[s * ld + i];
                store_out(z, (tok0 + t) * d + i, beta[t] * wa + cc[t] * sa - corr);
            }
        }
        __syncthreads();
        // chunk-end state
        const float bn = beta[n - 1], cn = cc[n - 1], Pn = P[n - 1];
        const float* Cn = C + (n - 1) * lc;
        for (size_t x = tid; x < nst; x += kThreads) {
            const int u = (int)(x / d), j = (int)(x % d);
            float uw = 0.f, us = 0.f;
            for (int s = 0; s < n; ++s) {
                const float g = D1[s * lh + u] * Ks[s * ld + j];
                uw += Cn[s] * g;
                us += pm[s] * g;
            }
            const float s1 = trackS ? S1[x] : 0.f;
            W1[x] = bn * W1[x] + cn * s1 - uw;
            if (trackS) S1[x] = Pn * s1 - us;
        }
        for (size_t x = tid; x < nst; x += kThreads) {
            const int i = (int)(x / hid), u = (int)(x % hid);
            float uw = 0.f, us = 0.f;
            for (int s = 0; s < n; ++s) {
                const float g = E[s * ld + i] * Ak[s * lh + u];
                uw += Cn[s] * g;
                us += pm[s] * g;
            }
            const float s2 = trackS ? S2[x] : 0.f;
            W2[x] = bn * W2[x] + cn * s2 - uw;
            if (trackS) S2[x] = Pn * s2 - us;
        }
        __syncthreads();
    }
}

}  // namespace

bool linear_simt_supported(const LinearArgs& a) {
    return a.dk <= 256 && linear_smem_floats(a.dk, a.chunk > kNB) * 4 <= 227 * 1024;
}

cudaError_t linear_simt_launch(const LinearArgs& a, cudaStream_t s) {
    const bool snap = a.chunk > kNB;
    const size_t smem = linear_smem_floats(a.dk, snap) * sizeof(float);
    dim3 grid(a.B * a.H, (a.dv + kRows - 1) / kRows);
    cudaError_t e;
    if (a.bf16) {
        e = cudaFuncSetAttribute(linear_simt_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        linear_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(a);
    } else {
        e = cudaFuncSetAttribute(linear_simt_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        linear_simt_kernel<float><<<grid, kThreads, smem, s>>>(a);
    }
    return cudaGetLastError();
}

bool mlp_simt_supported(const MlpArgs& a) {
    if (mlp_cluster_supported(a) || mlp_simt2_supported(a)) return true;
    const int nb = mlp_block_tokens(a.d, a.hidden);
    return nb >= 1 && a.chunk <= nb;
}

cudaError_t mlp_simt_launch(const MlpArgs& a, cudaStream_t s) {
    if (mlp_cluster_supported(a)) return mlp_cluster_launch(a, s);
    if (mlp_simt2_supported(a)) return mlp_simt2_launch(a, s);
    const int nb = mlp_block_tokens(a.d, a.hidden);
    const size_t smem = mlp_smem_floats(a.d, a.hidden, nb) * sizeof(float);
    dim3 grid(a.B * a.H);
    cudaError_t e;
    if (a.bf16) {
        e = cudaFuncSetAttribute(mlp_simt_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        mlp_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(a, nb);
    } else {
        e = cudaFuncSetAttribute(mlp_simt_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        mlp_simt_kernel<float><<<grid, kThreads, smem, s>>>(a, nb);
    }
    return cudaGetLastError();
}

}  // namespace ttm
