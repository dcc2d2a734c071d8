// Tensor-core (tcgen05 + TMA) chain and local passes of the scan's gradient
// (bf16 inputs, d_k = d_v in {64, 128}, chunks of 64 tokens).
//
// The local pass gives, for one chunk of n tokens with the chunk-start state
// (W, S) and the adjoint of the chunk-end state (dWe, dSe), the gradients of
// the chunk's q, k, v and gates ("Continual Learning: From Attention to
// Neural Memory" §4.5; the chunk form of "TTT layers 与 fast weights" §1.1
// eqs (7)-(9) with the momentum / decay unrolling of "论文速览 | Titans"
// §4.3, §4.5).  With E = K W^T - V (errors at the chunk start), the masked
// scores A~[t][s] = C[t][s] (q_t . k_s) (s <= t), DE[t][s] = dz_t . e_s and
// G = C o DE (s <= t):
//   De = -2 (A~^T dZ + diag(C[n-1]) K dWe^T + diag(pm) K dSe^T),   dV = -De
//   dQ = diag(beta) dZ W + diag(c) dZ S - 2 G K
//   dK = De W - 2 G^T Q - 2 diag(C[n-1]) E dWe - 2 diag(pm) E dSe
// and the gate gradients from dC = -2 (Q K^T) o DE (plus the end-state term
// on the last row), dbeta_t = dz_t . (W q_t), dc_t = dz_t . (S q_t),
// e_s . (dWe k_s), e_s . (dSe k_s) and <dWe, W>, <dWe, S>, <dSe, S>, carried
// back through the coefficient recurrences exactly as the CUDA-core pass
// does.
//
// Every contraction is a tcgen05 MMA with M = 128: the token-row products
// stack [K; Q] (or pad with rows that are never read back), and the products
// whose rows are tokens and whose result is d wide are taken transposed
// (dQ^T, dK^T: rows = key index j).  The state and adjoint matrices arrive in
// bf16 (the forward scan writes the checkpoints, the chain the adjoints) and
// load by TMA straight into their operand tiles, one half of their rows (the
// value index i) at a time; DE, De, dQ^T and dK^T accumulate over the halves
// in tensor memory.  One CTA of 256 threads per (sequence, chunk), every
// chunk at once.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "../../include/ttm.h"
#include "kernels.h"
#include "simt_common.cuh"
#include "tc_ptx.cuh"

namespace ttm {
namespace {

using namespace tc;

constexpr int kC = 64;              // tokens per chunk (== TMA tile height)
constexpr uint32_t kTile = 8192;    // 64 rows x 128 bytes (bf16)
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kLdc = kC + 1;        // row stride of the fp32 tables
constexpr int kQs = kC + 2;         // row stride of the bf16 score copy (33 words: no conflicts)
constexpr long long kWaitCycles = 4000000000LL;

// TMEM columns (each accumulator 64 columns; lanes = rows)
constexpr uint32_t kA1 = 0;     // [K; Q] W_I^T   (lanes 0-63: K W^T, 64-127: Q W^T); QK first
constexpr uint32_t kA2 = 64;    // [K; Q] S_I^T   (lanes 64-127: Q S^T)
constexpr uint32_t kA3 = 128;   // [K; Q] dWe_I^T (lanes 0-63: K dWe^T)
constexpr uint32_t kA4 = 192;   // [K; Q] dSe_I^T (lanes 0-63: K dSe^T)
constexpr uint32_t kDE = 256;   // DE (lanes t, columns s)
constexpr uint32_t kDeI = 320;  // De of the half (lanes s, columns i)
constexpr uint32_t kDQ = 384;   // dQ^T (lanes j, columns t)
constexpr uint32_t kDK = 448;   // dK^T (lanes j, columns s)

struct Layout {
    uint32_t kq, dz, vv, mat, ei, ec, ep, bz, cz, dei, at, gg, qkb, crec, vec, bars, total;
};

// [K_h][Q_h] per 64-column half of the keys (so [K; Q] is one 128-row
// operand); dZ and V per half of the value index; the four state / adjoint
// matrices of the current value half (rows i, bf16, one tile per key half);
// the bf16 operand tiles of the chunk; the chunk's coefficient record (as the
// forward scan's pre-pass wrote it); vectors.
__host__ __device__ constexpr Layout make_layout(int D) {
    Layout L{};
    uint32_t o = 0;
    const uint32_t NH = D / 64;
    L.kq = o;   o += NH * 2 * kTile;
    L.dz = o;   o += NH * kTile;
    L.vv = o;   o += NH * kTile;
    L.mat = o;  o += 4 * NH * kTile;     // W, S, dWe, dSe of the value half
    L.ei = o;   o += kTile;              // E of the half [s][i]
    L.ec = o;   o += kTile;              // -2 C[n-1][s] E
    L.ep = o;   o += kTile;              // -2 pm[s] E
    L.bz = o;   o += kTile;              // beta_t dZ [t][i]
    L.cz = o;   o += kTile;              // c_t dZ
    L.dei = o;  o += kTile;              // De of the half [s][i]
    L.at = o;   o += kTile;              // -2 A~ [t][s]
    L.gg = o;   o += kTile;              // -2 G [t][s]
    L.qkb = o;  o += kC * kQs * 2;       // Q K^T (bf16, [t][s], padded rows)
    L.crec = o; o += (kCoefRecBytes + 63) / 64 * 64;   // C table, beta, c, C[n-1], pm
    L.vec = o;  o += 16 * kC * 4;        // gate vectors
    L.bars = o; o += 64;
    L.total = o;
    return L;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack8(const float* x) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                      pack_bf16(x[6], x[7]));
}

__device__ __forceinline__ void unpack8(uint4 v, float* x) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4); }

struct Sync {
    uint64_t full, mma, mfull;
    long long limit;
    int abort;
    uint32_t tmem;
};

// Bounded wait by every thread of the block (uniform answer per warp).
__device__ __noinline__ bool wait_bar(Sync* Y, uint64_t* bar, uint32_t parity, int* status) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const long long t0 = clock64();
    bool ok = true;
    while (!mbar_try_wait_sleep(bar, parity, 20000)) {
        if (*(volatile int*)&Y->abort || clock64() - t0 > Y->limit) {
            *(volatile int*)&Y->abort = 1;
            atomicExch(status, TTM_ERR_TIMEOUT);
            ok = false;
            break;
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// The same bounded wait on an abort flag and a limit of any owner.
__device__ __noinline__ bool wait_flag(int* abort, long long limit, uint64_t* bar, uint32_t parity,
                                       int* status) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const long long t0 = clock64();
    bool ok = true;
    while (!mbar_try_wait_sleep(bar, parity, 20000)) {
        if (*(volatile int*)abort || clock64() - t0 > limit) {
            *(volatile int*)abort = 1;
            atomicExch(status, TTM_ERR_TIMEOUT);
            ok = false;
            break;
        }
    }
    return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_local_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap zmap, const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap ckmap, const __grid_constant__ CUtensorMap admap,
                    const BwdArgs a, const uint8_t* coef, int nch) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    constexpr Layout L = make_layout(D);
    constexpr int NH = D / 64, KS = D / 16;
    Sync* Y = reinterpret_cast<Sync*>(sm + L.bars);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seq = blockIdx.x / nch, c = blockIdx.x % nch;
    const int T = a.T;
    const int n = min(kC, T - c * kC);
    const size_t tok0 = (size_t)seq * T + (size_t)c * kC;
    int* status = a.status;

    uint8_t* kq = sm + L.kq;
    auto ktile = [&](int h) { return kq + h * 2 * kTile; };
    auto qtile = [&](int h) { return kq + h * 2 * kTile + kTile; };
    auto dztile = [&](int h) { return sm + L.dz + h * kTile; };
    auto vtile = [&](int h) { return sm + L.vv + h * kTile; };
    auto mtile = [&](int m, int h) { return sm + L.mat + (m * NH + h) * kTile; };   // m: W S dWe dSe
    uint8_t* ei = sm + L.ei;
    uint8_t* ec = sm + L.ec;
    uint8_t* ep = sm + L.ep;
    uint8_t* bz = sm + L.bz;
    uint8_t* cz = sm + L.cz;
    uint8_t* dei = sm + L.dei;
    uint8_t* at = sm + L.at;
    uint8_t* gg = sm + L.gg;
    __nv_bfloat16* qkb = reinterpret_cast<__nv_bfloat16*>(sm + L.qkb);
    const uint8_t* crec = sm + L.crec;
    // C[t][4g .. 4g+3] from the record's table (row t: 16-byte groups permuted by t % 16)
    auto cgroup = [&](int t, int g) {
        return *reinterpret_cast<const float4*>(crec + t * 256 + ((g ^ (t & 15)) << 4));
    };
    auto crow16 = [&](int t, int s0, float* w) {   // C[t][s0 .. s0+15], s0 % 16 == 0
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4 f = cgroup(t, s0 / 4 + g);
            w[4 * g] = f.x; w[4 * g + 1] = f.y; w[4 * g + 2] = f.z; w[4 * g + 3] = f.w;
        }
    };
    const float* beta = reinterpret_cast<const float*>(crec + kCoefVec + kCoefBeta);
    const float* cc = reinterpret_cast<const float*>(crec + kCoefVec + kCoefC);
    const float* cend = reinterpret_cast<const float*>(crec + kCoefVec + kCoefCend);
    const float* pm = reinterpret_cast<const float*>(crec + kCoefVec + kCoefPend);
    float* th = reinterpret_cast<float*>(sm + L.vec);
    float* et = th + kC;
    float* al = et + kC;
    float* dbeta = al + kC;
    float* dcc = dbeta + kC;
    float* dclast = dcc + kC;
    float* dpm = dclast + kC;
    float* dkeep = dpm + kC;
    float* deta = dkeep + kC;
    float* dth = deta + kC;
    float* scal = dth + kC;          // <dWe, W>, <dWe, S>, <dSe, S>

    // W, S (checkpoint) and dWe, dSe (adjoint) rows 64 I .. 64 I + 63 of this
    // chunk into the matrix tiles (one thread)
    int halves_issued = 0;
    auto load_half = [&](int I) {
        mbar_expect_tx(&Y->mfull, 4 * NH * kTile);
        const int z0 = (seq * nch + c) * 2;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            tma_load_3d(mtile(0, h), &ckmap, &Y->mfull, 64 * h, 64 * I, z0);
            tma_load_3d(mtile(1, h), &ckmap, &Y->mfull, 64 * h, 64 * I, z0 + 1);
            tma_load_3d(mtile(2, h), &admap, &Y->mfull, 64 * h, 64 * I, z0);
            tma_load_3d(mtile(3, h), &admap, &Y->mfull, 64 * h, 64 * I, z0 + 1);
        }
        ++halves_issued;
    };
    // a full chunk whose gates start on a 16-byte boundary takes them with the
    // tiles; otherwise threads load them
    const bool gate_bulk = n == kC && (tok0 & 3) == 0;
    if (tid == 0) {
        mbar_init(&Y->full, 1);
        mbar_init(&Y->mma, 1);
        mbar_init(&Y->mfull, 1);
        Y->limit = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;
        Y->abort = 0;
        fence_mbar_init();
        // every input copy starts before the tensor memory is allocated
        load_half(0);
        const uint32_t gbytes =
            gate_bulk ? kC * 4 * (1 + (a.eta ? 1 : 0) + (a.alpha ? 1 : 0)) : 0;
        mbar_expect_tx(&Y->full, 4 * NH * kTile + kCoefRecBytes + gbytes);
        bulk_load(sm + L.crec, coef + ((size_t)seq * nch + c) * kCoefRecBytes, kCoefRecBytes,
                  &Y->full);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            tma_load_3d(ktile(h), &kmap, &Y->full, 64 * h, c * kC, seq);
            tma_load_3d(qtile(h), &qmap, &Y->full, 64 * h, c * kC, seq);
            tma_load_3d(dztile(h), &zmap, &Y->full, 64 * h, c * kC, seq);
            tma_load_3d(vtile(h), &vmap, &Y->full, 64 * h, c * kC, seq);
        }
        if (gate_bulk) {
            bulk_load(th, a.theta + tok0, kC * 4, &Y->full);
            if (a.eta) bulk_load(et, a.eta + tok0, kC * 4, &Y->full);
            if (a.alpha) bulk_load(al, a.alpha + tok0, kC * 4, &Y->full);
        }
    }
    if (warp == 0) tmem_alloc(&Y->tmem, kTmemCols);
    if (tid < kC) {
        if (!gate_bulk) {
            th[tid] = tid < n ? a.theta[tok0 + tid] : 0.f;
            et[tid] = (tid < n && a.eta) ? a.eta[tok0 + tid] : 0.f;
            al[tid] = (tid < n && a.alpha) ? a.alpha[tok0 + tid] : 0.f;
        } else {
            if (!a.eta) et[tid] = 0.f;
            if (!a.alpha) al[tid] = 0.f;
        }
        dbeta[tid] = dcc[tid] = dclast[tid] = dpm[tid] = dkeep[tid] = deta[tid] = 0.f;
    }
    if (tid < 4) scal[tid] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = Y->tmem;
    const uint32_t tl = tmem + ((uint32_t)(warp & 3) * 32 << 16);   // this warp's TMEM lanes
    const int row = (warp & 3) * 32 + lane;                          // TMEM lane of this thread
    const int chalf = warp >> 2;                                     // column half of an epilogue


    uint32_t mma_phase = 0;
    bool ok = wait_bar(Y, &Y->full, 0, status);

    constexpr uint32_t idKK = idesc_bf16_f32(128, 64, 0, 0);   // A K-major, B K-major
    constexpr uint32_t idMM = idesc_bf16_f32(128, 64, 1, 1);   // both MN-major
    constexpr uint32_t idMK = idesc_bf16_f32(128, 64, 1, 0);   // A MN-major, B K-major

    // [K; Q] K^T -> lanes 64-127 of kA1: Q K^T
    if (warp == 0 && ok) {
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const uint32_t base = smem_u32(ktile(kk >> 2)) + (kk & 3) * 32;
                mma_bf16(tmem + kA1, sdesc(base, 16, 1024, 2), sdesc(base, 16, 1024, 2), idKK, kk > 0);
            }
            mma_commit(&Y->mma);
        }
        __syncwarp();
    }

    // the three inner products of the end-state term over value half I (from
    // the bf16 matrix tiles), and beta dZ, c dZ of the half
    auto prep_half = [&](int I) {
        float p0 = 0.f, p1 = 0.f, p2 = 0.f;
        constexpr int kChunks = 64 * (D / 8);                  // (row, 8-column chunk) pairs
        for (int x = tid; x < kChunks; x += kThreads) {
            const int i = x / (D / 8), c8 = x % (D / 8);
            const int h = c8 >> 3;
            const uint32_t off = swz(i, c8 & 7);
            float w[8], sv[8], gw[8], gs[8];
            unpack8(*reinterpret_cast<const uint4*>(mtile(0, h) + off), w);
            unpack8(*reinterpret_cast<const uint4*>(mtile(1, h) + off), sv);
            unpack8(*reinterpret_cast<const uint4*>(mtile(2, h) + off), gw);
            unpack8(*reinterpret_cast<const uint4*>(mtile(3, h) + off), gs);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                p0 = fmaf(gw[e], w[e], p0);
                p1 = fmaf(gw[e], sv[e], p1);
                p2 = fmaf(gs[e], sv[e], p2);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            p0 += __shfl_xor_sync(0xffffffffu, p0, off);
            p1 += __shfl_xor_sync(0xffffffffu, p1, off);
            p2 += __shfl_xor_sync(0xffffffffu, p2, off);
        }
        if (lane == 0) {
            atomicAdd(&scal[0], p0);
            atomicAdd(&scal[1], p1);
            atomicAdd(&scal[2], p2);
        }
        // beta_t dZ[t][i], c_t dZ[t][i] (same swizzled places as the dZ tile)
        for (int x = tid; x < 64 * 8; x += kThreads) {
            const int t = x >> 3, c8 = x & 7;
            const uint32_t off = swz(t, c8);
            float v[8], vb[8], vc[8];
            unpack8(*reinterpret_cast<const uint4*>(dztile(I) + off), v);
            const float bt = beta[t], ct = cc[t];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                vb[e] = bt * v[e];
                vc[e] = ct * v[e];
            }
            *reinterpret_cast<uint4*>(bz + off) = pack8(vb);
            *reinterpret_cast<uint4*>(cz + off) = pack8(vc);
        }
    };

    if (ok) ok = wait_bar(Y, &Y->mfull, 0, status);
    if (ok) prep_half(0);
    if (ok) ok = wait_bar(Y, &Y->mma, mma_phase++ & 1, status);
    if (ok && row >= 64) {
        // -2 A~[t][s] = -2 C[t][s] (q_t . k_s) for s <= t, and Q K^T in bf16
        tc_fence_after();
        const int t = row - 64;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int s0 = 32 * chalf + 16 * q;
            float r[16], x[16], cw[16];
            tmem_ld16(tl + kA1 + s0, r);
            crow16(t, s0, cw);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int s = s0 + e;
                x[e] = (s <= t && t < n) ? -2.f * cw[e] * r[e] : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 16; e += 2)
                *reinterpret_cast<uint32_t*>(qkb + t * kQs + s0 + e) = pack_bf16(r[e], r[e + 1]);
            *reinterpret_cast<uint4*>(at + swz(t, s0 / 8)) = pack8(x);
            *reinterpret_cast<uint4*>(at + swz(t, s0 / 8 + 1)) = pack8(x + 8);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    for (int I = 0; I < NH; ++I) {
        if (I > 0 && ok) {
            ok = wait_bar(Y, &Y->mfull, I & 1, status);
            if (ok) prep_half(I);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
        }
        // [K; Q] {W, S, dWe, dSe}_I^T
        if (warp == 0 && ok) {
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        const uint32_t abase = smem_u32(ktile(kk >> 2)) + (kk & 3) * 32;
                        const uint32_t bbase = smem_u32(mtile(m, kk >> 2)) + (kk & 3) * 32;
                        mma_bf16(tmem + kA1 + 64 * m, sdesc(abase, 16, 1024, 2),
                                 sdesc(bbase, 16, 1024, 2), idKK, kk > 0);
                    }
                }
                mma_commit(&Y->mma);
            }
            __syncwarp();
        }
        if (ok) ok = wait_bar(Y, &Y->mma, mma_phase++ & 1, status);
        if (ok) {
            tc_fence_after();
            if (row < 64) {
                // token s: E = K W^T - V, e_s . (dWe k_s), e_s . (dSe k_s), the scaled
                // copies of E, and -2 (C[n-1][s] dWK + pm[s] dSK) into the De accumulator
                const int s = row;
                const float cn = cend[s], pms = pm[s];
                float pw = 0.f, ps = 0.f;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int i0 = 32 * chalf + 16 * q;
                    float e[16], gw[16], gs[16], v[16];
                    tmem_ld16(tl + kA1 + i0, e);
                    tmem_ld16(tl + kA3 + i0, gw);
                    tmem_ld16(tl + kA4 + i0, gs);
                    unpack8(*reinterpret_cast<const uint4*>(vtile(I) + swz(s, i0 / 8)), v);
                    unpack8(*reinterpret_cast<const uint4*>(vtile(I) + swz(s, i0 / 8 + 1)), v + 8);
                    tmem_wait_ld();
                    float x1[16], x2[16];
                    uint32_t pre[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        e[k] = s < n ? e[k] - v[k] : 0.f;
                        pw = fmaf(e[k], gw[k], pw);
                        ps = fmaf(e[k], gs[k], ps);
                        x1[k] = -2.f * cn * e[k];
                        x2[k] = -2.f * pms * e[k];
                        pre[k] = __float_as_uint(s < n ? -2.f * (cn * gw[k] + pms * gs[k]) : 0.f);
                    }
                    *reinterpret_cast<uint4*>(ei + swz(s, i0 / 8)) = pack8(e);
                    *reinterpret_cast<uint4*>(ei + swz(s, i0 / 8 + 1)) = pack8(e + 8);
                    *reinterpret_cast<uint4*>(ec + swz(s, i0 / 8)) = pack8(x1);
                    *reinterpret_cast<uint4*>(ec + swz(s, i0 / 8 + 1)) = pack8(x1 + 8);
                    *reinterpret_cast<uint4*>(ep + swz(s, i0 / 8)) = pack8(x2);
                    *reinterpret_cast<uint4*>(ep + swz(s, i0 / 8 + 1)) = pack8(x2 + 8);
                    const uint32_t lo[8] = {pre[0], pre[1], pre[2], pre[3], pre[4], pre[5], pre[6], pre[7]};
                    const uint32_t hi[8] = {pre[8], pre[9], pre[10], pre[11], pre[12], pre[13], pre[14], pre[15]};
                    tmem_st8(tl + kDeI + i0, lo);
                    tmem_st8(tl + kDeI + i0 + 8, hi);
                }
                atomicAdd(&dclast[s], pw);
                atomicAdd(&dpm[s], ps);
                tmem_wait_st();
            } else {
                // token t: dz_t . (W q_t) and dz_t . (S q_t)
                const int t = row - 64;
                float pb = 0.f, pc = 0.f;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int i0 = 32 * chalf + 16 * q;
                    float qw[16], qs[16], z[16];
                    tmem_ld16(tl + kA1 + i0, qw);
                    tmem_ld16(tl + kA2 + i0, qs);
                    unpack8(*reinterpret_cast<const uint4*>(dztile(I) + swz(t, i0 / 8)), z);
                    unpack8(*reinterpret_cast<const uint4*>(dztile(I) + swz(t, i0 / 8 + 1)), z + 8);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        pb = fmaf(z[k], qw[k], pb);
                        pc = fmaf(z[k], qs[k], pc);
                    }
                }
                atomicAdd(&dbeta[t], pb);
                atomicAdd(&dcc[t], pc);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // DE += [dZ_I; .] E_I^T;  De_I += (-2 A~^T) dZ_I
        if (warp == 0 && ok) {
            tc_fence_after();
            if (elect_one()) {
                const uint32_t zb = smem_u32(dztile(I)), eb = smem_u32(ei), ab = smem_u32(at);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kDE, sdesc(zb + kk * 32, 16, 1024, 2), sdesc(eb + kk * 32, 16, 1024, 2),
                             idKK, (I > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kDeI, sdesc(ab + kk * 2048, kTile, 1024, 2),
                             sdesc(zb + kk * 2048, kTile, 1024, 2), idMM, 1u);
                mma_commit(&Y->mma);
            }
            __syncwarp();
        }
        if (ok) ok = wait_bar(Y, &Y->mma, mma_phase++ & 1, status);
        if (ok && row < 64) {
            // De of the half: dv = -De, and its bf16 tile [s][i]
            tc_fence_after();
            const int s = row;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int i0 = 32 * chalf + 16 * q;
                float r[16], nv[16];
                tmem_ld16(tl + kDeI + i0, r);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) nv[k] = -r[k];
                *reinterpret_cast<uint4*>(dei + swz(s, i0 / 8)) = pack8(r);
                *reinterpret_cast<uint4*>(dei + swz(s, i0 / 8 + 1)) = pack8(r + 8);
                if (s < n) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dv_) +
                                                          (tok0 + s) * D + 64 * I + i0);
                    dst[0] = pack8(nv);
                    dst[1] = pack8(nv + 8);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // dQ^T += W_I^T (beta dZ_I)^T + S_I^T (c dZ_I)^T;
        // dK^T += W_I^T De_I^T + dWe_I^T (-2 Cn E_I)^T + dSe_I^T (-2 pm E_I)^T
        if (warp == 0 && ok) {
            tc_fence_after();
            if (elect_one()) {
                const uint32_t mw = smem_u32(mtile(0, 0)), ms = smem_u32(mtile(1, 0));
                const uint32_t mgw = smem_u32(mtile(2, 0)), mgs = smem_u32(mtile(3, 0));
                const uint32_t bzb = smem_u32(bz), czb = smem_u32(cz), deb = smem_u32(dei);
                const uint32_t ecb = smem_u32(ec), epb = smem_u32(ep);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16(tmem + kDQ, sdesc(mw + kk * 2048, kTile, 1024, 2),
                             sdesc(bzb + kk * 32, 16, 1024, 2), idMK, (I > 0 || kk > 0) ? 1u : 0u);
                    mma_bf16(tmem + kDQ, sdesc(ms + kk * 2048, kTile, 1024, 2),
                             sdesc(czb + kk * 32, 16, 1024, 2), idMK, 1u);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16(tmem + kDK, sdesc(mw + kk * 2048, kTile, 1024, 2),
                             sdesc(deb + kk * 32, 16, 1024, 2), idMK, (I > 0 || kk > 0) ? 1u : 0u);
                    mma_bf16(tmem + kDK, sdesc(mgw + kk * 2048, kTile, 1024, 2),
                             sdesc(ecb + kk * 32, 16, 1024, 2), idMK, 1u);
                    mma_bf16(tmem + kDK, sdesc(mgs + kk * 2048, kTile, 1024, 2),
                             sdesc(epb + kk * 32, 16, 1024, 2), idMK, 1u);
                }
                mma_commit(&Y->mma);
            }
            __syncwarp();
        }
        // the next half overwrites the matrices and operand tiles
        if (ok) ok = wait_bar(Y, &Y->mma, mma_phase++ & 1, status);
        if (ok && tid == 0 && I + 1 < NH) {
            fence_proxy_async_smem();
            load_half(I + 1);
        }
    }

    // DE complete: dC = -2 (Q K^T) o DE (+ the end-state term on the last row)
    // and -2 G = -2 C o DE, for s <= t < n
    float* dC = reinterpret_cast<float*>(sm + L.mat);    // [t][kLdc], the matrices are done
    if (ok && row < 64) {
        tc_fence_after();
        const int t = row;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int s0 = 32 * chalf + 16 * q;
            float r[16], x[16], cw[16], qk[16];
            tmem_ld16(tl + kDE + s0, r);
            crow16(t, s0, cw);
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                const uint32_t u = *reinterpret_cast<const uint32_t*>(qkb + t * kQs + s0 + e);
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
                qk[e] = f.x;
                qk[e + 1] = f.y;
            }
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int s = s0 + e;
                const bool in = s <= t && t < n;
                const float de = in ? r[e] : 0.f;
                x[e] = -2.f * cw[e] * de;
                dC[t * kLdc + s] = -2.f * qk[e] * de -
                                   (t == n - 1 && s < n ? 2.f * dclast[s] : 0.f);
            }
            *reinterpret_cast<uint4*>(gg + swz(t, s0 / 8)) = pack8(x);
            *reinterpret_cast<uint4*>(gg + swz(t, s0 / 8 + 1)) = pack8(x + 8);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    __nv_bfloat16* stq = reinterpret_cast<__nv_bfloat16*>(sm + L.mat + kC * kLdc * 4);
    __nv_bfloat16* stk = stq + kC * D;
    // Two groups from here on, which meet again before the row sums: warps 2-3
    // walk the gate recurrences (they need dC, the end-state adjoints and the
    // gates only), the other six warps take the G products, the dQ / dK
    // epilogue and the stores.  The walks' tables live in tiles that no one
    // reads any more: Kc, Ec (rows read by other threads, padded) and Wm in
    // the operand tiles ei .. at, Mm in the dZ / V tiles; Wm and Mm are read
    // back only by the lane that wrote them.
    // (512 bytes in: at d = 64 the dq / dk staging above runs 256 bytes past the
    // matrix tiles)
    constexpr uint32_t kWalkOff = 512;
    static_assert(L.mat + kC * kLdc * 4 + 2 * kC * D * 2 <= L.ei + kWalkOff, "staging clear of the tables");
    float* Kc = reinterpret_cast<float*>(sm + L.ei + kWalkOff);
    float* Ec = Kc + kC * kLdc;
    float* Wm = Ec + kC * kLdc;                      // [t][kC]
    float* Mm = reinterpret_cast<float*>(sm + L.dz); // [t][kC]
    static_assert(kWalkOff + 2 * kC * kLdc * 4 + kC * kC * 4 <= 7 * kTile, "walk tables in ei .. at");
    static_assert(kC * kC * 4 <= 2 * (D / 64) * kTile, "Mm in the dZ / V tiles");
    constexpr uint32_t kBarRest = 1;                 // named barrier of the six warps
    if (warp != 2 && warp != 3) {
        // dQ^T += K^T (-2 G)^T;  dK^T += Q^T (-2 G)
        if (warp == 0 && ok) {
            tc_fence_after();
            if (elect_one()) {
                const uint32_t kb = smem_u32(ktile(0)), qb = smem_u32(qtile(0)), gb = smem_u32(gg);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16(tmem + kDQ, sdesc(kb + kk * 2048, 2 * kTile, 1024, 2),
                             sdesc(gb + kk * 32, 16, 1024, 2), idMK, 1u);
                    mma_bf16(tmem + kDK, sdesc(qb + kk * 2048, 2 * kTile, 1024, 2),
                             sdesc(gb + kk * 2048, kTile, 1024, 2), idMM, 1u);
                }
                mma_commit(&Y->mma);
            }
            __syncwarp();
        }
        if (ok) ok = wait_bar(Y, &Y->mma, mma_phase++ & 1, status);
        // dQ^T, dK^T (lanes j): transposed through shared memory into dq, dk rows;
        // warps 6-7 take both column halves of lanes 64-127
        if (ok && row < D) {
            tc_fence_after();
            const int j = row;
            const int nq = warp >= 6 ? 4 : 2, tb = warp >= 6 ? 0 : 32 * chalf;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (q < nq) {
                    const int t0 = tb + 16 * q;
                    float rq[16], rk[16];
                    tmem_ld16(tl + kDQ + t0, rq);
                    tmem_ld16(tl + kDK + t0, rk);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        stq[(t0 + e) * D + j] = __float2bfloat16_rn(rq[e]);
                        stk[(t0 + e) * D + j] = __float2bfloat16_rn(rk[e]);
                    }
                }
            }
        }
        named_bar_sync(kBarRest, 192);
        if (ok) {
            const int gt = tid < 64 ? tid : tid - 64;   // 0 .. 191 over the six warps
            constexpr int kRowV = D / 8;                 // 16-byte pieces per row
            for (int x = gt; x < n * kRowV; x += 192) {
                const int t = x / kRowV, p = x % kRowV;
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) + (tok0 + t) * D)[p] =
                    reinterpret_cast<const uint4*>(stq + t * D)[p];
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dk_) + (tok0 + t) * D)[p] =
                    reinterpret_cast<const uint4*>(stk + t * D)[p];
            }
        }
    } else if (ok) {
        // gate gradients.  C[t][s] = theta_s w(s,t) and pm[s] = theta_s m(s,n-1)
        // with m(s,t) = eta_t m(s,t-1), w(s,t) = (1 - alpha_t) w(s,t-1) + m(s,t),
        // w(s,s) = m(s,s) = 1.  One column s per lane, walking the rows: forward
        // for w, m and d theta_s, then backward for the adjoints of w and m, whose
        // products with w(s,t-1) and m(s,t-1), summed over s < t, give
        // d(1 - alpha_t) and d eta_t.
        // (a full chunk takes a copy with its length known at compile time)
        auto walk = [&](auto full) {
            const int nn = decltype(full)::value ? kC : n;
            const int s = (warp - 2) * 32 + lane;
            const float ths = th[s];
            // blocks of 8 rows: the block's loads, then its 8 dependent steps in
            // registers, then its stores (so no load waits behind a store)
            float m = 0.f, w = 0.f, g = 0.f;
    #pragma unroll
            for (int t0 = 0; t0 < kC; t0 += 8) {
                if (t0 < nn) {
                    float dcb[8], wb[8], mb[8], eb[8], kb[8];
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        dcb[u] = dC[(t0 + u) * kLdc + s];   // 0 past the chunk
                        eb[u] = et[t0 + u];
                        kb[u] = 1.f - al[t0 + u];
                    }
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int t = t0 + u;
                        const float e = eb[u], k1 = kb[u];
                        const float mn = t == s ? 1.f : e * m;     // stays 0 before the column starts
                        const float wn = t == s ? 1.f : fmaf(k1, w, mn);
                        const bool live = t < nn;
                        m = live ? mn : m;
                        w = live ? wn : w;
                        wb[u] = w;
                        mb[u] = m;
                        g = fmaf(dcb[u], w, g);
                    }
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        Wm[(t0 + u) * kC + s] = wb[u];
                        Mm[(t0 + u) * kC + s] = mb[u];
                    }
                }
            }
            dth[s] = g - 2.f * dpm[s] * m;
            float dw = s < nn ? ths * dC[(nn - 1) * kLdc + s] : 0.f;
            float dm = s < nn ? ths * (-2.f * dpm[s]) : 0.f;
    #pragma unroll
            for (int tb = kC - 1; tb >= 1; tb -= 8) {      // rows tb, tb-1, .., tb-7 (row 0 skipped)
                if (tb - 7 < nn) {
                    float wm[8], mm[8], dc[8], kc[8], ec[8], eb[8], kb[8];
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int t = tb - u;
                        if (t >= 1) {
                            wm[u] = Wm[(t - 1) * kC + s];
                            mm[u] = Mm[(t - 1) * kC + s];
                            dc[u] = dC[(t - 1) * kLdc + s];
                            eb[u] = et[t];
                            kb[u] = 1.f - al[t];
                        }
                    }
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int t = tb - u;
                        if (t >= 1) {
                            const float e = eb[u], k1 = kb[u];
                            const bool act = t < nn && t > s;
                            const float dm1 = dm + dw;
                            kc[u] = act ? dw * wm[u] : 0.f;
                            ec[u] = act ? dm1 * mm[u] : 0.f;
                            dm = act ? e * dm1 : dm;
                            dw = act ? fmaf(k1, dw, ths * dc[u]) : dw;
                        }
                    }
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int t = tb - u;
                        if (t >= 1) {
                            Kc[t * kLdc + s] = kc[u];
                            Ec[t * kLdc + s] = ec[u];
                        }
                    }
                }
            }
        
        };
        if (n == kC)
            walk(std::true_type{});
        else
            walk(std::false_type{});
    }
    __syncthreads();
    if (ok) {
        // sums over s < t, four threads per row
        const int t = tid >> 2, part = tid & 3;
        float gk = 0.f, ge = 0.f;
        if (t < n) {
            for (int s = part; s < t; s += 4) {
                gk += Kc[t * kLdc + s];
                ge += Ec[t * kLdc + s];
            }
        }
        gk += __shfl_xor_sync(0xffffffffu, gk, 1);
        ge += __shfl_xor_sync(0xffffffffu, ge, 1);
        gk += __shfl_xor_sync(0xffffffffu, gk, 2);
        ge += __shfl_xor_sync(0xffffffffu, ge, 2);
        if (part == 0 && t < n) {
            dkeep[t] += gk;
            deta[t] += ge;
        }
    }
    __syncthreads();
    if (ok && warp == 0) {
        // the prefix recurrences beta_t = (1 - alpha_t) beta_{t-1},
        // P_t = eta_t P_{t-1}, c_t = (1 - alpha_t) c_{t-1} + P_t taken back:
        // their adjoints obey r_t = a_t + g_{t+1} r_{t+1}, solved by a warp scan
        // with two tokens per lane
        const int t0 = 2 * lane, t1 = t0 + 1;
        const float kp0 = t0 < n ? 1.f - al[t0] : 0.f, kp1 = t1 < n ? 1.f - al[t1] : 0.f;
        const float e0 = t0 < n ? et[t0] : 0.f, e1 = t1 < n ? et[t1] : 0.f;
        const float kp_next = __shfl_down_sync(0xffffffffu, kp0, 1);
        const float e_next = __shfl_down_sync(0xffffffffu, e0, 1);
        const float kn1 = lane < 31 ? kp_next : 0.f, en1 = lane < 31 ? e_next : 0.f;
        // P_{t-1} of both tokens (multiplicative prefix scan, 1 past the chunk)
        float pp = (t0 < n ? e0 : 1.f) * (t1 < n ? e1 : 1.f);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, pp, off);
            if (lane >= off) pp *= v;
        }
        float pex = __shfl_up_sync(0xffffffffu, pp, 1);
        if (lane == 0) pex = 1.f;
        const float pprev0 = pex, pprev1 = pex * (t0 < n ? e0 : 1.f);
        auto rev = [&](float a0, float a1, float g0, float g1, float& r0, float& r1) {
            float B = fmaf(g0, a1, a0), A = g0 * g1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float A2 = __shfl_down_sync(0xffffffffu, A, off);
                const float B2 = __shfl_down_sync(0xffffffffu, B, off);
                if (lane + off < 32) {
                    B = fmaf(A, B2, B);
                    A = A * A2;
                }
            }
            r0 = B;
            const float nx = __shfl_down_sync(0xffffffffu, B, 1);
            r1 = fmaf(g1, lane < 31 ? nx : 0.f, a1);
        };
        auto av = [&](const float* v, int t, float last) {
            return t < n ? v[t] + (t == n - 1 ? last : 0.f) : 0.f;
        };
        float db0, db1, dcv0, dcv1, dp0, dp1;
        rev(av(dbeta, t0, scal[0]), av(dbeta, t1, scal[0]), kp1, kn1, db0, db1);
        rev(av(dcc, t0, scal[1]), av(dcc, t1, scal[1]), kp1, kn1, dcv0, dcv1);
        rev(t0 < n ? dcv0 + (t0 == n - 1 ? scal[2] : 0.f) : 0.f,
            t1 < n ? dcv1 + (t1 == n - 1 ? scal[2] : 0.f) : 0.f, e1, en1, dp0, dp1);
        if (t0 < n) {
            dkeep[t0] += dcv0 * (t0 > 0 ? cc[t0 - 1] : 0.f) + db0 * (t0 > 0 ? beta[t0 - 1] : 1.f);
            deta[t0] += dp0 * pprev0;
        }
        if (t1 < n) {
            dkeep[t1] += dcv1 * cc[t0] + db1 * beta[t0];
            deta[t1] += dp1 * pprev1;
        }
    }
    __syncthreads();
    if (ok) {
        for (int t = tid; t < n; t += kThreads) {
            a.dtheta[tok0 + t] = dth[t];
            if (a.deta) a.deta[tok0 + t] = deta[t];
            if (a.dalpha) a.dalpha[tok0 + t] = -dkeep[t];
        }
    }
    if (tid == 0 && !ok) {
        // copies in flight before the kernel's shared memory goes
        const long long t0 = clock64();
        while (!mbar_try_wait(&Y->full, 0) && clock64() - t0 < Y->limit) {
        }
        if (halves_issued > 0) {
            const long long t1 = clock64();
            while (!mbar_try_wait(&Y->mfull, (halves_issued - 1) & 1) && clock64() - t1 < Y->limit) {
            }
        }
    }
    if (warp == 0) {
        // every MMA (also after an abort) completes before TMEM is released
        if (elect_one()) mma_commit(&Y->mma);
        __syncwarp();
        const long long t0 = clock64();
        if (lane == 0)
            while (!mbar_try_wait(&Y->mma, mma_phase & 1) && clock64() - t0 < Y->limit) {
            }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ chain
//
// The adjoint of the state at every chunk end, chunks in reverse, for a slice
// of 16 rows i of (dW, dS) (rows evolve independently).  Per chunk, with the
// masked score tile A~ and the coefficient vectors (beta, c, C[n-1][.], pm,
// beta_n, c_n, P_n) that the forward scan left in the workspace:
//   dWK = K dW^T, dSK = K dS^T                       [K; .] [dW; dS]^T  (MMA)
//   de  = -2 (A~^T dZ + C_n o dWK + pm o dSK)         A~^T dZ             (MMA)
//   dW <- beta_n dW + (Q^T (beta o dZ) + K^T de)^T,    (Q^T, K^T MN-major; MMA)
//   dS <- c_n dW + P_n dS + (Q^T (c o dZ))^T
// A~^T dZ and Q^T [beta o dZ | c o dZ] depend on the inputs alone, so they are
// computed one chunk ahead into alternating tensor-memory buffers; the serial
// path per chunk is K [dW; dS]^T -> de -> K^T de -> the update.  These thin
// products run at about a hundred cycles per 16-deep MMA step whatever their
// width, so the chunk's step count (8 + 4 + 4 + 4) sets its time.
//
// Roles (320 threads):
//   warps 0-3  state: thread j holds column j of the slice's 16 rows of dW and
//              dS in fp32 registers, applies the update and writes the bf16
//              copy [dW; dS]^T for the next chunk's first product; warps 0-1
//              (TMEM lanes 0-63 = tokens s) also form de.
//   warps 4-7  the next chunk's dZ slice and [beta dZ | c dZ] tiles.
//   warp 8     issues every MMA, ordered so that the input-only products of
//              a chunk run while the state warps work on the previous one.
//   warp 9     TMA loads into three input stages: a stage is refilled three
//              chunks ahead once the state warps release it after its update.
// Hand-offs between roles are named barriers that both sides sync on (state ->
// issuer: the adjoint copy; de warps -> issuer: the de tile; tile warps ->
// issuer: the dZ tiles) and MMA-completion mbarriers the other way; stage
// release and refill are mbarriers.  Every wait on an mbarrier is bounded;
// after a timeout every role runs out its loop doing no work, and since every
// role passes the same named barriers in the same order, they stay in
// lockstep.

constexpr int kSl = 16;                                          // rows of the slice
constexpr int kNS = 3;                                           // input stages
constexpr int kChainThreads = 320;
constexpr uint32_t kVecSlot = (kCoefVecBytes + 63) / 64 * 64;
constexpr uint32_t kBarWs = 1, kBarDe = 2, kBarTiles = 3;        // named barriers

struct ChainLayout {
    uint32_t kq, at, dzs, vec, dzt, bct, det, ws, total;
};

__host__ __device__ constexpr ChainLayout chain_layout(int D) {
    ChainLayout L{};
    uint32_t o = 0;
    const uint32_t NH = D / 64;
    L.kq = o;  o += kNS * NH * 2 * kTile;   // stages of [K_h][Q_h]
    L.at = o;  o += kNS * kTile;            // stages of A~ [t][s] (swizzled, as stored)
    L.dzs = o; o += kNS * kC * kSl * 2;     // stages of the dZ slice (64 x 16 bf16)
    L.vec = o; o += kNS * kVecSlot;         // stages of the coefficient vectors
    o = (o + 1023) / 1024 * 1024;
    L.dzt = o; o += 2 * kTile;              // dZ slice [t][i] (16 of 64 columns), 2 buffers
    L.bct = o; o += 2 * kTile;              // [beta_t dZ | c_t dZ] [t][32 columns], 2 buffers
    L.det = o; o += kTile;                  // de [s][i]
    L.ws = o;  o += (uint32_t)D * 128;      // [dW; dS]^T bf16 [j][i'] (32 of 64 columns)
    L.total = o + 128;                      // barriers
    return L;
}

struct ChainSync {
    uint64_t full[kNS], sfree[kNS], mma1, mma3;
    long long limit;
    int abort;
    uint32_t tmem;
};

template <int D>
__global__ void __launch_bounds__(kChainThreads, 1)
bwd_chain_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap zmap, const BwdArgs a, float* ws,
                    size_t off_adj, const uint8_t* coef, const uint8_t* tiles, size_t off_part,
                    int nch) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    constexpr ChainLayout L = chain_layout(D);
    constexpr int NH = D / 64, KS = D / 16;
    static_assert(sizeof(ChainSync) <= 128, "chain barriers");
    ChainSync* Y = reinterpret_cast<ChainSync*>(sm + L.total - 128);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsl = D / kSl;
    const int seq = blockIdx.x / nsl, r0 = (blockIdx.x % nsl) * kSl;
    const int T = a.T;
    const size_t sd = (size_t)D * D;
    int* status = a.status;

    auto kt = [&](int st, int h) { return sm + L.kq + (st * NH + h) * 2 * kTile; };
    auto qt = [&](int st, int h) { return kt(st, h) + kTile; };
    auto atb = [&](int st) { return sm + L.at + st * kTile; };
    auto dzs = [&](int st) { return sm + L.dzs + st * kC * kSl * 2; };
    auto vecb = [&](int st) { return reinterpret_cast<const float*>(sm + L.vec + st * kVecSlot); };
    auto dzt = [&](int b) { return sm + L.dzt + b * kTile; };
    auto bct = [&](int b) { return sm + L.bct + b * kTile; };
    uint8_t* det = sm + L.det;
    uint8_t* wsm = sm + L.ws;
    auto chunk_len = [&](int k) { return min(kC, T - (nch - 1 - k) * kC); };

    if (tid == 0) {
        for (int st = 0; st < kNS; ++st) {
            mbar_init(&Y->full[st], 1);
            mbar_init(&Y->sfree[st], 4);   // one arrival per state warp
        }
        mbar_init(&Y->mma1, 1);
        mbar_init(&Y->mma3, 1);
        Y->limit = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;
        Y->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&Y->tmem, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = Y->tmem;
    // TMEM columns: [K; Q][dW; dS]^T, then A~^T dZ and the Q^T . dZ pair per buffer
    constexpr uint32_t kAc1 = 0;
    auto kAc2 = [](int b) { return 32u + 16u * (uint32_t)b; };
    auto kAc3 = [](int b) { return 64u + 32u * (uint32_t)b; };
    bool ok = true;

    if (warp < 4) {
        // ------------------------------------------------------------ state
        const uint32_t tl = tmem + ((uint32_t)warp * 32 << 16);
        const int j = tid;
        const bool own = j < D;
        float dw[kSl], dsv[kSl];
#pragma unroll
        for (int i = 0; i < kSl; ++i) {
            const size_t g = (size_t)seq * sd + (size_t)(r0 + i) * D + j;
            dw[i] = (own && a.dW) ? a.dW[g] : 0.f;
            dsv[i] = (own && a.dS) ? a.dS[g] : 0.f;
        }
        auto write_ws = [&]() {
            if (!own) return;
            *reinterpret_cast<uint4*>(wsm + swz(j, 0)) = pack8(dw);
            *reinterpret_cast<uint4*>(wsm + swz(j, 1)) = pack8(dw + 8);
            *reinterpret_cast<uint4*>(wsm + swz(j, 2)) = pack8(dsv);
            *reinterpret_cast<uint4*>(wsm + swz(j, 3)) = pack8(dsv + 8);
        };
        write_ws();
        fence_proxy_async_smem();
        named_bar_sync(kBarWs, 160);
        for (int k = 0; k < nch; ++k) {
            const int c = nch - 1 - k, st = k % kNS, b = k & 1;
            const int n = chunk_len(k);
            const float* vclast = vecb(st) + kCoefCend / 4;
            const float* vpm = vecb(st) + kCoefPend / 4;
            const float* vscal = vecb(st) + kCoefScal / 4;   // beta_n, c_n, P_n, n
            // the chunk's coefficient vectors have landed (long since, as a rule)
            if (ok) ok = wait_flag(&Y->abort, Y->limit, &Y->full[st], (k / kNS) & 1, status);
            // this chunk's end adjoint, for the local pass
            if (own && ok) {
                __nv_bfloat16* adj = reinterpret_cast<__nv_bfloat16*>(ws + off_adj) +
                                     ((size_t)seq * nch + c) * 2 * sd;
#pragma unroll
                for (int i = 0; i < kSl; ++i) {
                    adj[(size_t)(r0 + i) * D + j] = __float2bfloat16_rn(dw[i]);
                    adj[sd + (size_t)(r0 + i) * D + j] = __float2bfloat16_rn(dsv[i]);
                }
            }
            if (warp < 2) {
                // de[s][i] = -2 ((A~^T dZ)[s][i] + C_n[s] dWK + pm[s] dSK), s < n
                if (ok) ok = wait_flag(&Y->abort, Y->limit, &Y->mma1, k & 1, status);
                if (ok) {
                    tc_fence_after();
                    const int sidx = j;
                    float gw[16], gs[16], ad[16], de[16];
                    tmem_ld16(tl + kAc1, gw);
                    tmem_ld16(tl + kAc1 + 16, gs);
                    tmem_ld16(tl + kAc2(b), ad);
                    tmem_wait_ld();
                    const float cl = vclast[sidx], pmv = vpm[sidx];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        de[e] = sidx < n ? -2.f * (ad[e] + cl * gw[e] + pmv * gs[e]) : 0.f;
                    *reinterpret_cast<uint4*>(det + swz(sidx, 0)) = pack8(de);
                    *reinterpret_cast<uint4*>(det + swz(sidx, 1)) = pack8(de + 8);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(kBarDe, 96);
            }
            // dW <- beta_n dW + .,  dS <- c_n dW + P_n dS + .  (column j)
            if (ok) ok = wait_flag(&Y->abort, Y->limit, &Y->mma3, k & 1, status);
            if (ok) {
                tc_fence_after();
                float uw[16], us[16];
                tmem_ld16(tl + kAc3(b), uw);
                tmem_ld16(tl + kAc3(b) + 16, us);
                tmem_wait_ld();
                const float bn = vscal[0], cn = vscal[1], Pn = vscal[2];
                if (own) {
#pragma unroll
                    for (int i = 0; i < kSl; ++i) {
                        const float w = dw[i];
                        dw[i] = fmaf(bn, w, uw[i]);
                        dsv[i] = fmaf(cn, w, fmaf(Pn, dsv[i], us[i]));
                    }
                }
                write_ws();
            }
            if (k + 1 < nch) {
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(kBarWs, 160);
            }
            // this warp is done with the chunk's stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&Y->sfree[st]);
        }
        // adjoint of the initial state: per sequence, or a per-sequence partial
        // that a reduction sums over the batch when W0 / S0 are shared
        if (own && ok) {
            float* oW;
            float* oS;
            size_t base;
            if (a.shared) {
                oW = ws + off_part;
                oS = oW + sd;
                base = (size_t)seq * 2 * sd;
            } else {
                oW = a.dW0;
                oS = a.dS0;
                base = (size_t)seq * sd;
            }
#pragma unroll
            for (int i = 0; i < kSl; ++i) {
                const size_t g = base + (size_t)(r0 + i) * D + j;
                oW[g] = dw[i];
                if (oS) oS[g] = dsv[i];
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ tiles
        const int p = tid - 128;
        for (int k = 0; k < nch; ++k) {
            const int st = k % kNS, b = k & 1;
            const int n = chunk_len(k);
            // buffer b was last read by the chunk k-2 products, which complete
            // before the first product of chunk k-1
            if (k >= 1 && ok) ok = wait_flag(&Y->abort, Y->limit, &Y->mma1, (k - 1) & 1, status);
            if (ok) ok = wait_flag(&Y->abort, Y->limit, &Y->full[st], (k / kNS) & 1, status);
            if (ok) {
                const float* vbeta = vecb(st) + kCoefBeta / 4;
                const float* vc = vecb(st) + kCoefC / 4;
                const int t = p >> 1, c8 = p & 1;     // 64 tokens x 2 eight-column groups
                float z[8], zb[8], zc[8];
                unpack8(*reinterpret_cast<const uint4*>(dzs(st) + t * kSl * 2 + 16 * c8), z);
                const float bt = t < n ? vbeta[t] : 0.f, ct = t < n ? vc[t] : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    zb[e] = bt * z[e];
                    zc[e] = ct * z[e];
                }
                *reinterpret_cast<uint4*>(dzt(b) + swz(t, c8)) = pack8(z);
                *reinterpret_cast<uint4*>(bct(b) + swz(t, c8)) = pack8(zb);
                *reinterpret_cast<uint4*>(bct(b) + swz(t, 2 + c8)) = pack8(zc);
            }
            fence_proxy_async_smem();
            named_bar_sync(kBarTiles, 160);
        }
    } else if (warp == 8) {
        // ----------------------------------------------------------- issuer
        constexpr uint32_t id1 = idesc_bf16_f32(128, 32, 0, 1);   // [K; Q] [dW; dS]^T
        constexpr uint32_t id16 = idesc_bf16_f32(128, 16, 1, 1);  // MN-major A and B, N = 16
        constexpr uint32_t id32 = idesc_bf16_f32(128, 32, 1, 1);  // MN-major A and B, N = 32
        auto live = [&]() { return ok && !*(volatile int*)&Y->abort; };
        // A~^T dZ of chunk k (for its de)
        auto issue_scores = [&](int k) {
            const int st = k % kNS, b = k & 1;
            tc_fence_after();
            if (elect_one()) {
                const uint32_t aa = smem_u32(atb(st)), za = smem_u32(dzt(b));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kAc2(b), sdesc(aa + kk * 2048, kTile, 1024, 2),
                             sdesc(za + kk * 2048, kTile, 1024, 2), id16, kk > 0);
            }
            __syncwarp();
        };
        int n3 = 0;   // commits to mma3
        named_bar_sync(kBarTiles, 160);
        if (live()) ok = wait_flag(&Y->abort, Y->limit, &Y->full[0], 0, status);
        if (live()) issue_scores(0);
        for (int k = 0; k < nch; ++k) {
            const int st = k % kNS, b = k & 1;
            named_bar_sync(kBarWs, 160);
            ok = live();
            if (ok) ok = wait_flag(&Y->abort, Y->limit, &Y->full[st], (k / kNS) & 1, status);
            if (ok) {
                tc_fence_after();
                if (elect_one()) {
                    // [K; Q] [dW; dS]^T (lanes 0-63: dWK, dSK)
                    const uint32_t wsa = smem_u32(wsm);
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        const uint32_t abase = smem_u32(kt(st, kk >> 2)) + (kk & 3) * 32;
                        mma_bf16(tmem + kAc1, sdesc(abase, 16, 1024, 2),
                                 sdesc(wsa + kk * 2048, 8192, 1024, 2), id1, kk > 0);
                    }
                    mma_commit(&Y->mma1);
                    // Q^T [beta dZ | c dZ], while the de warps work
                    const uint32_t qa = smem_u32(qt(st, 0)), bcb = smem_u32(bct(b));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + kAc3(b), sdesc(qa + kk * 2048, 2 * kTile, 1024, 2),
                                 sdesc(bcb + kk * 2048, kTile, 1024, 2), id32, kk > 0);
                }
                __syncwarp();
            }
            named_bar_sync(kBarDe, 96);
            ok = live();
            // + K^T de onto Q^T (beta dZ)
            if (ok) {
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t ka = smem_u32(kt(st, 0)), deb = smem_u32(det);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + kAc3(b), sdesc(ka + kk * 2048, 2 * kTile, 1024, 2),
                                 sdesc(deb + kk * 2048, kTile, 1024, 2), id16, 1u);
                    mma_commit(&Y->mma3);
                }
                __syncwarp();
                ++n3;
            }
            if (k + 1 < nch) {
                // the next chunk's scores, while the state warps update
                named_bar_sync(kBarTiles, 160);
                ok = live();
                const int st1 = (k + 1) % kNS;
                if (ok) ok = wait_flag(&Y->abort, Y->limit, &Y->full[st1], ((k + 1) / kNS) & 1, status);
                if (ok) issue_scores(k + 1);
            }
        }
        // one more commit on mma3 completes its phase n3 once every MMA this
        // thread issued has completed (before tensor memory goes)
        if (elect_one()) mma_commit(&Y->mma3);
        __syncwarp();
        if (lane == 0) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&Y->mma3, n3 & 1) && clock64() - t0 < Y->limit) {
            }
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------------- loader
        auto issue_loads = [&](int k) {
            const int c = nch - 1 - k, st = k % kNS;
            // (a.debug_stall = k + 1: the test hook announces 16 bytes more than
            // it copies, so this stage's barrier never completes)
            mbar_expect_tx(&Y->full[st], 2 * NH * kTile + kTile + kC * kSl * 2 + kCoefVecBytes +
                                             (k + 1 == a.debug_stall ? 16u : 0u));
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                tma_load_3d(kt(st, h), &kmap, &Y->full[st], 64 * h, c * kC, seq);
                tma_load_3d(qt(st, h), &qmap, &Y->full[st], 64 * h, c * kC, seq);
            }
            tma_load_3d(dzs(st), &zmap, &Y->full[st], r0, c * kC, seq);
            const size_t rec = (size_t)seq * nch + c;
            bulk_load(atb(st), tiles + rec * kTile, kTile, &Y->full[st]);
            bulk_load(sm + L.vec + st * kVecSlot, coef + rec * kCoefRecBytes + kCoefVec,
                      kCoefVecBytes, &Y->full[st]);
        };
        int issued = min(kNS, nch);
        if (lane == 0)
            for (int k = 0; k < issued; ++k) issue_loads(k);
        __syncwarp();
        for (int k = 0; k + kNS < nch; ++k) {
            // chunk k's stage, once the state warps have updated with it
            if (ok) ok = wait_flag(&Y->abort, Y->limit, &Y->sfree[k % kNS], (k / kNS) & 1, status);
            if (!ok) break;
            if (lane == 0) issue_loads(k + kNS);
            __syncwarp();
            issued = k + kNS + 1;
        }
        // every copy lands before shared memory goes
        if (lane == 0) {
            for (int k = max(0, issued - kNS); k < issued; ++k) {
                const long long t0 = clock64();
                while (!mbar_try_wait(&Y->full[k % kNS], (k / kNS) & 1) && clock64() - t0 < Y->limit) {
                }
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace

bool bwd_local_tc_supported(const BwdArgs& a) {
    // matrices of the checkpoints as the 32-bit third coordinate of a TMA tile
    const long long nmat = (long long)a.B * a.H * ((a.T + kC - 1) / kC) * 2;
    return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128) && a.chunk == kC && a.T >= 1 &&
           nmat < (1LL << 31);
}

cudaError_t bwd_chain_tc_launch(const BwdArgs& a, float* ws, size_t off_adj, const void* coef,
                                const void* tiles, size_t off_part, cudaStream_t s) {
    const int D = a.dk, BH = a.B * a.H;
    const int nch = (a.T + kC - 1) / kC;
    CUtensorMap qm, km, zm;
    if (!make_token_tile_map(&qm, a.q, BH, a.T, D, 64, true) ||
        !make_token_tile_map(&km, a.k, BH, a.T, D, 64, true) ||
        !make_token_tile_map(&zm, a.dz, BH, a.T, D, kSl, false))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(BH * (D / kSl)));
    if (D == 128) {
        const size_t smem = chain_layout(128).total + 1024;
        cudaError_t e = cudaFuncSetAttribute(bwd_chain_tc_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        bwd_chain_tc_kernel<128><<<grid, kChainThreads, smem, s>>>(qm, km, zm, a, ws, off_adj,
                                                              static_cast<const uint8_t*>(coef),
                                                              static_cast<const uint8_t*>(tiles),
                                                              off_part, nch);
    } else {
        const size_t smem = chain_layout(64).total + 1024;
        cudaError_t e = cudaFuncSetAttribute(bwd_chain_tc_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        bwd_chain_tc_kernel<64><<<grid, kChainThreads, smem, s>>>(qm, km, zm, a, ws, off_adj,
                                                             static_cast<const uint8_t*>(coef),
                                                             static_cast<const uint8_t*>(tiles),
                                                             off_part, nch);
    }
    return cudaGetLastError();
}

cudaError_t bwd_local_tc_launch(const BwdArgs& a, const void* ckpt, const void* adj,
                                const void* coef, cudaStream_t s) {
    const int D = a.dk, BH = a.B * a.H;
    const int nch = (a.T + kC - 1) / kC;
    CUtensorMap qm, km, zm, vm, cm, am;
    // the checkpoints and adjoints as (64 columns j) x (64 rows i) tiles of the
    // matrices [seq][chunk][W | S]
    const int nmat = BH * nch * 2;
    if (!make_token_tile_map(&qm, a.q, BH, a.T, D, 64, true) ||
        !make_token_tile_map(&km, a.k, BH, a.T, D, 64, true) ||
        !make_token_tile_map(&zm, a.dz, BH, a.T, D, 64, true) ||
        !make_token_tile_map(&vm, a.v, BH, a.T, D, 64, true) ||
        !make_token_tile_map(&cm, ckpt, nmat, D, D, 64, true) ||
        !make_token_tile_map(&am, adj, nmat, D, D, 64, true))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(BH * nch));
    const uint8_t* cf = static_cast<const uint8_t*>(coef);
    if (D == 128) {
        const size_t smem = make_layout(128).total + 1024;
        cudaError_t e = cudaFuncSetAttribute(bwd_local_tc_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        bwd_local_tc_kernel<128><<<grid, kThreads, smem, s>>>(qm, km, zm, vm, cm, am, a, cf, nch);
    } else {
        const size_t smem = make_layout(64).total + 1024;
        cudaError_t e = cudaFuncSetAttribute(bwd_local_tc_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        bwd_local_tc_kernel<64><<<grid, kThreads, smem, s>>>(qm, km, zm, vm, cm, am, a, cf, nch);
    }
    return cudaGetLastError();
}

}  // namespace ttm
