// Tensor-core (tcgen05 + TMA + 2-CTA cluster) kernel of the 2-layer MLP memory
// scan: f(x) = W2 GELU(W1 x), W1 [256 x 64], W2 [64 x 256], chunks of 16
// tokens, bf16 inputs, fp32 state.
//
// Method ("论文速览 | Titans" §4.3-§4.5 for the momentum / forgetting unrolling;
// "TTT layers 与 fast weights" §1.1 eqs (7)-(9) for the matrix form of one
// chunk), with the chunk-start state (W1, S1, W2, S2), the chunk's rows K, Q,
// V and the gate coefficients beta_t, c_t, P_t, C[t][s], Pm[t][s] of the
// chunk (defined in scan_simt.cu):
//
//   H  = W1 K^T,  A = GELU(H),  E = 2 (W2 A - V^T)        errors at the chunk start
//   D1 = (W2^T E) o GELU'(H)                              hidden-side error
//   Hq = beta_t W1 q_t + c_t S1 q_t - sum_{s<=t} C[t][s] (q_t.k_s) D1_s
//   z_t = beta_t W2 GELU(Hq)_t + c_t S2 GELU(Hq)_t
//         - sum_{s<=t} C[t][s] (GELU(Hq)_t . A_s) E_s
//   W1' = beta_n W1 + c_n S1 - D1 diag(C[n]) K,  S1' = P_n S1 - D1 diag(Pm[n]) K
//   W2' = beta_n W2 + c_n S2 - E diag(C[n]) A^T,  S2' = P_n S2 - E diag(Pm[n]) A^T
//
// Decomposition.  The fp32 state of one sequence (4 x 64 KB) does not fit one
// SM, so a cluster of two CTAs runs each sequence and CTA r owns the hidden
// units 128 r .. 128 r + 127: its rows of W1 / S1 and its columns of W2 / S2.
// Every product then stays local except Y = W2 A and the read-out W2 GELU(Hq),
// whose sums over the hidden units need the peer's half: the partial Y (4 KB)
// crosses the cluster once per chunk through distributed shared memory
// (st.async with transaction-count completion), and each CTA finishes half of
// the chunk's outputs from both partial read-outs.
//
// State layout.  The fp32 state lives in tensor memory, lane = hidden unit,
// columns W1 [j], S1 [j], W2^T [i], S2^T [i]; the update MMAs accumulate into
// it directly (after an elementwise pass applies beta_n, c_n, P_n).  bf16
// copies for the MMAs: W1, S1 as tensor-memory A operands (fast to issue), W2^T
// and S2^T in shared memory (needed as MN-major operands with M = d).
//
// Roles (448 threads):
//   warps 0-3   chain: H -> GELU -> Y -> exchange -> E -> W2^T E -> D1, then
//               issue the read pre-activations Hq and the W1 / S1 update; thread
//               = hidden unit (tensor-memory lane).  Warp 0 issues the MMAs.
//   warps 4-7   state: bf16 copies of the state, the elementwise beta / c / P
//               pass, initial load and final store.
//   warps 8-11  read side: GELU(Hq), scores GELU(Hq) A^T, read-out MMAs and the
//               outputs z (half the tokens of each chunk per CTA).
//   warp 12     coefficients from the gates, scaled copies of K and Q, the
//               Q K^T scores.
//   warp 13     producer: TMA loads of K, V, Q.
//
// Every wait is bounded.  A wait that gives up sets the device status word to
// TTM_ERR_TIMEOUT and raises an abort flag in both CTAs of the cluster; every
// role then only runs out its loop (named barriers stay balanced), MMAs and
// copies in flight are drained, tensor memory is freed and the kernel returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "../../include/ttm.h"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace ttm {
namespace {

using namespace tc;

constexpr int kC = 16;        // tokens per chunk
constexpr int kD = 64;        // width of keys, values and outputs
constexpr int kHid = 256;     // hidden units
constexpr int kHalf = 128;    // hidden units per CTA
constexpr int kThreads = 448;
constexpr int kNS = 3;        // input pipeline stages
constexpr uint32_t kTmemCols = 512;

// Tensor-memory columns.  fp32 state (lane = hidden unit of this CTA):
constexpr uint32_t TW1 = 0, TS1 = 64, TW2 = 128, TS2 = 192;
// accumulators
constexpr uint32_t TH = 256;    // H = W1 K^T                  [u][t]
constexpr uint32_t TBK = 272;   // W2^T E                      [u][t]
constexpr uint32_t TY = 288;    // partial W2 A (M = 64)       [i][t]
constexpr uint32_t THQ = 304;   // read pre-activations        [u][t]
constexpr uint32_t TZS = 320;   // [W2; S2] GELU(Hq) (M = 128)  [i | 64 + i][t]
constexpr uint32_t TZC = 336;   // read correction (M = 64)    [i][t]
constexpr uint32_t TSC = 352;   // GELU(Hq) A^T (M = 64)       [t][s]
constexpr uint32_t TQK = 368;   // Q K^T (M = 64)              [t][s]
// bf16 A operands (two values per column)
constexpr uint32_t TW1B = 384;  // W1 [u][j]
constexpr uint32_t TS1B = 416;  // S1 [u][j]
constexpr uint32_t TDL = 448;   // D1 [u][s]
constexpr uint32_t TAK = 456;   // A  [u][s]

// Shared-memory map (offsets from a 1024-byte aligned base).  All operand
// tiles are rows of 128 bytes in the 128-byte swizzle pattern.
constexpr uint32_t kStageBytes = 12288;
constexpr uint32_t kStK = 0;       // K [16][64]
constexpr uint32_t kStV = 2048;    // V [16][64]
constexpr uint32_t kStQ = 4096;    // Q [64][64], rows 16..63 stay zero (M = 64 operand)
constexpr uint32_t OFF_W2B = kNS * kStageBytes;   // 2 slots x (W2^T [128][64], S2^T [128][64])
constexpr uint32_t kW2BSlot = 32768;
constexpr uint32_t OFF_AQ = OFF_W2B + 2 * kW2BSlot;   // GELU(Hq) [t][u]: 2 atoms x [64][64], rows 16..63 zero
constexpr uint32_t OFF_AK = OFF_AQ + 16384;          // 2 slots x A [t][u]: 2 atoms x [16][64]
constexpr uint32_t OFF_ES = OFF_AK + 8192;           // 2 slots x E [t][i]
constexpr uint32_t OFF_EC = OFF_ES + 4096;           // [-C_n E | -Pm_n E] [t][i], 2 atoms
constexpr uint32_t OFF_KC = OFF_EC + 4096;           // 2 slots x [-C_n K | -Pm_n K] [t][j], 2 atoms
constexpr uint32_t OFF_QB = OFF_KC + 8192;           // 2 slots x (beta Q, c Q, M1) [t][.]
constexpr uint32_t kQBSlot = 6144;
constexpr uint32_t OFF_M2 = OFF_QB + 2 * kQBSlot;    // read correction weights [t][s]
constexpr uint32_t OFF_YR = OFF_M2 + 2048;           // 2 slots x peer's partial Y [i][16] fp32
constexpr uint32_t OFF_ZP = OFF_YR + 8192;           // 3 read-out parts [t][64] fp32
constexpr uint32_t OFF_ZR = OFF_ZP + 12288;          // 2 slots x peer's read-out [8][64] fp32
constexpr uint32_t OFF_REC = OFF_ZR + 4096;          // 2 slots x coefficient record
constexpr uint32_t kRecSlot = 1536;
constexpr uint32_t kSmemBytes = OFF_REC + 2 * kRecSlot;

// coefficient record
constexpr uint32_t REC_C = 0;        // C[t][s] fp32, row-major 16 x 16
constexpr uint32_t REC_BETA = 1024;  // beta_t
constexpr uint32_t REC_CV = 1088;    // c_t
constexpr uint32_t REC_CN = 1152;    // C[n-1][s]
constexpr uint32_t REC_PN = 1216;    // Pm[n-1][s]
constexpr uint32_t REC_SCAL = 1280;  // beta_{n-1}, c_{n-1}, P_{n-1}, n

struct Bars {
    uint64_t full[kNS], empty[kNS];
    uint64_t prep_ready[2], prep_free[2], rd_done[2], w2b_ready[2], ybar[2], zbar[2];
    uint64_t init_done, w1_copied, scaled1, scaled2;
    uint64_t h_done, y_done, bk_done, u1_done, hq_done, hq_free, sc_done, z_done, qk_done;
    uint64_t drain[3];
    uint32_t tmem_base;
    int abort;
};

constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

// ------------------------------------------------------------ cluster helpers

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// 16-byte store into the peer CTA's shared memory that counts its bytes on
// the peer's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(addr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
        : "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok = 0;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// ------------------------------------------------------------ tensor memory


// ------------------------------------------------------------------- waits

__device__ __forceinline__ void raise_abort(Bars* B, int* status, uint32_t peer) {
    *(volatile int*)&B->abort = 1;
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_addr(&B->abort, peer)), "r"(1)
                 : "memory");
    atomicExch(status, TTM_ERR_TIMEOUT);
}

// Bounded wait; false once it gave up or another role (of either CTA) aborted.
template <bool kCluster>
__device__ __forceinline__ bool wait_bar(Bars* B, uint64_t* bar, uint32_t parity, int* status,
                                         uint32_t peer) {
    if (kCluster ? try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    uint32_t polls = 0;
    while (!(kCluster ? try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))) {
        if ((++polls & 63u) == 0) {
            if (*(volatile int*)&B->abort) return false;
            if (clock64() - t0 > kWaitCycles) {
                raise_abort(B, status, peer);
                return false;
            }
        }
    }
    return true;
}

// Warp-uniform wait: one lane's timeout never splits the warp before a
// .sync.aligned instruction.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_all(Bars* B, uint64_t* bar, uint32_t parity, int* status,
                                         uint32_t peer) {
    if (__all_sync(0xffffffffu, kCluster ? try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)))
        return true;
    return __all_sync(0xffffffffu, wait_bar<kCluster>(B, bar, parity, status, peer));
}

// Wait used while draining: ignores the abort flag, gives up after the limit.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) break;
}

// ------------------------------------------------------------- small helpers

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_bf16(uint8_t* p, float x) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float ld_bf16(const uint8_t* p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

// 16 consecutive floats (16-byte aligned) into registers.
__device__ __forceinline__ void ld_f32x16(const uint8_t* p, float (&r)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 f = reinterpret_cast<const float4*>(p)[j];
        r[4 * j] = f.x;
        r[4 * j + 1] = f.y;
        r[4 * j + 2] = f.z;
        r[4 * j + 3] = f.w;
    }
}

// 8 consecutive bf16 values of row `row` from column `col` (multiple of 8) of
// a 128-byte-swizzled tile.
__device__ __forceinline__ void st_chunk(uint8_t* tile, int row, int col, const float* x) {
    uint4 v;
    v.x = pack_bf16(x[0], x[1]);
    v.y = pack_bf16(x[2], x[3]);
    v.z = pack_bf16(x[4], x[5]);
    v.w = pack_bf16(x[6], x[7]);
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, col)) = v;
}

// 16-byte chunk of 8 bf16 values scaled by s.
__device__ __forceinline__ uint4 scale_chunk(uint4 v, float s) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w[i]);
        const float2 f = __bfloat1622float2(h);
        w[i] = pack_bf16(f.x * s, f.y * s);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

// GELU(x) = x Phi(x) and GELU'(x) = Phi(x) + x phi(x) of the erf-based GELU.
// Phi comes from erf by Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26: for z >= 0, erf(z) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5))))
// e^{-z^2} with t = 1 / (1 + p z), |error| <= 1.5e-7.  It is branch-free, so the
// evaluations of one epilogue overlap in the pipeline, and e^{-x^2/2} serves
// both Phi and the density phi.
__device__ __forceinline__ void gelu_parts(float x, float& Phi, float& ez) {
    const float z = fabsf(x) * 0.70710678118654752f;
    const float t = __fdividef(1.f, fmaf(0.3275911f, z, 1.f));
    float poly = fmaf(t, 1.061405429f, -1.453152027f);
    poly = fmaf(t, poly, 1.421413741f);
    poly = fmaf(t, poly, -0.284496736f);
    poly = fmaf(t, poly, 0.254829592f);
    poly *= t;
    ez = __expf(-z * z);                  // e^{-x^2 / 2}
    const float q = 0.5f * poly * ez;     // Phi(-|x|)
    Phi = x >= 0.f ? 1.f - q : q;
}

__device__ __forceinline__ float gelu(float x) {
    float P, e;
    gelu_parts(x, P, e);
    return x * P;
}

__device__ __forceinline__ void gelu_and_grad(float x, float& g, float& dg) {
    float P, e;
    gelu_parts(x, P, e);
    g = x * P;
    dg = fmaf(x * 0.3989422804014327f, e, P);
}

namespace {

// fp32 columns [src, src + 64) of this warp's 32 lanes -> bf16 pairs in
// columns [dst, dst + 32).
__device__ __forceinline__ void tmem_to_bf16(uint32_t lanebase, uint32_t src, uint32_t dst) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float r[32];
        tmem_ld16(lanebase + src + 32 * h, *reinterpret_cast<float(*)[16]>(r));
        tmem_ld16(lanebase + src + 32 * h + 16, *reinterpret_cast<float(*)[16]>(r + 16));
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            uint32_t p[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) p[j] = pack_bf16(r[16 * g + 2 * j], r[16 * g + 2 * j + 1]);
            tmem_st8(lanebase + dst + 16 * h + 8 * g, p);
        }
    }
    tmem_wait_st();
}

// Inclusive scan of affine maps x -> A x + B along lanes (later lanes outside).
__device__ __forceinline__ void scan_affine(float& A, float& Bv, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float A2 = __shfl_up_sync(0xffffffffu, A, off);
        const float B2 = __shfl_up_sync(0xffffffffu, Bv, off);
        if (lane >= off) {
            Bv = A * B2 + Bv;
            A = A * A2;
        }
    }
}

// --------------------------------------------------------------- the kernel

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mlp_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
              const __grid_constant__ CUtensorMap vmap, const MlpArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ Bars bars;
    Bars* B = &bars;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int seq = blockIdx.x >> 1;
    const int bb = seq / a.H, hh = seq % a.H;
    const int T = a.T;
    const int nch = (T + kC - 1) / kC;
    int* status = a.status;

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&B->full[s], 1);
            mbar_init(&B->empty[s], 2);      // coefficient warp + chain
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&B->prep_ready[b], 1);
            mbar_init(&B->prep_free[b], 2);  // chain + read side
            mbar_init(&B->rd_done[b], 1);
            mbar_init(&B->w2b_ready[b], 1);
            mbar_init(&B->ybar[b], 1);
            mbar_init(&B->zbar[b], 1);
        }
        uint64_t* ones[] = {&B->init_done, &B->w1_copied, &B->scaled1, &B->scaled2,
                            &B->h_done,    &B->y_done,    &B->bk_done, &B->u1_done,
                            &B->hq_done,   &B->hq_free,   &B->sc_done, &B->z_done,
                            &B->qk_done,   &B->drain[0],  &B->drain[1], &B->drain[2]};
        for (uint64_t* p : ones) mbar_init(p, 1);
        B->abort = 0;
        fence_mbar_init();
    }
    // rows 16..63 of the M = 64 operands (Q stages, GELU(Hq)) stay zero
    for (int s = 0; s < kNS; ++s)
        for (int o = tid * 16; o < 6144; o += kThreads * 16)
            *reinterpret_cast<uint4*>(sm + s * kStageBytes + kStQ + 2048 + o) = make_uint4(0, 0, 0, 0);
    for (int h = 0; h < 2; ++h)
        for (int o = tid * 16; o < 6144; o += kThreads * 16)
            *reinterpret_cast<uint4*>(sm + OFF_AQ + h * 8192 + 2048 + o) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 0) tmem_alloc(&B->tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // the peer's barriers exist before anything is sent to them
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;
    const uint32_t lq = (uint32_t)(warp & 3) * 32;       // TMEM sub-partition of this warp
    const uint32_t tl = tmem + (lq << 16);                // TMEM address of lane lq, column 0
    const int u = (warp & 3) * 32 + lane;                 // hidden unit of this thread (warps 0-11)
    const size_t init = (size_t)(a.shared ? 0 : bb) * a.H + hh;

    auto stage = [&](int s) { return sm + s * kStageBytes; };
    auto rec = [&](int b) { return sm + OFF_REC + b * kRecSlot; };
    auto recf = [&](int b, uint32_t off) { return reinterpret_cast<const float*>(rec(b) + off); };

    constexpr uint32_t idN16 = idesc_bf16_f32(128, 16, 0, 0);    // M 128, N 16, both K-major
    constexpr uint32_t idUpd = idesc_bf16_f32(128, 128, 0, 1);   // state updates, B MN-major
    constexpr uint32_t idY = idesc_bf16_f32(64, 16, 1, 0);       // M 64, A MN-major
    constexpr uint32_t idM64 = idesc_bf16_f32(64, 16, 0, 0);     // M 64, both K-major
    constexpr uint32_t idZS = idesc_bf16_f32(128, 16, 1, 0);     // stacked [W2; S2], A MN-major

    if (warp < 4) {
        // ---------------------------------------------------------- chain
        bool ok = true;
        float gp[kC];   // GELU'(H) of this hidden unit, kept until the D1 epilogue
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1, st = c % kNS;
            const uint32_t pb = (c >> 1) & 1;
            uint8_t* stg = stage(st);
            // (0) state(c) complete: bf16 copy of W1 for the MMAs
            if (ok) ok = wait_all(B, c == 0 ? &B->init_done : &B->u1_done, c == 0 ? 0u : (uint32_t)((c - 1) & 1), status, peer);
            if (ok) {
                tc_fence_after();
                tmem_to_bf16(tl, TW1, TW1B);
            }
            tc_fence_before();
            named_bar_sync(1, 128);
            if (tid == 0 && ok) {
                if (c >= 1) mbar_arrive(&B->prep_free[(c - 1) & 1]);
                mbar_arrive(&B->w1_copied);
            }
            // (1) H = W1 K^T
            if (warp == 0) {
                if (ok) ok = wait_all(B, &B->full[st], (c / kNS) & 1, status, peer);
                if (ok) {
                    tc_fence_after();
                    const uint32_t ka = smem_u32(stg + kStK);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_tmem_a(tmem + TH, tmem + TW1B + 8 * kk, sdesc(ka + 32 * kk, 16, 1024, 2),
                                       idN16, kk > 0);
                        mma_commit(&B->h_done);
                    }
                    __syncwarp();
                }
            }
            // (2) A = GELU(H), GELU'(H)
            if (ok) ok = wait_all(B, &B->h_done, c & 1, status, peer);
            if (ok && c >= 2) ok = wait_all(B, &B->rd_done[b], ((c - 2) >> 1) & 1, status, peer);
            if (ok) {
                tc_fence_after();
                float h[kC];
                tmem_ld16(tl + TH, h);
                tmem_wait_ld();
                uint8_t* akt = sm + OFF_AK + b * 4096 + (u >> 6) * 2048;
                float av[kC];
#pragma unroll
                for (int t = 0; t < kC; ++t) gelu_and_grad(h[t], av[t], gp[t]);
                uint32_t ap[8];
#pragma unroll
                for (int t = 0; t < kC; t += 2) ap[t >> 1] = pack_bf16(av[t], av[t + 1]);
                tmem_st8(tl + TAK, ap);
#pragma unroll
                for (int t = 0; t < kC; t += 2) {
                    const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162*>(&ap[t >> 1]);
                    *reinterpret_cast<__nv_bfloat16*>(akt + sw128_offset(t, u & 63)) = pr.x;
                    *reinterpret_cast<__nv_bfloat16*>(akt + sw128_offset(t + 1, u & 63)) = pr.y;
                }
                tmem_wait_st();
                fence_proxy_async_smem();
            }
            tc_fence_before();
            named_bar_sync(1, 128);
            // (3) partial Y = W2 A over this CTA's hidden units
            if (warp == 0) {
                if (ok) ok = wait_all(B, &B->w2b_ready[b], pb, status, peer);
                if (ok) {
                    tc_fence_after();
                    const uint32_t w2 = smem_u32(sm + OFF_W2B + b * kW2BSlot);
                    const uint32_t ak = smem_u32(sm + OFF_AK + b * 4096);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16(tmem + TY, sdesc(w2 + 2048 * kk, 16384, 1024, 2),
                                     sdesc(ak + 2048 * (kk >> 2) + 32 * (kk & 3), 16, 1024, 2), idY,
                                     kk > 0);
                        mma_commit(&B->y_done);
                    }
                    __syncwarp();
                }
            }
            // (4) exchange the partial Y with the peer; E = 2 (Y - V)
            if (tid == 0 && ok) mbar_expect_tx(&B->ybar[b], 4096);
            if (ok) ok = wait_all(B, &B->y_done, c & 1, status, peer);
            if (ok) ok = wait_all(B, &B->prep_ready[b], pb, status, peer);
            float y[kC];
            const int irow = (warp << 4) + lane;   // output row i (M = 64 layout), lanes < 16
            if (ok) {
                tc_fence_after();
                tmem_ld16(tl + TY, y);
                tmem_wait_ld();
                if (lane < 16) {
                    const uint32_t dst = peer_addr(sm + OFF_YR + b * 4096 + irow * 64, peer);
                    const uint32_t rb = peer_addr(&B->ybar[b], peer);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        st_async_v4(dst + 16 * j,
                                    make_float4(y[4 * j], y[4 * j + 1], y[4 * j + 2], y[4 * j + 3]), rb);
                }
            }
            if (ok) ok = wait_all<true>(B, &B->ybar[b], pb, status, peer);
            if (ok && lane < 16) {
                // every load first: the stores below could otherwise serialise them
                float yp[kC], cn[kC], pn[kC], vv[kC];
                ld_f32x16(sm + OFF_YR + b * 4096 + irow * 64, yp);
                ld_f32x16(rec(b) + REC_CN, cn);
                ld_f32x16(rec(b) + REC_PN, pn);
#pragma unroll
                for (int t = 0; t < kC; ++t) vv[t] = ld_bf16(stg + kStV + sw128_offset(t, irow));
                uint8_t* es = sm + OFF_ES + b * 2048;
                uint8_t* ec = sm + OFF_EC;
#pragma unroll
                for (int t = 0; t < kC; ++t) {
                    const uint32_t o = sw128_offset(t, irow);
                    const float e = 2.f * (y[t] + yp[t] - vv[t]);
                    st_bf16(es + o, e);
                    st_bf16(ec + o, -cn[t] * e);
                    st_bf16(ec + 2048 + o, -pn[t] * e);
                }
                fence_proxy_async_smem();
            }
            named_bar_sync(1, 128);
            if (tid == 0 && ok) mbar_arrive(&B->empty[st]);
            // (5) W2^T E, and the W2 / S2 update (accumulated into the state)
            if (warp == 0) {
                if (ok) ok = wait_all(B, &B->scaled2, c & 1, status, peer);
                if (ok) {
                    tc_fence_after();
                    const uint32_t w2 = smem_u32(sm + OFF_W2B + b * kW2BSlot);
                    const uint32_t es = smem_u32(sm + OFF_ES + b * 2048);
                    const uint32_t ec = smem_u32(sm + OFF_EC);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16(tmem + TBK, sdesc(w2 + 32 * kk, 16, 1024, 2),
                                     sdesc(es + 32 * kk, 16, 1024, 2), idN16, kk > 0);
                        mma_tmem_a(tmem + TW2, tmem + TAK, sdesc(ec, 2048, 1024, 2), idUpd, 1);
                        mma_commit(&B->bk_done);
                    }
                    __syncwarp();
                }
            }
            // (6) D1 = (W2^T E) o GELU'(H)
            if (ok) ok = wait_all(B, &B->bk_done, c & 1, status, peer);
            if (ok) {
                tc_fence_after();
                float bk[kC];
                tmem_ld16(tl + TBK, bk);
                tmem_wait_ld();
                uint32_t dp[8];
#pragma unroll
                for (int t = 0; t < kC; t += 2) dp[t >> 1] = pack_bf16(bk[t] * gp[t], bk[t + 1] * gp[t + 1]);
                tmem_st8(tl + TDL, dp);
                tmem_wait_st();
            }
            tc_fence_before();
            named_bar_sync(1, 128);
            // (7) read pre-activations Hq, then the W1 / S1 update
            if (warp == 0) {
                if (ok && c >= 1) ok = wait_all(B, &B->hq_free, (c - 1) & 1, status, peer);
                if (ok) ok = wait_all(B, &B->scaled1, c & 1, status, peer);
                if (ok) {
                    tc_fence_after();
                    const uint32_t qb = smem_u32(sm + OFF_QB + b * kQBSlot);
                    const uint32_t kc = smem_u32(sm + OFF_KC + b * 4096);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_tmem_a(tmem + THQ, tmem + TW1B + 8 * kk, sdesc(qb + 32 * kk, 16, 1024, 2),
                                       idN16, kk > 0);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_tmem_a(tmem + THQ, tmem + TS1B + 8 * kk,
                                       sdesc(qb + 2048 + 32 * kk, 16, 1024, 2), idN16, 1);
                        mma_tmem_a(tmem + THQ, tmem + TDL, sdesc(qb + 4096, 16, 1024, 2), idN16, 1);
                        mma_commit(&B->hq_done);
                        mma_tmem_a(tmem + TW1, tmem + TDL, sdesc(kc, 2048, 1024, 2), idUpd, 1);
                        mma_commit(&B->u1_done);
                    }
                    __syncwarp();
                }
            }
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------- state
        bool ok = true;
        const int ug = kHalf * (int)rank + u;   // hidden unit in the sequence
        {
            const float* w1 = a.W1_0 + (init * kHid + ug) * kD;
            const float* s1 = a.S1_0 ? a.S1_0 + (init * kHid + ug) * kD : nullptr;
            const float* w2 = a.W2_0 + init * kD * kHid + ug;
            const float* s2 = a.S2_0 ? a.S2_0 + init * kD * kHid + ug : nullptr;
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
                float r[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = w1[16 * g + j];
                tmem_st16(tl + TW1 + 16 * g, r);
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = s1 ? s1[16 * g + j] : 0.f;
                tmem_st16(tl + TS1 + 16 * g, r);
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = w2[(size_t)(16 * g + j) * kHid];
                tmem_st16(tl + TW2 + 16 * g, r);
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = s2 ? s2[(size_t)(16 * g + j) * kHid] : 0.f;
                tmem_st16(tl + TS2 + 16 * g, r);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        named_bar_sync(2, 128);
        if (tid == 128) mbar_arrive(&B->init_done);
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            const uint32_t pb = (c >> 1) & 1;
            // (a) bf16 copies of W2^T / S2^T (state(c)) into shared memory
            if (ok && c >= 1) ok = wait_all(B, &B->bk_done, (c - 1) & 1, status, peer);
            if (ok && c >= 2) ok = wait_all(B, &B->rd_done[b], ((c - 2) >> 1) & 1, status, peer);
            if (ok) {
                tc_fence_after();
                uint8_t* w2b = sm + OFF_W2B + b * kW2BSlot;
#pragma unroll 1
                for (int m = 0; m < 2; ++m) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float r[32];
                        tmem_ld16(tl + (m ? TS2 : TW2) + 32 * h, *reinterpret_cast<float(*)[16]>(r));
                        tmem_ld16(tl + (m ? TS2 : TW2) + 32 * h + 16,
                                  *reinterpret_cast<float(*)[16]>(r + 16));
                        tmem_wait_ld();
#pragma unroll
                        for (int g = 0; g < 4; ++g) st_chunk(w2b + m * 16384, u, 32 * h + 8 * g, r + 8 * g);
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            named_bar_sync(2, 128);
            if (tid == 128 && ok) mbar_arrive(&B->w2b_ready[b]);
            // (b) W2 <- beta_n W2 + c_n S2, S2 <- P_n S2 (chunk c's coefficients)
            if (ok) ok = wait_all(B, &B->prep_ready[b], pb, status, peer);
            if (ok) {
                tc_fence_after();
                const float* sc = recf(b, REC_SCAL);
                const float bn = sc[0], cn = sc[1], Pn = sc[2];
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    float w[16], s[16];
                    tmem_ld16(tl + TW2 + 16 * g, w);
                    tmem_ld16(tl + TS2 + 16 * g, s);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        w[j] = fmaf(bn, w[j], cn * s[j]);
                        s[j] = Pn * s[j];
                    }
                    tmem_st16(tl + TW2 + 16 * g, w);
                    tmem_st16(tl + TS2 + 16 * g, s);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            named_bar_sync(2, 128);
            if (tid == 128 && ok) mbar_arrive(&B->scaled2);
            // (c) bf16 copy of S1 (state(c)), then scale W1 / S1 once the chain
            //     has copied W1
            if (ok && c >= 1) ok = wait_all(B, &B->u1_done, (c - 1) & 1, status, peer);
            if (ok) {
                tc_fence_after();
                tmem_to_bf16(tl, TS1, TS1B);
            }
            if (ok) ok = wait_all(B, &B->w1_copied, c & 1, status, peer);
            if (ok) {
                tc_fence_after();
                const float* sc = recf(b, REC_SCAL);
                const float bn = sc[0], cn = sc[1], Pn = sc[2];
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    float w[16], s[16];
                    tmem_ld16(tl + TW1 + 16 * g, w);
                    tmem_ld16(tl + TS1 + 16 * g, s);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        w[j] = fmaf(bn, w[j], cn * s[j]);
                        s[j] = Pn * s[j];
                    }
                    tmem_st16(tl + TW1 + 16 * g, w);
                    tmem_st16(tl + TS1 + 16 * g, s);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            named_bar_sync(2, 128);
            if (tid == 128 && ok) mbar_arrive(&B->scaled1);
        }
        // final state
        if (ok && nch > 0) ok = wait_all(B, &B->bk_done, (nch - 1) & 1, status, peer);
        if (ok && nch > 0) ok = wait_all(B, &B->u1_done, (nch - 1) & 1, status, peer);
        if (ok) {
            tc_fence_after();
            float* w1 = a.W1_out + ((size_t)seq * kHid + ug) * kD;
            float* s1 = a.S1_out ? a.S1_out + ((size_t)seq * kHid + ug) * kD : nullptr;
            float* w2 = a.W2_out + (size_t)seq * kD * kHid + ug;
            float* s2 = a.S2_out ? a.S2_out + (size_t)seq * kD * kHid + ug : nullptr;
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
                float r[16];
                tmem_ld16(tl + TW1 + 16 * g, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) w1[16 * g + j] = r[j];
                tmem_ld16(tl + TW2 + 16 * g, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) w2[(size_t)(16 * g + j) * kHid] = r[j];
                tmem_ld16(tl + TS1 + 16 * g, r);
                tmem_wait_ld();
                if (s1)
#pragma unroll
                    for (int j = 0; j < 16; ++j) s1[16 * g + j] = r[j];
                tmem_ld16(tl + TS2 + 16 * g, r);
                tmem_wait_ld();
                if (s2)
#pragma unroll
                    for (int j = 0; j < 16; ++j) s2[(size_t)(16 * g + j) * kHid] = r[j];
            }
        }
    } else if (warp < 12) {
        // ------------------------------------------------------ read side
        bool ok = true;
        const int t8 = u >> 4, i0 = (u & 15) * 4;   // (token, 4 outputs) of the output pass
        float* P0 = reinterpret_cast<float*>(sm + OFF_ZP);
        float* P1 = P0 + kC * kD;
        float* P2 = P1 + kC * kD;
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            const uint32_t pb = (c >> 1) & 1;
            if (ok) ok = wait_all(B, &B->prep_ready[b], pb, status, peer);
            // (a) GELU(Hq) into the M = 64 operand tile
            if (ok) ok = wait_all(B, &B->hq_done, c & 1, status, peer);
            if (ok) {
                tc_fence_after();
                float hq[kC];
                tmem_ld16(tl + THQ, hq);
                tmem_wait_ld();
                uint8_t* aq = sm + OFF_AQ + (u >> 6) * 8192;
                float gv[kC];
#pragma unroll
                for (int t = 0; t < kC; ++t) gv[t] = gelu(hq[t]);
#pragma unroll
                for (int t = 0; t < kC; ++t) st_bf16(aq + sw128_offset(t, u & 63), gv[t]);
                fence_proxy_async_smem();
            }
            tc_fence_before();
            named_bar_sync(3, 128);
            if (tid == 256 && ok) mbar_arrive(&B->hq_free);
            // (b) scores GELU(Hq) A^T, weights, read-out MMAs (warp 8)
            if (warp == 8 && ok) {
                tc_fence_after();
                const uint32_t aq = smem_u32(sm + OFF_AQ);
                const uint32_t ak = smem_u32(sm + OFF_AK + b * 4096);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + TSC, sdesc(aq + 8192 * (kk >> 2) + 32 * (kk & 3), 16, 1024, 2),
                                 sdesc(ak + 2048 * (kk >> 2) + 32 * (kk & 3), 16, 1024, 2), idM64,
                                 kk > 0);
                    mma_commit(&B->sc_done);
                }
                __syncwarp();
                ok = wait_all(B, &B->sc_done, c & 1, status, peer);
                if (ok) {
                    tc_fence_after();
                    float sc[kC];
                    tmem_ld16(tl + TSC, sc);
                    tmem_wait_ld();
                    if (lane < 16) {
                        const int t = lane;
                        float crow[kC], w[kC];
                        ld_f32x16(rec(b) + REC_C + t * kC * 4, crow);
#pragma unroll
                        for (int s = 0; s < kC; ++s) w[s] = s <= t ? -crow[s] * sc[s] : 0.f;
                        uint8_t* m2 = sm + OFF_M2;
                        st_chunk(m2, t, 0, w);
                        st_chunk(m2, t, 8, w + 8);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    const uint32_t w2 = smem_u32(sm + OFF_W2B + b * kW2BSlot);
                    const uint32_t es = smem_u32(sm + OFF_ES + b * 2048);
                    const uint32_t m2 = smem_u32(sm + OFF_M2);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16(tmem + TZS, sdesc(w2 + 2048 * kk, 16384, 1024, 2),
                                     sdesc(aq + 8192 * (kk >> 2) + 32 * (kk & 3), 16, 1024, 2), idZS,
                                     kk > 0);
                        mma_bf16(tmem + TZC, sdesc(es, 16, 1024, 2), sdesc(m2, 16, 1024, 2), idY, 0);
                        mma_commit(&B->z_done);
                    }
                    __syncwarp();
                }
            }
            // (c) this CTA's read-out parts
            if (ok) ok = wait_all(B, &B->z_done, c & 1, status, peer);
            if (ok) {
                tc_fence_after();
                float zs[kC], zc[kC];
                tmem_ld16(tl + TZS, zs);
                tmem_ld16(tl + TZC, zc);
                tmem_wait_ld();
                float beta[kC], cv[kC];
                ld_f32x16(rec(b) + REC_BETA, beta);
                ld_f32x16(rec(b) + REC_CV, cv);
                if (u < 64) {
#pragma unroll
                    for (int t = 0; t < kC; ++t) P0[t * kD + u] = beta[t] * zs[t];
                } else {
#pragma unroll
                    for (int t = 0; t < kC; ++t) P1[t * kD + u - 64] = cv[t] * zs[t];
                }
                if (lane < 16) {
                    const int i = ((warp & 3) << 4) + lane;
#pragma unroll
                    for (int t = 0; t < kC; ++t) P2[t * kD + i] = zc[t];
                }
            }
            tc_fence_before();
            named_bar_sync(3, 128);
            if (tid == 256 && ok) {
                mbar_arrive(&B->rd_done[b]);
                mbar_arrive(&B->prep_free[b]);
                mbar_expect_tx(&B->zbar[b], 2048);
            }
            // (d) send the peer's tokens, finish this CTA's 8 tokens
            if (ok) {
                const int tp = 8 * (int)peer + t8;
                const float4 p0 = *reinterpret_cast<const float4*>(P0 + tp * kD + i0);
                const float4 p1 = *reinterpret_cast<const float4*>(P1 + tp * kD + i0);
                const float4 p2 = *reinterpret_cast<const float4*>(P2 + tp * kD + i0);
                st_async_v4(peer_addr(sm + OFF_ZR + b * 2048 + (t8 * kD + i0) * 4, peer),
                            make_float4(p0.x + p1.x + p2.x, p0.y + p1.y + p2.y, p0.z + p1.z + p2.z,
                                        p0.w + p1.w + p2.w),
                            peer_addr(&B->zbar[b], peer));
            }
            if (ok) ok = wait_all<true>(B, &B->zbar[b], pb, status, peer);
            if (ok) {
                const int to = 8 * (int)rank + t8;
                const float4 p0 = *reinterpret_cast<const float4*>(P0 + to * kD + i0);
                const float4 p1 = *reinterpret_cast<const float4*>(P1 + to * kD + i0);
                const float4 p2 = *reinterpret_cast<const float4*>(P2 + to * kD + i0);
                const float4 pr = *reinterpret_cast<const float4*>(
                    sm + OFF_ZR + b * 2048 + (t8 * kD + i0) * 4);
                const int tok = c * kC + to;
                if (tok < T) {
                    uint2 o;
                    o.x = pack_bf16(p0.x + p1.x + p2.x + pr.x, p0.y + p1.y + p2.y + pr.y);
                    o.y = pack_bf16(p0.z + p1.z + p2.z + pr.z, p0.w + p1.w + p2.w + pr.w);
                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.z) +
                                              ((size_t)seq * T + tok) * kD + i0) = o;
                }
            }
            named_bar_sync(3, 128);
        }
    } else if (warp == 12) {
        // ---------------------------------------------------- coefficients
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const int b = c & 1, st = c % kNS;
            if (c >= 2) ok = wait_all(B, &B->prep_free[b], ((c - 2) >> 1) & 1, status, peer);
            if (!ok) break;
            const int n = min(kC, T - c * kC);
            const bool valid = lane < n;
            const size_t tok = (size_t)seq * T + (size_t)c * kC + lane;
            // padded tokens are neutral (theta 0, eta = keep = 1)
            const float th = valid ? a.theta[tok] : 0.f;
            const float et = valid ? (a.eta ? a.eta[tok] : 0.f) : 1.f;
            const float kp = valid ? 1.f - (a.alpha ? a.alpha[tok] : 0.f) : 1.f;
            float Ab = kp, Bb = 0.f;
            scan_affine(Ab, Bb, lane);              // beta_t = prod keep
            float Ap = et, Bp = 0.f;
            scan_affine(Ap, Bp, lane);              // P_t = prod eta
            float Ac = kp, Bc = Ap;
            scan_affine(Ac, Bc, lane);              // c_t = keep_t c_{t-1} + P_t
            const float beta = Ab, P = Ap, cv = Bc;
            const float bn = __shfl_sync(0xffffffffu, beta, n - 1);
            const float cn = __shfl_sync(0xffffffffu, cv, n - 1);
            const float Pn = __shfl_sync(0xffffffffu, P, n - 1);
            // C[t][s] = theta_s w(s,t), Pm[t][s] = theta_s m(s,t); lane = column s
            uint8_t* r = rec(b);
            float m = 0.f, w = 0.f, cend = 0.f, pend = 0.f;
#pragma unroll
            for (int t = 0; t < kC; ++t) {
                const float e = __shfl_sync(0xffffffffu, et, t);
                const float k1 = __shfl_sync(0xffffffffu, kp, t);
                m = fmaf(e, m, lane == t ? 1.f : 0.f);
                w = fmaf(k1, w, m);
                if (lane < kC) reinterpret_cast<float*>(r + REC_C)[t * kC + lane] = th * w;
                if (t == n - 1) {
                    cend = th * w;
                    pend = th * m;
                }
            }
            if (lane < kC) {
                reinterpret_cast<float*>(r + REC_BETA)[lane] = beta;
                reinterpret_cast<float*>(r + REC_CV)[lane] = cv;
                reinterpret_cast<float*>(r + REC_CN)[lane] = cend;
                reinterpret_cast<float*>(r + REC_PN)[lane] = pend;
            }
            if (lane == 0)
                *reinterpret_cast<float4*>(r + REC_SCAL) = make_float4(bn, cn, Pn, (float)n);
            __syncwarp();
            ok = wait_all(B, &B->full[st], (c / kNS) & 1, status, peer);
            if (!ok) break;
            tc_fence_after();
            uint8_t* stg = stage(st);
            // Q K^T (M = 64; Q rows 16..63 are zero)
            {
                const uint32_t qa = smem_u32(stg + kStQ), ka = smem_u32(stg + kStK);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + TQK, sdesc(qa + 32 * kk, 16, 1024, 2),
                                 sdesc(ka + 32 * kk, 16, 1024, 2), idM64, kk > 0);
                    mma_commit(&B->qk_done);
                }
                __syncwarp();
            }
            // scaled copies: [-C_n K | -Pm_n K] (update operand), beta Q, c Q
            {
                const float* cnv = recf(b, REC_CN);
                const float* pnv = recf(b, REC_PN);
                const float* bv = recf(b, REC_BETA);
                const float* cvv = recf(b, REC_CV);
                uint8_t* kc = sm + OFF_KC + b * 4096;
                uint8_t* qb = sm + OFF_QB + b * kQBSlot;
                uint4 kv[4], qv[4];
                float sk[4], sp[4], sb[4], sc[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int x = lane + 32 * r, t = x >> 3;
                    const uint32_t o = sw128_offset(t, (x & 7) * 8);
                    kv[r] = *reinterpret_cast<const uint4*>(stg + kStK + o);
                    qv[r] = *reinterpret_cast<const uint4*>(stg + kStQ + o);
                    sk[r] = -cnv[t];
                    sp[r] = -pnv[t];
                    sb[r] = bv[t];
                    sc[r] = cvv[t];
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int x = lane + 32 * r, t = x >> 3;
                    const uint32_t o = sw128_offset(t, (x & 7) * 8);
                    *reinterpret_cast<uint4*>(kc + o) = scale_chunk(kv[r], sk[r]);
                    *reinterpret_cast<uint4*>(kc + 2048 + o) = scale_chunk(kv[r], sp[r]);
                    *reinterpret_cast<uint4*>(qb + o) = scale_chunk(qv[r], sb[r]);
                    *reinterpret_cast<uint4*>(qb + 2048 + o) = scale_chunk(qv[r], sc[r]);
                }
            }
            ok = wait_all(B, &B->qk_done, c & 1, status, peer);
            if (!ok) break;
            tc_fence_after();
            {
                float sq[kC];
                tmem_ld16(tl + TQK, sq);
                tmem_wait_ld();
                if (lane < kC) {
                    const int t = lane;
                    float crow[kC], w1[kC];
                    ld_f32x16(rec(b) + REC_C + t * kC * 4, crow);
#pragma unroll
                    for (int s = 0; s < kC; ++s) w1[s] = s <= t ? -crow[s] * sq[s] : 0.f;
                    uint8_t* m1 = sm + OFF_QB + b * kQBSlot + 4096;
                    st_chunk(m1, t, 0, w1);
                    st_chunk(m1, t, 8, w1 + 8);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&B->empty[st]);
                mbar_arrive(&B->prep_ready[b]);
            }
        }
    } else {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int st = c % kNS;
                if (c >= kNS && !wait_bar<false>(B, &B->empty[st], ((c / kNS) - 1) & 1, status, peer))
                    break;
                mbar_expect_tx(&B->full[st], 3 * 2048);
                uint8_t* stg = stage(st);
                tma_load_3d(stg + kStK, &kmap, &B->full[st], 0, c * kC, seq);
                tma_load_3d(stg + kStV, &vmap, &B->full[st], 0, c * kC, seq);
                tma_load_3d(stg + kStQ, &qmap, &B->full[st], 0, c * kC, seq);
                issued = c + 1;
            }
            // every issued stage's copies land before the CTA exits
            for (int c = (issued > kNS ? issued - kNS : 0); c < issued; ++c)
                wait_drain(&B->full[c % kNS], (c / kNS) & 1);
        }
        __syncwarp();
    }

    // drain the MMAs of the three issuing warps before tensor memory is freed
    if (warp == 0 || warp == 8 || warp == 12) {
        uint64_t* d = &B->drain[warp == 0 ? 0 : (warp == 8 ? 1 : 2)];
        if (elect_one()) mma_commit(d);
        __syncwarp();
        if (lane == 0) wait_drain(d, 0);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no DSMEM traffic towards a CTA that has exited
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D view [sequences][T][64] of a bf16 tensor, 16-row tiles, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int BH, int T) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)T * kD * 2};
    cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

namespace {
__global__ void gelu_eval_kernel(const float* x, float* y, float* dy, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float g, d;
    gelu_and_grad(x[i], g, d);
    y[i] = g;
    if (dy) dy[i] = d;
}
}  // namespace

cudaError_t mlp_gelu_launch(const float* x, float* y, float* dy, int n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    gelu_eval_kernel<<<(n + 255) / 256, 256, 0, s>>>(x, y, dy, n);
    return cudaGetLastError();
}

bool mlp_tc_supported(const MlpArgs& a) {
    return a.bf16 && a.d == kD && a.hidden == kHid && a.chunk == kC && a.T >= 1;
}

cudaError_t mlp_tc_launch(const MlpArgs& a, cudaStream_t s) {
    const int BH = a.B * a.H;
    CUtensorMap km, qm, vm;
    if (!make_map(&km, a.k, BH, a.T) || !make_map(&qm, a.q, BH, a.T) ||
        !make_map(&vm, a.v, BH, a.T))
        return cudaErrorInvalidValue;
    const size_t smem = kSmemBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(mlp_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    mlp_tc_kernel<<<2 * BH, kThreads, smem, s>>>(km, qm, vm, a);
    return cudaGetLastError();
}

}  // namespace ttm
