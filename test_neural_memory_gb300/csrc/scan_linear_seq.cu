// Tensor-core (tcgen05 + TMA) scan of the linear / Titans memory for
// d_k = d_v = 64 with one CTA per sequence, in 64-token tiles whose gradient
// points fall every b in {16, 32} tokens (mini-batch TTT with b = 16 is the
// TTT-Linear setting, "TTT layers 与 fast weights" §1.1 eqs (6)-(9)).
//
// Method.  Let tile g hold tokens t = 0..n-1 (n <= 64) with the state (W_g, S_g)
// at its start, keys K, queries Q, values V (rows = tokens) and the tile's
// decay / momentum coefficients beta_t, c_t, C[t][s] ("论文速览 | Titans"
// §4.3-§4.5; C[t][s] = theta_s w(s, t) is the weight of token s's gradient in
// the state after token t).  Token t takes its gradient at the state left
// before its sub-chunk, which starts at sigma(t) = b floor(t / b), so
//
//   e_t = beta'_t W_g k_t + c'_t S_g k_t - v_t
//         - 2 sum_{s < sigma(t)} C[sigma(t)-1][s] (k_s . k_t) e_s,
//   beta'_t = beta_{sigma(t)-1} (1 for sigma = 0), c'_t = c_{sigma(t)-1} (0).
//
// In matrix form (I + L) E = R0 with R0 = diag(beta') K W^T + diag(c') K S^T - V
// and L[t][s] = 2 C[sigma(t)-1][s] (k_s . k_t), strictly block-lower with
// b x b blocks, so E = N R0 with N = (I + L)^-1 = (I - L)(I + L^2) (at most four
// blocks: L^4 = 0).  The reads and the carry are the chunk form of the tile:
//
//   Z       = diag(beta) Q W^T + diag(c) Q S^T - 2 (A~ N) R0,
//             A~ = mask_{s<=t}(Q K^T) o C
//   W_{g+1}^T = beta_n W^T + c_n S^T - 2 (K^T diag(C[n-1]) N) R0
//   S_{g+1}^T = P_n S^T            - 2 (K^T diag(Pm)     N) R0,
//             Pm[s] = theta_s prod_{j=s+1..n-1} eta_j.
//
// E itself is never formed: A~ N, Y_C = K^T diag(C[n-1]) N and
// Y_P = K^T diag(Pm) N depend only on the tile's inputs and gates, so the
// state's own chain per tile is two tensor-core products,
//   C1: [Q; K] [W; S]^T      (reads and the state part of R0),
//   C3: [A~N; Y_C; 0; Y_P] R0 (the read correction and the carry),
// with an epilogue after each; everything else is prepared beside it.
//
// Roles (512 threads, one CTA per (b, h) sequence, all 64 rows of the state):
//   warps 0,1       reads: token t = TMEM lane 0..63, all 64 columns
//   warps 2,3,6,7   state: E1 (R0 for token = TMEM lane 64..127) and E3 (the
//                   update; thread j holds W[r][j], S[r][j] for 32 rows r in
//                   fp32 registers and writes their bf16 copy)
//   warps 4,5,10,11 preparation, first group, one tile ahead of the chain:
//                   gates (loaded a tile early), C[t][s] by columns (one lane
//                   per column) with the vector scans beside it, then from
//                   the scores [Q; K] K^T the weighted rows of A~ and L, (I - L),
//                   and row-scaled copies of K (the MN-major operand
//                   K^T diag C, K^T diag Pm)
//   warps 8,9,14,15 preparation, second group: N applied to those operands by
//                   two MMA rounds ((I - L), then I + L^2), one tile behind the
//                   first group, so the two groups' latencies overlap
//   warp 12         TMA producer (Q, K, V tiles of 64 tokens, three stages)
//   warp 13         issues C1 and C3, and the next tile's score MMA
// Every wait is bounded; a wait that runs out sets the status word, all roles
// run out their loops without further work, copies and MMAs drain, TMEM is
// freed and the kernel returns.
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

constexpr int kD = 64;              // d_k = d_v
constexpr int kTile = 64;           // tokens per tile
constexpr int kThreads = 512;
constexpr int kNS = 3;              // input stages
constexpr uint32_t kTileBytes = 8192;                 // 64 rows x 128 bytes of bf16
constexpr uint32_t kStageBytes = 3 * kTileBytes;      // Q, K, V
constexpr uint32_t kOpBytes = 32768;                  // a 256-row A operand
constexpr uint32_t kTmemCols = 512;

// TMEM columns
constexpr uint32_t kC1 = 0;      // [Q; K] [W; S]^T: 64 (W) + 64 (S) columns
constexpr uint32_t kC3 = 128;    // [A~N; Y_C] R0 (64) and [0; Y_P] R0 (64)
constexpr uint32_t kP1 = 256;    // 2 x 64: [Q; K] K^T of two tiles
constexpr uint32_t kPR = 384;    // preparation rounds: 2 x 64

// Per-tile vectors (floats) in a slot of shared memory.
constexpr int vTh = 0, vEt = 64, vKp = 128, vBeta = 192, vCv = 256, vBp = 320, vCp = 384,
              vCn = 448, vPm = 512, vScal = 576;     // scal: beta_n, c_n, P_n, n
constexpr uint32_t kVecBytes = 4096;

struct Bars {
    uint64_t full[kNS], empty[kNS];
    uint64_t c1_done, c1_free, r0_ready, c3_free, ws_ready, pr_done;
    uint64_t ay_ready[2], c3_done[2], vec_ready[2], vec_free[2], p1_done[2], p1_free[2], ops_ready[2];
    uint64_t ap_free;
    uint64_t drain[2];
    long long wait_limit;
    uint32_t tmem_base;
    int abort;
};

struct Layout {
    uint32_t stages, ay, ap, r0, ws, il, b2, vec, bars, total;
};

__host__ __device__ constexpr Layout make_layout() {
    Layout L{};
    uint32_t o = 0;
    L.stages = o; o += kNS * kStageBytes;
    L.ay = o;     o += 2 * kOpBytes;       // A operand of C3 (two tiles in flight)
    L.ap = o;     o += kOpBytes;           // between the two preparation rounds
    L.r0 = o;     o += kTileBytes;         // R0 [s][r] (MN-major B)
    L.ws = o;     o += 2 * kTileBytes;     // bf16 W^T [j][r] then S^T [j][r] (MN-major B)
    L.il = o;     o += 2 * kTileBytes;     // (I - L) [s][u] (MN-major B), two tiles in flight
    L.b2 = o;     o += kTileBytes;         // (I + L^2) [s][u] (MN-major B)
    L.vec = o;    o += 2 * kVecBytes;
    L.bars = o;   o += (uint32_t)((sizeof(Bars) + 15) & ~size_t(15));
    L.total = o;
    return L;
}

constexpr long long kWaitCycles = 4000000000LL;   // default limit, ~2 s at 2 GHz

__device__ __noinline__ bool wait_bar_slow(Bars* B, uint64_t* bar, uint32_t parity, int* status) {
    const long long t0 = clock64();
    const long long limit = B->wait_limit;
    uint32_t polls = 0;
    while (!mbar_try_wait_sleep(bar, parity, 20000)) {
        if ((++polls & 3u) == 0) {
            if (*(volatile int*)&B->abort) return false;
            if (clock64() - t0 > limit) {
                *(volatile int*)&B->abort = 1;
                atomicExch(status, TTM_ERR_TIMEOUT);
                return false;
            }
        }
    }
    return true;
}

__device__ __forceinline__ bool wait_bar(Bars* B, uint64_t* bar, uint32_t parity, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(B, bar, parity, status);
}

// Warp-uniform bounded wait (every lane gets the same answer).
__device__ __noinline__ bool wait_all_slow(Bars* B, uint64_t* bar, uint32_t parity, int* status) {
    return __all_sync(0xffffffffu, wait_bar_slow(B, bar, parity, status));
}

__device__ __forceinline__ bool wait_all(Bars* B, uint64_t* bar, uint32_t parity, int* status) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    return wait_all_slow(B, bar, parity, status);
}

__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) break;
}

__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 8 consecutive bf16 values of row `row` from column `col` (a multiple of 8)
// of a 128-byte-swizzled tile.
__device__ __forceinline__ void st_chunk(uint8_t* tile, int row, int col, const float* x) {
    uint4 v;
    v.x = pack_bf16(x[0], x[1]);
    v.y = pack_bf16(x[2], x[3]);
    v.z = pack_bf16(x[4], x[5]);
    v.w = pack_bf16(x[6], x[7]);
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, col)) = v;
}

__device__ __forceinline__ void ld_chunk(const uint8_t* tile, int row, int col, float* x) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128_offset(row, col));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// 32 lanes x 32 consecutive 32-bit TMEM columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
    uint32_t u[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]),
          "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
          "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]),
          "=r"(u[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __uint_as_float(u[i]);
}

// Inclusive scan of affine maps x -> A x + B along lanes (later lanes outside).
__device__ __forceinline__ void scan_affine_up(float& A, float& B, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float A2 = __shfl_up_sync(0xffffffffu, A, off);
        const float B2 = __shfl_up_sync(0xffffffffu, B, off);
        if (lane >= off) {
            B = A * B2 + B;
            A = A * A2;
        }
    }
}

// Four K steps (K = 64) of one M = 128 MMA with both operands in shared
// memory, B MN-major ([k][n] rows of 128 bytes, N atoms 8 KB apart); A
// K-major (rows of the M index) or MN-major ([k][m], M atoms 8 KB apart).
__device__ __forceinline__ void mma_k64_ka(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_bf16(d, sdesc(a + kk * 32, 16, 1024, 2), sdesc(b + kk * 2048, 8192, 1024, 2), idesc,
                 kk > 0);
}

__device__ __forceinline__ void mma_k64_ma(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_bf16(d, sdesc(a + kk * 2048, 8192, 1024, 2), sdesc(b + kk * 2048, 8192, 1024, 2), idesc,
                 kk > 0);
}

// Index of C[t][s] in the tile's fp32 coefficient table: row t at 64 t floats,
// its sixteen groups of four XOR-permuted by t % 16, so that the column walk
// (one column per lane) and the row reads (one row per thread) are both free
// of bank conflicts.
__device__ __forceinline__ int c_index(int t, int s) {
    return t * 64 + ((((s >> 2) ^ (t & 15))) << 2) + (s & 3);
}

template <bool kTitans>
__global__ void __launch_bounds__(kThreads, 1)
linear_seq_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const LinearArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    constexpr Layout L = make_layout();
    Bars* B = reinterpret_cast<Bars*>(sm + L.bars);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seq = blockIdx.x;
    const int bb = seq / a.H, hh = seq % a.H;
    const int T = a.T;
    const int nt = (T + kTile - 1) / kTile;
    const int bsub = a.chunk;
    int* status = a.status;

    auto stage = [&](int s) { return sm + L.stages + s * kStageBytes; };   // Q | K | V
    auto ay = [&](int s) { return sm + L.ay + s * kOpBytes; };
    uint8_t* ap = sm + L.ap;
    uint8_t* r0 = sm + L.r0;
    uint8_t* wsW = sm + L.ws;
    uint8_t* wsS = wsW + kTileBytes;
    uint8_t* il = sm + L.il;
    uint8_t* b2 = sm + L.b2;
    auto vec = [&](int v) { return reinterpret_cast<float*>(sm + L.vec + v * kVecBytes); };

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&B->full[s], 1);
            mbar_init(&B->empty[s], 2);        // state warps + preparation warps
        }
        mbar_init(&B->c1_done, 1);
        mbar_init(&B->c1_free, 2);             // read warps
        mbar_init(&B->r0_ready, 4);            // state warps
        mbar_init(&B->c3_free, 2);             // read warps
        mbar_init(&B->ws_ready, 4);            // state warps
        mbar_init(&B->pr_done, 1);
        mbar_init(&B->ap_free, 1);             // second preparation group
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B->ay_ready[i], 1);
            mbar_init(&B->c3_done[i], 1);
            mbar_init(&B->vec_ready[i], 1);    // the scan warp
            mbar_init(&B->vec_free[i], 6);     // read warps + state warps
            mbar_init(&B->p1_done[i], 1);
            mbar_init(&B->ops_ready[i], 1);    // first preparation group
            mbar_init(&B->p1_free[i], 1);      // first preparation group (scores read)
        }
        for (int i = 0; i < 2; ++i) mbar_init(&B->drain[i], 1);
        B->wait_limit = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;
        B->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&B->tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(warp & 3) * 32 << 16);   // this warp's TMEM lanes

    constexpr uint32_t idC1 = idesc_bf16_f32(128, kTitans ? 128 : 64, 0, 1);
    constexpr uint32_t idK = idesc_bf16_f32(128, 64, 0, 0);   // B K-major
    constexpr uint32_t idM = idesc_bf16_f32(128, 64, 0, 1);   // B MN-major
    constexpr uint32_t idMM = idesc_bf16_f32(128, 64, 1, 1);  // A and B MN-major

    const bool is_read = warp < 2;
    const bool is_state = warp == 2 || warp == 3 || warp == 6 || warp == 7;
    const bool is_p1 = warp == 4 || warp == 5 || warp == 10 || warp == 11;
    const bool is_p2 = warp == 8 || warp == 9 || warp == 14 || warp == 15;

    if (is_read) {
        // ------------------------------------------------------------- reads
        // token t = TMEM lane 0..63, all 64 columns.  C3 of a tile is issued
        // after the state's E1, which waited for C1, so once C3 is complete both
        // products of the tile are in tensor memory.
        const int t = 32 * warp + lane;
        bool ok = true;
        for (int g = 0; g < nt; ++g) {
            const int v = g & 1;
            const int n = min(kTile, T - g * kTile);
            if (ok) ok = wait_all(B, &B->vec_ready[v], (g >> 1) & 1, status);
            if (ok) ok = wait_all(B, &B->c3_done[v], (g >> 1) & 1, status);
            if (ok) {
                const float bt = vec(v)[vBeta + t];
                const float ct = kTitans ? vec(v)[vCv + t] : 0.f;
                tc_fence_after();
                uint4* zr = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.z) +
                                                     ((size_t)seq * T + (size_t)g * kTile + t) * kD);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float qw[16], qs[16], dz[16];
                    tmem_ld16(tl + kC1 + 16 * q, qw);
                    if (kTitans) tmem_ld16(tl + kC1 + 64 + 16 * q, qs);
                    tmem_ld16(tl + kC3 + 16 * q, dz);
                    tmem_wait_ld();
                    float zz[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        zz[i] = fmaf(-2.f, dz[i], bt * qw[i]);
                        if (kTitans) zz[i] = fmaf(ct, qs[i], zz[i]);
                    }
                    if (t < n) {
                        zr[2 * q] = make_uint4(pack_bf16(zz[0], zz[1]), pack_bf16(zz[2], zz[3]),
                                               pack_bf16(zz[4], zz[5]), pack_bf16(zz[6], zz[7]));
                        zr[2 * q + 1] = make_uint4(pack_bf16(zz[8], zz[9]), pack_bf16(zz[10], zz[11]),
                                                   pack_bf16(zz[12], zz[13]), pack_bf16(zz[14], zz[15]));
                    }
                }
                tc_fence_before();
                warp_arrive(&B->c1_free);
                warp_arrive(&B->c3_free);
                warp_arrive(&B->vec_free[v]);
            }
        }
    } else if (is_state) {
        // ------------------------------------------------------------- state
        const int h = warp >> 2;
        const int j = 32 * ((warp & 3) - 2) + lane;   // E1: token; E3: key index
        const size_t init = (size_t)(a.shared ? 0 : bb) * a.H + hh;
        float w[32], s[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const size_t idx = (init * kD + 32 * h + i) * (size_t)kD + j;
            w[i] = a.W0[idx];
            s[i] = (kTitans && a.S0) ? a.S0[idx] : 0.f;
        }
        auto write_ws = [&]() {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                st_chunk(wsW, j, 32 * h + 8 * q, w + 8 * q);
                if (kTitans) st_chunk(wsS, j, 32 * h + 8 * q, s + 8 * q);
            }
        };
        write_ws();
        fence_proxy_async_smem();
        warp_arrive(&B->ws_ready);
        bool ok = true;
        for (int g = 0; g < nt; ++g) {
            const int st = g % kNS, v = g & 1;
            if (ok) ok = wait_all(B, &B->full[st], (g / kNS) & 1, status);
            if (ok) ok = wait_all(B, &B->c1_done, g & 1, status);
            if (ok) ok = wait_all(B, &B->vec_ready[v], (g >> 1) & 1, status);
            if (ok) {
                // E1: R0 for token j, rows 32h .. 32h + 31, sixteen at a time
                tc_fence_after();
                const uint8_t* vt = stage(st) + 2 * kTileBytes;
                const float bp = vec(v)[vBp + j];
                const float cp = kTitans ? vec(v)[vCp + j] : 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c0 = 32 * h + 16 * half;
                    float kw[16], ks[16], vv[16];
                    tmem_ld16(tl + kC1 + c0, kw);
                    if (kTitans) tmem_ld16(tl + kC1 + 64 + c0, ks);
                    ld_chunk(vt, j, c0, vv);
                    ld_chunk(vt, j, c0 + 8, vv + 8);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        kw[i] = bp * kw[i] - vv[i];
                        if (kTitans) kw[i] = fmaf(cp, ks[i], kw[i]);
                    }
                    st_chunk(r0, j, c0, kw);
                    st_chunk(r0, j, c0 + 8, kw + 8);
                }
                tc_fence_before();
                fence_proxy_async_smem();
                warp_arrive(&B->r0_ready);
            }
            named_bar_sync(1, 128);
            if (tid == 64 && ok) mbar_arrive(&B->empty[st]);   // V and the C1 reads are done
            if (ok) ok = wait_all(B, &B->c3_done[v], (g >> 1) & 1, status);
            if (ok) {
                // E3: the carry for key index j, sixteen rows at a time
                tc_fence_after();
                const float4 sc = *reinterpret_cast<const float4*>(vec(v) + vScal);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float dc[16], dp[16];
                    tmem_ld16(tl + kC3 + 32 * h + 16 * half, dc);
                    if (kTitans) tmem_ld16(tl + kC3 + 64 + 32 * h + 16 * half, dp);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int ii = 16 * half + i;
                        if (kTitans) {
                            const float wn = sc.x * w[ii] + sc.y * s[ii] - 2.f * dc[i];
                            s[ii] = sc.z * s[ii] - 2.f * dp[i];
                            w[ii] = wn;
                        } else {
                            w[ii] = sc.x * w[ii] - 2.f * dc[i];
                        }
                    }
                }
                tc_fence_before();
                write_ws();
                fence_proxy_async_smem();
                warp_arrive(&B->ws_ready);
                warp_arrive(&B->vec_free[v]);
            }
        }
        if (ok && a.W_out) {
            const size_t dst = (size_t)seq * kD * kD;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const size_t idx = dst + (size_t)(32 * h + i) * kD + j;
                a.W_out[idx] = w[i];
                if (a.S_out) a.S_out[idx] = s[i];
            }
        }
    } else if (is_p1) {
        // ----------------------------------------- preparation, first group
        // Gates, coefficients, the scores and the weighted rows of tile g
        // (one tile ahead of the chain); the second group applies N to them.
        const int p = 32 * (warp & 3) + lane;    // TMEM lane 0..127 (warps 4, 5, 10, 11)
        const bool qside = p < 64;
        const int tr = qside ? p : p - 64;
        float* Ctab = reinterpret_cast<float*>(ap);   // the tile's C (fp32), until round 1
        const bool gated = a.eta || a.alpha;
        bool ok = true;
        // gates of token tr of tile gg (padded tokens: theta 0, eta = keep = 1),
        // loaded one tile ahead so that their latency overlaps a tile's work
        float th_n = 0.f, et_n = 1.f, kp_n = 1.f;
        auto load_gates = [&](int gg) {
            th_n = 0.f;
            et_n = 1.f;
            kp_n = 1.f;
            if (qside && gg < nt && gg * kTile + tr < T) {
                const size_t gi = gate_index(a, (size_t)seq, gg * kTile + tr);
                th_n = a.theta[gi];
                et_n = a.eta ? a.eta[gi] : 0.f;
                kp_n = 1.f - (a.alpha ? a.alpha[gi] : 0.f);
            }
        };
        if (!kTitans) {
            // the momentum operand rows stay zero without momentum
            const float zero8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (!qside)
                for (int c8 = 0; c8 < 8; ++c8)
                    for (int sl = 0; sl < 2; ++sl)
                        st_chunk(ay(sl) + 128 * 128 + kTileBytes, tr, 8 * c8, zero8);
        }
        load_gates(0);
        for (int g = 0; g < nt; ++g) {
            const int v = g & 1, st = g % kNS;
            const int n = min(kTile, T - g * kTile);
            float* V = vec(v);
            uint8_t* X = ay(v);                  // [A~; L] rows 0..127 (K-major), then the C3 operand
            uint8_t* KCP = X + 128 * 128;        // [s][j]: K scaled by C[n-1][s], then by Pm[s]
            uint8_t* ilv = il + v * kTileBytes;  // (I - L) of this tile
            if (ok && g >= 2) ok = wait_all(B, &B->vec_free[v], ((g - 2) >> 1) & 1, status);
            if (ok && g >= 2) ok = wait_all(B, &B->c3_done[v], ((g - 2) >> 1) & 1, status);
            if (ok && qside) {
                V[vTh + tr] = th_n;
                V[vEt + tr] = et_n;
                V[vKp + tr] = kp_n;
            }
            load_gates(g + 1);
            named_bar_sync(3, 128);
            if (ok && gated && (warp == 4 || warp == 5)) {
                // the coefficient table shares its buffer with the second group's
                // operand between its rounds: wait until that group is done with it
                if (g >= 1) ok = wait_all(B, &B->ap_free, (g - 1) & 1, status);
            }
            if (ok && gated && (warp == 4 || warp == 5)) {
                // C[t][s] = theta_s w(s, t) by columns (lane = column s, rows in
                // order): m(s,t) = eta_t m(s,t-1), w(s,t) = keep_t w(s,t-1) + m(s,t),
                // both 0 before row s and 1 at it; above the diagonal C is 0.
                // The rows' gates are loaded sixteen at a time into registers, so
                // no load sits on the recurrence.
                const int sc = lane + 32 * (warp & 3);
                const float ths = V[vTh + sc];
                float m = 0.f, wv = 0.f, ce = 0.f;
                float* __restrict__ ct = Ctab;
#pragma unroll 1
                for (int tb = 0; tb < kTile; tb += 16) {
                    float e[16], k1[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 ev = *reinterpret_cast<const float4*>(V + vEt + tb + 4 * i);
                        const float4 kv = *reinterpret_cast<const float4*>(V + vKp + tb + 4 * i);
                        e[4 * i] = ev.x; e[4 * i + 1] = ev.y; e[4 * i + 2] = ev.z; e[4 * i + 3] = ev.w;
                        k1[4 * i] = kv.x; k1[4 * i + 1] = kv.y; k1[4 * i + 2] = kv.z; k1[4 * i + 3] = kv.w;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = tb + i;
                        m = fmaf(e[i], m, t == sc ? 1.f : 0.f);
                        wv = fmaf(k1[i], wv, m);
                        const float c = ths * wv;
                        ct[c_index(t, sc)] = c;
                        ce = t == n - 1 ? c : ce;
                    }
                }
                V[vCn + sc] = ce;              // C[n-1][s]
                V[vPm + sc] = ths * m;         // theta_s prod_{j=s+1..n-1} eta_j (padded eta = 1)
            }
            if (ok && !gated && (warp == 4 || warp == 5)) {
                // no momentum and no forgetting: C[t][s] = theta_s for s <= t
                const int sc = lane + 32 * (warp & 3);
                const float ths = V[vTh + sc];
                V[vCn + sc] = sc <= n - 1 ? ths : 0.f;
                V[vPm + sc] = sc == n - 1 ? ths : 0.f;
            }
            if (ok && !gated && warp == 10) {
                // beta = 1, c = 0, P = 0 throughout
                V[vBeta + lane] = 1.f;
                V[vBeta + lane + 32] = 1.f;
                V[vCv + lane] = 0.f;
                V[vCv + lane + 32] = 0.f;
                V[vBp + lane] = 1.f;
                V[vBp + lane + 32] = 1.f;
                V[vCp + lane] = 0.f;
                V[vCp + lane + 32] = 0.f;
                if (lane == 0) *reinterpret_cast<float4*>(V + vScal) = make_float4(1.f, 0.f, 0.f, (float)n);
                warp_arrive(&B->vec_ready[v]);
            }
            if (ok && gated && warp == 10) {
                // beta_t = prod keep, P_t = prod eta, c_t = keep_t c_{t-1} + P_t;
                // lane l owns tokens 2l, 2l + 1
                const int t0 = 2 * lane, t1 = t0 + 1;
                const float et0 = V[vEt + t0], et1 = V[vEt + t1];
                const float kp0 = V[vKp + t0], kp1 = V[vKp + t1];
                float Ab = kp0 * kp1, Bb = 0.f, Ap = et0 * et1, Bp = 0.f;
                scan_affine_up(Ab, Bb, lane);
                scan_affine_up(Ap, Bp, lane);
                float pre_b = __shfl_up_sync(0xffffffffu, Ab, 1);
                float pre_p = __shfl_up_sync(0xffffffffu, Ap, 1);
                if (lane == 0) pre_b = pre_p = 1.f;
                const float be0 = pre_b * kp0, be1 = be0 * kp1;
                const float P0 = pre_p * et0, P1 = P0 * et1;
                float Ac = kp1 * kp0, Bc = kp1 * P0 + P1;
                scan_affine_up(Ac, Bc, lane);
                float cpre = __shfl_up_sync(0xffffffffu, Bc, 1);
                if (lane == 0) cpre = 0.f;
                const float c0 = kp0 * cpre + P0, c1 = kp1 * c0 + P1;
                V[vBeta + t0] = be0;
                V[vBeta + t1] = be1;
                V[vCv + t0] = c0;
                V[vCv + t1] = c1;
                // beta', c': the values at the token before the sub-chunk's start
                // (t0 and t1 share a sub-chunk: b is even)
                const int src = bsub * (t0 / bsub) - 1;
                const int sl = src < 0 ? 0 : src >> 1;
                const float sb0 = __shfl_sync(0xffffffffu, be0, sl), sb1 = __shfl_sync(0xffffffffu, be1, sl);
                const float sc0 = __shfl_sync(0xffffffffu, c0, sl), sc1 = __shfl_sync(0xffffffffu, c1, sl);
                const float bp = src < 0 ? 1.f : ((src & 1) ? sb1 : sb0);
                const float cp = src < 0 ? 0.f : ((src & 1) ? sc1 : sc0);
                V[vBp + t0] = bp;
                V[vBp + t1] = bp;
                V[vCp + t0] = cp;
                V[vCp + t1] = cp;
                const int ln = (n - 1) >> 1, un = (n - 1) & 1;
                const float bn = __shfl_sync(0xffffffffu, un ? be1 : be0, ln);
                const float cn = __shfl_sync(0xffffffffu, un ? c1 : c0, ln);
                const float Pn = __shfl_sync(0xffffffffu, un ? P1 : P0, ln);
                if (lane == 0)
                    *reinterpret_cast<float4*>(V + vScal) = make_float4(bn, cn, Pn, (float)n);
                // the reads and the state only need these vectors: publish them now
                warp_arrive(&B->vec_ready[v]);
            }
            named_bar_sync(3, 128);
            // weighted scores: row p of [A~; L] and row tr of (I - L); K rows
            // scaled by C[n-1][s] (Q side) and Pm[s] (K side)
            if (ok) ok = wait_all(B, &B->p1_done[v], (g >> 1) & 1, status);
            if (ok) {
                tc_fence_after();
                const int r = qside ? tr : bsub * (tr / bsub) - 1;   // row of C used
                const float scale = qside ? 1.f : 2.f;
#pragma unroll 1
                for (int q4 = 0; q4 < 4; ++q4) {
                    float raw[16], cr[16], val[16];
                    tmem_ld16(tl + kP1 + 64 * v + 16 * q4, raw);
#pragma unroll
                    for (int gq = 0; gq < 4; ++gq) {
                        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (gated) {
                            if (r >= 0) f = *reinterpret_cast<const float4*>(Ctab + c_index(r, 16 * q4 + 4 * gq));
                        } else {
                            // theta_s below and on the diagonal of row r
                            const int s0 = 16 * q4 + 4 * gq;
                            f = *reinterpret_cast<const float4*>(V + vTh + s0);
                            f.x = s0 <= r ? f.x : 0.f;
                            f.y = s0 + 1 <= r ? f.y : 0.f;
                            f.z = s0 + 2 <= r ? f.z : 0.f;
                            f.w = s0 + 3 <= r ? f.w : 0.f;
                        }
                        cr[4 * gq] = f.x;
                        cr[4 * gq + 1] = f.y;
                        cr[4 * gq + 2] = f.z;
                        cr[4 * gq + 3] = f.w;
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) val[i] = scale * cr[i] * raw[i];
                    st_chunk(X, p, 16 * q4, val);
                    st_chunk(X, p, 16 * q4 + 8, val + 8);
                    if (!qside) {
                        float iv[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) iv[i] = (16 * q4 + i == tr ? 1.f : 0.f) - val[i];
                        st_chunk(ilv, tr, 16 * q4, iv);
                        st_chunk(ilv, tr, 16 * q4 + 8, iv + 8);
                    }
                }
                if (qside || kTitans) {
                    const uint8_t* kt = stage(st) + kTileBytes;
                    const float f = V[(qside ? vCn : vPm) + tr];
                    uint8_t* dst = KCP + (qside ? 0u : kTileBytes);
#pragma unroll 2
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float x[8];
                        ld_chunk(kt, tr, 8 * c8, x);
#pragma unroll
                        for (int i = 0; i < 8; ++i) x[i] *= f;
                        st_chunk(dst, tr, 8 * c8, x);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(3, 128);
            if (ok && p == 0) {
                mbar_arrive(&B->empty[st]);      // the scores and K reads are done
                mbar_arrive(&B->p1_free[v]);     // the score accumulator may be reused
                mbar_arrive(&B->ops_ready[v]);   // the second group may start on this tile
            }
        }
    } else if (is_p2) {
        // ---------------------------------------- preparation, second group
        // N = (I - L)(I + L^2) applied to [A~; K^T diag C; K^T diag Pm] of tile
        // g by two MMA rounds, while the first group prepares tile g + 1.
        const int p = 32 * (warp & 3) + lane;    // TMEM lane 0..127 (warps 8, 9, 14, 15)
        const bool issuer = warp == 8;
        const bool qside = p < 64;
        const int tr = qside ? p : p - 64;
        bool ok = true;
        uint32_t pr_phase = 0;
        for (int g = 0; g < nt; ++g) {
            const int v = g & 1;
            uint8_t* X = ay(v);
            uint8_t* KCP = X + 128 * 128;
            uint8_t* ilv = il + v * kTileBytes;
            if (ok) ok = wait_all(B, &B->ops_ready[v], (g >> 1) & 1, status);
            tc_fence_after();
            if (bsub < kTile) {
                // round 1: [A~; L] (I - L) and [K^T diag C; K^T diag Pm] (I - L)
                if (issuer && ok) {
                    tc_fence_after();
                    if (elect_one()) {
                        mma_k64_ka(tmem + kPR, smem_u32(X), smem_u32(ilv), idM);
                        mma_k64_ma(tmem + kPR + 64, smem_u32(KCP), smem_u32(ilv), idMM);
                        mma_commit(&B->pr_done);
                    }
                    __syncwarp();
                }
                if (ok) ok = wait_all(B, &B->pr_done, pr_phase & 1, status);
                ++pr_phase;
                if (ok) {
                    tc_fence_after();
                    // b = 32: N = I - L, so this round gives the C3 operand itself
                    uint8_t* dst = bsub == 32 ? X : ap;
#pragma unroll 1
                    for (int hh2 = 0; hh2 < 2; ++hh2) {
                        float d1[32], d2[32];
                        tmem_ld32(tl + kPR + 32 * hh2, d1);
                        tmem_ld32(tl + kPR + 64 + 32 * hh2, d2);
                        tmem_wait_ld();
                        if (qside) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                st_chunk(dst, p, 32 * hh2 + 8 * q, d1 + 8 * q);        // A~ (I - L)
                                st_chunk(dst, 64 + p, 32 * hh2 + 8 * q, d2 + 8 * q);   // Y0_C (I - L)
                            }
                        } else {
                            if (kTitans) {
#pragma unroll
                                for (int q = 0; q < 4; ++q)                            // Y0_P (I - L)
                                    st_chunk(dst, 192 + tr, 32 * hh2 + 8 * q, d2 + 8 * q);
                            }
                            if (bsub == 16) {
                                // I + L^2 = I + L - (L - L^2), with the bf16 L the MMA used
                                float x[32];
#pragma unroll
                                for (int q = 0; q < 4; ++q) ld_chunk(X, p, 32 * hh2 + 8 * q, x + 8 * q);
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    const int u = 32 * hh2 + i;
                                    x[i] = (u == tr ? 1.f : 0.f) + x[i] - d1[i];
                                }
#pragma unroll
                                for (int q = 0; q < 4; ++q) st_chunk(b2, tr, 32 * hh2 + 8 * q, x + 8 * q);
                            }
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(5, 128);
                if (bsub == 16) {
                    // round 2: [A~(I-L); Y0_C(I-L)] (I + L^2) and [.; Y0_P(I-L)] (I + L^2)
                    if (issuer && ok) {
                        tc_fence_after();
                        if (elect_one()) {
                            mma_k64_ka(tmem + kPR, smem_u32(ap), smem_u32(b2), idM);
                            if (kTitans)
                                mma_k64_ka(tmem + kPR + 64, smem_u32(ap) + 128 * 128, smem_u32(b2), idM);
                            mma_commit(&B->pr_done);
                        }
                        __syncwarp();
                    }
                    if (ok) ok = wait_all(B, &B->pr_done, pr_phase & 1, status);
                    ++pr_phase;
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int hh2 = 0; hh2 < 2; ++hh2) {
                            float d1[32], d2[32];
                            tmem_ld32(tl + kPR + 32 * hh2, d1);
                            if (kTitans) tmem_ld32(tl + kPR + 64 + 32 * hh2, d2);
                            tmem_wait_ld();
#pragma unroll
                            for (int q = 0; q < 4; ++q) st_chunk(X, p, 32 * hh2 + 8 * q, d1 + 8 * q);
                            if (!qside && kTitans) {
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    st_chunk(X, 192 + tr, 32 * hh2 + 8 * q, d2 + 8 * q);
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    named_bar_sync(5, 128);
                }
            }
            if (ok && p == 0) {
                mbar_arrive(&B->ap_free);
                mbar_arrive(&B->ay_ready[v]);
            }
        }
    } else if (warp == 12) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            constexpr int kPrefetch = 4;
            auto prefetch = [&](int g) {
                if (g >= nt) return;
                tma_prefetch_l2_3d(&qmap, 0, g * kTile, seq);
                tma_prefetch_l2_3d(&kmap, 0, g * kTile, seq);
                tma_prefetch_l2_3d(&vmap, 0, g * kTile, seq);
            };
            for (int g = 0; g < kPrefetch; ++g) prefetch(g);
            int issued = 0;
            for (int g = 0; g < nt; ++g) {
                const int st = g % kNS;
                prefetch(g + kPrefetch);
                if (g >= kNS && !wait_bar(B, &B->empty[st], ((g / kNS) - 1) & 1, status)) break;
                mbar_expect_tx(&B->full[st], kStageBytes + (g + 1 == a.debug_stall ? 16u : 0u));
                tma_load_3d(stage(st), &qmap, &B->full[st], 0, g * kTile, seq);
                tma_load_3d(stage(st) + kTileBytes, &kmap, &B->full[st], 0, g * kTile, seq);
                tma_load_3d(stage(st) + 2 * kTileBytes, &vmap, &B->full[st], 0, g * kTile, seq);
                issued = g + 1;
            }
            for (int g = (issued > kNS ? issued - kNS : 0); g < issued; ++g)
                wait_drain(&B->full[g % kNS], (g / kNS) & 1, B->wait_limit);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------- chain MMA issue
        // Also issues the score MMA [Q; K] K^T of the next tile, so that the
        // wait for a free tensor pipe stays off the preparation's path.
        bool ok = true;
        auto issue_scores = [&](int g2) -> bool {
            const int st2 = g2 % kNS;
            if (!wait_all(B, &B->full[st2], (g2 / kNS) & 1, status)) return false;
            if (g2 >= 2 && !wait_all(B, &B->p1_free[g2 & 1], ((g2 - 2) >> 1) & 1, status)) return false;
            tc_fence_after();
            if (elect_one()) {
                const uint32_t sa = smem_u32(stage(st2));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kP1 + 64 * (g2 & 1), sdesc(sa + kk * 32, 16, 1024, 2),
                             sdesc(sa + kTileBytes + kk * 32, 16, 1024, 2), idK, kk > 0);
                mma_commit(&B->p1_done[g2 & 1]);
            }
            __syncwarp();
            return true;
        };
        ok = issue_scores(0);
        for (int g = 0; g < nt; ++g) {
            const int st = g % kNS, v = g & 1;
            if (ok) ok = wait_all(B, &B->full[st], (g / kNS) & 1, status);
            if (ok) ok = wait_all(B, &B->ws_ready, g & 1, status);
            if (ok && g >= 1) ok = wait_all(B, &B->c1_free, (g - 1) & 1, status);
            if (ok) {
                tc_fence_after();
                if (elect_one()) {
                    // C1 = [Q; K] [W; S]^T (B: W^T then S^T, 8 KB apart)
                    mma_k64_ka(tmem + kC1, smem_u32(stage(st)), smem_u32(wsW), idC1);
                    mma_commit(&B->c1_done);
                }
                __syncwarp();
            }
            // the next tile's scores now if its operands have landed, else after C3
            bool scored = g + 1 >= nt;
            if (ok && !scored &&
                __all_sync(0xffffffffu, mbar_try_wait(&B->full[(g + 1) % kNS], ((g + 1) / kNS) & 1))) {
                ok = issue_scores(g + 1);
                scored = true;
            }
            if (ok) ok = wait_all(B, &B->r0_ready, g & 1, status);
            if (ok) ok = wait_all(B, &B->ay_ready[v], (g >> 1) & 1, status);
            if (ok && g >= 1) ok = wait_all(B, &B->c3_free, (g - 1) & 1, status);
            if (ok) {
                tc_fence_after();
                if (elect_one()) {
                    // C3 = [A~N; Y_C] R0 (and [.; Y_P] R0)
                    mma_k64_ka(tmem + kC3, smem_u32(ay(v)), smem_u32(r0), idM);
                    if (kTitans)
                        mma_k64_ka(tmem + kC3 + 64, smem_u32(ay(v)) + 128 * 128, smem_u32(r0), idM);
                    mma_commit(&B->c3_done[v]);
                }
                __syncwarp();
            }
            if (ok && !scored) ok = issue_scores(g + 1);
        }
    }

    // drain the MMAs of the two issuing warps before TMEM is released
    if (warp == 8 || warp == 13) {
        uint64_t* d = &B->drain[warp == 8 ? 0 : 1];
        if (elect_one()) mma_commit(d);
        __syncwarp();
        if (lane == 0) wait_drain(d, 0, B->wait_limit);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool linear_seq_supported(const LinearArgs& a) {
    return a.bf16 && a.dk == kD && a.dv == kD && (a.chunk == 16 || a.chunk == 32) && a.T >= 1 &&
           !a.ckpt && a.z;
}

cudaError_t linear_seq_launch(const LinearArgs& a, cudaStream_t s) {
    const int BH = a.B * a.H;
    CUtensorMap qm, km, vm;
    if (!make_token_tile_map(&qm, a.q, BH, a.T, kD, 64, true) ||
        !make_token_tile_map(&km, a.k, BH, a.T, kD, 64, true) ||
        !make_token_tile_map(&vm, a.v, BH, a.T, kD, 64, true))
        return cudaErrorInvalidValue;
    constexpr Layout L = make_layout();
    const size_t smem = L.total + 1024;
    const bool titans = a.eta || a.alpha || a.S0 || a.S_out;
    if (titans) {
        cudaError_t e = cudaFuncSetAttribute(linear_seq_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        linear_seq_kernel<true><<<BH, kThreads, smem, s>>>(qm, km, vm, a);
    } else {
        cudaError_t e = cudaFuncSetAttribute(linear_seq_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        linear_seq_kernel<false><<<BH, kThreads, smem, s>>>(qm, km, vm, a);
    }
    return cudaGetLastError();
}

}  // namespace ttm
