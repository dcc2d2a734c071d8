// Tensor-core (tcgen05 + TMA) kernel of the chunked linear / Titans memory scan.
//
// Method (per sequence, chunks of 64 tokens; "TTT layers 与 fast weights" §1.1
// eqs (7)-(9) for the matrix form of one chunk, "论文速览 | Titans" §4.3-§4.5
// for the decay / momentum unrolling): with the chunk-start state (W, S), the
// chunk's keys K, queries Q, values V (rows = tokens) and the per-chunk
// coefficients beta_t, c_t, P_t, C[t][s] (see scan_simt.cu for their
// definition),
//
//   E^T  = K W^T - V                       errors at the chunk-start state
//   z_t  = beta_t (Q W^T)_t + c_t (Q S^T)_t - 2 sum_{s<=t} C[t][s] (q_t.k_s) e_s
//   W'   = beta_n W + c_n S - 2 (E diag(C[n][.]) K)
//   S'   = P_n S        - 2 (E diag(Pm[n][.]) K)
//
// Every row of W (and S) evolves independently of the others (its error only
// involves that row), so one CTA owns a slice of 16 rows of one sequence's
// memory and runs the whole sequence; the grid covers (sequence, slice).
//
// The per-chunk coefficients depend only on the gates, so a pre-pass kernel
// (one warp per sequence and chunk) writes them into the caller's workspace:
// the 64 x 64 matrix C (fp32) and the vectors beta_t, c_t, C[n-1][s],
// Pm[n-1][s] and the chunk-end scalars.  The scan kernel copies each chunk's
// record into its pipeline stage next to the K, Q and V tiles.
//
// Roles inside a CTA of the scan kernel (256 threads):
//   warps 0-3  chain.  Thread j holds W[r0..r0+15][j] and S[r0..r0+15][j] in
//              fp32 registers for the whole sequence.  Warps 0-1 (thread =
//              token) turn K W^T into the errors and the scaled error
//              operands; all four apply the state carry; warp 0 issues the
//              two chain MMAs itself after named barriers.
//   warp 4     producer: TMA loads of K, Q (128-byte swizzle) and the V
//              slice, bulk copy of the coefficient record.
//   warp 5     read-side MMA issuer (scores two chunks ahead, corrections)
//              and TMEM owner.
//   warps 6-9  weight the scores by C (warp w takes the 16 tokens of TMEM
//              sub-partition w % 4); warps 6-7 then form the outputs z.
//
// Tensor-core contractions per chunk (A operands are M = 128 rows: the K tile
// and the Q tile are stacked so one instruction covers both):
//   MMA1  [K;Q] . [W;S]^T      -> K W^T (errors), Q W^T, Q S^T     (chain)
//   MMA2  K^T . [C_n E^T | Pm_n E^T] -> the state updates           (chain)
//   MMAqk [K;Q] . K^T          -> Q K^T (scores), one chunk ahead
//   MMAz  A~ . E^T             -> the causal correction of the reads
// Operands are bf16, accumulators fp32 in tensor memory; the fp32 state
// masters never leave registers.
//
// Every wait is bounded: a wait that exceeds its limit sets the device status
// word to TTM_ERR_TIMEOUT, every role stops, in-flight copies and MMAs are
// drained, TMEM is freed and the kernel returns.
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

constexpr int kChunk = 64;      // tokens per chunk (== TMA tile height)
constexpr int kRows = 16;       // rows of W per CTA
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;

// TMEM column map
constexpr uint32_t kAcc1 = 0;     // 2 x 32 columns: [K W^T | K S^T] on lanes 0-63, [Q W^T | Q S^T] on 64-127
constexpr uint32_t kAcc2 = 64;    // 32 columns: W / S updates (lane = d_k index)
constexpr uint32_t kAccQK = 128;  // 3 x 64 columns: Q K^T (M = 64 layout: 16 tokens per sub-partition)
constexpr uint32_t kAccZ = 320;   // 2 x 16 columns: A~ E^T on lanes 64-127

// Per-chunk coefficient record (workspace and pipeline stage).  C[t][s] =
// theta_s w(s,t) (zero above the diagonal) is stored row-major in fp32 with
// the 16-byte chunks of row t XOR-permuted by t % 16, so that 32 threads
// reading 32 different rows stay free of bank conflicts.
constexpr uint32_t kRecC = 0;                    // 64 x 64 fp32
constexpr uint32_t kRecBeta = 16384;             // beta_t
constexpr uint32_t kRecCvec = kRecBeta + 256;    // c_t
constexpr uint32_t kRecCend = kRecCvec + 256;    // C[n-1][s]
constexpr uint32_t kRecPend = kRecCend + 256;    // theta_s m(s, n-1)
constexpr uint32_t kRecScal = kRecPend + 256;    // beta_{n-1}, c_{n-1}, P_{n-1}, n
constexpr uint32_t kRecBytes = kRecScal + 16;    // 17424 (a multiple of 16)

__host__ __device__ constexpr uint32_t c_offset(int t, int s) {
    return (uint32_t)t * 256u + (uint32_t)(((s >> 2) ^ (t & 15)) << 4) + (uint32_t)(s & 3) * 4u;
}

struct Layout {
    int D, NS;
    uint32_t kq_bytes, off_v, off_rec, stage_bytes;
    uint32_t off_ws, off_b2, off_at0, off_et0, off_at1, off_et1, total;
};

// Shared-memory map.  Each A~ tile (8 KB, the 64 rows of the scores) is
// preceded by another 8 KB buffer: its MMA reads 128 rows starting 8 KB
// earlier and only the upper 64 rows of that product are used.
__host__ __device__ constexpr Layout make_layout(int D) {
    Layout L{};
    L.D = D;
    L.NS = D == 128 ? 3 : 4;
    L.kq_bytes = (D / 64) * 16384u;   // per 64-column half: K (8 KB) then Q (8 KB)
    L.off_v = L.kq_bytes;             // V slice, 64 x 16 bf16
    L.off_rec = L.kq_bytes + 2048u;   // coefficient record
    L.stage_bytes = (L.off_rec + kRecBytes + 1023u) & ~1023u;
    uint32_t off = L.NS * L.stage_bytes;
    L.off_ws = off;  off += D * 128u;        // [W;S] operand, row = d_k index
    L.off_b2 = off;  off += kChunk * 128u;   // [C E^T | Pm E^T], row = token
    L.off_at0 = off; off += kChunk * 128u;   // A~ (chunk parity 0)
    L.off_et0 = off; off += kChunk * 128u;   // E^T (chunk parity 0)
    L.off_at1 = off; off += kChunk * 128u;
    L.off_et1 = off; off += kChunk * 128u;
    L.total = off;
    return L;
}

struct Bars {
    uint64_t full[4], empty[4];
    uint64_t mma1_done[2], mma2_done[2], acc1_free[2], at_ready[2], z_done[2], accz_free[2];
    uint64_t qk_done[3], qk_free[3];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

struct TcParams {
    LinearArgs a;
    int nslices;
};

constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_bar(Bars* B, uint64_t* bar, uint32_t parity, int* status) {
    const long long t0 = clock64();
    uint32_t polls = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++polls & 63u) == 0) {
            if (*(volatile int*)&B->abort) return false;
            if (clock64() - t0 > kWaitCycles) {
                *(volatile int*)&B->abort = 1;
                atomicExch(status, TTM_ERR_TIMEOUT);
                return false;
            }
        }
    }
    return true;
}

// Warp-uniform variant: every lane of the warp gets the same answer, so a
// timeout seen by one lane never splits the warp before a .sync.aligned op.
__device__ __forceinline__ bool wait_all(Bars* B, uint64_t* bar, uint32_t parity, int* status) {
    return __all_sync(0xffffffffu, wait_bar(B, bar, parity, status));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Stores 8 consecutive bf16 values (one 16-byte chunk) of row `row` starting
// at column `col` (multiple of 8) into a 128-byte-swizzled tile.
__device__ __forceinline__ void st_chunk(uint8_t* tile, int row, int col, const float* x) {
    uint4 v;
    v.x = pack_bf16(x[0], x[1]);
    v.y = pack_bf16(x[2], x[3]);
    v.z = pack_bf16(x[4], x[5]);
    v.w = pack_bf16(x[6], x[7]);
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, col)) = v;
}

// ---------------------------------------------------------------- warp scans

// Inclusive scan of affine maps x -> A x + B along lanes (lane order = token
// order); the composition puts later lanes outside.
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

// ------------------------------------------------------- coefficient warp

// One warp computes all coefficients of one chunk of n tokens from its raw
// gates g; it first makes the padded tokens neutral in place (eta 1,
// alpha 0; theta is masked where read):
//  * forward scans (lane l owns tokens 2l, 2l+1): beta_t = prod keep,
//    P_t = prod eta, c_t = keep_t c_{t-1} + P_t;
//  * the matrix C[t][s] = theta_s w(s,t) with, per column s, the forward
//    recurrences m(s,t) = eta_t m(s,t-1), w(s,t) = keep_t w(s,t-1) + m(s,t),

// ------------------------------------------------------- coefficient pre-pass

// One warp per (sequence, chunk) of n tokens.  Padded tokens have theta 0
// and eta = keep = 1 (neutral).
//  * forward scans (lane l owns tokens 2l, 2l+1): beta_t = prod keep,
//    P_t = prod eta, c_t = keep_t c_{t-1} + P_t;
//  * C[t][s] = theta_s w(s,t) with, per column s, the forward recurrences
//    m(s,t) = eta_t m(s,t-1), w(s,t) = keep_t w(s,t-1) + m(s,t),
//    m(s,s) = w(s,s) = 1.  Lane l owns columns l and l + 32; all lanes walk
//    the rows together.  A column holds m = w = 0 before its start row and the
//    start enters as an additive unit, so a step is two dependent FMAs and the
//    rows above the diagonal come out as exact zeros.  With neutral gates
//    past the last token m stops changing, so the final m is m(s, n-1).
__global__ void __launch_bounds__(128) linear_coef_kernel(const LinearArgs a, int nch) {
    const int lane = threadIdx.x & 31;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long BH = (long long)a.B * a.H;
    if (wid >= BH * nch) return;
    const int seq = (int)(wid / nch), c = (int)(wid % nch);
    const int T = a.T;
    const int n = min(kChunk, T - c * kChunk);
    const size_t tok0 = (size_t)seq * T + (size_t)c * kChunk;
    uint8_t* rec = static_cast<uint8_t*>(a.workspace) + (size_t)wid * kRecBytes;

    auto eta_at = [&](int t) { return t < n ? (a.eta ? a.eta[tok0 + t] : 0.f) : 1.f; };
    auto keep_at = [&](int t) { return t < n ? 1.f - (a.alpha ? a.alpha[tok0 + t] : 0.f) : 1.f; };
    auto theta_at = [&](int t) { return t < n ? a.theta[tok0 + t] : 0.f; };

    // forward scans
    const int t0 = 2 * lane, t1 = t0 + 1;
    const float et0 = eta_at(t0), et1 = eta_at(t1), kp0 = keep_at(t0), kp1 = keep_at(t1);
    float Ab = kp0 * kp1, Bb = 0.f;
    float Ap = et0 * et1, Bp = 0.f;
    scan_affine_up(Ab, Bb, lane);
    scan_affine_up(Ap, Bp, lane);
    float pre_b = __shfl_up_sync(0xffffffffu, Ab, 1);
    float pre_p = __shfl_up_sync(0xffffffffu, Ap, 1);
    if (lane == 0) pre_b = pre_p = 1.f;
    const float beta0 = pre_b * kp0, beta1 = beta0 * kp1;
    const float P0 = pre_p * et0, P1 = P0 * et1;
    float Ac = kp1 * kp0, Bc = kp1 * P0 + P1;
    scan_affine_up(Ac, Bc, lane);
    float cpre = __shfl_up_sync(0xffffffffu, Bc, 1);
    if (lane == 0) cpre = 0.f;
    const float c0 = kp0 * cpre + P0, c1 = kp1 * c0 + P1;
    float* beta = reinterpret_cast<float*>(rec + kRecBeta);
    float* cvec = reinterpret_cast<float*>(rec + kRecCvec);
    reinterpret_cast<float2*>(beta)[lane] = make_float2(beta0, beta1);
    reinterpret_cast<float2*>(cvec)[lane] = make_float2(c0, c1);
    const int ln = (n - 1) >> 1, un = (n - 1) & 1;
    const float bn = __shfl_sync(0xffffffffu, un ? beta1 : beta0, ln);
    const float cn = __shfl_sync(0xffffffffu, un ? c1 : c0, ln);
    const float Pn = __shfl_sync(0xffffffffu, un ? P1 : P0, ln);
    if (lane == 0)
        *reinterpret_cast<float4*>(rec + kRecScal) = make_float4(bn, cn, Pn, (float)n);

    // C matrix
    const int s0 = lane, s1 = lane + 32;
    const float th0 = theta_at(s0), th1 = theta_at(s1);
    const float e_lo = eta_at(s0), e_hi = eta_at(s1), k_lo = keep_at(s0), k_hi = keep_at(s1);
    float m0 = 0.f, w0 = 0.f, m1 = 0.f, w1 = 0.f, ce0 = 0.f, ce1 = 0.f;
#pragma unroll
    for (int t = 0; t < kChunk; ++t) {
        const float e = __shfl_sync(0xffffffffu, t < 32 ? e_lo : e_hi, t & 31);
        const float k1 = __shfl_sync(0xffffffffu, t < 32 ? k_lo : k_hi, t & 31);
        const float d = (lane == (t & 31)) ? 1.f : 0.f;   // start of column t
        if (t < 32) {
            m0 = fmaf(e, m0, d);
            m1 = e * m1;
        } else {
            m0 = e * m0;
            m1 = fmaf(e, m1, d);
        }
        w0 = fmaf(k1, w0, m0);
        w1 = fmaf(k1, w1, m1);
        const float v0 = th0 * w0, v1 = th1 * w1;
        *reinterpret_cast<float*>(rec + kRecC + c_offset(t, s0)) = v0;
        *reinterpret_cast<float*>(rec + kRecC + c_offset(t, s1)) = v1;
        if (t == n - 1) {
            ce0 = v0;
            ce1 = v1;
        }
    }
    float* cend = reinterpret_cast<float*>(rec + kRecCend);
    float* pend = reinterpret_cast<float*>(rec + kRecPend);
    cend[s0] = ce0;
    cend[s1] = ce1;
    pend[s0] = th0 * m0;
    pend[s1] = th1 * m1;
}

// ------------------------------------------------------------- scan kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
linear_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap vmap, const TcParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ Bars bars;
    Bars* B = &bars;
    constexpr Layout L = make_layout(D);
    const LinearArgs& a = P.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = blockIdx.x % P.nslices;
    const int seq = blockIdx.x / P.nslices;
    const int bb = seq / a.H, hh = seq % a.H;
    const int r0 = slice * kRows;
    const int T = a.T;
    const int nch = (T + kChunk - 1) / kChunk;
    int* status = a.status;

    auto stage = [&](int s) { return sm + s * L.stage_bytes; };
    auto vtile = [&](int s) { return stage(s) + L.off_v; };
    auto rec = [&](int s) { return stage(s) + L.off_rec; };
    auto recf = [&](int s, uint32_t off) { return reinterpret_cast<const float*>(rec(s) + off); };
    uint8_t* ws = sm + L.off_ws;
    uint8_t* b2 = sm + L.off_b2;
    auto et = [&](int b) { return sm + (b ? L.off_et1 : L.off_et0); };
    auto at = [&](int b) { return sm + (b ? L.off_at1 : L.off_at0); };

    if (tid == 0) {
        for (int s = 0; s < L.NS; ++s) {
            mbar_init(&B->full[s], 1);
            // chain 128 + read side 128 + chain MMA commit 1 + score MMA commit 1
            mbar_init(&B->empty[s], 128 + 128 + 1 + 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&B->mma1_done[b], 1);
            mbar_init(&B->mma2_done[b], 1);
            mbar_init(&B->acc1_free[b], 64);
            mbar_init(&B->at_ready[b], 128);
            mbar_init(&B->z_done[b], 1);
            mbar_init(&B->accz_free[b], 64);
        }
        for (int b = 0; b < 3; ++b) {
            mbar_init(&B->qk_done[b], 1);
            mbar_init(&B->qk_free[b], 128);
        }
        mbar_init(&B->drain, 1);
        B->abort = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(&B->tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;

    const uint32_t id1 = idesc_bf16_f32(128, 32, 0, 1);
    const uint32_t id2 = idesc_bf16_f32(128, 32, 1, 1);

    if (warp < 4) {
        // ----------------------------------------------------- chain warps
        // Every thread runs every iteration and reaches every named barrier,
        // also after an abort (then it only skips work), so the barriers
        // stay balanced.
        const int j = tid;
        const bool own = j < D;
        const size_t init = (size_t)(a.shared ? 0 : bb) * a.H + hh;
        float w[kRows], s[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const size_t idx = (init * D + r0 + i) * (size_t)D + j;
            w[i] = own ? a.W0[idx] : 0.f;
            s[i] = (own && a.S0) ? a.S0[idx] : 0.f;
        }
        auto write_ws = [&]() {
            if (!own) return;
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) st_chunk(ws, j, 8 * c8, w + 8 * c8);
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) st_chunk(ws, j, 16 + 8 * c8, s + 8 * c8);
        };
        const uint32_t ws_a = smem_u32(ws), b2_a = smem_u32(b2);
        // MMA1(c): [K;Q] . [W;S]^T, issued by warp 0 once [W;S] is in place
        auto issue_mma1 = [&](int c, bool ok) -> bool {
            if (warp != 0 || nch == 0) return ok;
            const int st = c % L.NS, b = c & 1;
            if (ok) ok = wait_all(B, &B->full[st], (c / L.NS) & 1, status);
            if (ok && c >= 2) ok = wait_all(B, &B->acc1_free[b], ((c - 2) >> 1) & 1, status);
            if (!ok) return false;
            tc_fence_after();
            const uint32_t base = smem_u32(stage(st));
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ad = base + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + kAcc1 + b * 32, sdesc(ad, 16, 1024, 2),
                             sdesc(ws_a + kk * 2048, 8192, 1024, 2), id1, kk > 0);
                }
                mma_commit(&B->mma1_done[b]);
            }
            __syncwarp();
            return true;
        };
        write_ws();
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        bool ok = issue_mma1(0, true);
        for (int c = 0; c < nch; ++c) {
            const int st = c % L.NS, b = c & 1;
            if (ok) ok = wait_all(B, &B->full[st], (c / L.NS) & 1, status);
            if (warp < 2) {
                // Epi1: errors of token t at the chunk-start state
                const int t = j;
                if (ok) ok = wait_all(B, &B->mma1_done[b], (c >> 1) & 1, status);
                if (ok && c >= 2) ok = wait_all(B, &B->z_done[b], ((c - 2) >> 1) & 1, status);
                if (ok) {
                    const float ce = recf(st, kRecCend)[t], pe = recf(st, kRecPend)[t];
                    tc_fence_after();
                    float kw[16];
                    tmem_ld16(tmem_addr(tmem, warp * 32, kAcc1 + b * 32), kw);
                    const uint4* vrow = reinterpret_cast<const uint4*>(vtile(st) + t * 32);
                    const uint4 v0 = vrow[0], v1 = vrow[1];
                    tmem_wait_ld();
                    const __nv_bfloat162* vb0 = reinterpret_cast<const __nv_bfloat162*>(&v0);
                    const __nv_bfloat162* vb1 = reinterpret_cast<const __nv_bfloat162*>(&v1);
                    float e[16], ec[16], ep[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f0 = __bfloat1622float2(vb0[i]);
                        const float2 f1 = __bfloat1622float2(vb1[i]);
                        e[2 * i] = kw[2 * i] - f0.x;
                        e[2 * i + 1] = kw[2 * i + 1] - f0.y;
                        e[8 + 2 * i] = kw[8 + 2 * i] - f1.x;
                        e[8 + 2 * i + 1] = kw[8 + 2 * i + 1] - f1.y;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        ec[i] = ce * e[i];
                        ep[i] = pe * e[i];
                    }
                    st_chunk(b2, t, 0, ec);
                    st_chunk(b2, t, 8, ec + 8);
                    st_chunk(b2, t, 16, ep);
                    st_chunk(b2, t, 24, ep + 8);
                    st_chunk(et(b), t, 0, e);
                    st_chunk(et(b), t, 8, e + 8);
                    fence_proxy_async_smem();
                    tc_fence_before();
                }
                named_bar_sync(2, 64);
                // MMA2(c): K^T . [C E^T | Pm E^T]
                if (warp == 0 && ok) {
                    tc_fence_after();
                    const uint32_t base = smem_u32(stage(st));
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kChunk / 16; ++kk)
                            mma_bf16(tmem + kAcc2,
                                     sdesc(base + kk * 2048, D == 128 ? 16384 : 8192, 1024, 2),
                                     sdesc(b2_a + kk * 2048, 8192, 1024, 2), id2, kk > 0);
                        mma_commit(&B->mma2_done[b]);
                        mma_commit(&B->empty[st]);
                    }
                    __syncwarp();
                }
            }
            // Epi2: state carry
            if (ok) ok = wait_all(B, &B->mma2_done[b], (c >> 1) & 1, status);
            if (ok) {
                const float* sc = recf(st, kRecScal);
                const float bn = sc[0], cn = sc[1], Pn = sc[2];
                mbar_arrive(&B->empty[st]);
                tc_fence_after();
                if (own) {
                    float uw[16], us[16];
                    tmem_ld16(tmem_addr(tmem, warp * 32, kAcc2), uw);
                    tmem_ld16(tmem_addr(tmem, warp * 32, kAcc2 + 16), us);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < kRows; ++i) {
                        const float wn = bn * w[i] + cn * s[i] - 2.f * uw[i];
                        s[i] = Pn * s[i] - 2.f * us[i];
                        w[i] = wn;
                    }
                }
                if (c + 1 < nch) {
                    write_ws();
                    fence_proxy_async_smem();
                }
                tc_fence_before();
            }
            named_bar_sync(1, 128);
            if (c + 1 < nch) ok = issue_mma1(c + 1, ok);
        }
        if (own) {
            const size_t dst = (size_t)seq * D * D;
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                a.W_out[dst + (size_t)(r0 + i) * D + j] = w[i];
                if (a.S_out) a.S_out[dst + (size_t)(r0 + i) * D + j] = s[i];
            }
        }
    } else if (warp == 4) {
        // --------------------------------------------------------- producer
        if (lane == 0) {
            const uint32_t tx = L.kq_bytes + kChunk * kRows * 2 + kRecBytes;
            const uint8_t* recs = static_cast<const uint8_t*>(a.workspace) +
                                  (size_t)seq * nch * kRecBytes;
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int st = c % L.NS;
                if (c >= L.NS && !wait_bar(B, &B->empty[st], ((c / L.NS) - 1) & 1, status)) break;
                mbar_expect_tx(&B->full[st], tx);
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    tma_load_3d(stage(st) + h * 16384, &kmap, &B->full[st], 64 * h, c * kChunk, seq);
                    tma_load_3d(stage(st) + h * 16384 + 8192, &qmap, &B->full[st], 64 * h,
                                c * kChunk, seq);
                }
                tma_load_3d(vtile(st), &vmap, &B->full[st], r0, c * kChunk, seq);
                bulk_load(rec(st), recs + (size_t)c * kRecBytes, kRecBytes, &B->full[st]);
                issued = c + 1;
            }
            // drain: every issued stage's copies must have landed before exit
            for (int c = (issued > L.NS ? issued - L.NS : 0); c < issued; ++c) {
                const long long t0 = clock64();
                while (!mbar_try_wait(&B->full[c % L.NS], (c / L.NS) & 1))
                    if (clock64() - t0 > kWaitCycles) break;
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------ read-side MMA issuer
        // The correction MMA of chunk c-1 goes right after MMA1(c) completes
        // (it runs while the errors of chunk c are formed); the scores run two
        // chunks ahead, issued after MMA2(c) completes (during the carry).
        if (nch > 0) {
            const uint32_t idqk = idesc_bf16_f32(64, 64, 0, 0);
            const uint32_t idz = idesc_bf16_f32(128, 16, 0, 1);
            auto issue_qk = [&](int c) -> bool {
                const int q = c % 3, st = c % L.NS;
                bool ok = wait_all(B, &B->full[st], (c / L.NS) & 1, status);
                if (ok && c >= 3) ok = wait_all(B, &B->qk_free[q], ((c - 3) / 3) & 1, status);
                if (!ok) return false;
                tc_fence_after();
                const uint32_t base = smem_u32(stage(st));
                const uint32_t d = tmem + kAccQK + q * 64;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t half = base + (kk >> 2) * 16384 + (kk & 3) * 32;
                        // A = the 64 Q rows (8 KB after the K rows), B = the 64 K rows
                        mma_bf16(d, sdesc(half + 8192, 16, 1024, 2), sdesc(half, 16, 1024, 2), idqk,
                                 kk > 0);
                    }
                    mma_commit(&B->qk_done[q]);
                    mma_commit(&B->empty[st]);
                }
                __syncwarp();
                return true;
            };
            auto issue_z = [&](int c) -> bool {
                const int b = c & 1;
                bool ok = wait_all(B, &B->at_ready[b], (c >> 1) & 1, status);
                if (ok && c >= 2) ok = wait_all(B, &B->accz_free[b], ((c - 2) >> 1) & 1, status);
                if (!ok) return false;
                tc_fence_after();
                // 128-row A operand starting 8 KB before the 64 rows of A~
                const uint32_t at_a = smem_u32(at(b)) - 8192, et_a = smem_u32(et(b));
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kChunk / 16; ++kk)
                        mma_bf16(tmem + kAccZ + b * 16, sdesc(at_a + kk * 32, 16, 1024, 2),
                                 sdesc(et_a + kk * 2048, 8192, 1024, 2), idz, kk > 0);
                    mma_commit(&B->z_done[b]);
                }
                __syncwarp();
                return true;
            };
            bool ok = issue_qk(0);
            if (ok && nch > 1) ok = issue_qk(1);
            for (int c = 0; c < nch && ok; ++c) {
                ok = wait_all(B, &B->mma1_done[c & 1], (c >> 1) & 1, status);
                if (ok && c >= 1) ok = issue_z(c - 1);
                if (ok) ok = wait_all(B, &B->mma2_done[c & 1], (c >> 1) & 1, status);
                if (ok && c + 2 < nch) ok = issue_qk(c + 2);
            }
            if (ok) issue_z(nch - 1);
            // drain: all MMAs issued by this thread complete before TMEM is
            // released (the chain's own MMAs were waited for by the chain)
            if (elect_one()) mma_commit(&B->drain);
            __syncwarp();
            const long long t0 = clock64();
            while (!mbar_try_wait(&B->drain, 0))
                if (clock64() - t0 > kWaitCycles) break;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ read side (6-9)
        // Score weighting: warp w owns TMEM sub-partition p = w % 4, i.e. the
        // tokens 16p + lane (lane < 16) of the M = 64 score accumulator.
        const int p = warp & 3;
        const int ta = 16 * p + lane;        // token of this lane in A~ (lane < 16)
        const bool zw = warp < 8;            // warps 6-7 also form the outputs
        const int t = tid - 192;             // output token of warps 6-7 (TMEM lane 64 + t)
        const int wl = (warp & 3) * 32;
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const int st = c % L.NS, b = c & 1, q = c % 3;
            ok = wait_all(B, &B->full[st], (c / L.NS) & 1, status);
            if (ok) ok = wait_all(B, &B->qk_done[q], (c / 3) & 1, status);
            if (ok && c >= 2) ok = wait_all(B, &B->z_done[b], ((c - 2) >> 1) & 1, status);
            if (!ok) break;
            tc_fence_after();
            // A~[t][s] = C[t][s] (q_t . k_s); C is zero above the diagonal
            const uint8_t* crow = rec(st) + kRecC + ta * 256;
            uint8_t* arow = at(b);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float r[16];
                tmem_ld16(tmem_addr(tmem, wl, kAccQK + q * 64 + 16 * q4), r);
                float cv[16];
                if (lane < 16) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float4 f = *reinterpret_cast<const float4*>(
                            crow + (((4 * q4 + jj) ^ (ta & 15)) << 4));
                        cv[4 * jj] = f.x;
                        cv[4 * jj + 1] = f.y;
                        cv[4 * jj + 2] = f.z;
                        cv[4 * jj + 3] = f.w;
                    }
                }
                tmem_wait_ld();
                if (lane < 16) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) r[i] *= cv[i];
                    st_chunk(arow, ta, 16 * q4, r);
                    st_chunk(arow, ta, 16 * q4 + 8, r + 8);
                }
            }
            tc_fence_before();
            mbar_arrive(&B->qk_free[q]);
            fence_proxy_async_smem();
            mbar_arrive(&B->at_ready[b]);
            if (!zw) {
                mbar_arrive(&B->empty[st]);
                continue;
            }
            const float bt = recf(st, kRecBeta)[t], ct = recf(st, kRecCvec)[t];
            const int n = (int)recf(st, kRecScal)[3];
            mbar_arrive(&B->empty[st]);
            // reads: z_t = beta_t Q W^T + c_t Q S^T - 2 A~ E^T
            ok = wait_all(B, &B->mma1_done[b], (c >> 1) & 1, status);
            if (!ok) break;
            tc_fence_after();
            float qw[16], qs[16], ae[16];
            tmem_ld16(tmem_addr(tmem, wl, kAcc1 + b * 32), qw);
            tmem_ld16(tmem_addr(tmem, wl, kAcc1 + b * 32 + 16), qs);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&B->acc1_free[b]);
            ok = wait_all(B, &B->z_done[b], (c >> 1) & 1, status);
            if (!ok) break;
            tc_fence_after();
            tmem_ld16(tmem_addr(tmem, wl, kAccZ + b * 16), ae);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&B->accz_free[b]);
            if (t < n) {
                float zz[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) zz[i] = bt * qw[i] + ct * qs[i] - 2.f * ae[i];
                uint4 o0, o1;
                o0.x = pack_bf16(zz[0], zz[1]);   o0.y = pack_bf16(zz[2], zz[3]);
                o0.z = pack_bf16(zz[4], zz[5]);   o0.w = pack_bf16(zz[6], zz[7]);
                o1.x = pack_bf16(zz[8], zz[9]);   o1.y = pack_bf16(zz[10], zz[11]);
                o1.z = pack_bf16(zz[12], zz[13]); o1.w = pack_bf16(zz[14], zz[15]);
                __nv_bfloat16* zr = static_cast<__nv_bfloat16*>(a.z) +
                                    ((size_t)seq * T + (size_t)c * kChunk + t) * D + r0;
                reinterpret_cast<uint4*>(zr)[0] = o0;
                reinterpret_cast<uint4*>(zr)[1] = o1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
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

// 3-D view [sequences][T][D] of a bf16 tensor, tile box {bx, 64, 1}.
bool make_map(CUtensorMap* m, const void* ptr, int BH, int T, int D, int bx, bool swz) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)bx, (cuuint32_t)kChunk, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

bool linear_tc_supported(const LinearArgs& a) {
    return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128) && a.chunk == kChunk &&
           a.T >= 1;
}

size_t linear_tc_workspace_bytes(const LinearArgs& a) {
    const size_t nch = ((size_t)a.T + kChunk - 1) / kChunk;
    return (size_t)a.B * a.H * nch * kRecBytes;
}

cudaError_t linear_tc_launch(const LinearArgs& a, cudaStream_t s) {
    const int D = a.dk, BH = a.B * a.H;
    const int nch = (a.T + kChunk - 1) / kChunk;
    if (!a.workspace || a.workspace_bytes < linear_tc_workspace_bytes(a) ||
        (reinterpret_cast<uintptr_t>(a.workspace) & 15u))
        return cudaErrorInvalidValue;
    {
        const long long warps = (long long)BH * nch;
        const unsigned blocks = (unsigned)((warps + 3) / 4);
        linear_coef_kernel<<<blocks, 128, 0, s>>>(a, nch);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    CUtensorMap km, qm, vm;
    if (!make_map(&km, a.k, BH, a.T, D, 64, true) || !make_map(&qm, a.q, BH, a.T, D, 64, true) ||
        !make_map(&vm, a.v, BH, a.T, D, kRows, false))
        return cudaErrorInvalidValue;
    TcParams p{a, D / kRows};
    const Layout L = make_layout(D);
    const size_t smem = L.total + 1024;
    dim3 grid(BH * (D / kRows));
    if (D == 128) {
        cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        linear_tc_kernel<128><<<grid, kThreads, smem, s>>>(km, qm, vm, p);
    } else {
        cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        linear_tc_kernel<64><<<grid, kThreads, smem, s>>>(km, qm, vm, p);
    }
    return cudaGetLastError();
}

}  // namespace ttm
