// Tensor-core (tcgen05 + TMA) kernel of the chunked linear / Titans memory scan.
//
// Method (per sequence, chunks of 64 tokens; "TTT layers 与 fast weights" §1.1
// eqs (7)-(9) for the matrix form of one chunk, "论文速览 | Titans" §4.3-§4.5
// for the decay / momentum unrolling): with the chunk-start state (W_c, S_c),
// the chunk's keys K_c, queries Q_c, values V_c (rows = tokens) and the
// chunk coefficients beta_t, c_t, P_t, C[t][s], Pm[t][s] (see scan_simt.cu),
//
//   E_c  = K_c W_c^T - V_c                           errors at the chunk start
//   z_t  = beta_t (Q W^T)_t + c_t (Q S^T)_t - 2 sum_{s<=t} C[t][s] (q_t.k_s) e_s
//   W_{c+1} = beta_n W_c + c_n S_c - 2 E_c^T diag(C[n]) K_c
//   S_{c+1} = P_n S_c            - 2 E_c^T diag(Pm[n]) K_c
//
// Serial chain.  Substituting the carry into the next chunk's errors gives
//
//   E_{c+1} = beta_n K_{c+1} W_c^T + c_n K_{c+1} S_c^T
//             - 2 (K_{c+1} K_c^T diag(C[n])) E_c - V_{c+1},
//
// whose first two terms only need the state at the start of chunk c and whose
// matrix M_c = K_{c+1} K_c^T diag(C[n]) only needs the inputs.  So the chain
// from one chunk's errors to the next is a single tensor-core product M_c E_c
// plus an elementwise epilogue; the state carry itself (an MMA and a register
// update) runs beside it, one chunk ahead of where its result is needed.
//
// Stacked operands.  The queries of chunk c and the keys of chunk c+1 sit next
// to each other in shared memory (a ring of [K_0][Q_0][K_1][Q_1]... tiles with
// the first key tile duplicated at the end), so one 128-row A operand
// [Q_c; K_{c+1}] serves
//   scores  [Q_c; K_{c+1}] K_c^T       -> A~_c = mask(Q K^T) o C and M_c
//   state   [Q_c; K_{c+1}] [W_c; S_c]^T -> Q W^T, Q S^T (reads) and the two
//                                          state terms of E_{c+1}
// and the chain product [A~_c; M_c] E_c gives the read correction of chunk c
// and the recursion term of E_{c+1} in one go.
//
// Every row of W (and S) evolves independently of the others, so one CTA owns
// a slice of 16 rows of one sequence's memory and runs the whole sequence; the
// grid covers (sequence, slice).  The per-chunk coefficients depend only on
// the gates and come from a pre-pass kernel (one warp per sequence and chunk)
// through the caller's workspace.
//
// Roles inside a CTA (512 threads):
//   warps 0-3   state: thread j holds column j of the 16 W rows and 16 S rows
//               in fp32 registers, applies the carry and writes the bf16 copy
//               [W; S] for the state MMA, which warp 0 issues.
//   warps 4-5   outputs z (token = TMEM lane 0-63).
//   warps 6-7,  error chain (token of the next chunk = TMEM lane 64-127; warps
//   14-15       6-7 take columns 0-7 of a row, warps 14-15 columns 8-15);
//               warp 6 issues the chain MMA, warp 7 then the carry MMA.
//   warps 8-11  score weighting (TMEM sub-partition = warp % 4); warp 8
//               issues the score MMAs ahead of the chain.
//   warp 12     producer: TMA loads of K, Q, the V slice and the coefficient
//               record, L2 prefetch four chunks ahead.
//   warp 13     idle.
//
// Every wait is bounded: a wait that exceeds its limit sets the device status
// word to TTM_ERR_TIMEOUT, every role runs out its loop doing no further work
// (named barriers stay balanced), in-flight copies and MMAs are drained, TMEM
// is freed and the kernel returns.
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
constexpr int kThreads = 512;
constexpr int kNS = 3;          // pipeline stages
constexpr uint32_t kTmemCols = 512;

// TMEM column map (M = 128 accumulators: row = TMEM lane)
constexpr uint32_t kAcc1 = 0;     // 2 x 32: [Q_c; K_{c+1}] [W_c; S_c]^T
constexpr uint32_t kAccS = 64;    // 2 x 64: [Q_c; K_{c+1}] K_c^T (raw scores)
constexpr uint32_t kAcc2 = 192;   // 2 x 32: K_c^T [C E | Pm E] (lane = d_k index)
constexpr uint32_t kAcc3 = 256;   // 2 x 16: [A~_c; M_c] E_c
constexpr uint32_t kAM = 288;     // 2 x 32: [A~_c; M_c] as a bf16 A operand (two values per column)

// Per-chunk coefficient record (workspace, staged whole into shared memory).
// C[t][s] = theta_s w(s,t) (zero above the diagonal) in fp32, row t at
// t * 256 bytes with its sixteen 16-byte groups XOR-permuted by t % 16 (so the
// weighting threads, one row each, read without bank conflicts), then vectors
// over the chunk's tokens and four scalars.
constexpr uint32_t kRecC = 0;                    // 64 x 64 fp32
constexpr uint32_t kVBeta = 16384;               // beta_t
constexpr uint32_t kVCvec = kVBeta + 256;        // c_t
constexpr uint32_t kVCend = kVBeta + 512;        // C[n-1][s]
constexpr uint32_t kVPend = kVBeta + 768;        // theta_s m(s, n-1)
constexpr uint32_t kVScal = kVBeta + 1024;       // beta_{n-1}, c_{n-1}, P_{n-1}, n
constexpr uint32_t kRecBytes = kVScal + 16;      // 17424 (a multiple of 16)
constexpr uint32_t kVecSlot = 17472;             // staged copy, 64-byte aligned slots

static_assert(kRecBytes == kCoefRecBytes && kVBeta == kCoefVec && kVCvec == kCoefVec + kCoefC &&
                  kVCend == kCoefVec + kCoefCend && kVPend == kCoefVec + kCoefPend &&
                  kVScal == kCoefVec + kCoefScal,
              "coefficient record layout");

__host__ __device__ constexpr uint32_t c_offset(int t, int s) {
    return (uint32_t)t * 256u + (uint32_t)(((s >> 2) ^ (t & 15)) << 4) + (uint32_t)(s & 3) * 4u;
}

constexpr uint32_t kTile = 8192;                          // 64 rows x 128 bytes
constexpr uint32_t kRingBytes = (2 * kNS + 1) * kTile;    // [K_0][Q_0]...[K_2][Q_2][K_0 copy]

struct Bars {
    uint64_t full[kNS], empty[kNS];
    uint64_t acc1_ready[2], acc1_free[2], sc_ready[2], am_ready[2];
    uint64_t mma3_done[2], acc3_free[2], mma2_done[2], acc2_free[2], mma3_issued;
    uint64_t drain[4];
    long long wait_limit;   // SM clock cycles a wait may take before it gives up
    uint32_t tmem_base;
    int abort;
};

struct Layout {
    uint32_t off_ete, off_ring, off_etcp, off_ws, off_v, off_rec, off_bars, total;
};

// Shared-memory map.  The error tile E (8 KB) sits right before the key /
// query ring, so the first state MMA, whose A operand starts one tile before
// the first key tile, reads valid memory.
__host__ __device__ constexpr Layout make_layout(int D) {
    Layout L{};
    uint32_t off = 0;
    L.off_ete = off;  off += kTile;                        // E_c [t][r] (16 of 64 columns)
    L.off_ring = off; off += (D / 64) * kRingBytes;       // one ring per 64-column half
    L.off_etcp = off; off += 2 * kTile;                    // 2 x [C E | Pm E] [t][r'] (32 columns)
    L.off_ws = off;   off += D * 128;                      // [W; S]^T bf16 [j][r'] (32 of 64 columns)
    L.off_v = off;    off += kNS * 2048;                   // V slice [t][16]
    L.off_rec = off;  off += kNS * kVecSlot;               // coefficient record
    L.off_bars = off; off += (sizeof(Bars) + 15) & ~size_t(15);   // mbarriers (no static smem)
    L.total = off;
    return L;
}


struct TcParams {
    LinearArgs a;
    int nslices;
};

constexpr long long kWaitCycles = 4000000000LL;  // default limit, ~2 s at 2 GHz

// Bounded wait that also gives up once another role has aborted (the slow
// path, out of line: ~25 call sites share one copy of it).
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
    if (mbar_try_wait(bar, parity)) return true;   // already complete: no clock, no loop
    return wait_bar_slow(B, bar, parity, status);
}

// Warp-uniform variant: every lane of the warp gets the same answer, so a
// timeout seen by one lane never splits the warp before a .sync.aligned op.
// A converged warp reads the phase once for all lanes, so a completed phase
// needs only the vote.
__device__ __noinline__ bool wait_all_slow(Bars* B, uint64_t* bar, uint32_t parity, int* status) {
    return __all_sync(0xffffffffu, wait_bar_slow(B, bar, parity, status));
}

__device__ __forceinline__ bool wait_all(Bars* B, uint64_t* bar, uint32_t parity, int* status) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    return wait_all_slow(B, bar, parity, status);
}

// Wait used while draining: ignores the abort flag, gives up after the limit.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) break;
}

// One arrival for the whole warp, after every lane's prior work (the lanes
// converge first, which orders their memory and tcgen05 operations).
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
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

__device__ __forceinline__ void unpack8(uint4 v, float* x) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// Use index of a double-buffered slot by chunk x >= -1 (slot x & 1): chunks
// -1, 1, 3, ... and 0, 2, 4, ... count up separately.
__device__ __forceinline__ uint32_t use_parity(int x) { return (uint32_t)(((x + 1) >> 1) & 1); }

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
    uint8_t* rec = static_cast<uint8_t*>(a.workspace) + (size_t)wid * kRecBytes;
    uint8_t* vec = rec;

    auto gi = [&](int t) { return gate_index(a, (size_t)seq, c * kChunk + t); };
    auto eta_at = [&](int t) { return t < n ? (a.eta ? a.eta[gi(t)] : 0.f) : 1.f; };
    auto keep_at = [&](int t) { return t < n ? 1.f - (a.alpha ? a.alpha[gi(t)] : 0.f) : 1.f; };
    auto theta_at = [&](int t) { return t < n ? a.theta[gi(t)] : 0.f; };

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
    reinterpret_cast<float2*>(vec + kVBeta)[lane] = make_float2(beta0, beta1);
    reinterpret_cast<float2*>(vec + kVCvec)[lane] = make_float2(c0, c1);
    const int ln = (n - 1) >> 1, un = (n - 1) & 1;
    const float bn = __shfl_sync(0xffffffffu, un ? beta1 : beta0, ln);
    const float cn = __shfl_sync(0xffffffffu, un ? c1 : c0, ln);
    const float Pn = __shfl_sync(0xffffffffu, un ? P1 : P0, ln);
    if (lane == 0)
        *reinterpret_cast<float4*>(vec + kVScal) = make_float4(bn, cn, Pn, (float)n);

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
    float* cend = reinterpret_cast<float*>(vec + kVCend);
    float* pend = reinterpret_cast<float*>(vec + kVPend);
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
    constexpr Layout L = make_layout(D);
    Bars* B = reinterpret_cast<Bars*>(sm + L.off_bars);
    constexpr int NH = D / 64;         // 64-column halves
    constexpr int KS = D / 16;         // K steps over d
    const LinearArgs& a = P.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = blockIdx.x % P.nslices;
    const int seq = blockIdx.x / P.nslices;
    const int bb = seq / a.H, hh = seq % a.H;
    const int r0 = slice * kRows;
    const int T = a.T;
    const int nch = (T + kChunk - 1) / kChunk;
    int* status = a.status;
    const uint8_t* recs = static_cast<const uint8_t*>(a.workspace) + (size_t)seq * nch * kRecBytes;

    auto ring = [&](int h) { return sm + L.off_ring + h * kRingBytes; };
    auto ktile = [&](int h, int s) { return ring(h) + 2 * s * kTile; };
    auto qtile = [&](int h, int s) { return ring(h) + (2 * s + 1) * kTile; };
    auto vtile = [&](int s) { return sm + L.off_v + s * 2048; };
    auto vec = [&](int s) { return sm + L.off_rec + s * kVecSlot; };
    auto vecf = [&](int s, uint32_t off) { return reinterpret_cast<const float*>(vec(s) + off); };
    uint8_t* ete = sm + L.off_ete;
    auto etcp = [&](int b) { return sm + L.off_etcp + b * kTile; };
    uint8_t* ws = sm + L.off_ws;

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&B->full[s], 1);
            mbar_init(&B->empty[s], 2);          // outputs + state
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&B->acc1_ready[b], 1);
            mbar_init(&B->acc1_free[b], 6);      // error chain 4 warps + outputs 2
            mbar_init(&B->sc_ready[b], 1);
            mbar_init(&B->mma3_done[b], 1);
            mbar_init(&B->acc3_free[b], 6);      // error chain 4 warps + outputs 2
            mbar_init(&B->mma2_done[b], 1);
            mbar_init(&B->acc2_free[b], 4);      // state warps
        }
        mbar_init(&B->am_ready[0], 4);           // weighting warps
        mbar_init(&B->am_ready[1], 4);
        mbar_init(&B->mma3_issued, 1);           // chain MMA queued (carry MMA goes after it)
        for (int i = 0; i < 4; ++i) mbar_init(&B->drain[i], 1);
        B->wait_limit = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;
        B->abort = 0;
        fence_mbar_init();
    }
    if (warp == 4) tmem_alloc(&B->tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(warp & 3) * 32 << 16);   // this warp's TMEM lanes

    // [Q_c; K_{c+1}] K-major operand address for K step kk (c = -1: the rows
    // before the first key tile, whose products are never read)
    auto qk_a = [&](int c, int kk) -> uint32_t {
        const int h = kk >> 2;
        const uint8_t* base = c < 0 ? ktile(h, 0) - kTile : qtile(h, c % kNS);
        return smem_u32(base) + (kk & 3) * 32;
    };
    // Every MMA sequence below is unrolled so its descriptors are fixed at
    // compile time: issued from a rolled loop, one MMA left the issuing thread
    // every ~90 cycles, against ~40-50 (the pipe's own rate) unrolled.
    constexpr uint32_t id1 = idesc_bf16_f32(128, 32, 0, 1);   // state MMA, B MN-major
    constexpr uint32_t idS = idesc_bf16_f32(128, 64, 0, 0);   // scores
    constexpr uint32_t id2 = idesc_bf16_f32(128, 32, 1, 1);   // carry: A = K^T, B = [C E | Pm E]
    constexpr uint32_t id3 = idesc_bf16_f32(128, 16, 0, 1);   // chain: [A~; M] E

    if (warp < 4) {
        // ------------------------------------------------------------ state
        // Every thread runs every iteration and reaches every named barrier,
        // also after an abort (then it only skips work).
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
        // the state operand MN-major: row j holds W[.][j] then S[.][j], so
        // thread j writes its column with four 16-byte stores
        auto write_ws = [&]() {
            if (!own) return;
            st_chunk(ws, j, 0, w);
            st_chunk(ws, j, 8, w + 8);
            st_chunk(ws, j, 16, s);
            st_chunk(ws, j, 24, s + 8);
        };
        // state MMA of chunk x (x = -1, 0 use the initial state)
        auto issue_state = [&](int x, bool ok) -> bool {
            if (warp != 0) return ok;
            if (ok && x >= 0) ok = wait_all(B, &B->full[x % kNS], (x / kNS) & 1, status);
            if (ok && x + 1 < nch) ok = wait_all(B, &B->full[(x + 1) % kNS], ((x + 1) / kNS) & 1, status);
            if (ok && x >= 1) ok = wait_all(B, &B->acc1_free[x & 1], use_parity(x - 2), status);
            if (!ok) return false;
            tc_fence_after();
            const uint32_t wsa = smem_u32(ws);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk)
                    mma_bf16(tmem + kAcc1 + (x & 1) * 32, sdesc(qk_a(x, kk), 16, 1024, 2),
                             sdesc(wsa + kk * 2048, 8192, 1024, 2), id1, kk > 0);
                mma_commit(&B->acc1_ready[x & 1]);
            }
            __syncwarp();
            return true;
        };
        write_ws();
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        bool ok = issue_state(-1, true);
        ok = issue_state(0, ok);
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1, st = c % kNS;
            if (a.ckpt && own && ok) {
                // the state at this chunk's start, for the gradient passes
                const size_t o = ((size_t)seq * nch + c) * 2 * (size_t)D * D + (size_t)r0 * D + j;
                if (a.ckpt_bf16) {
                    __nv_bfloat16* ck = reinterpret_cast<__nv_bfloat16*>(a.ckpt) + o;
#pragma unroll
                    for (int i = 0; i < kRows; ++i) {
                        ck[(size_t)i * D] = __float2bfloat16_rn(w[i]);
                        ck[(size_t)D * D + (size_t)i * D] = __float2bfloat16_rn(s[i]);
                    }
                } else {
                    float* ck = a.ckpt + o;
#pragma unroll
                    for (int i = 0; i < kRows; ++i) {
                        ck[(size_t)i * D] = w[i];
                        ck[(size_t)D * D + (size_t)i * D] = s[i];
                    }
                }
            }
            if (ok) ok = wait_all(B, &B->full[st], (c / kNS) & 1, status);
            if (ok) ok = wait_all(B, &B->mma2_done[b], (c >> 1) & 1, status);
            if (ok) {
                tc_fence_after();
                float uw[16], us[16];
                tmem_ld16(tl + kAcc2 + b * 32, uw);
                tmem_ld16(tl + kAcc2 + b * 32 + 16, us);
                const float4 sc = *reinterpret_cast<const float4*>(vec(st) + kVScal);
                tmem_wait_ld();
                tc_fence_before();
                warp_arrive(&B->acc2_free[b]);
                // the carry MMA (the last reader of K_c) is complete and the
                // scalars are in registers: this role is done with the stage
                if (tid == 0) mbar_arrive(&B->empty[st]);
                if (own) {
#pragma unroll
                    for (int i = 0; i < kRows; ++i) {
                        const float wn = sc.x * w[i] + sc.y * s[i] - 2.f * uw[i];
                        s[i] = sc.z * s[i] - 2.f * us[i];
                        w[i] = wn;
                    }
                }
                if (c + 1 < nch) {
                    // the state MMA of chunk c still reads the previous copy
                    ok = wait_all(B, &B->acc1_ready[b], use_parity(c), status);
                    if (ok) {
                        write_ws();
                        fence_proxy_async_smem();
                    }
                }
            }
            named_bar_sync(1, 128);
            if (c + 1 < nch) ok = issue_state(c + 1, ok);
        }
        if (own && ok && a.W_out) {
            const size_t dst = (size_t)seq * D * D;
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                a.W_out[dst + (size_t)(r0 + i) * D + j] = w[i];
                if (a.S_out) a.S_out[dst + (size_t)(r0 + i) * D + j] = s[i];
            }
        }
    } else if (warp < 6) {
        // ---------------------------------------------------------- outputs
        const int t = tid - 128;                 // token = TMEM lane 0..63
        bool ok = true;
        warp_arrive(&B->acc1_free[1]);           // the chunk -1 state product has no reads
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1, st = c % kNS;
            if (ok) ok = wait_all(B, &B->full[st], (c / kNS) & 1, status);
            if (ok) ok = wait_all(B, &B->acc1_ready[b], use_parity(c), status);
            if (ok) ok = wait_all(B, &B->mma3_done[b], (c >> 1) & 1, status);
            if (ok) {
                tc_fence_after();
                float qw[16], qs[16], ae[16];
                tmem_ld16(tl + kAcc1 + b * 32, qw);
                tmem_ld16(tl + kAcc1 + b * 32 + 16, qs);
                tmem_ld16(tl + kAcc3 + b * 16, ae);
                const float bt = vecf(st, kVBeta)[t], ct = vecf(st, kVCvec)[t];
                const int n = (int)vecf(st, kVScal)[3];
                tmem_wait_ld();
                tc_fence_before();
                warp_arrive(&B->acc1_free[b]);
                warp_arrive(&B->acc3_free[b]);
                if (t < n && a.z) {
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
            named_bar_sync(3, 64);
            if (tid == 128 && ok) mbar_arrive(&B->empty[st]);
        }
    } else if (warp < 8 || warp >= 14) {
        // ------------------------------------------------------ error chain
        // Thread t' produces half h of row t' of E_x (columns 8h .. 8h + 7) for
        // x = 0, 1, ...: from the state product of chunk x-1 (lanes 64-127:
        // K_x W^T, K_x S^T) and, for x >= 1, the chain product M_{x-1} E_{x-1}.
        // Warps 6-7 take h = 0, warps 14-15 (same TMEM lanes) h = 1.
        const int t = lane + 32 * ((warp & 3) - 2);   // token = TMEM lane 64 + t
        const int h = warp >= 14 ? 1 : 0;
        bool ok = true;
        float bn = 1.f, cn = 0.f;                // carry coefficients of chunk x-1
        for (int x = 0; x < nch; ++x) {
            const int st = x % kNS, pb = (x - 1) & 1;
            if (ok) ok = wait_all(B, &B->full[st], (x / kNS) & 1, status);
            if (ok) ok = wait_all(B, &B->acc1_ready[pb], use_parity(x - 1), status);
            if (ok && x >= 1) ok = wait_all(B, &B->mma3_done[pb], ((x - 1) >> 1) & 1, status);
            float e[8];
            if (ok) {
                tc_fence_after();
                float f[8], g[8], m[8];
                tmem_ld8(tl + kAcc1 + pb * 32 + 8 * h, f);
                tmem_ld8(tl + kAcc1 + pb * 32 + 16 + 8 * h, g);
                if (x >= 1) tmem_ld8(tl + kAcc3 + pb * 16 + 8 * h, m);
                float v[8];
                unpack8(reinterpret_cast<const uint4*>(vtile(st) + t * 32)[h], v);
                tmem_wait_ld();
                tc_fence_before();
                warp_arrive(&B->acc1_free[pb]);
                if (x >= 1) {
                    warp_arrive(&B->acc3_free[pb]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) e[i] = bn * f[i] + cn * g[i] - 2.f * m[i] - v[i];
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) e[i] = f[i] - v[i];
                }
                const float4 sc = *reinterpret_cast<const float4*>(vec(st) + kVScal);
                const float ce = vecf(st, kVCend)[t], pe = vecf(st, kVPend)[t];
                bn = sc.x;
                cn = sc.y;
                // the carry MMA of chunk x-2 read this [C E | Pm E] buffer; the
                // chain MMA of chunk x-1 (complete) read the E tile
                if (x >= 2) ok = wait_all(B, &B->mma2_done[x & 1], ((x - 2) >> 1) & 1, status);
                if (ok) {
                    float ec[8], ep[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        ec[i] = ce * e[i];
                        ep[i] = pe * e[i];
                    }
                    uint8_t* cp = etcp(x & 1);
                    st_chunk(ete, t, 8 * h, e);
                    st_chunk(cp, t, 8 * h, ec);
                    st_chunk(cp, t, 16 + 8 * h, ep);
                    fence_proxy_async_smem();
                }
            }
            named_bar_sync(2, 128);
            // chain MMA of chunk x (warp 6), then the carry MMA (warp 7), so the
            // chain product is first in the tensor pipe and warp 6 is free to
            // wait for it at once
            const int b = x & 1;
            if (warp == 6) {
                if (ok) ok = wait_all(B, &B->am_ready[b], (x >> 1) & 1, status);
                if (ok && x >= 2) ok = wait_all(B, &B->acc3_free[b], ((x - 2) >> 1) & 1, status);
                if (ok) {
                    tc_fence_after();
                    const uint32_t et = smem_u32(ete);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kChunk / 16; ++kk)
                            mma_tmem_a(tmem + kAcc3 + b * 16, tmem + kAM + b * 32 + kk * 8,
                                       sdesc(et + kk * 2048, 8192, 1024, 2), id3, kk > 0);
                        mma_commit(&B->mma3_done[b]);
                        mbar_arrive(&B->mma3_issued);
                    }
                    __syncwarp();
                }
            } else if (warp == 7) {
                if (ok) ok = wait_all(B, &B->mma3_issued, x & 1, status);
                if (ok && x >= 2) ok = wait_all(B, &B->acc2_free[b], ((x - 2) >> 1) & 1, status);
                if (ok) {
                    tc_fence_after();
                    const uint32_t ecp = smem_u32(etcp(b)), kb = smem_u32(ktile(0, st));
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kChunk / 16; ++kk)
                            mma_bf16(tmem + kAcc2 + b * 32,
                                     sdesc(kb + kk * 2048, D == 128 ? kRingBytes : kTile, 1024, 2),
                                     sdesc(ecp + kk * 2048, 8192, 1024, 2), id2, kk > 0);
                        mma_commit(&B->mma2_done[b]);
                    }
                    __syncwarp();
                }
            }
        }
    } else if (warp < 12) {
        // -------------------------------------------------------- weighting
        // Row m of the scores: m < 64 -> A~[m][s] = C[m][s] (q_m . k_s) with
        // row m of the chunk's coefficient table; m >= 64 ->
        // M[m-64][s] = C[n-1][s] (k'_{m-64} . k_s).
        const int m = (warp & 3) * 32 + lane;
        // the first slice of each sequence also stores the score tiles
        uint8_t* tile_out = (a.score_tiles && slice == 0 && m < 64)
                                ? static_cast<uint8_t*>(a.score_tiles) + (size_t)seq * nch * 8192 + m * 128
                                : nullptr;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1, st = c % kNS;
            if (warp == 8) {
                if (ok) ok = wait_all(B, &B->full[st], (c / kNS) & 1, status);
                if (ok && c + 1 < nch)
                    ok = wait_all(B, &B->full[(c + 1) % kNS], ((c + 1) / kNS) & 1, status);
                if (ok) {
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < KS; ++kk)
                            mma_bf16(tmem + kAccS + b * 64, sdesc(qk_a(c, kk), 16, 1024, 2),
                                     sdesc(smem_u32(ktile(kk >> 2, st)) + (kk & 3) * 32, 16, 1024, 2),
                                     idS, kk > 0);
                        mma_commit(&B->sc_ready[b]);
                    }
                    __syncwarp();
                }
            }
            if (ok && warp != 8) ok = wait_all(B, &B->full[st], (c / kNS) & 1, status);
            if (ok) ok = wait_all(B, &B->sc_ready[b], (c >> 1) & 1, status);
            // the chain MMA of chunk c-2 read this buffer's previous contents
            if (ok && c >= 2) ok = wait_all(B, &B->mma3_done[b], ((c - 2) >> 1) & 1, status);
            if (ok) {
                tc_fence_after();
                // weights of this row: row m of the table (m < 64) or C[n-1][.]
                const float* wrow = m < 64 ? vecf(st, kRecC + m * 256) : vecf(st, kVCend);
                const int sw = m < 64 ? (m & 15) : 0;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float r[16], wt[16];
                    tmem_ld16(tl + kAccS + b * 64 + 16 * q4, r);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const float4 f = *reinterpret_cast<const float4*>(wrow + (((4 * q4 + g) ^ sw) << 2));
                        wt[4 * g] = f.x;
                        wt[4 * g + 1] = f.y;
                        wt[4 * g + 2] = f.z;
                        wt[4 * g + 3] = f.w;
                    }
                    tmem_wait_ld();
                    uint32_t p[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        p[i] = pack_bf16(r[2 * i] * wt[2 * i], r[2 * i + 1] * wt[2 * i + 1]);
                    tmem_st8(tl + kAM + b * 32 + 8 * q4, p);
                    if (tile_out) {
                        uint8_t* row = tile_out + (size_t)c * 8192;
                        *reinterpret_cast<uint4*>(row + (((2 * q4) ^ (m & 7)) << 4)) =
                            make_uint4(p[0], p[1], p[2], p[3]);
                        *reinterpret_cast<uint4*>(row + (((2 * q4 + 1) ^ (m & 7)) << 4)) =
                            make_uint4(p[4], p[5], p[6], p[7]);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                warp_arrive(&B->am_ready[b]);
            }
            named_bar_sync(4, 128);
        }
    } else if (warp == 12) {
        // --------------------------------------------------------- producer
        if (lane == 0) {
            // tiles of chunk c are requested into L2 kPrefetch chunks before
            // their load, so the load itself is an L2 hit
            constexpr int kPrefetch = 4;
            auto prefetch = [&](int c) {
                if (c >= nch) return;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    tma_prefetch_l2_3d(&kmap, 64 * h, c * kChunk, seq);
                    tma_prefetch_l2_3d(&qmap, 64 * h, c * kChunk, seq);
                }
                tma_prefetch_l2_3d(&vmap, r0, c * kChunk, seq);
                bulk_prefetch_l2(recs + (size_t)c * kRecBytes, kRecBytes);
            };
            for (int c = 0; c < kPrefetch; ++c) prefetch(c);
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int st = c % kNS;
                prefetch(c + kPrefetch);
                if (c >= kNS && !wait_bar(B, &B->empty[st], ((c / kNS) - 1) & 1, status)) break;
                const uint32_t tx = (st == 0 ? 3 : 2) * NH * kTile + kChunk * kRows * 2 + kRecBytes +
                                    (c + 1 == a.debug_stall ? 16u : 0u);
                mbar_expect_tx(&B->full[st], tx);
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    tma_load_3d(ktile(h, st), &kmap, &B->full[st], 64 * h, c * kChunk, seq);
                    tma_load_3d(qtile(h, st), &qmap, &B->full[st], 64 * h, c * kChunk, seq);
                    if (st == 0)   // the copy after the last query tile of the ring
                        tma_load_3d(ktile(h, kNS), &kmap, &B->full[st], 64 * h, c * kChunk, seq);
                }
                tma_load_3d(vtile(st), &vmap, &B->full[st], r0, c * kChunk, seq);
                bulk_load(vec(st), recs + (size_t)c * kRecBytes, kRecBytes, &B->full[st]);
                issued = c + 1;
            }
            // drain: every issued stage's copies must have landed before exit
            for (int c = (issued > kNS ? issued - kNS : 0); c < issued; ++c)
                wait_drain(&B->full[c % kNS], (c / kNS) & 1, B->wait_limit);
        }
        __syncwarp();
    }

    // drain the MMAs of the three issuing warps before TMEM is released
    if (warp == 0 || warp == 6 || warp == 7 || warp == 8) {
        uint64_t* d = &B->drain[warp == 0 ? 0 : (warp == 6 ? 1 : (warp == 7 ? 3 : 2))];
        if (elect_one()) mma_commit(d);
        __syncwarp();
        if (lane == 0) wait_drain(d, 0, B->wait_limit);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, kTmemCols);
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

bool make_map(CUtensorMap* m, const void* ptr, int BH, int T, int D, int bx, bool swz) {
    return make_token_tile_map(m, ptr, BH, T, D, bx, swz);
}

}  // namespace

// 3-D view [sequences][T][D] of a bf16 tensor, tile box {bx, 64, 1}.
bool make_token_tile_map(void* map, const void* ptr, int BH, int T, int D, int bx, bool swz) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)bx, (cuuint32_t)kChunk, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

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
