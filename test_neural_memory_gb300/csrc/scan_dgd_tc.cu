// Tensor-core (tcgen05 + TMA) kernels of the DGD memory scan in chunk form.
//
// Method ("Nested Learning" §8.1 eq (88) with the L2 objective of eq (93),
// chunk-wise as §8.2 takes it, each token read before its write as eq (86)
// prints y_t = M_{t-1} q_t): every row w of the memory evolves on its own; with
// w_c the row at the start of a chunk of n <= 64 tokens,
//   w_t = alpha_t w_{t-1} - g_t k_t,   g_t = eta_t ((w_{t-1} + w_c) . k_t - v_t),
//   z_t = w_{t-1} . q_t.
// Unrolling the chunk with a_t = prod_{tau<=t} alpha_tau (a_{-1} = 1) and the
// retention between the write of token s and the read at token t,
// R[t][s] = prod_{tau=s+1..t-1} alpha_tau (s < t),
//   w_{t-1} = a_{t-1} w_c - sum_{s<t} R[t][s] g_s k_s,
// so the chunk's gradients solve a unit lower-triangular system
//   (I + L) g = R0,   L[t][s] = eta_t R[t][s] (k_s . k_t)   (s < t),
//   R0_t = eta_t ((a_{t-1} + 1) (w_c . k_t) - v_t),
// and with N = (I + L)^-1, A~[t][s] = R[t][s] (q_t . k_s) (s < t) and
// r_s = prod_{tau=s+1..n-1} alpha_tau:
//   z_t   = a_{t-1} (w_c . q_t) - (A~ N R0)_t,
//   w_end = a_{n-1} w_c - sum_s r_s (N R0)_s k_s.
// For all rows at once (rows of the memory = columns of R0; W_c^T is d_k x d_v):
//   R0      = diag(eta (a_- + 1)) K W_c^T - diag(eta) V
//   Z       = diag(a_-) Q W_c^T - (A~ N) R0
//   W_end^T = a_{n-1} W_c^T - (K^T diag(r) N) R0.
// The two operators A~N and Y = K^T diag(r) N depend only on the chunk's keys,
// queries and gates.
//
// Pre-pass (dgd_prep_kernel, one CTA per (sequence, chunk), every chunk at
// once): the scores [Q; K] K^T on the tensor cores; the rows of A~ and L from
// them and the gates; N by forward substitution in fp32 (one thread per
// column); then A~N and Y on the tensor cores (bf16 operands, fp32
// accumulation).  It writes them in bf16 to the workspace in the 128-byte
// swizzled K-major layout the scan's MMAs read, with the chunk's vectors.
//
// Scan (dgd_tc_kernel): one CTA per (sequence, slice of 16 rows of the
// memory) runs the whole sequence.  Per chunk the state's chain is two
// products: C1 = [Q; K] W_c^T (reads and gradient terms) -> R0 (epilogue) ->
// C3 = Y R0 (the update) -> W_{c+1} (registers) -> its bf16 copy for the next
// C1; the read correction (A~N) R0 is issued right after Y R0, off that chain.
//
// Roles of the scan CTA (288 threads):
//   warps 0-3  state: thread j holds column j of the slice's 16 rows in fp32
//              registers and writes their bf16 copy; warp 0 issues C1.
//   warps 4-5  outputs z (token = TMEM lane 0..63).
//   warps 6-7  R0 (token = TMEM lane 64..127); warp 6 issues C3.
//   warp 8     producer: TMA loads of Q, K, the V slice and the chunk's record.
// Every wait is bounded: a wait that runs out sets the status word to
// TTM_ERR_TIMEOUT, every role runs out its loop without further work, copies
// and MMAs drain, TMEM is freed and the kernel returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/ttm.h"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace ttm {
namespace {

using namespace tc;

constexpr int kChunk = 64;          // tokens per chunk (== TMA tile height)
constexpr int kRows = 16;           // rows of the memory per scan CTA
constexpr uint32_t kTile = 8192;    // 64 rows x 128 bytes

// Per-chunk record (workspace): A~N (64 rows), Y (d_k rows), 128-byte rows of
// 64 bf16 values in the 128-byte swizzle, then fp32 vectors over the chunk's
// tokens and two scalars.
__host__ __device__ constexpr uint32_t rec_vec(int D) { return kTile + (uint32_t)D * 128u; }
__host__ __device__ constexpr uint32_t rec_bytes(int D) { return rec_vec(D) + 1024u; }
constexpr uint32_t kVAprev = 0;       // a_{t-1}
constexpr uint32_t kVEa1 = 256;       // eta_t (a_{t-1} + 1)
constexpr uint32_t kVEta = 512;       // eta_t
constexpr uint32_t kVScal = 768;      // a_{n-1}, n

constexpr long long kWaitCycles = 4000000000LL;   // default limit, ~2 s at 2 GHz

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack8(const float* x) {
    uint4 v;
    v.x = pack_bf16(x[0], x[1]);
    v.y = pack_bf16(x[2], x[3]);
    v.z = pack_bf16(x[4], x[5]);
    v.w = pack_bf16(x[6], x[7]);
    return v;
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

// 8 consecutive bf16 values of row `row` from column `col` (a multiple of 8)
// of a 128-byte-swizzled tile.
__device__ __forceinline__ void st_chunk(uint8_t* tile, int row, int col, const float* x) {
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, col)) = pack8(x);
}

// A whole 64-value row (128 bytes) in the 128-byte swizzle, to shared or
// global memory; `base` is 1024-byte aligned relative to the pattern.
__device__ __forceinline__ void st_row64(uint8_t* base, int row, const float* x) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(base + (size_t)row * 128 + ((c ^ (row & 7)) << 4)) = pack8(x + 8 * c);
}

// ----------------------------------------------------------- bounded waits

struct Abort {
    long long wait_limit;
    int abort;
};

__device__ __noinline__ bool wait_bar_slow(Abort* A, uint64_t* bar, uint32_t parity, int* status) {
    const long long t0 = clock64();
    const long long limit = A->wait_limit;
    uint32_t polls = 0;
    while (!mbar_try_wait_sleep(bar, parity, 20000)) {
        if ((++polls & 3u) == 0) {
            if (*(volatile int*)&A->abort) return false;
            if (clock64() - t0 > limit) {
                *(volatile int*)&A->abort = 1;
                atomicExch(status, TTM_ERR_TIMEOUT);
                return false;
            }
        }
    }
    return true;
}

// Warp-uniform bounded wait (every lane gets the same answer).
__device__ __noinline__ bool wait_all_slow(Abort* A, uint64_t* bar, uint32_t parity, int* status) {
    return __all_sync(0xffffffffu, wait_bar_slow(A, bar, parity, status));
}

__device__ __forceinline__ bool wait_all(Abort* A, uint64_t* bar, uint32_t parity, int* status) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    return wait_all_slow(A, bar, parity, status);
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

// ----------------------------------------------------------------- pre-pass

struct PrepBars {
    uint64_t full, mma, drain;
    Abort A;
    uint32_t tmem_base;
};

struct PrepLayout {
    uint32_t off_qk, off_aop, off_L, off_g, off_bars, total;
};

constexpr int kLStride = 68;    // floats per row of L (16-byte rows offsets apart: no bank conflicts)

// [Q h][K h] per 64-column half (so [Q; K] is one 128-row operand; once the
// scores are taken, the row-scaled keys diag(r) K, the MN-major operand
// K^T diag(r), take the place of the query tiles), then [A~][N^T] (K-major,
// 64 rows each), L (fp32), the gate vectors.
__host__ __device__ constexpr PrepLayout prep_layout(int D) {
    PrepLayout L{};
    uint32_t off = 0;
    L.off_qk = off;   off += (D / 64) * 2 * kTile;
    L.off_aop = off;  off += 2 * kTile;
    L.off_L = off;    off += 64 * kLStride * 4;
    L.off_g = off;    off += 4 * 256;           // alpha, eta, r, a_{t-1}
    L.off_bars = off; off += (sizeof(PrepBars) + 15) & ~size_t(15);
    L.total = off;
    return L;
}

constexpr int kPrepThreads = 256;
constexpr uint32_t kPrepTmemCols = 128;

template <int D>
__global__ void __launch_bounds__(kPrepThreads)
dgd_prep_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const DgdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    constexpr PrepLayout L = prep_layout(D);
    constexpr int NH = D / 64, KS = D / 16;
    PrepBars* B = reinterpret_cast<PrepBars*>(sm + L.off_bars);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = (a.T + kChunk - 1) / kChunk;
    const int seq = blockIdx.x / nch, c = blockIdx.x % nch;
    const int n = min(kChunk, a.T - c * kChunk);
    int* status = a.status;
    uint8_t* qk = sm + L.off_qk;
    uint8_t* aop = sm + L.off_aop;      // A~ rows 0..63, then N^T rows 64..127
    uint8_t* ks = qk;                   // diag(r) K over the query tiles (stride 2 tiles)
    float* Lf = reinterpret_cast<float*>(sm + L.off_L);
    float* g_al = reinterpret_cast<float*>(sm + L.off_g);
    float* g_et = g_al + 64;
    float* g_r = g_al + 128;
    float* g_ap = g_al + 192;

    if (tid == 0) {
        mbar_init(&B->full, 1);
        mbar_init(&B->mma, 1);
        mbar_init(&B->drain, 1);
        B->A.wait_limit = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;
        B->A.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&B->tmem_base, kPrepTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(warp & 3) * 32 << 16);

    if (tid == 0) {
        mbar_expect_tx(&B->full, NH * 2 * kTile);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            tma_load_3d(qk + h * 2 * kTile, &qmap, &B->full, 64 * h, c * kChunk, seq);
            tma_load_3d(qk + h * 2 * kTile + kTile, &kmap, &B->full, 64 * h, c * kChunk, seq);
        }
    }
    // gates; past the chunk's last token alpha = 1 and eta = 0 (neutral)
    if (tid < kChunk) {
        const size_t gi = (size_t)seq * a.T + (size_t)c * kChunk + tid;
        g_al[tid] = tid < n ? a.alpha[gi] : 1.f;
        g_et[tid] = tid < n ? a.eta[gi] : 0.f;
    }
    __syncthreads();
    if (tid == 0) {
        float p = 1.f;                       // a_{t-1}
        for (int t = 0; t < kChunk; ++t) {
            g_ap[t] = p;
            p *= g_al[t];
        }
    } else if (tid == 32) {
        float p = 1.f;                       // r_s = prod_{tau > s} alpha_tau
        for (int s = kChunk - 1; s >= 0; --s) {
            g_r[s] = p;
            p *= g_al[s];
        }
    }
    bool ok = wait_all(&B->A, &B->full, 0, status);
    if (warp == 0 && ok) {
        tc_fence_after();
        if (elect_one()) {
            constexpr uint32_t idS = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const uint32_t base = smem_u32(qk + (kk >> 2) * 2 * kTile) + (kk & 3) * 32;
                mma_bf16(tmem, sdesc(base, 16, 1024, 2), sdesc(base + kTile, 16, 1024, 2), idS,
                         kk > 0);
            }
            mma_commit(&B->mma);
        }
        __syncwarp();
    }
    __syncthreads();                         // the gate vectors are in place

    if (warp < 4) {
        // row p of the scores: q_p . k_s (p < 64) or k_t . k_s (t = p - 64);
        // R[t][s] walked down from s = t - 1 (R = 1 there): R[t][s-1] = alpha_s R[t][s]
        const int p = tid;
        const bool qrow = p < 64;
        const int t = qrow ? p : p - 64;
        if (ok) ok = wait_all(&B->A, &B->mma, 0, status);
        if (ok) {
            tc_fence_after();
            float S[kChunk];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float r[16];
                tmem_ld16(tl + 16 * q4, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) S[16 * q4 + i] = r[i];
            }
            const float scale = qrow ? 1.f : g_et[t];
            float R = 1.f;
#pragma unroll
            for (int s = kChunk - 1; s >= 0; --s) {
                const bool below = s < t;
                S[s] = below ? scale * R * S[s] : 0.f;
                if (below) R *= g_al[s];
            }
            if (qrow) {
                st_row64(aop, t, S);
            } else {
#pragma unroll
                for (int s4 = 0; s4 < kChunk / 4; ++s4)
                    reinterpret_cast<float4*>(Lf + t * kLStride)[s4] =
                        make_float4(S[4 * s4], S[4 * s4 + 1], S[4 * s4 + 2], S[4 * s4 + 3]);
            }
        }
    } else {
        // row-scaled keys r_s k_s (same swizzled positions as the key tiles),
        // over the query tiles once the score MMA has read them
        const int u = tid - 128;
        if (ok) ok = wait_all(&B->A, &B->mma, 0, status);
#pragma unroll
        for (int i = 0; i < 4 * NH; ++i) {
            if (!ok) break;
            const int idx = u + 128 * i;            // 16-byte chunk: half, row, chunk
            const int h = idx >> 9, row = (idx >> 3) & 63, ch = idx & 7;
            const uint32_t off = (uint32_t)h * 2 * kTile + row * 128 + ch * 16;
            const uint8_t* src = qk + h * 2 * kTile + kTile + row * 128 + ch * 16;
            float x[8];
            unpack8(*reinterpret_cast<const uint4*>(src), x);
            const float rs = g_r[row];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] *= rs;
            *reinterpret_cast<uint4*>(ks + off) = pack8(x);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    if (warp < 2 && ok) {
        // column j of N = (I + L)^-1: x_t = [t == j] - sum_{s<t} L[t][s] x_s
        // (x_s = 0 for s < j), then row j of N^T
        const int j = tid;
        float x[kChunk];
#pragma unroll
        for (int t = 0; t < kChunk; ++t) {
            float acc0 = t == j ? 1.f : 0.f, acc1 = 0.f;
            const float4* Lr = reinterpret_cast<const float4*>(Lf + t * kLStride);
#pragma unroll
            for (int s4 = 0; s4 < (t + 3) / 4; ++s4) {
                const float4 l = Lr[s4];
                const int s = 4 * s4;
                if (s < t) acc0 = fmaf(-l.x, x[s], acc0);
                if (s + 1 < t) acc1 = fmaf(-l.y, x[s + 1], acc1);
                if (s + 2 < t) acc0 = fmaf(-l.z, x[s + 2], acc0);
                if (s + 3 < t) acc1 = fmaf(-l.w, x[s + 3], acc1);
            }
            x[t] = acc0 + acc1;
        }
        st_row64(aop + kTile, j, x);
    }
    fence_proxy_async_smem();
    __syncthreads();

    if (warp == 0 && ok) {
        tc_fence_after();
        if (elect_one()) {
            constexpr uint32_t idA = idesc_bf16_f32(128, 64, 0, 0);   // [A~; N^T] N
            constexpr uint32_t idY = idesc_bf16_f32(128, 64, 1, 0);   // (diag(r) K)^T N
            const uint32_t aa = smem_u32(aop), nb = smem_u32(aop + kTile), kb = smem_u32(ks);
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk)
                mma_bf16(tmem, sdesc(aa + kk * 32, 16, 1024, 2), sdesc(nb + kk * 32, 16, 1024, 2),
                         idA, kk > 0);
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk)
                mma_bf16(tmem + 64, sdesc(kb + kk * 2048, 2 * kTile, 1024, 2),
                         sdesc(nb + kk * 32, 16, 1024, 2), idY, kk > 0);
            mma_commit(&B->mma);
        }
        __syncwarp();
    }

    uint8_t* rec = static_cast<uint8_t*>(a.workspace) + ((size_t)seq * nch + c) * rec_bytes(D);
    if (warp < 4) {
        const int p = tid;
        if (ok) ok = wait_all(&B->A, &B->mma, 1, status);
        if (ok) {
            tc_fence_after();
            float x[kChunk];
            if (p < 64) {                         // warp-uniform
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float r[16];
                    tmem_ld16(tl + 16 * q4, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[16 * q4 + i] = r[i];
                }
                st_row64(rec, p, x);
            }
            if (p < D) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float r[16];
                    tmem_ld16(tl + 64 + 16 * q4, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[16 * q4 + i] = r[i];
                }
                st_row64(rec + kTile, p, x);
            }
        }
    }
    if (tid < kChunk) {
        float* v = reinterpret_cast<float*>(rec + rec_vec(D));
        v[kVAprev / 4 + tid] = g_ap[tid];
        v[kVEa1 / 4 + tid] = g_et[tid] * (g_ap[tid] + 1.f);
        v[kVEta / 4 + tid] = g_et[tid];
        if (tid == 0) {
            v[kVScal / 4] = g_ap[kChunk - 1] * g_al[kChunk - 1];   // a_{n-1} (neutral past n)
            v[kVScal / 4 + 1] = (float)n;
            v[kVScal / 4 + 2] = 0.f;
            v[kVScal / 4 + 3] = 0.f;
        }
    }
    if (tid == 0 && !ok) wait_drain(&B->full, 0, B->A.wait_limit);   // copies in flight
    if (warp == 0) {
        // every MMA (also any left after an abort) completes before TMEM goes
        if (elect_one()) mma_commit(&B->drain);
        __syncwarp();
        if (lane == 0) wait_drain(&B->drain, 0, B->A.wait_limit);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// --------------------------------------------------------------------- scan

constexpr int kScanThreads = 288;
constexpr uint32_t kScanTmemCols = 128;
constexpr int kMaxNS = 4;

__host__ __device__ constexpr int scan_stages(int D) { return D == 128 ? 3 : 4; }
// stage: [Q h][K h] per half, the record, the V slice (64 x 16 bf16)
__host__ __device__ constexpr uint32_t stage_bytes(int D) {
    return (uint32_t)(D / 64) * 2 * kTile + rec_bytes(D) + 2048u;
}

struct ScanBars {
    uint64_t full[kMaxNS], empty[kMaxNS];
    uint64_t acc1_ready[2], acc1_free[2], c3_done, c3z_done[2], accz_free[2];
    uint64_t drain[2];
    Abort A;
    uint32_t tmem_base;
};

struct ScanLayout {
    uint32_t off_stage, off_ws, off_r0, off_bars, total;
};

// The stages first, then the state copy and the R0 tile: the 128-row A
// operands that start inside a record (rows past the record are never read
// back) stay inside the allocation.
__host__ __device__ constexpr ScanLayout scan_layout(int D) {
    ScanLayout L{};
    uint32_t off = 0;
    L.off_stage = off; off += scan_stages(D) * stage_bytes(D);
    L.off_ws = off;    off += (uint32_t)D * 128;        // W_c^T bf16 [j][r] (16 of 64 columns)
    L.off_r0 = off;    off += kTile;                    // R0 bf16 [t][r] (16 of 64 columns)
    L.off_bars = off;  off += (sizeof(ScanBars) + 15) & ~size_t(15);
    L.total = off;
    return L;
}

// TMEM columns: C1 accumulators (2 x 16: Q W^T lanes 0-63, K W^T lanes
// 64-127), Y R0 (16, lane = d_k index), A~N R0 (2 x 16, lanes 0-63).
constexpr uint32_t kAcc1 = 0, kAccY = 32, kAccZ = 48;

template <int D>
__global__ void __launch_bounds__(kScanThreads, 1)
dgd_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap, const DgdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    constexpr ScanLayout L = scan_layout(D);
    constexpr int NH = D / 64, KS = D / 16, NS = scan_stages(D);
    constexpr uint32_t SB = stage_bytes(D), RB = rec_bytes(D);
    ScanBars* B = reinterpret_cast<ScanBars*>(sm + L.off_bars);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsl = D / kRows;
    const int slice = blockIdx.x % nsl, seq = blockIdx.x / nsl;
    const int bb = seq / a.H, hh = seq % a.H;
    const int r0 = slice * kRows;
    const int T = a.T;
    const int nch = (T + kChunk - 1) / kChunk;
    int* status = a.status;
    const uint8_t* recs = static_cast<const uint8_t*>(a.workspace) + (size_t)seq * nch * RB;

    auto stage = [&](int s) { return sm + L.off_stage + s * SB; };
    auto rec = [&](int s) { return stage(s) + NH * 2 * kTile; };
    auto vecf = [&](int s) { return reinterpret_cast<const float*>(rec(s) + rec_vec(D)); };
    auto vtile = [&](int s) { return rec(s) + RB; };
    uint8_t* ws = sm + L.off_ws;
    uint8_t* r0t = sm + L.off_r0;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&B->full[s], 1);
            mbar_init(&B->empty[s], 2);          // state + outputs
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&B->acc1_ready[b], 1);
            mbar_init(&B->acc1_free[b], 2);      // output warps
            mbar_init(&B->c3z_done[b], 1);
            mbar_init(&B->accz_free[b], 2);      // output warps
            mbar_init(&B->drain[b], 1);
        }
        mbar_init(&B->c3_done, 1);
        B->A.wait_limit = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;
        B->A.abort = 0;
        fence_mbar_init();
    }
    if (warp == 4) tmem_alloc(&B->tmem_base, kScanTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(warp & 3) * 32 << 16);

    constexpr uint32_t id1 = idesc_bf16_f32(128, 16, 0, 1);   // [Q; K] W^T, B MN-major
    constexpr uint32_t id3 = idesc_bf16_f32(128, 16, 0, 1);   // [A~N; Y] R0

    if (warp < 4) {
        // ------------------------------------------------------------ state
        const int j = tid;
        const bool own = j < D;
        const size_t init = (size_t)(a.shared ? 0 : bb) * a.H + hh;
        float w[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            w[i] = own ? a.W0[(init * D + r0 + i) * (size_t)D + j] : 0.f;
        auto write_ws = [&]() {
            if (!own) return;
            st_chunk(ws, j, 0, w);
            st_chunk(ws, j, 8, w + 8);
        };
        auto issue_c1 = [&](int c, bool ok) -> bool {
            if (warp != 0) return ok;
            if (ok) ok = wait_all(&B->A, &B->full[c % NS], (c / NS) & 1, status);
            if (ok && c >= 2) ok = wait_all(&B->A, &B->acc1_free[c & 1], ((c - 2) >> 1) & 1, status);
            if (!ok) return false;
            tc_fence_after();
            if (elect_one()) {
                const uint32_t wsa = smem_u32(ws);
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint32_t qa = smem_u32(stage(c % NS) + (kk >> 2) * 2 * kTile) + (kk & 3) * 32;
                    mma_bf16(tmem + kAcc1 + (c & 1) * 16, sdesc(qa, 16, 1024, 2),
                             sdesc(wsa + kk * 2048, 8192, 1024, 2), id1, kk > 0);
                }
                mma_commit(&B->acc1_ready[c & 1]);
            }
            __syncwarp();
            return true;
        };
        write_ws();
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        bool ok = issue_c1(0, true);
        for (int c = 0; c < nch; ++c) {
            const int st = c % NS;
            if (ok) ok = wait_all(&B->A, &B->c3_done, c & 1, status);
            if (ok) {
                tc_fence_after();
                float u[16];
                tmem_ld16(tl + kAccY, u);
                const float aend = vecf(st)[kVScal / 4];
                tmem_wait_ld();
                tc_fence_before();
                // C1 and C3 of this chunk are complete: the stage is consumed
                if (tid == 0) mbar_arrive(&B->empty[st]);
                if (own) {
#pragma unroll
                    for (int i = 0; i < kRows; ++i) w[i] = fmaf(aend, w[i], -u[i]);
                }
                if (c + 1 < nch) {
                    write_ws();
                    fence_proxy_async_smem();
                }
            }
            named_bar_sync(1, 128);
            if (c + 1 < nch) ok = issue_c1(c + 1, ok);
        }
        if (own && ok) {
            const size_t dst = (size_t)seq * D * D;
#pragma unroll
            for (int i = 0; i < kRows; ++i) a.W_out[dst + (size_t)(r0 + i) * D + j] = w[i];
        }
    } else if (warp < 6) {
        // ---------------------------------------------------------- outputs
        const int t = tid - 128;                 // token = TMEM lane 0..63
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int st = c % NS, b = c & 1;
            if (ok) ok = wait_all(&B->A, &B->full[st], (c / NS) & 1, status);
            if (ok) ok = wait_all(&B->A, &B->acc1_ready[b], (c >> 1) & 1, status);
            if (ok) ok = wait_all(&B->A, &B->c3z_done[b], (c >> 1) & 1, status);
            if (ok) {
                tc_fence_after();
                float qw[16], az[16];
                tmem_ld16(tl + kAcc1 + b * 16, qw);
                tmem_ld16(tl + kAccZ + b * 16, az);
                const float ap = vecf(st)[kVAprev / 4 + t];
                const int n = (int)vecf(st)[kVScal / 4 + 1];
                tmem_wait_ld();
                tc_fence_before();
                warp_arrive(&B->acc1_free[b]);
                warp_arrive(&B->accz_free[b]);
                if (t < n) {
                    float zz[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) zz[i] = fmaf(ap, qw[i], -az[i]);
                    uint4* zr = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.z) +
                                                         ((size_t)seq * T + (size_t)c * kChunk + t) * D + r0);
                    zr[0] = pack8(zz);
                    zr[1] = pack8(zz + 8);
                }
            }
            named_bar_sync(3, 64);
            if (tid == 128 && ok) mbar_arrive(&B->empty[st]);
        }
    } else if (warp < 8) {
        // --------------------------------------------------------------- R0
        const int t = tid - 192;                 // token = TMEM lane 64 + t
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int st = c % NS, b = c & 1;
            if (ok) ok = wait_all(&B->A, &B->full[st], (c / NS) & 1, status);
            if (ok) ok = wait_all(&B->A, &B->acc1_ready[b], (c >> 1) & 1, status);
            float r[16];
            if (ok) {
                tc_fence_after();
                float kw[16], v[16];
                tmem_ld16(tl + kAcc1 + b * 16, kw);
                const float ea1 = vecf(st)[kVEa1 / 4 + t], et = vecf(st)[kVEta / 4 + t];
                const uint4* vr = reinterpret_cast<const uint4*>(vtile(st) + t * 32);
                unpack8(vr[0], v);
                unpack8(vr[1], v + 8);
                tmem_wait_ld();
                tc_fence_before();
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = fmaf(ea1, kw[i], -et * v[i]);
                // the previous chunk's read-correction product (committed after the
                // state's) has read the R0 tile
                if (c >= 1)
                    ok = wait_all(&B->A, &B->c3z_done[(c - 1) & 1], ((c - 1) >> 1) & 1, status);
            }
            if (ok) {
                st_chunk(r0t, t, 0, r);
                st_chunk(r0t, t, 8, r + 8);
                fence_proxy_async_smem();
            }
            named_bar_sync(2, 64);
            if (warp == 6) {
                if (ok && c >= 2) ok = wait_all(&B->A, &B->accz_free[b], ((c - 2) >> 1) & 1, status);
                if (ok) {
                    tc_fence_after();
                    if (elect_one()) {
                        const uint32_t ra = smem_u32(rec(st)), rb = smem_u32(r0t);
                        // Y R0 (Y rows from the record's second block), then
                        // [A~N; Y rows 0..63] R0 (lanes 0-63 are the correction)
#pragma unroll
                        for (int kk = 0; kk < kChunk / 16; ++kk)
                            mma_bf16(tmem + kAccY, sdesc(ra + kTile + kk * 32, 16, 1024, 2),
                                     sdesc(rb + kk * 2048, 8192, 1024, 2), id3, kk > 0);
                        mma_commit(&B->c3_done);        // the state's product first
#pragma unroll
                        for (int kk = 0; kk < kChunk / 16; ++kk)
                            mma_bf16(tmem + kAccZ + b * 16, sdesc(ra + kk * 32, 16, 1024, 2),
                                     sdesc(rb + kk * 2048, 8192, 1024, 2), id3, kk > 0);
                        mma_commit(&B->c3z_done[b]);
                    }
                    __syncwarp();
                }
            }
        }
    } else {
        // --------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int st = c % NS;
                if (c >= NS && !wait_bar_slow(&B->A, &B->empty[st], ((c / NS) - 1) & 1, status)) break;
                mbar_expect_tx(&B->full[st], NH * 2 * kTile + RB + kChunk * kRows * 2);
                uint8_t* sg = stage(st);
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    tma_load_3d(sg + h * 2 * kTile, &qmap, &B->full[st], 64 * h, c * kChunk, seq);
                    tma_load_3d(sg + h * 2 * kTile + kTile, &kmap, &B->full[st], 64 * h, c * kChunk, seq);
                }
                bulk_load(rec(st), recs + (size_t)c * RB, RB, &B->full[st]);
                tma_load_3d(vtile(st), &vmap, &B->full[st], r0, c * kChunk, seq);
                issued = c + 1;
            }
            for (int c = (issued > NS ? issued - NS : 0); c < issued; ++c)
                wait_drain(&B->full[c % NS], (c / NS) & 1, B->A.wait_limit);
        }
        __syncwarp();
    }

    // drain the MMAs of the two issuing warps before TMEM is released
    if (warp == 0 || warp == 6) {
        uint64_t* d = &B->drain[warp == 0 ? 0 : 1];
        if (elect_one()) mma_commit(d);
        __syncwarp();
        if (lane == 0) wait_drain(d, 0, B->A.wait_limit);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, kScanTmemCols);
}

}  // namespace

// ---------------------------------------------------------------------- host

bool dgd_tc_supported(const DgdArgs& a) {
    return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128) && a.chunk == kChunk &&
           a.T >= 1;
}

size_t dgd_tc_workspace_bytes(const DgdArgs& a) {
    const size_t nch = ((size_t)a.T + kChunk - 1) / kChunk;
    return (size_t)a.B * a.H * nch * rec_bytes(a.dk);
}

namespace {
template <int D>
cudaError_t launch_d(const DgdArgs& a, cudaStream_t s) {
    const int BH = a.B * a.H, nch = (a.T + kChunk - 1) / kChunk;
    CUtensorMap qm, km, vm;
    if (!make_token_tile_map(&qm, a.q, BH, a.T, D, 64, true) ||
        !make_token_tile_map(&km, a.k, BH, a.T, D, 64, true) ||
        !make_token_tile_map(&vm, a.v, BH, a.T, D, kRows, false))
        return cudaErrorInvalidValue;
    {
        const size_t smem = prep_layout(D).total + 1024;
        cudaError_t e = cudaFuncSetAttribute(dgd_prep_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        dgd_prep_kernel<D><<<(unsigned)(BH * nch), kPrepThreads, smem, s>>>(qm, km, a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t smem = scan_layout(D).total + 1024;
    cudaError_t e = cudaFuncSetAttribute(dgd_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dgd_tc_kernel<D><<<(unsigned)(BH * (D / kRows)), kScanThreads, smem, s>>>(qm, km, vm, a);
    return cudaGetLastError();
}
}  // namespace

cudaError_t dgd_tc_launch(const DgdArgs& a, cudaStream_t s) {
    if (!a.workspace || a.workspace_bytes < dgd_tc_workspace_bytes(a) ||
        (reinterpret_cast<uintptr_t>(a.workspace) & 15u))
        return cudaErrorInvalidValue;
    return a.dk == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace ttm
