// Gradient of the chunked linear / Titans memory scan.
//
// The outer loss trains the projections, the rates and W0 through the inner
// updates, so the gradient follows the chain of state transitions backward
// ("Continual Learning: From Attention to Neural Memory" §4.5; the pages ask
// for the primal / dual and finite-difference gradient checks in
// "TTT layers 与 fast weights" §1.2).  It is taken here through the chunk
// ("dual") form that the forward scan uses ("TTT layers 与 fast weights" §1.1
// eqs (7)-(9); momentum and decay unrolled as in "论文速览 | Titans" §4.3 and
// §4.5).  Inside a chunk of n tokens starting from (W, S), with e_s = W k_s - v_s,
// A[t][s] = C[t][s] (k_s . q_t) for s <= t:
//
//   z_t   = beta_t W q_t + c_t S q_t - 2 sum_{s<=t} A[t][s] e_s
//   W_end = beta_n W + c_n S - 2 sum_s C[n][s] e_s k_s^T
//   S_end = P_n S - 2 sum_s pm[s] e_s k_s^T,     pm[s] = theta_s m(s, n)
//
// (index n = the chunk's last token).  Given the adjoints dz_t, dWe = dL/dW_end
// and dSe = dL/dS_end, the chunk's backward is
//
//   de_s  = -2 sum_{t>=s} A[t][s] dz_t - 2 C[n][s] dWe k_s - 2 pm[s] dSe k_s,  dv_s = -de_s
//   dW    = beta_n dWe + sum_t beta_t dz_t q_t^T + sum_s de_s k_s^T            (chunk start)
//   dS    = c_n dWe + P_n dSe + sum_t c_t dz_t q_t^T
//   dq_t  = beta_t W^T dz_t + c_t S^T dz_t - 2 sum_{s<=t} C[t][s] (dz_t . e_s) k_s
//   dk_s  = W^T de_s - 2 sum_{t>=s} C[t][s] (dz_t . e_s) q_t - 2 C[n][s] dWe^T e_s
//           - 2 pm[s] dSe^T e_s
//
// and the adjoints of the coefficients (dC, dpm, dbeta, dc, dP) are carried
// back through their defining recurrences to theta, eta and alpha.
//
// Three passes (plus the forward scan, which writes the state at every chunk
// start):
//   records  one CTA per (sequence, chunk): coefficients and A, stored;
//   chain    one CTA per (sequence, slice of rows), chunks in reverse: the
//            adjoint (dW, dS) at every chunk end.  It needs no forward state
//            (the chunk map is affine in the state), only A, the coefficients,
//            q, k and dz; rows are independent, as in the forward;
//   local    one CTA per (sequence, chunk), all chunks at once: dq, dk, dv and
//            the gate gradients from the chunk's start state and end adjoint.
// The records pass and the fp32 CUDA-core chain and local passes below serve
// every shape; for bf16 inputs with d_k = d_v in {64, 128} and chunks of 64 the
// chain and local passes run on the tensor cores instead (scan_bwd_tc.cu).
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

__device__ __forceinline__ float warp_sum_f(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

constexpr int kBT = 256;      // threads per CTA
constexpr int kMaxBC = 64;    // largest chunk
constexpr int kMaxDK = 128;   // widest key
constexpr int kR2 = 16;       // rows of the adjoint per chain CTA
constexpr int kR3 = 16;       // rows per tile in the local pass
constexpr int kBT3 = 512;     // threads per local-pass CTA

// Workspace carve-up (floats).  ckpt and adj hold [seq][chunk][W | S][dv][dk];
// rec holds per (seq, chunk): A [bc][bc], beta [bc], cc [bc], clast [bc],
// pm [bc], P_n.
struct BwdLayout {
    int nch, bc;
    size_t sd, rec_f;
    size_t ckpt, adj, rec, part, tcws, total;
};

BwdLayout bwd_layout(const BwdArgs& a) {
    BwdLayout L;
    L.bc = a.chunk;
    L.nch = (a.T + a.chunk - 1) / a.chunk;
    L.sd = (size_t)a.dv * a.dk;
    L.rec_f = ((size_t)L.bc * L.bc + 4 * (size_t)L.bc + 1 + 3) / 4 * 4;
    const size_t nseq = (size_t)a.B * a.H;
    L.ckpt = 0;
    L.adj = L.ckpt + nseq * L.nch * 2 * L.sd;
    L.rec = L.adj + nseq * L.nch * 2 * L.sd;
    L.part = L.rec + nseq * L.nch * L.rec_f;
    L.tcws = L.part + (a.shared ? nseq * 2 * L.sd : 0);
    L.total = L.tcws;
    if (a.fwd_tc) {   // the tensor-core scan's own coefficient records
        LinearArgs f{};
        f.B = a.B; f.H = a.H; f.T = a.T; f.dk = a.dk; f.dv = a.dv; f.chunk = a.chunk;
        f.bf16 = a.bf16;
        L.tcws = (L.tcws + 3) / 4 * 4;   // 16-byte aligned
        L.total = L.tcws + (linear_tc_workspace_bytes(f) + 3) / 4;
    }
    return L;
}

// ------------------------------------------------------------------------
// records: coefficients and the score-times-coefficient table A per chunk
// ------------------------------------------------------------------------

template <typename Tin>
__global__ void __launch_bounds__(kBT) bwd_records_kernel(const BwdArgs a, const BwdLayout L,
                                                          float* ws) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const int seq = blockIdx.x, c = blockIdx.y;
    const int dk = a.dk, bc = L.bc, ldk = dk + 4;   // 16-byte aligned rows
    const int t0 = c * bc, n = min(bc, a.T - t0);
    float* Qs = sm;                    // [bc][ldk]
    float* Ks = Qs + bc * ldk;         // [bc][ldk]
    float* C = Ks + bc * ldk;          // [bc][bc + 1]
    float* th = C + bc * (bc + 1);
    float* et = th + bc;
    float* al = et + bc;
    float* beta = al + bc;
    float* P = beta + bc;
    float* cc = P + bc;
    float* pm = cc + bc;
    const Tin* q = static_cast<const Tin*>(a.q);
    const Tin* k = static_cast<const Tin*>(a.k);
    const size_t tok0 = (size_t)seq * a.T + t0;
    for (int x = tid; x < bc * dk; x += kBT) {
        const int s = x / dk, j = x % dk;
        Qs[s * ldk + j] = s < n ? load_in(q, (tok0 + s) * dk + j) : 0.f;
        Ks[s * ldk + j] = s < n ? load_in(k, (tok0 + s) * dk + j) : 0.f;
    }
    for (int s = tid; s < bc; s += kBT) {
        th[s] = s < n ? a.theta[tok0 + s] : 0.f;
        et[s] = (s < n && a.eta) ? a.eta[tok0 + s] : 0.f;
        al[s] = (s < n && a.alpha) ? a.alpha[tok0 + s] : 0.f;
    }
    __syncthreads();
    block_coefficients(n, bc, th, et, al, beta, P, cc, C, bc + 1, pm);
    float* rec = ws + L.rec + ((size_t)seq * L.nch + c) * L.rec_f;
    for (int x = tid; x < bc * bc; x += kBT) {
        const int t = x / bc, s = x % bc;
        float acc = 0.f;
        if (s <= t && t < n) {
            for (int j = 0; j < dk; j += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(Qs + t * ldk + j);
                const float4 b4 = *reinterpret_cast<const float4*>(Ks + s * ldk + j);
                acc += a4.x * b4.x + a4.y * b4.y + a4.z * b4.z + a4.w * b4.w;
            }
            acc *= C[t * (bc + 1) + s];
        }
        rec[x] = acc;
    }
    float* vec = rec + (size_t)bc * bc;
    for (int s = tid; s < bc; s += kBT) {
        vec[s] = s < n ? beta[s] : 0.f;
        vec[bc + s] = s < n ? cc[s] : 0.f;
        vec[2 * bc + s] = s < n ? C[(n - 1) * (bc + 1) + s] : 0.f;
        vec[3 * bc + s] = s < n ? pm[s] : 0.f;
    }
    if (tid == 0) vec[4 * bc] = P[n - 1];
}

// ------------------------------------------------------------------------
// chain: the adjoint of the state at every chunk end, chunks in reverse
// ------------------------------------------------------------------------

constexpr int kBT2 = 512;     // threads per chain CTA (one per SM)

// 16-byte pieces of q (and of k) per thread and chunk, at most
template <typename Tin>
constexpr int pieces_per_thread() {
    return (kMaxBC * kMaxDK / (16 / (int)sizeof(Tin)) + kBT2 - 1) / kBT2;
}

// A chunk's inputs to the chain, held in registers while the previous chunk
// computes: q and k rows as 16-byte pieces, the record's A table and vectors,
// and the slice's dz.
template <typename Tin>
struct ChainPrefetch {
    static constexpr int kPre = pieces_per_thread<Tin>();
    uint4 q[kPre], k[kPre];
    float4 A[2];
    float vec, dz[2];
};

template <typename Tin>
__device__ __forceinline__ void chain_fetch(ChainPrefetch<Tin>& f, const BwdArgs& a,
                                            const BwdLayout& L, const float* ws, int seq, int c,
                                            int r0, int nr) {
    const int tid = threadIdx.x, dk = a.dk, bc = L.bc;
    const int t0 = c * bc, n = min(bc, a.T - t0);
    const size_t tok0 = (size_t)seq * a.T + t0;
    constexpr int per = 16 / sizeof(Tin);                  // elements per piece
    const int nvec = n * dk / per;
    const uint4* q = reinterpret_cast<const uint4*>(static_cast<const Tin*>(a.q) + tok0 * dk);
    const uint4* k = reinterpret_cast<const uint4*>(static_cast<const Tin*>(a.k) + tok0 * dk);
#pragma unroll
    for (int u = 0; u < ChainPrefetch<Tin>::kPre; ++u) {
        const int v = tid + u * kBT2;
        f.q[u] = v < nvec ? __ldg(q + v) : make_uint4(0, 0, 0, 0);
        f.k[u] = v < nvec ? __ldg(k + v) : make_uint4(0, 0, 0, 0);
    }
    const float* rec = ws + L.rec + ((size_t)seq * L.nch + c) * L.rec_f;
    const float4* rec4 = reinterpret_cast<const float4*>(rec);
#pragma unroll
    for (int u = 0; u < 2; ++u) {   // the record's A table: bc^2 floats, read as 4-float pieces
        const int v = tid + u * kBT2;
        f.A[u] = v < (bc * bc + 3) / 4 ? __ldg(rec4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    f.vec = tid < 4 * bc + 1 ? __ldg(rec + (size_t)bc * bc + tid) : 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int x = tid + u * kBT2, s = x / kR2, i = x % kR2;
        f.dz[u] = (s < n && i < nr)
                      ? load_in(static_cast<const Tin*>(a.dz), (tok0 + s) * a.dv + r0 + i)
                      : 0.f;
    }
}

// dst is 16-byte aligned (rows of dk + 4 floats, pieces of 4 or 8 values).
__device__ __forceinline__ void unpack_piece(const uint4& p, float* dst, const float*) {
    *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(&p);
}
__device__ __forceinline__ void unpack_piece(const uint4& p, float* dst, const __nv_bfloat16*) {
    float4* d4 = reinterpret_cast<float4*>(dst);
    d4[0] = make_float4(__uint_as_float(p.x << 16), __uint_as_float(p.x & 0xffff0000u),
                        __uint_as_float(p.y << 16), __uint_as_float(p.y & 0xffff0000u));
    d4[1] = make_float4(__uint_as_float(p.z << 16), __uint_as_float(p.z & 0xffff0000u),
                        __uint_as_float(p.w << 16), __uint_as_float(p.w & 0xffff0000u));
}

// ------------------------------------------------------------------------
// chain: the adjoint of the state at every chunk end, chunks in reverse
// ------------------------------------------------------------------------

// Shared-memory carve-up of the chain pass (floats; every region a multiple of
// 4 floats so that 16-byte rows stay aligned).
struct ChainSmem {
    int ldk;                       // row stride of q, k and the adjoint rows: dk + 4
    size_t Qs, Ks, A, dZ, bz, cz, de, dWK, dSK, dW, dS, vec, total;
};

__host__ __device__ inline ChainSmem chain_smem(int bc, int dk) {
    auto up = [](size_t x) { return (x + 3) / 4 * 4; };
    ChainSmem m;
    m.ldk = dk + 4;
    size_t o = 0;
    // q and k, later reused for the update's four token-group partial sums of
    // W and S ([4][2][kR2][dk]): the region holds the larger of the two
    const size_t qk = 2 * up((size_t)bc * m.ldk), parts = 8 * (size_t)kR2 * dk;
    m.Qs = o;
    m.Ks = o + up((size_t)bc * m.ldk);
    o += qk > parts ? qk : parts;
    m.A = o; o += up((size_t)bc * (bc + 1));
    m.dZ = o; o += up((size_t)bc * kR2);
    m.bz = o; o += up((size_t)bc * kR2);
    m.cz = o; o += up((size_t)bc * kR2);
    m.de = o; o += up((size_t)bc * kR2);
    m.dWK = o; o += up((size_t)bc * kR2);
    m.dSK = o; o += up((size_t)bc * kR2);
    m.dW = o; o += up((size_t)kR2 * m.ldk);
    m.dS = o; o += up((size_t)kR2 * m.ldk);
    m.vec = o; o += up(4 * (size_t)bc + 1);
    m.total = o;
    return m;
}

// One CTA per (sequence, slice of kR2 = 16 rows), chunks in reverse.  Per chunk:
//   keys:   dWK[s][i] = (dWe k_s)_i, dSK likewise  (thread: one key s, rows 2p, 2p+1,
//           16-byte steps along the key)
//   errors: de[s][i] = -2 (sum_{t>=s} A[t][s] dz_t[i] + C_n[s] dWK + pm[s] dSK)
//   update: dW = beta_n dW + sum_t (beta_t dz_t[i] q_t + de_t[i] k_t),
//           dS = c_n dW + P_n dS + sum_t c_t dz_t[i] q_t
//           (thread: row i = tid / 32, columns 4 (tid % 32) .. + 3; per token one
//           16-byte load of q and of k and three broadcasts)
template <typename Tin>
__global__ void __launch_bounds__(kBT2, 1) bwd_chain_kernel(const BwdArgs a, const BwdLayout L,
                                                            float* ws) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const int seq = blockIdx.x;
    const int dk = a.dk, dv = a.dv, bc = L.bc;
    const int r0 = blockIdx.y * kR2, nr = min(kR2, dv - r0);
    constexpr int per = 16 / sizeof(Tin);
    const ChainSmem M = chain_smem(bc, dk);
    const int ldk = M.ldk;
    float* Qs = sm + M.Qs;
    float* Ks = sm + M.Ks;
    float* A = sm + M.A;
    float* dZ = sm + M.dZ;      // [bc][kR2]
    float* bz = sm + M.bz;      // beta_t dz_t[i]
    float* cz = sm + M.cz;      // c_t dz_t[i]
    float* de = sm + M.de;
    float* dWK = sm + M.dWK;
    float* dSK = sm + M.dSK;
    float* dW = sm + M.dW;      // [kR2][ldk] running adjoint of W
    float* dS = sm + M.dS;
    float* vec = sm + M.vec;    // beta, cc, clast, pm [bc] each, P_n

    const size_t sd = L.sd;
    for (int x = tid; x < kR2 * dk; x += kBT2) {
        const int i = x / dk, j = x % dk;
        const size_t g = (size_t)seq * sd + (size_t)(r0 + i) * dk + j;
        dW[i * ldk + j] = (i < nr && a.dW) ? a.dW[g] : 0.f;
        dS[i * ldk + j] = (i < nr && a.dS) ? a.dS[g] : 0.f;
    }
    ChainPrefetch<Tin> f;
    chain_fetch<Tin>(f, a, L, ws, seq, L.nch - 1, r0, nr);
    const int ks = tid >> 3, kp = tid & 7;          // errors phase: key, row pair
    // keys phase: key = tid % 64 across the lanes, row pair = tid / 64 uniform per
    // warp, so the adjoint rows are broadcast reads and the key rows conflict-free
    const int kk = tid & 63, kq = tid >> 6;
    const int uj = (tid & 31) * 4;                  // update phase: first column of the lane
    for (int c = L.nch - 1; c >= 0; --c) {
        const int t0 = c * bc, n = min(bc, a.T - t0);
        __syncthreads();   // the previous chunk is done with every buffer
        {   // this chunk's inputs from the prefetch registers into shared memory
            const int nvec = bc * dk / per;
#pragma unroll
            for (int u = 0; u < ChainPrefetch<Tin>::kPre; ++u) {
                const int v = tid + u * kBT2;
                if (v < nvec) {
                    const int e0 = v * per, srow = e0 / dk, j = e0 % dk;
                    unpack_piece(f.q[u], Qs + srow * ldk + j, static_cast<const Tin*>(nullptr));
                    unpack_piece(f.k[u], Ks + srow * ldk + j, static_cast<const Tin*>(nullptr));
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int v = tid + u * kBT2;
                const float x4[4] = {f.A[u].x, f.A[u].y, f.A[u].z, f.A[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int idx = 4 * v + e;   // element t * bc + s of the table
                    if (idx < bc * bc) A[(idx / bc) * (bc + 1) + idx % bc] = x4[e];
                }
                const int x = tid + u * kBT2;
                if (x < bc * kR2) dZ[x] = f.dz[u];
            }
            if (tid < 4 * bc + 1) vec[tid] = f.vec;
        }
        // this chunk's end adjoint, for the local pass
        float* adj = ws + L.adj + ((size_t)seq * L.nch + c) * 2 * sd;
        for (int x = tid; x < nr * dk; x += kBT2) {
            const int i = x / dk, j = x % dk;
            adj[(size_t)(r0 + i) * dk + j] = dW[i * ldk + j];
            adj[sd + (size_t)(r0 + i) * dk + j] = dS[i * ldk + j];
        }
        __syncthreads();
        if (c > 0) chain_fetch<Tin>(f, a, L, ws, seq, c - 1, r0, nr);   // overlaps the compute
        const float* beta = vec;
        const float* cc = vec + bc;
        const float* clast = vec + 2 * bc;
        const float* pm = vec + 3 * bc;
        const float Pn = vec[4 * bc];
        if (kk < bc) {   // keys against the end adjoints; scaled dz for the update
            const int ks = kk, i0 = 2 * kq, i1 = i0 + 1;
            float uw0 = 0.f, uw1 = 0.f, us0 = 0.f, us1 = 0.f;
            for (int j = 0; j < dk; j += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(Ks + ks * ldk + j);
                const float4 w0 = *reinterpret_cast<const float4*>(dW + i0 * ldk + j);
                const float4 w1 = *reinterpret_cast<const float4*>(dW + i1 * ldk + j);
                const float4 s0 = *reinterpret_cast<const float4*>(dS + i0 * ldk + j);
                const float4 s1 = *reinterpret_cast<const float4*>(dS + i1 * ldk + j);
                uw0 += k4.x * w0.x + k4.y * w0.y + k4.z * w0.z + k4.w * w0.w;
                uw1 += k4.x * w1.x + k4.y * w1.y + k4.z * w1.z + k4.w * w1.w;
                us0 += k4.x * s0.x + k4.y * s0.y + k4.z * s0.z + k4.w * s0.w;
                us1 += k4.x * s1.x + k4.y * s1.y + k4.z * s1.z + k4.w * s1.w;
            }
            dWK[ks * kR2 + i0] = uw0;
            dWK[ks * kR2 + i1] = uw1;
            dSK[ks * kR2 + i0] = us0;
            dSK[ks * kR2 + i1] = us1;
            const float z0 = dZ[ks * kR2 + i0], z1 = dZ[ks * kR2 + i1];
            const bool live = ks < n;
            bz[ks * kR2 + i0] = live ? beta[ks] * z0 : 0.f;
            bz[ks * kR2 + i1] = live ? beta[ks] * z1 : 0.f;
            cz[ks * kR2 + i0] = live ? cc[ks] * z0 : 0.f;
            cz[ks * kR2 + i1] = live ? cc[ks] * z1 : 0.f;
        }
        __syncthreads();
        if (ks < bc) {   // errors
            const int i0 = 2 * kp;
            float a0 = 0.f, a1 = 0.f;
            for (int t = ks; t < n; ++t) {
                const float at = A[t * (bc + 1) + ks];
                const float2 z = *reinterpret_cast<const float2*>(dZ + t * kR2 + i0);
                a0 += at * z.x;
                a1 += at * z.y;
            }
            const bool live = ks < n;
            de[ks * kR2 + i0] = live ? -2.f * (a0 + clast[ks] * dWK[ks * kR2 + i0] +
                                               pm[ks] * dSK[ks * kR2 + i0]) : 0.f;
            de[ks * kR2 + i0 + 1] = live ? -2.f * (a1 + clast[ks] * dWK[ks * kR2 + i0 + 1] +
                                                   pm[ks] * dSK[ks * kR2 + i0 + 1]) : 0.f;
        }
        __syncthreads();
        // State-adjoint update: warp w owns rows 4 (w % 4) .. + 3 and tokens
        // 16 (w / 4) .. + 15; lane l columns 4 l .. + 3.  The four token groups'
        // partial sums meet in the q / k buffers once every warp is done reading them.
        float gw[4][4], gs[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) gw[r][e] = gs[r][e] = 0.f;
        const int uw = tid >> 5, rg = (uw & 3) * 4, tg = uw >> 2;
        const int tq0 = tg * 16, tq1 = min(n, tq0 + 16);
        if (uj < dk) {
            for (int t = tq0; t < tq1; ++t) {
                const float4 q4 = *reinterpret_cast<const float4*>(Qs + t * ldk + uj);
                const float4 k4 = *reinterpret_cast<const float4*>(Ks + t * ldk + uj);
                const float4 b4 = *reinterpret_cast<const float4*>(bz + t * kR2 + rg);
                const float4 e4 = *reinterpret_cast<const float4*>(de + t * kR2 + rg);
                const float4 c4 = *reinterpret_cast<const float4*>(cz + t * kR2 + rg);
                const float qv[4] = {q4.x, q4.y, q4.z, q4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
                const float bv[4] = {b4.x, b4.y, b4.z, b4.w}, ev[4] = {e4.x, e4.y, e4.z, e4.w};
                const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        gw[r][e] = fmaf(bv[r], qv[e], fmaf(ev[r], kv[e], gw[r][e]));
                        gs[r][e] = fmaf(cv[r], qv[e], gs[r][e]);
                    }
            }
        }
        __syncthreads();   // every warp is done with q and k
        float* part = Qs;  // [4 token groups][W | S][kR2][dk]
        if (uj < dk) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float* pw = part + ((tg * 2 + 0) * kR2 + rg + r) * dk + uj;
                float* ps = part + ((tg * 2 + 1) * kR2 + rg + r) * dk + uj;
                *reinterpret_cast<float4*>(pw) = make_float4(gw[r][0], gw[r][1], gw[r][2], gw[r][3]);
                *reinterpret_cast<float4*>(ps) = make_float4(gs[r][0], gs[r][1], gs[r][2], gs[r][3]);
            }
        }
        __syncthreads();
        {
            const float bn = beta[n - 1], cn = cc[n - 1];
            for (int x = tid; x < kR2 * dk; x += kBT2) {
                const int i = x / dk, j = x % dk;
                float sw = 0.f, ss = 0.f;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    sw += part[((g * 2 + 0) * kR2 + i) * dk + j];
                    ss += part[((g * 2 + 1) * kR2 + i) * dk + j];
                }
                const float w = dW[i * ldk + j], sv = dS[i * ldk + j];
                dW[i * ldk + j] = bn * w + sw;
                dS[i * ldk + j] = cn * w + Pn * sv + ss;
            }
        }
    }
    __syncthreads();
    // adjoint of the initial state: per sequence, or a per-sequence partial
    // that a reduction sums over the batch when W0 / S0 are shared
    float* oW;
    float* oS;
    size_t base;
    if (a.shared) {
        oW = ws + L.part;
        oS = oW + sd;
        base = (size_t)seq * 2 * sd;
    } else {
        oW = a.dW0;
        oS = a.dS0;
        base = (size_t)seq * sd;
    }
    for (int x = tid; x < nr * dk; x += kBT2) {
        const int i = x / dk, j = x % dk;
        const size_t g = base + (size_t)(r0 + i) * dk + j;
        oW[g] = dW[i * ldk + j];
        if (oS) oS[g] = dS[i * ldk + j];
    }
}

// No tokens: the initial state is the final one, so its adjoint is the
// final state's (summed over the batch when W0 / S0 are shared).
__global__ void bwd_empty_kernel(const BwdArgs a, size_t sd) {
    const size_t x = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t nout = (size_t)(a.shared ? 1 : a.B) * a.H * sd;
    if (x >= nout) return;
    float gw = 0.f, gs = 0.f;
    const int nb = a.shared ? a.B : 1;
    for (int b = 0; b < nb; ++b) {
        const size_t src = x + (size_t)b * a.H * sd;
        gw += a.dW ? a.dW[src] : 0.f;
        gs += a.dS ? a.dS[src] : 0.f;
    }
    a.dW0[x] = gw;
    if (a.dS0) a.dS0[x] = gs;
}

// Sums the per-sequence adjoints of a batch-shared W0 / S0 over the batch.
__global__ void bwd_shared_reduce_kernel(const BwdArgs a, const BwdLayout L, const float* ws) {
    const size_t sd = L.sd;
    const size_t x = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= (size_t)a.H * sd) return;
    const int h = (int)(x / sd);
    const size_t e = x % sd;
    float gw = 0.f, gs = 0.f;
    for (int b = 0; b < a.B; ++b) {
        const float* p = ws + L.part + ((size_t)b * a.H + h) * 2 * sd;
        gw += p[e];
        gs += p[sd + e];
    }
    a.dW0[x] = gw;
    if (a.dS0) a.dS0[x] = gs;
}

// ------------------------------------------------------------------------
// local: dq, dk, dv and the gate gradients of one chunk
// ------------------------------------------------------------------------

// Shared-memory carve-up of the local pass (floats).  Rows of q, k and the
// state tiles are dk + 4 floats (16-byte aligned for vector loads); every
// region starts on a 4-float boundary.  The q / k buffers are reused at the end
// for the two [bc][bc + 1] tables of the gate gradients, so that region holds
// the larger of the two uses.
struct LocalSmem {
    int ldk, ldb;
    size_t Qs, Ks, QK, Cm, Xm, Wr, Sr, dWr, dSr, dZt, Et, dWK, dSK, de, vec, total;
};

__host__ __device__ inline LocalSmem local_smem(int bc, int dk) {
    auto up = [](size_t x) { return (x + 3) / 4 * 4; };
    LocalSmem m;
    m.ldk = dk + 4;
    m.ldb = bc + 1;
    const size_t ldr = kR3 + 1;
    const size_t qk = 2 * (size_t)bc * m.ldk, tables = 2 * (size_t)bc * m.ldb;
    size_t o = 0;
    m.Qs = o;
    m.Ks = o + (size_t)bc * m.ldk;
    o += up(qk > tables ? qk : tables);
    m.QK = o; o += up((size_t)bc * m.ldb);
    m.Cm = o; o += up((size_t)bc * m.ldb);
    m.Xm = o; o += up((size_t)bc * m.ldb);
    m.Wr = o; o += (size_t)kR3 * m.ldk;
    m.Sr = o; o += (size_t)kR3 * m.ldk;
    m.dWr = o; o += (size_t)kR3 * m.ldk;
    m.dSr = o; o += (size_t)kR3 * m.ldk;
    m.dZt = o; o += up(bc * ldr);
    m.Et = o; o += up(bc * ldr);
    m.dWK = o; o += up(bc * ldr);
    m.dSK = o; o += up(bc * ldr);
    m.de = o; o += up(bc * ldr);
    m.vec = o; o += up(14 * (size_t)bc + 4);
    m.total = o;
    return m;
}

size_t local_smem_floats(int bc, int dk) { return local_smem(bc, dk).total; }

// A thread owns rows t = 4 tg + a (a < 4) and columns j = jg + 32 bb (bb < 4)
// of dq / dk (tg = tid / 32, jg = tid % 32), and the 4 x 2 block of
// DE[t][s] = dz_t . e_s with s = jg + 32 bb (bb < 2).
template <typename Tin>
__global__ void __launch_bounds__(kBT3, 1) bwd_local_kernel(const BwdArgs a, const BwdLayout L,
                                                           const float* ws) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const int seq = blockIdx.x, c = blockIdx.y;
    const LocalSmem M = local_smem(L.bc, a.dk);
    const int dk = a.dk, dv = a.dv, bc = L.bc, ldk = M.ldk, ldb = M.ldb;
    constexpr int ldr = kR3 + 1;
    const int t0 = c * bc, n = min(bc, a.T - t0);
    const size_t tok0 = (size_t)seq * a.T + t0;
    const size_t sd = L.sd;

    float* Qs = sm + M.Qs;             // [bc][ldk]
    float* Ks = sm + M.Ks;             // [bc][ldk]
    float* QK = sm + M.QK;             // [bc][ldb]  q_t . k_s (s <= t), later dC
    float* Cm = sm + M.Cm;             // [bc][ldb]  C[t][s]
    float* Xm = sm + M.Xm;             // [bc][ldb]  A = C QK, later C DE
    float* Wr = sm + M.Wr;             // [kR3][ldk] tile of W (chunk start)
    float* Sr = sm + M.Sr;             //            tile of S
    float* dWr = sm + M.dWr;           //            tile of dWe (chunk end adjoint)
    float* dSr = sm + M.dSr;           //            tile of dSe
    float* dZt = sm + M.dZt;           // [bc][ldr]
    float* Et = sm + M.Et;             // [bc][ldr]  e_s, rows of the tile
    float* dWK = sm + M.dWK;           // [bc][ldr]  (dWe k_s)_i
    float* dSK = sm + M.dSK;           // [bc][ldr]  (dSe k_s)_i
    float* de = sm + M.de;             // [bc][ldr]
    float* th = sm + M.vec;
    float* et = th + bc;
    float* al = et + bc;
    float* beta = al + bc;
    float* P = beta + bc;
    float* cc = P + bc;
    float* pm = cc + bc;
    float* dbeta = pm + bc;
    float* dcc = dbeta + bc;
    float* dclast = dcc + bc;          // sum_i e_s[i] (dWe k_s)[i]
    float* dpm = dclast + bc;          // sum_i e_s[i] (dSe k_s)[i]
    float* dkeep = dpm + bc;
    float* deta = dkeep + bc;
    float* dth = deta + bc;
    float* scal = dth + bc;            // <dWe, W>, <dWe, S>, <dSe, S>

    const Tin* q = static_cast<const Tin*>(a.q);
    const Tin* k = static_cast<const Tin*>(a.k);
    const Tin* v = static_cast<const Tin*>(a.v);
    const Tin* dz = static_cast<const Tin*>(a.dz);

    for (int x = tid; x < bc * dk; x += kBT3) {
        const int s = x / dk, j = x % dk;
        Qs[s * ldk + j] = s < n ? load_in(q, (tok0 + s) * dk + j) : 0.f;
        Ks[s * ldk + j] = s < n ? load_in(k, (tok0 + s) * dk + j) : 0.f;
    }
    for (int s = tid; s < bc; s += kBT3) {
        th[s] = s < n ? a.theta[tok0 + s] : 0.f;
        et[s] = (s < n && a.eta) ? a.eta[tok0 + s] : 0.f;
        al[s] = (s < n && a.alpha) ? a.alpha[tok0 + s] : 0.f;
        dbeta[s] = dcc[s] = dclast[s] = dpm[s] = dkeep[s] = deta[s] = 0.f;
    }
    if (tid < 4) scal[tid] = 0.f;
    __syncthreads();
    block_coefficients(n, bc, th, et, al, beta, P, cc, Cm, ldb, pm);
    for (int x = tid; x < bc * bc; x += kBT3) {
        const int t = x / bc, s = x % bc;
        float acc = 0.f;
        if (s <= t && t < n)
            for (int j = 0; j < dk; j += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(Qs + t * ldk + j);
                const float4 b4 = *reinterpret_cast<const float4*>(Ks + s * ldk + j);
                acc += a4.x * b4.x + a4.y * b4.y + a4.z * b4.z + a4.w * b4.w;
            }
        QK[t * ldb + s] = acc;
        Xm[t * ldb + s] = acc * Cm[t * ldb + s];
    }

    const int tg = tid >> 5, jg = tid & 31;
    float U[4][4], V[4][4], DK[4][4], DE[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) U[r][bb] = V[r][bb] = DK[r][bb] = 0.f;
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) DE[r][bb] = 0.f;
    }

    const float* ck = ws + L.ckpt + ((size_t)seq * L.nch + c) * 2 * sd;
    const float* ad = ws + L.adj + ((size_t)seq * L.nch + c) * 2 * sd;
    for (int r0 = 0; r0 < dv; r0 += kR3) {
        const int nr = min(kR3, dv - r0);
        __syncthreads();   // the previous tile is consumed (and the tables above are built)
        for (int x = tid; x < kR3 * dk; x += kBT3) {
            const int i = x / dk, j = x % dk;
            const size_t g = (size_t)(r0 + i) * dk + j;
            const bool in = i < nr;
            Wr[i * ldk + j] = in ? ck[g] : 0.f;
            Sr[i * ldk + j] = in ? ck[sd + g] : 0.f;
            dWr[i * ldk + j] = in ? ad[g] : 0.f;
            dSr[i * ldk + j] = in ? ad[sd + g] : 0.f;
        }
        for (int x = tid; x < bc * kR3; x += kBT3) {
            const int s = x / kR3, i = x % kR3;
            dZt[s * ldr + i] = (s < n && i < nr) ? load_in(dz, (tok0 + s) * dv + r0 + i) : 0.f;
        }
        __syncthreads();
        {   // errors at the chunk start and the end adjoints applied to each key:
            // row i = warp (its W, dWe, dSe rows are broadcast reads), keys lane and
            // lane + 32 (conflict-free rows of k)
            const int i = tid >> 5, lane = tid & 31;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int s = lane + 32 * r;
                float e = 0.f, uw = 0.f, us = 0.f;
                for (int j = 0; j < (s < bc ? dk : 0); j += 4) {
                    const float4 k4 = *reinterpret_cast<const float4*>(Ks + s * ldk + j);
                    const float4 w4 = *reinterpret_cast<const float4*>(Wr + i * ldk + j);
                    const float4 g4 = *reinterpret_cast<const float4*>(dWr + i * ldk + j);
                    const float4 h4 = *reinterpret_cast<const float4*>(dSr + i * ldk + j);
                    e += k4.x * w4.x + k4.y * w4.y + k4.z * w4.z + k4.w * w4.w;
                    uw += k4.x * g4.x + k4.y * g4.y + k4.z * g4.z + k4.w * g4.w;
                    us += k4.x * h4.x + k4.y * h4.y + k4.z * h4.z + k4.w * h4.w;
                }
                if (s < bc) {
                    const bool live = s < n && i < nr;
                    Et[s * ldr + i] = live ? e - load_in(v, (tok0 + s) * dv + r0 + i) : 0.f;
                    dWK[s * ldr + i] = uw;
                    dSK[s * ldr + i] = us;
                }
            }
        }
        {   // <dWe, W>, <dWe, S>, <dSe, S> over the tile
            float p0 = 0.f, p1 = 0.f, p2 = 0.f;
            for (int x = tid; x < kR3 * dk; x += kBT3) {
                const int i = x / dk, j = x % dk;
                const float w = Wr[i * ldk + j], sv = Sr[i * ldk + j], gw = dWr[i * ldk + j];
                p0 += gw * w;
                p1 += gw * sv;
                p2 += dSr[i * ldk + j] * sv;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                p0 += __shfl_xor_sync(0xffffffffu, p0, off);
                p1 += __shfl_xor_sync(0xffffffffu, p1, off);
                p2 += __shfl_xor_sync(0xffffffffu, p2, off);
            }
            if ((tid & 31) == 0) {
                atomicAdd(&scal[0], p0);
                atomicAdd(&scal[1], p1);
                atomicAdd(&scal[2], p2);
            }
        }
        __syncthreads();
        for (int sk = tid; sk < n; sk += kBT3) {   // sum over the tile's rows, per key
            float pw = 0.f, ps = 0.f;
#pragma unroll
            for (int i = 0; i < kR3; ++i) {
                const float e = Et[sk * ldr + i];
                pw += e * dWK[sk * ldr + i];
                ps += e * dSK[sk * ldr + i];
            }
            dclast[sk] += pw;
            dpm[sk] += ps;
        }
        {   // de_s and dv_s
            const int i = tid & 15, sg = tid >> 4;
            const float* clast = Cm + (n - 1) * ldb;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int s = sg * 2 + r;
                if (s >= bc) continue;
                float acc = 0.f;
                for (int t = s; t < n; ++t) acc += Xm[t * ldb + s] * dZt[t * ldr + i];
                const float g = s < n ? -2.f * (acc + clast[s] * dWK[s * ldr + i] +
                                                pm[s] * dSK[s * ldr + i])
                                      : 0.f;
                de[s * ldr + i] = g;
                if (s < n && i < nr) store_out(static_cast<Tin*>(a.dv_), (tok0 + s) * dv + r0 + i, -g);
            }
        }
        __syncthreads();
        {   // owned blocks: U += dZ^T W, V += dZ^T S, DK += de W - 2 C_n e dWe - 2 pm e dSe,
            // DE += dZ E^T over the tile's rows
            const float* clast = Cm + (n - 1) * ldb;
            float cl[4], pmv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = tg * 4 + r;
                cl[r] = t < n ? -2.f * clast[t] : 0.f;
                pmv[r] = t < n ? -2.f * pm[t] : 0.f;
            }
            for (int i = 0; i < kR3; ++i) {
                float zt[4], dea[4], ea[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int t = tg * 4 + r;
                    zt[r] = t < bc ? dZt[t * ldr + i] : 0.f;
                    dea[r] = t < bc ? de[t * ldr + i] : 0.f;
                    ea[r] = t < bc ? Et[t * ldr + i] : 0.f;
                }
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    const int j = jg + 32 * bb;
                    if (j >= dk) break;
                    const float w = Wr[i * ldk + j], sv = Sr[i * ldk + j];
                    const float gw = dWr[i * ldk + j], gs = dSr[i * ldk + j];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        U[r][bb] += zt[r] * w;
                        V[r][bb] += zt[r] * sv;
                        DK[r][bb] += dea[r] * w + cl[r] * ea[r] * gw + pmv[r] * ea[r] * gs;
                    }
                }
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int s = jg + 32 * bb;
                    if (s >= bc) break;
                    const float es = Et[s * ldr + i];
#pragma unroll
                    for (int r = 0; r < 4; ++r) DE[r][bb] += zt[r] * es;
                }
            }
        }
    }
    __syncthreads();
    // DE complete: dC[t][s] = -2 QK DE (+ the end-state term on the last row),
    // and C DE for the remaining dq / dk terms
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
            const int t = tg * 4 + r, s = jg + 32 * bb;
            if (t < bc && s < bc) {
                const float d = (s <= t && t < n) ? DE[r][bb] : 0.f;
                const float g = -2.f * QK[t * ldb + s] * d - (t == n - 1 && s < n ? 2.f * dclast[s] : 0.f);
                Xm[t * ldb + s] = Cm[t * ldb + s] * d;
                QK[t * ldb + s] = g;
            }
        }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = tg * 4 + r;
        if (t >= n) continue;
        float pb = 0.f, pc = 0.f;
        // the score terms of the four columns, each score read once
        float sq[4] = {0.f, 0.f, 0.f, 0.f}, sk[4] = {0.f, 0.f, 0.f, 0.f};
        const int jmax = dk - jg;   // columns jg + 32 bb < dk
        for (int s2 = 0; s2 <= t; ++s2) {
            const float x = Xm[t * ldb + s2];
#pragma unroll
            for (int bb = 0; bb < 4; ++bb)
                if (32 * bb < jmax) sq[bb] += x * Ks[s2 * ldk + jg + 32 * bb];
        }
        for (int u = t; u < n; ++u) {
            const float x = Xm[u * ldb + t];
#pragma unroll
            for (int bb = 0; bb < 4; ++bb)
                if (32 * bb < jmax) sk[bb] += x * Qs[u * ldk + jg + 32 * bb];
        }
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
            const int j = jg + 32 * bb;
            if (j >= dk) break;
            const float qv = Qs[t * ldk + j];
            pb += qv * U[r][bb];
            pc += qv * V[r][bb];
            store_out(static_cast<Tin*>(a.dq), (tok0 + t) * dk + j,
                      beta[t] * U[r][bb] + cc[t] * V[r][bb] - 2.f * sq[bb]);
            store_out(static_cast<Tin*>(a.dk_), (tok0 + t) * dk + j, DK[r][bb] - 2.f * sk[bb]);
        }
        // the warp owns rows 4 tg .. 4 tg + 3: its lanes' partial sums are the whole
        pb = warp_sum_f(pb);
        pc = warp_sum_f(pc);
        if (jg == 0) {
            dbeta[t] = pb;
            dcc[t] = pc;
        }
    }
    __syncthreads();
    // gate gradients: C[t][s] = theta_s w(s,t), pm[s] = theta_s m(s,n-1) with
    // m(s,t) = eta_t m(s,t-1), w(s,t) = (1 - alpha_t) w(s,t-1) + m(s,t)
    // (w(s,s) = m(s,s) = 1); tables of w and m reuse the q / k buffers.
    float* Wm = Qs;                    // [bc][ldb]  w(s,t) at [t][s]
    float* Mm = Wm + bc * ldb;         // [bc][ldb]  m(s,t) at [t][s]
    const float* dC = QK;
    float* Kc = Xm;                    // [bc][ldb]  contributions of column s to dkeep[t]
    float* Ec = Cm;                    // [bc][ldb]  contributions of column s to deta[t]
    for (int s = tid; s < bc; s += kBT3)
        for (int t = 0; t < bc; ++t) Kc[t * ldb + s] = Ec[t * ldb + s] = 0.f;
    for (int s = tid; s < n; s += kBT3) {
        float m = 1.f, w = 1.f;
        Wm[s * ldb + s] = 1.f;
        Mm[s * ldb + s] = 1.f;
        for (int t = s + 1; t < n; ++t) {
            m = et[t] * m;
            w = (1.f - al[t]) * w + m;
            Wm[t * ldb + s] = w;
            Mm[t * ldb + s] = m;
        }
    }
    __syncthreads();
    for (int s = tid; s < n; s += kBT3) {
        const float ths = th[s];
        float g = -2.f * dpm[s] * Mm[(n - 1) * ldb + s];   // d pm[s] / d theta_s
        for (int t = s; t < n; ++t) g += dC[t * ldb + s] * Wm[t * ldb + s];
        dth[s] = g;
        float dw = ths * dC[(n - 1) * ldb + s];            // adjoint of w(s, n-1)
        float dm = ths * (-2.f * dpm[s]);                  // adjoint of m(s, n-1), direct part
        for (int t = n - 1; t > s; --t) {
            Kc[t * ldb + s] = dw * Wm[(t - 1) * ldb + s];
            dm += dw;                                      // w(s,t) = ... + m(s,t)
            Ec[t * ldb + s] = dm * Mm[(t - 1) * ldb + s];
            dm = et[t] * dm;
            dw = (1.f - al[t]) * dw + ths * dC[(t - 1) * ldb + s];
        }
    }
    __syncthreads();
    for (int t = tid; t < n; t += kBT3) {   // sum every column's contribution per token
        float gk = 0.f, ge = 0.f;
        for (int s = 0; s < t; ++s) {
            gk += Kc[t * ldb + s];
            ge += Ec[t * ldb + s];
        }
        dkeep[t] += gk;
        deta[t] += ge;
    }
    __syncthreads();
    if (tid == 0) {
        // beta_t = keep_t beta_{t-1}, P_t = eta_t P_{t-1}, c_t = keep_t c_{t-1} + P_t;
        // the end state adds beta_n <dWe,W>, c_n <dWe,S> and P_n <dSe,S>
        float rb = 0.f, rc = 0.f, rp = 0.f;
        for (int t = n - 1; t >= 0; --t) {
            const bool last = t == n - 1;
            const float db = dbeta[t] + rb + (last ? scal[0] : 0.f);
            const float dc = dcc[t] + rc + (last ? scal[1] : 0.f);
            const float dp = rp + dc + (last ? scal[2] : 0.f);
            const float keep = 1.f - al[t];
            const float cprev = t > 0 ? cc[t - 1] : 0.f;
            const float bprev = t > 0 ? beta[t - 1] : 1.f;
            const float pprev = t > 0 ? P[t - 1] : 1.f;
            dkeep[t] += dc * cprev + db * bprev;
            deta[t] += dp * pprev;
            rc = keep * dc;
            rb = keep * db;
            rp = et[t] * dp;
        }
    }
    __syncthreads();
    for (int t = tid; t < n; t += kBT3) {
        a.dtheta[tok0 + t] = dth[t];
        if (a.deta) a.deta[tok0 + t] = deta[t];
        if (a.dalpha) a.dalpha[tok0 + t] = -dkeep[t];
    }
}

size_t records_smem_floats(int bc, int dk) {
    return 2 * (size_t)bc * (dk + 4) + (size_t)bc * (bc + 1) + 7 * (size_t)bc;
}

size_t chain_smem_floats(int bc, int dk) { return chain_smem(bc, dk).total; }

template <typename Tin>
cudaError_t launch_passes(const BwdArgs& a, const BwdLayout& L, cudaStream_t s, int* launches) {
    float* ws = static_cast<float*>(a.workspace);
    // forward scan writing the state at every chunk start
    LinearArgs f{};
    f.B = a.B; f.H = a.H; f.T = a.T; f.dk = a.dk; f.dv = a.dv; f.chunk = a.chunk;
    f.bf16 = a.bf16;
    f.q = a.q; f.k = a.k; f.v = a.v;
    f.eta = a.eta; f.theta = a.theta; f.alpha = a.alpha;
    f.W0 = a.W0; f.S0 = a.S0; f.shared = a.shared;
    f.ckpt = ws + L.ckpt;
    // the tensor-core passes take the scan's masked score tiles (in the space
    // of the records, which they do not use) and its coefficient records
    if (a.local_tc) {
        f.score_tiles = ws + L.rec;
        f.ckpt_bf16 = 1;   // the tensor-core local pass loads bf16 checkpoints by TMA
    }
    cudaError_t e;
    if (a.fwd_tc) {
        f.workspace = ws + L.tcws;
        f.workspace_bytes = linear_tc_workspace_bytes(f);
        f.status = a.status;
        e = linear_tc_launch(f, s);
        *launches += 2;   // coefficient pre-pass and scan
    } else {
        e = linear_simt_launch(f, s);
        ++*launches;
    }
    if (e != cudaSuccess) return e;

    const int nseq = a.B * a.H;
    const size_t sm0 = records_smem_floats(L.bc, a.dk) * sizeof(float);
    const size_t sm2 = chain_smem_floats(L.bc, a.dk) * sizeof(float);
    const size_t sm3 = local_smem_floats(L.bc, a.dk) * sizeof(float);
    if ((e = cudaFuncSetAttribute(bwd_records_kernel<Tin>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm0)) ||
        (e = cudaFuncSetAttribute(bwd_chain_kernel<Tin>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) ||
        (e = cudaFuncSetAttribute(bwd_local_kernel<Tin>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)))
        return e;
    if (a.local_tc) {
        // chain and local passes on the tensor cores
        if ((e = bwd_chain_tc_launch(a, ws, L.adj, ws + L.tcws, ws + L.rec, L.part, s)) !=
            cudaSuccess)
            return e;
        if ((e = bwd_local_tc_launch(a, ws + L.ckpt, ws + L.adj, ws + L.tcws, s)) != cudaSuccess)
            return e;
        *launches += 2;
    } else {
        bwd_records_kernel<Tin><<<dim3(nseq, L.nch), kBT, sm0, s>>>(a, L, ws);
        bwd_chain_kernel<Tin><<<dim3(nseq, (a.dv + kR2 - 1) / kR2), kBT2, sm2, s>>>(a, L, ws);
        bwd_local_kernel<Tin><<<dim3(nseq, L.nch), kBT3, sm3, s>>>(a, L, ws);
        *launches += 3;
    }
    if (a.shared) {
        const size_t n = (size_t)a.H * L.sd;
        bwd_shared_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, L, ws);
        ++*launches;
    }
    return cudaGetLastError();
}

}  // namespace

bool linear_bwd_supported(const BwdArgs& a) {
    LinearArgs f{};
    f.dk = a.dk; f.chunk = a.chunk;
    return a.chunk >= 1 && a.chunk <= kMaxBC && a.dk >= 1 && a.dk <= kMaxDK &&
           linear_simt_supported(f) &&
           local_smem_floats(a.chunk, a.dk) * sizeof(float) <= 227 * 1024;
}

size_t linear_bwd_workspace_bytes(const BwdArgs& a) { return bwd_layout(a).total * sizeof(float); }

cudaError_t linear_bwd_launch(const BwdArgs& a, cudaStream_t s, int* launches) {
    const BwdLayout L = bwd_layout(a);
    if (a.T == 0) {
        const size_t n = (size_t)(a.shared ? 1 : a.B) * a.H * L.sd;
        bwd_empty_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, L.sd);
        ++*launches;
        return cudaGetLastError();
    }
    return a.bf16 ? launch_passes<__nv_bfloat16>(a, L, s, launches)
                  : launch_passes<float>(a, L, s, launches);
}

}  // namespace ttm
