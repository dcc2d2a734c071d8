// Device helpers shared by the CUDA-core kernels (forward scan and gradient):
// element loads / stores in the input dtype, the GELU of the 2-layer memory and
// the per-block coefficients of the chunk recurrences.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>

namespace ttm {
namespace simt {

__device__ __forceinline__ float load_in(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_in(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_out(float* p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// Exact GELU x/2 (1 + erf(x / sqrt 2)) of the 2-layer memory and its
// derivative, with CUDA's erff / expf.
__device__ __forceinline__ float gelu(float x) {
    return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
}
__device__ __forceinline__ float gelu_grad(float x) {
    return 0.5f * (1.f + erff(x * 0.70710678118654752f)) +
           x * 0.39894228040143268f * expf(-0.5f * x * x);
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

// Per-block coefficients.  th/et/al hold the n gates of the block; writes
// beta, P, cc (prefix forms), C[t][s] (ld = ldc, s <= t, zero above) and
// pm[s] = theta_s m(s, n-1).  Runs on the whole block; ends with a barrier.
__device__ inline void block_coefficients(int n, int nb, const float* th, const float* et,
                                          const float* al, float* beta, float* P, float* cc,
                                          float* C, int ldc, float* pm) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        float b = 1.f, p = 1.f, c = 0.f;
        for (int t = 0; t < n; ++t) {
            const float keep = 1.f - al[t];
            b *= keep;
            p *= et[t];
            c = keep * c + p;
            beta[t] = b;
            P[t] = p;
            cc[t] = c;
        }
    }
    for (int s = tid; s < nb; s += blockDim.x) {
        if (s >= n) {
            for (int t = 0; t < nb; ++t) C[t * ldc + s] = 0.f;
            pm[s] = 0.f;
            continue;
        }
        for (int t = 0; t < s; ++t) C[t * ldc + s] = 0.f;
        float m = 1.f, w = 1.f;
        C[s * ldc + s] = th[s];
        for (int t = s + 1; t < n; ++t) {
            m = et[t] * m;
            w = (1.f - al[t]) * w + m;
            C[t * ldc + s] = th[s] * w;
        }
        for (int t = n; t < nb; ++t) C[t * ldc + s] = 0.f;
        pm[s] = th[s] * m;
    }
    __syncthreads();
}

}  // namespace simt
}  // namespace ttm
