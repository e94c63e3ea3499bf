// ns_common.cuh -- the momentum / norm pass shared by both Newton-Schulz paths.
#pragma once

#include "common.cuh"

namespace dion {
namespace {   // internal linkage: one copy per translation unit

// Momentum and Frobenius norms.  Block bh = (matrix b, head h) covers rows
// [0, m) x columns [h*hd, (h+1)*hd).  If M != NULL: M <- mu M + G, y = M;
// else y = G.  nrm[bh] += sum y^2 (nrm zeroed beforehand).
template <typename T>
__global__ void __launch_bounds__(256) ns_prep_kernel(int m, int n, int hd, int heads, const T* G, float* M, float mu,
                                                      float* nrm)
{
    __shared__ float red[256];
    const int bh = blockIdx.y, b = bh / heads, h = bh % heads;
    const long long base = (long long)b * m * n + (long long)h * hd;
    const long long cnt = (long long)m * hd;
    float s = 0.f;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < cnt; e += (long long)gridDim.x * blockDim.x) {
        const long long o = base + (e / hd) * n + (e % hd);
        float y = to_f(G[o]);
        if (M) {
            y = fmaf(mu, M[o], y);
            M[o] = y;
        }
        s = fmaf(y, y, s);
    }
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) atomicAdd(&nrm[bh], red[0]);
}

// Eight consecutive values of a row as float (T = float or bf16), and back.
__device__ __forceinline__ void ld8(const float* p, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4*>(p), c = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
}
__device__ __forceinline__ void ld8(const bf16* p, float (&v)[8])
{
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __bfloat162float(h[e]);
}
__device__ __forceinline__ void st8(float* p, const float (&v)[8])
{
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void st8(bf16* p, const float (&v)[8])
{
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// ns_prep_kernel with eight columns per thread (hd % 8 == 0, n % 8 == 0,
// 16-byte aligned rows): 32-bit row / unit indexing and vector accesses.
template <typename T>
__global__ void __launch_bounds__(256) ns_prep_vec_kernel(int m, int n, int hd, int heads, const T* G, float* M,
                                                          float mu, float* nrm)
{
    __shared__ float red[8];
    const int bh = blockIdx.y, b = bh / heads, h = bh % heads;
    const size_t base = (size_t)b * m * n + (size_t)h * hd;
    const int upr = hd >> 3, cnt = m * upr;
    float s = 0.f;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < cnt; e += gridDim.x * blockDim.x) {
        const int i = e / upr, c = (e - i * upr) * 8;
        const size_t o = base + (size_t)i * n + c;
        float y[8];
        ld8(G + o, y);
        if (M) {
            float mv[8];
            ld8(M + o, mv);
#pragma unroll
            for (int t = 0; t < 8; ++t) y[t] = fmaf(mu, mv[t], y[t]);
            st8(M + o, y);
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) s = fmaf(y[t], y[t], s);
    }
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
        atomicAdd(&nrm[bh], t);
    }
}

}  // namespace
}  // namespace dion
