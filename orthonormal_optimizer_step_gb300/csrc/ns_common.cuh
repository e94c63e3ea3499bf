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

}  // namespace
}  // namespace dion
