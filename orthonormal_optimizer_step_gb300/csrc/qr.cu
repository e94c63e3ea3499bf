// qr.cu -- batched CholeskyQR2 of tall m x r panels in float32.
//
// Dion orthonormalizes the m x r panel P = B Q at every step ("Dion: The
// distributed orthonormal update revolution is here": power iteration needs an
// orthonormal basis of the iterate).  One CholeskyQR pass is
//     S = P^T P,   S = L L^T,   P <- P L^{-T};
// two passes (CholeskyQR2) bring ||P^T P - I|| to float32 rounding level for
// panels with condition number up to ~1e3.  The Gram and the triangular
// application are batched GEMMs; the r x r factorization runs one CTA per
// matrix.
//
// Rank deficiency: a pivot d <= r * 6e-8 * max(diag S) (or non-finite) marks
// column j dependent.  Its column of L is zeroed and its column of L^{-T} is
// set to zero, so the corresponding column of the new P is exactly zero and
// the remaining columns stay orthonormal; the status word records the event.
#include "internal.h"
#include "simt_gemm.cuh"

namespace dion {

template <bool kSmem>
__global__ void __launch_bounds__(1024) chol_inv_kernel(int r, float* S, float* W, int* dead_g, int* status)
{
    extern __shared__ float smem[];
    __shared__ float s_piv, s_thr;
    __shared__ int s_dead, s_bad;
    const int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
    float* Sg = S + (size_t)b * r * r;
    float* Wg = W + (size_t)b * r * r;
    int* dead = dead_g + (size_t)b * r;
    float* L = kSmem ? smem : Sg;
    if (kSmem)
        for (int e = tid; e < r * r; e += nt) L[e] = Sg[e];
    __syncthreads();
    if (tid == 0) {
        float mx = 0.f;
        for (int i = 0; i < r; ++i) {
            const float d = L[(size_t)i * r + i];
            if (d > mx) mx = d;
        }
        s_thr = mx * (float)r * 6e-8f;
        s_bad = 0;
    }
    __syncthreads();
    for (int j = 0; j < r; ++j) {
        if (tid == 0) {
            const float d = L[(size_t)j * r + j];
            const bool fin = isfinite(d);
            const bool ok = fin && d > s_thr;
            if (!ok) s_bad |= fin ? kStatusPivot : kStatusNonFinite;
            s_dead = !ok;
            s_piv = ok ? sqrtf(d) : 1.f;
            L[(size_t)j * r + j] = s_piv;
            dead[j] = !ok;
        }
        __syncthreads();
        const float piv = s_piv;
        const int dj = s_dead;
        for (int i = j + 1 + tid; i < r; i += nt) {
            float* p = &L[(size_t)i * r + j];
            *p = dj ? 0.f : *p / piv;
        }
        __syncthreads();
        const int w = r - j - 1;
        if (!dj) {
            for (int e = tid; e < w * w; e += nt) {
                const int ii = j + 1 + e / w, kk = j + 1 + e % w;
                if (kk <= ii) L[(size_t)ii * r + kk] -= L[(size_t)ii * r + j] * L[(size_t)kk * r + j];
            }
        }
        __syncthreads();
    }
    // W = L^{-T}: row c of W is column c of L^{-1} (forward substitution).
    for (int c = tid; c < r; c += nt) {
        float* wrow = Wg + (size_t)c * r;
        for (int i = 0; i < c; ++i) wrow[i] = 0.f;
        for (int i = c; i < r; ++i) {
            float s = (i == c) ? 1.f : 0.f;
            for (int k = c; k < i; ++k) s -= L[(size_t)i * r + k] * wrow[k];
            wrow[i] = dead[i] ? 0.f : s / L[(size_t)i * r + i];
        }
    }
    if (tid == 0 && s_bad) atomicOr(status, s_bad);
}

static cudaError_t chol_inv(int batch, int r, float* S, float* W, int* dead, int* status, cudaStream_t st)
{
    const size_t smem = (size_t)r * r * sizeof(float);
    if (smem <= 200 * 1024) {
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(chol_inv_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 200 * 1024);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        return launch("chol_inv_smem", chol_inv_kernel<true>, dim3(batch), dim3(1024), smem, st, r, S, W, dead,
                      status);
    }
    return launch("chol_inv_global", chol_inv_kernel<false>, dim3(batch), dim3(1024), 0, st, r, S, W, dead, status);
}

cudaError_t qr_cholesky2(int batch, int m, int r, long long ldp, float* P, float* Ptmp, float* S, float* W,
                         int* dead, int* status, cudaStream_t st)
{
    const long long sp = (long long)m * ldp, ss = (long long)r * r;
    float* src = P;
    float* dst = Ptmp;
    for (int pass = 0; pass < 2; ++pass) {
        cudaError_t e = gemm_simt<1>("qr_gram", batch, r, r, m, LdA<float, false>{src, sp, ldp},
                                     LdB<float, true>{src, sp, ldp}, LdB<float, true>{src, sp, ldp},
                                     EpStore{S, ss, r}, st);
        if (e != cudaSuccess) return e;
        e = chol_inv(batch, r, S, W, dead, status, st);
        if (e != cudaSuccess) return e;
        e = gemm_simt<1>("qr_apply", batch, m, r, r, LdA<float, true>{src, sp, ldp}, LdB<float, true>{W, ss, r},
                         LdB<float, true>{W, ss, r}, EpStore{dst, sp, ldp}, st);
        if (e != cudaSuccess) return e;
        float* t = src; src = dst; dst = t;
    }
    return cudaSuccess;  // two passes: the result is back in P
}

}  // namespace dion
