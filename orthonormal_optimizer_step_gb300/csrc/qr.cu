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
// Rank deficiency: a pivot d <= 1e-6 * S_jj (the column's own squared norm;
// d / S_jj is the squared sine of its angle to the span of the columns before
// it), or a non-finite pivot, marks column j dependent.  Its column of L is
// zeroed and its column of L^{-T} is set to zero, so the corresponding column
// of the new P is exactly zero and the remaining columns stay orthonormal; the
// status word records the event.
#include "internal.h"
#include "simt_gemm.cuh"

namespace dion {

// One CTA per matrix: Cholesky S = L L^T and W = L^{-T}, both blocked by 32.
//   Cholesky (right-looking), per 32-column block J:
//     warp 0 factors the diagonal block in registers (lane = row; columns
//     are broadcast with shuffles), one thread per row solves the panel below
//     it in registers, and the trailing lower triangle is updated with one
//     warp per row.
//   Inverse Z = L^{-1} (lower), written transposed as W = Z^T:
//     diagonal blocks Z_II = L_II^{-1} (one warp each, registers),
//     then block diagonals d = 1, 2, ...: Z_IJ = -Z_II sum_{K=J}^{I-1} L_IK Z_KJ,
//     with the partial sums parked in the (finally zeroed) lower part of W.
// kSmem: L lives in shared memory with row pitch r + 1 (no bank conflicts);
// otherwise it is factored in place in global memory (pitch r).
template <bool kSmem>
__global__ void __launch_bounds__(512) chol_inv_kernel(int r, float* S, float* W, int* dead_g, int* status)
{
    extern __shared__ float smem[];
    __shared__ int s_bad;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
    const int nwarps = nt >> 5;
    float* Sg = S + (size_t)b * r * r;
    float* Wg = W + (size_t)b * r * r;
    int* dead = dead_g + (size_t)b * r;
    const int ld = kSmem ? r + 1 : r;
    float* L = kSmem ? smem : Sg;
    float* d0 = kSmem ? smem + (size_t)r * ld : smem;     // original diagonal
    if (kSmem)
        for (int e = tid; e < r * r; e += nt) L[(size_t)(e / r) * ld + (e % r)] = Sg[e];
    for (int i = tid; i < r; i += nt) d0[i] = Sg[(size_t)i * r + i];
    if (tid == 0) s_bad = 0;
    __syncthreads();
#define Lx(i, k) L[(size_t)(i) * ld + (k)]

    for (int J = 0; J < r; J += 32) {
        const int jb = min(32, r - J);
        if (warp == 0) {
            // diagonal block in registers: lane = row, a[k] = L(J + lane, J + k)
            float a[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) a[k] = (lane < jb && k < jb) ? Lx(J + lane, J + k) : 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if (c < jb) {
                    const float d = __shfl_sync(0xffffffffu, a[c], c);
                    const bool fin = isfinite(d);
                    const bool ok = fin && d > 1e-6f * d0[J + c];
                    const float piv = ok ? sqrtf(d) : 1.f;
                    if (lane == 0) {
                        dead[J + c] = !ok;
                        if (!ok) s_bad |= fin ? kStatusPivot : kStatusNonFinite;
                    }
                    const float lv = (lane > c) ? (ok ? a[c] / piv : 0.f) : (lane == c ? piv : a[c]);
                    a[c] = lv;
#pragma unroll
                    for (int k = c + 1; k < 32; ++k) {
                        const float lkc = __shfl_sync(0xffffffffu, lv, k);     // L(J + k, J + c)
                        if (lane >= k && lane > c) a[k] = fmaf(-lv, lkc, a[k]);
                    }
                }
            }
            if (lane < jb)
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (k < jb) Lx(J + lane, J + k) = a[k];
        }
        __syncthreads();
        // panel below the diagonal block: one thread per row, row held in registers
        for (int i = J + jb + tid; i < r; i += nt) {
            float a[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) a[c] = (c < jb) ? Lx(i, J + c) : 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if (c < jb) {
                    float s = a[c];
#pragma unroll
                    for (int k = 0; k < c; ++k) s = fmaf(-a[k], Lx(J + c, J + k), s);
                    a[c] = dead[J + c] ? 0.f : s / Lx(J + c, J + c);
                }
            }
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (c < jb) Lx(i, J + c) = a[c];
        }
        __syncthreads();
        // trailing lower triangle: one warp per row i, lanes over k
        const int t0 = J + jb;
        for (int i = t0 + warp; i < r; i += nwarps) {
            float li[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) li[c] = (c < jb) ? Lx(i, J + c) : 0.f;
            for (int k = t0 + lane; k <= i; k += 32) {
                float s = 0.f;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (c < jb) s = fmaf(li[c], Lx(k, J + c), s);
                Lx(i, k) -= s;
            }
        }
        __syncthreads();
    }

    // ---- inverse: W = L^{-T}
    const int nb = (r + 31) / 32;
#define Wx(i, k) Wg[(size_t)(i) * r + (k)]
    for (int I = warp; I < nb; I += nwarps) {
        const int I0 = I * 32, ib = min(32, r - I0);
        const int c = lane;
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float s = (i == c) ? 1.f : 0.f;
            if (i < ib) {                       // rows of L beyond r do not exist
#pragma unroll
                for (int k = 0; k < i; ++k)
                    if (k >= c) s = fmaf(-Lx(I0 + i, I0 + k), z[k], s);
            }
            const bool valid = i >= c && i < ib && c < ib;
            z[i] = (valid && !dead[I0 + i]) ? s / Lx(I0 + i, I0 + i) : 0.f;
        }
        if (c < ib)
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ib) Wx(I0 + c, I0 + i) = z[i];          // W[c][i] = Z[i][c]
    }
    __syncthreads();
    for (int d = 1; d < nb; ++d) {
        // T_IJ = sum_{K=J}^{I-1} L_IK Z_KJ  -> parked at W block (I, J).  The
        // lane index runs over a, so the W row read below is a broadcast.
        for (int e = tid; e < (nb - d) * 1024; e += nt) {
            const int I = d + e / 1024, J = I - d, a = e % 32, bb = (e % 1024) / 32;
            const int I0 = I * 32, J0 = J * 32;
            if (I0 + a >= r || J0 + bb >= r) continue;
            float s = 0.f;
            for (int k = J0; k < I0; ++k) s = fmaf(Lx(I0 + a, k), Wx(J0 + bb, k), s);   // Z[k][J0+bb] = W[J0+bb][k]
            Wx(I0 + a, J0 + bb) = s;
        }
        __syncthreads();
        // Z_IJ = -Z_II T_IJ  -> W block (J, I)
        for (int e = tid; e < (nb - d) * 1024; e += nt) {
            const int I = d + e / 1024, J = I - d, a = (e % 1024) / 32, bb = e % 32;
            const int I0 = I * 32, J0 = J * 32;
            if (I0 + a >= r || J0 + bb >= r) continue;
            float s = 0.f;
            for (int k = 0; k <= a; ++k) s = fmaf(Wx(I0 + k, I0 + a), Wx(I0 + k, J0 + bb), s);  // Z_II[a][k] = W[I0+k][I0+a]
            Wx(J0 + bb, I0 + a) = dead[I0 + a] ? 0.f : -s;
        }
        __syncthreads();
    }
    for (int e = tid; e < r * r; e += nt) {
        const int i = e / r, k = e % r;
        if (k < i) Wx(i, k) = 0.f;
    }
#undef Wx
#undef Lx
    if (tid == 0 && s_bad) atomicOr(status, s_bad);
}

static cudaError_t chol_inv(int batch, int r, float* S, float* W, int* dead, int* status, cudaStream_t st)
{
    const size_t smem = ((size_t)r * (r + 1) + r) * sizeof(float);
    if (smem <= 210 * 1024) {
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(chol_inv_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 210 * 1024);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        return launch("chol_inv_smem", chol_inv_kernel<true>, dim3(batch), dim3(512), smem, st, r, S, W, dead,
                      status);
    }
    return launch("chol_inv_global", chol_inv_kernel<false>, dim3(batch), dim3(512), (size_t)r * sizeof(float), st,
                  r, S, W, dead, status);
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
