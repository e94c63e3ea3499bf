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
//   Inverse, in place, block columns from the last to the first: the
//     diagonal block is inverted in registers (one warp, lane = column), and
//     the panel below it becomes -(trailing inverse) * panel * (block inverse).
//   W receives L^{-1} row-major (upper part zero).
// kSmem: L lives in shared memory with row pitch r + 1 (no bank conflicts);
// otherwise it is factored in place in global memory (pitch r).
// Sin holds nparts partial Gram matrices per matrix (summed on load); Swork is
// the in-place factor of the global variant.  Output: W = L^{-1} as float32
// (W != NULL), or as three bf16 terms Z3[3b + t] (pitch ldz, columns up to ldz,
// Z = Z3[0] + Z3[1] + Z3[2] to float32 accuracy) for the tensor-core apply.
template <bool kSmem>
__global__ void __launch_bounds__(512) chol_inv_kernel(int r, const float* Sin, int nparts, float* Swork, float* Wbuf,
                                                       float* W, bf16* Z3, int ldz, int* dead_g, int* status)
{
    extern __shared__ float smem[];
    __shared__ int s_bad;
    __shared__ float s_emax;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
    const int nwarps = nt >> 5;
    const size_t rr = (size_t)r * r;
    const float* Sb = Sin + (size_t)b * nparts * rr;
    float* Sg = Swork + (size_t)b * rr;
    float* Wg = Wbuf + (size_t)b * rr;
    int* dead = dead_g + (size_t)b * r;
    const int ld = kSmem ? r + 1 : r;
    float* L = kSmem ? smem : Sg;
    float* d0 = kSmem ? smem + (size_t)r * ld : smem;     // original diagonal
    int* deadsm = (int*)(d0 + r);                          // dependent-column flags
#define Lx0(i) (kSmem ? L[(size_t)(i) * ld + (i)] : Sg[(size_t)(i) * r + (i)])
    float* T = kSmem ? (float*)(deadsm + r) : Wg;         // (r - 32) x 32 scratch of the inverse
    for (int e = tid; e < r * r; e += nt) {
        float v = Sb[e];
        for (int q = 1; q < nparts; ++q) v += Sb[(size_t)q * rr + e];
        if (kSmem) L[(size_t)(e / r) * ld + (e % r)] = v;
        else Sg[e] = v;
    }
    __syncthreads();
    for (int i = tid; i < r; i += nt) d0[i] = Lx0(i);
    if (tid == 0) { s_bad = 0; s_emax = 0.f; }
    __syncthreads();
#define Lx(i, k) L[(size_t)(i) * ld + (k)]

    // Near-identity Gram (the second CholeskyQR pass of a well-conditioned
    // panel): S = I + E with max|E| <= 1e-4.  Then L = I + F with
    // F = strictly_lower(E) + diag(E)/2 + O(E^2), and L^{-1} = I - F + O(E^2),
    // so the factorization is skipped; the O(E^2) <= 1e-8 terms are below
    // float32 rounding of the result.
    {
        float em = 0.f;
        for (int e = tid; e < r * r; e += nt) {
            const int i = e / r, k = e % r;
            const float v = Lx(i, k) - (i == k ? 1.f : 0.f);
            em = fmaxf(em, isfinite(v) ? fabsf(v) : 1e30f);
        }
        for (int o = 16; o > 0; o >>= 1) em = fmaxf(em, __shfl_xor_sync(0xffffffffu, em, o));
        if (lane == 0) atomicMax((int*)&s_emax, __float_as_int(em));   // em >= 0: int order = float order
        __syncthreads();
        if (s_emax <= 1e-4f) {
            for (int i = tid; i < r; i += nt) dead[i] = 0;
            if (W) {
                float* Wo = W + (size_t)b * rr;
                for (int e = tid; e < r * r; e += nt) {
                    const int i = e / r, k = e % r;
                    Wo[e] = (k < i) ? -Lx(i, k) : (k == i ? 1.f - 0.5f * (Lx(i, i) - 1.f) : 0.f);
                }
            } else {
                const size_t zs = (size_t)r * ldz;
                bf16* z0 = Z3 + (size_t)3 * b * zs;
                for (int e = tid; e < r * ldz; e += nt) {
                    const int i = e / ldz, k = e % ldz;
                    const float v = (k < i) ? -Lx(i, k) : (k == i ? 1.f - 0.5f * (Lx(i, i) - 1.f) : 0.f);
                    const bf16 h1 = __float2bfloat16_rn(v);
                    const float r1 = v - __bfloat162float(h1);
                    const bf16 h2 = __float2bfloat16_rn(r1);
                    z0[e] = h1;
                    z0[zs + e] = h2;
                    z0[2 * zs + e] = __float2bfloat16_rn(r1 - __bfloat162float(h2));
                }
            }
            return;
        }
    }

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
                        deadsm[J + c] = !ok;
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
                    a[c] = deadsm[J + c] ? 0.f : s / Lx(J + c, J + c);
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

    // ---- in-place inverse L <- L^{-1}, block columns from the last one back:
    //   Z_JJ = L_JJ^{-1};  panel <- -(L^{-1} of the trailing part) * panel * Z_JJ
    for (int J = ((r - 1) / 32) * 32; J >= 0; J -= 32) {
        const int jb = min(32, r - J), t0 = J + jb, nt_rows = r - t0;
        // T = Linv_trail * panel  (rows t0..r-1, 32 columns), one warp per row
        for (int i = t0 + warp; i < r; i += nwarps) {
            float s = 0.f;
            if (lane < jb)
                for (int k = t0; k <= i; ++k) s = fmaf(Lx(i, k), Lx(k, J + lane), s);
            T[(size_t)(i - t0) * 32 + lane] = s;
        }
        if (warp == 0) {
            // Z_JJ: lane c computes column c by forward substitution (registers)
            const int c = lane;
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float v = (i == c) ? 1.f : 0.f;
                if (i < jb) {
#pragma unroll
                    for (int k = 0; k < i; ++k)
                        if (k >= c) v = fmaf(-Lx(J + i, J + k), z[k], v);
                }
                z[i] = (i >= c && i < jb && c < jb) ? v / Lx(J + i, J + i) : 0.f;
            }
            __syncwarp();
            if (c < jb)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i >= c && i < jb) Lx(J + i, J + c) = z[i];
        }
        __syncthreads();
        // panel <- -T * Z_JJ
        for (int i = t0 + warp; i < r; i += nwarps) {
            if (lane < jb) {
                float s = 0.f;
                for (int k = lane; k < jb; ++k) s = fmaf(T[(size_t)(i - t0) * 32 + k], Lx(J + k, J + lane), s);
                Lx(i, J + lane) = -s;
            }
        }
        (void)nt_rows;
        __syncthreads();
    }
    // W = L^{-1} row-major with a zero upper part; rows of dependent columns are zero,
    // so the apply P <- P W^T leaves those columns of P at zero.
    if (W) {
        float* Wo = W + (size_t)b * rr;
        for (int e = tid; e < r * r; e += nt) {
            const int i = e / r, k = e % r;
            Wo[e] = (k <= i && !deadsm[i]) ? Lx(i, k) : 0.f;
        }
    } else {
        const size_t zs = (size_t)r * ldz;
        bf16* z0 = Z3 + (size_t)3 * b * zs;
        for (int e = tid; e < r * ldz; e += nt) {
            const int i = e / ldz, k = e % ldz;
            const float v = (k <= i && k < r && !deadsm[i]) ? Lx(i, k) : 0.f;
            const bf16 h1 = __float2bfloat16_rn(v);
            const float r1 = v - __bfloat162float(h1);
            const bf16 h2 = __float2bfloat16_rn(r1);
            const bf16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
            z0[e] = h1;
            z0[zs + e] = h2;
            z0[2 * zs + e] = h3;
        }
    }
#undef Lx0
#undef Lx
    if (tid == 0 && s_bad) atomicOr(status, s_bad);
}

static size_t chol_smem_bytes(int r, bool in_smem)
{
    const size_t scratch = (size_t)(r > 32 ? r - 32 : 0) * 32;
    return in_smem ? ((size_t)r * (r + 1) + r + r + scratch) * sizeof(float) : (size_t)2 * r * sizeof(float);
}

cudaError_t chol_inv(int batch, int r, const float* Sin, int nparts, float* Swork, float* Wbuf, float* W, bf16* Z3,
                     int ldz, int* dead, int* status, cudaStream_t st)
{
    const size_t smem = chol_smem_bytes(r, true);
    if (smem <= 225 * 1024) {
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(chol_inv_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 225 * 1024);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        return launch("chol_inv_smem", chol_inv_kernel<true>, dim3(batch), dim3(512), smem, st, r, Sin, nparts, Swork,
                      Wbuf, W, Z3, ldz, dead, status);
    }
    return launch("chol_inv_global", chol_inv_kernel<false>, dim3(batch), dim3(512), chol_smem_bytes(r, false), st, r,
                  Sin, nparts, Swork, Wbuf, W, Z3, ldz, dead, status);
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
        e = chol_inv(batch, r, S, 1, S, W, W, nullptr, 0, dead, status, st);
        if (e != cudaSuccess) return e;
        // P <- P L^{-T}: B(k, j) = L^{-1}[j][k]
        e = gemm_simt<1>("qr_apply", batch, m, r, r, LdA<float, true>{src, sp, ldp}, LdB<float, false>{W, ss, r},
                         LdB<float, false>{W, ss, r}, EpStore{dst, sp, ldp}, st);
        if (e != cudaSuccess) return e;
        float* t = src; src = dst; dst = t;
    }
    return cudaSuccess;  // two passes: the result is back in P
}

}  // namespace dion
