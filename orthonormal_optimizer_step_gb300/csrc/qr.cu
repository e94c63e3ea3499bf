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
__global__ void __launch_bounds__(512, 1) chol_inv_kernel(int r, const float* Sin, int nparts, float* Swork, float* Wbuf,
                                                       float* W, bf16* Z3, int ldz, int* dead_g, int* status,
                                                       const int* emax_pre)
{
    extern __shared__ float smem[];
    __shared__ int s_bad;
    __shared__ float s_emax;
    __shared__ __align__(16) float colw[64];
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
    float* rinv_all = (float*)(deadsm + r);                // reciprocal pivots 1 / L(j, j) (0 if dependent)
#define Lx0(i) (kSmem ? L[(size_t)(i) * ld + (i)] : Sg[(size_t)(i) * r + (i)])
    float* T = kSmem ? rinv_all + r : Wg;                  // (r - 32) x 32 scratch of the inverse
    // The near-identity inverse was already written by qr_near_identity_kernel
    // (emax_pre = max|S - I| of this matrix): nothing left to do.
    if (emax_pre && __int_as_float(emax_pre[b]) <= 1e-4f) {
        for (int i = tid; i < r; i += nt) dead[i] = 0;
        return;
    }
    for (int i = warp; i < r; i += nwarps) {
        for (int k = lane; k < r; k += 32) {
            const size_t e = (size_t)i * r + k;
            float v = Sb[e];
            for (int q = 1; q < nparts; ++q) v += Sb[(size_t)q * rr + e];
            if (kSmem) L[(size_t)i * ld + k] = v;
            else Sg[e] = v;
        }
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

    // The loops below are kept rolled (modest unrolling only): the factorization
    // is a long chain of short dependent steps, and compact code keeps them in
    // the instruction cache.
    for (int J = 0; J < r; J += 32) {
        const int jb = min(32, r - J);
        if (warp == 0) {
            // Diagonal block, lane = row.  w[j] holds L(J + lane, J + c + j):
            // the current column is always w[0], and the window shifts by one
            // column per step, so every register index is a compile-time
            // constant inside a rolled loop.
            float w[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = (lane < jb && j < jb) ? Lx(J + lane, J + j) : 0.f;
            for (int c = 0; c < jb; ++c) {
                const float d = __shfl_sync(0xffffffffu, w[0], c);
                const bool fin = isfinite(d);
                const bool ok = fin && d > 1e-6f * d0[J + c];
                const float rinv = ok ? rsqrtf(d) : 0.f;
                const float lv = (lane > c) ? w[0] * rinv : (lane == c ? (ok ? d * rinv : 1.f) : 0.f);
                if (lane == 0) {
                    deadsm[J + c] = !ok;
                    rinv_all[J + c] = rinv;
                    if (!ok) s_bad |= fin ? kStatusPivot : kStatusNonFinite;
                }
                if (lane >= c && lane < jb) Lx(J + lane, J + c) = lv;
                // column c relative to the step: colw[32 + j] = L(J + c + j, J + c)
                colw[32 + lane - c] = lv;
                __syncwarp();
                float cb[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 v4 = *reinterpret_cast<const float4*>(&colw[32 + j]);
                    cb[j] = v4.x; cb[j + 1] = v4.y; cb[j + 2] = v4.z; cb[j + 3] = v4.w;
                }
#pragma unroll
                for (int j = 1; j < 32; ++j)
                    if (lane > c && lane >= c + j) w[j] = fmaf(-lv, cb[j], w[j]);
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 31; ++j) w[j] = w[j + 1];
                w[31] = 0.f;
            }
        }
        __syncthreads();
        // panel below the diagonal block: one thread per row, x L_JJ^T = row
        for (int i = J + jb + tid; i < r; i += nt) {
            float a[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) a[c] = (c < jb) ? Lx(i, J + c) : 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if (c < jb) {
                    float lr[32];
#pragma unroll
                    for (int k = 0; k < c; ++k) lr[k] = Lx(J + c, J + k);
                    float s4[4] = {a[c], 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < c; ++k) s4[k & 3] = fmaf(-a[k], lr[k], s4[k & 3]);
                    a[c] = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * rinv_all[J + c];
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
            const float* li = &Lx(i, J);
            for (int k = t0 + lane; k <= i; k += 32) {
                const float* lk = &Lx(k, J);
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
                int c = 0;
                for (; c + 3 < jb; c += 4) {
                    s4[0] = fmaf(li[c], lk[c], s4[0]);
                    s4[1] = fmaf(li[c + 1], lk[c + 1], s4[1]);
                    s4[2] = fmaf(li[c + 2], lk[c + 2], s4[2]);
                    s4[3] = fmaf(li[c + 3], lk[c + 3], s4[3]);
                }
                for (; c < jb; ++c) s4[0] = fmaf(li[c], lk[c], s4[0]);
                Lx(i, k) -= (s4[0] + s4[1]) + (s4[2] + s4[3]);
            }
        }
        __syncthreads();
    }

    // ---- diagonal blocks Z_II = L_II^{-1}, all at once (one warp per block):
    // lane c computes column c right-looking; acc[j] is the partial right-hand
    // side of row i + j.
    for (int I = warp; I * 32 < r; I += nwarps) {
        const int J = I * 32, jb = min(32, r - J), c = lane;
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = (j == c) ? 1.f : 0.f;
        float zc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            zc[i] = 0.f;
            if (i < jb) {
                const float z = (i >= c && c < jb) ? acc[0] * rinv_all[J + i] : 0.f;
                zc[i] = z;
#pragma unroll
                for (int j = 1; j < 32; ++j) {
                    const float l = Lx(J + min(i + j, jb - 1), J + i);
                    acc[j] = (i + j < jb) ? fmaf(-l, z, acc[j]) : acc[j];
                }
            }
#pragma unroll
            for (int j = 0; j < 31; ++j) acc[j] = acc[j + 1];
            acc[31] = 0.f;
        }
        __syncwarp();
        if (c < jb)
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i >= c && i < jb) Lx(J + i, J + c) = zc[i];
    }
    __syncthreads();

    // ---- in-place inverse L <- L^{-1}, block columns from the last one back:
    //   Z_JJ = L_JJ^{-1};  panel <- -(L^{-1} of the trailing part) * panel * Z_JJ
    for (int J = ((r - 1) / 32) * 32; J >= 0; J -= 32) {
        const int jb = min(32, r - J), t0 = J + jb;
        // T = Linv_trail * panel  (rows t0..r-1, 32 columns), one warp per row
        for (int i = t0 + warp; i < r; i += nwarps) {
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
            if (lane < jb) {
                int k = t0;
                for (; k + 3 <= i; k += 4) {
                    s0 = fmaf(Lx(i, k), Lx(k, J + lane), s0);
                    s1 = fmaf(Lx(i, k + 1), Lx(k + 1, J + lane), s1);
                    s2 = fmaf(Lx(i, k + 2), Lx(k + 2, J + lane), s2);
                    s3 = fmaf(Lx(i, k + 3), Lx(k + 3, J + lane), s3);
                }
                for (; k <= i; ++k) s0 = fmaf(Lx(i, k), Lx(k, J + lane), s0);
            }
            T[(size_t)(i - t0) * 32 + lane] = (s0 + s1) + (s2 + s3);
        }
        __syncthreads();
        // panel <- -T * Z_JJ
        for (int i = t0 + warp; i < r; i += nwarps) {
            if (lane < jb) {
                const float* Ti = T + (size_t)(i - t0) * 32;
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
                int k = lane;
                for (; k + 3 < jb; k += 4) {
                    s4[0] = fmaf(Ti[k], Lx(J + k, J + lane), s4[0]);
                    s4[1] = fmaf(Ti[k + 1], Lx(J + k + 1, J + lane), s4[1]);
                    s4[2] = fmaf(Ti[k + 2], Lx(J + k + 2, J + lane), s4[2]);
                    s4[3] = fmaf(Ti[k + 3], Lx(J + k + 3, J + lane), s4[3]);
                }
                for (; k < jb; ++k) s4[0] = fmaf(Ti[k], Lx(J + k, J + lane), s4[0]);
                Lx(i, J + lane) = -((s4[0] + s4[1]) + (s4[2] + s4[3]));
            }
        }
        __syncthreads();
    }
    for (int i = tid; i < r; i += nt) dead[i] = deadsm[i];
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
    return in_smem ? ((size_t)r * (r + 1) + 3 * (size_t)r + scratch) * sizeof(float) : (size_t)3 * r * sizeof(float);
}

cudaError_t chol_inv(const char* name, int batch, int r, const float* Sin, int nparts, float* Swork, float* Wbuf, float* W, bf16* Z3,
                     int ldz, int* dead, int* status, cudaStream_t st, const int* emax_pre)
{
    const size_t smem = chol_smem_bytes(r, true);
    if (smem <= 215 * 1024) {
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(chol_inv_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 215 * 1024);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        return launch(name, chol_inv_kernel<true>, dim3(batch), dim3(512), smem, st, r, Sin, nparts, Swork,
                      Wbuf, W, Z3, ldz, dead, status, emax_pre);
    }
    static bool gattr = false;
    if (!gattr) {   // 3 r floats of dynamic shared memory: up to 48 KB at r = 4096, plus the static part
        cudaError_t e = cudaFuncSetAttribute(chol_inv_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             96 * 1024);
        if (e != cudaSuccess) return e;
        gattr = true;
    }
    if (chol_smem_bytes(r, false) > 96 * 1024) return cudaErrorInvalidValue;
    return launch(name, chol_inv_kernel<false>, dim3(batch), dim3(512), chol_smem_bytes(r, false), st, r,
                  Sin, nparts, Swork, Wbuf, W, Z3, ldz, dead, status, emax_pre);
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
        e = chol_inv(pass == 0 ? "chol_inv_pass1" : "chol_inv_pass2", batch, r, S, 1, S, W, W, nullptr, 0, dead,
                     status, st);
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
