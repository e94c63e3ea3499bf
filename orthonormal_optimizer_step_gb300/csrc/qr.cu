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
// This kernel serves ranks above kGjMaxR on the float32 path, with kSmem =
// false: L is factored in place in global memory (pitch r).  (kSmem = true
// keeps L in shared memory with row pitch r + 1; that only fits ranks that
// chol_gj_kernel handles faster.)
// Sin holds nparts partial Gram matrices per matrix (summed on load); Swork is
// the in-place factor of the global variant.  Output: W = L^{-1} as float32
// (W != NULL), or as three bf16 terms Z3[3b + t] (pitch ldz, columns up to ldz,
// Z = Z3[0] + Z3[1] + Z3[2] to float32 accuracy) for the tensor-core apply.
template <bool kSmem>
__global__ void __launch_bounds__(512, 1) chol_inv_kernel(int r, const float* Sin, int nparts, float* Swork, float* Wbuf,
                                                       float* W, bf16* Z3, int ldz, int* dead_g, int* status,
                                                       const int* emax_pre, CholIn in)
{
    extern __shared__ float smem[];
    __shared__ int s_bad;
    __shared__ float s_emax;
    __shared__ __align__(16) float colw[64];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
    const int nwarps = nt >> 5;
    const size_t rr = (size_t)r * r;
    const float* Sb = Sin + (size_t)b * in.mstride;
    float* Sg = Swork + (size_t)b * rr;
    float* Wg = Wbuf + (size_t)b * rr;
    int* dead = dead_g + (size_t)b * in.dstride;
    const int ld = kSmem ? r + 1 : r;
    float* L = kSmem ? smem : Sg;
    float* d0 = kSmem ? smem + (size_t)r * ld : smem;     // original diagonal
    int* deadsm = (int*)(d0 + r);                          // dependent-column flags
    float* rinv_all = (float*)(deadsm + r);                // reciprocal pivots 1 / L(j, j) (0 if dependent)
#define Lx0(i) (kSmem ? L[(size_t)(i) * ld + (i)] : Sg[(size_t)(i) * r + (i)])
    float* T = kSmem ? rinv_all + r : Wg;                  // (r - 32) x 32 scratch of the inverse
    // The near-identity inverse was already written by qr_near_identity_kernel
    // (emax_pre = max|S - I| of this matrix): nothing left to do.
    if (emax_pre && __int_as_float(emax_pre[b]) <= kNearIdentityTol) {
        for (int i = tid; i < r; i += nt) dead[i] = 0;
        return;
    }
    for (int i = warp; i < r; i += nwarps) {
        for (int k = lane; k < r; k += 32) {
            const size_t e = (size_t)i * r + k, ei = (size_t)i * in.lds + k;
            float v = Sb[ei];
            for (int q = 1; q < nparts; ++q) v += Sb[(size_t)q * in.pstride + ei];
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
        if (s_emax <= kNearIdentityTol) {
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
    if (tid == 0 && s_bad) {
        atomicOr(status + (size_t)b * in.sstride, s_bad);
        if (in.any) atomicOr(in.any, 1);
    }
}

// ---- Register-resident inverse Cholesky for r <= kGjMaxR, one CTA per matrix.
//
// The lower triangle of S is cut into 8 x 8 blocks, one per thread, held in
// registers (padding rows beyond r are the identity).  Pivot step k
// eliminates column k of S = L1 D L1^T (L1 unit lower, D the pivots): every
// row i > k with multiplier g_i = S(i, k) / d_k takes
//     A(i, j) -= g_i u_j    for every column j of the row,
// where the step's broadcast vector is u = [E(k, 0 .. k-1), d_k + 1,
// S(k+1 .., k)].  Right of column k this forms the Schur complement; left of
// it the same update applies the row operation to E = L1^{-1}, which is kept
// in place (u_k = d_k + 1 turns A(i, k) = S(i, k) into E(i, k) = -g_i).  After
// the last step L^{-1} = D^{-1/2} E.  u is double-buffered, so each step takes
// one barrier.  A dependent column k (pivot test as in chol_inv_kernel) gets
// g = 0: nothing is eliminated with it, its entries of E are set to zero, and
// its row and column of L^{-1} are zero.
constexpr int kGjMaxR = 248;     // 31 block rows: 496 blocks <= 512 threads
constexpr int kGjStageRows = 64; // rows per pass through the shared staging buffer
constexpr int kGjMaxParts = 6;   // partial Gram matrices summed on load

__global__ void __launch_bounds__(512, 1) chol_gj_kernel(int r, const float* Sin, int nparts, float* W, bf16* Z3,
                                                        int ldz, int* dead_g, int* status, const int* emax_pre,
                                                        CholIn in)
{
    constexpr int kV = kGjMaxR + 8;
    extern __shared__ __align__(16) float stage[];   // kGjStageRows x sp staging rows
    __shared__ __align__(16) float ubuf[2][2][kV];
    __shared__ float piv[kV];
    __shared__ float d0[kV];
    __shared__ int deadsm[kV];
    __shared__ int s_bad;
    __shared__ float s_emax;
    const int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
    int* dead = dead_g + (size_t)b * in.dstride;
    // the near-identity inverse was already written (emax_pre = max|S - I| of this matrix)
    if (emax_pre && __int_as_float(emax_pre[b]) <= kNearIdentityTol) {
        for (int i = tid; i < r; i += nt) dead[i] = 0;
        return;
    }
    const float* Sb = Sin + (size_t)b * in.mstride;
    const int nbr = (r + 7) >> 3, nblk = nbr * (nbr + 1) / 2;
    const int cpad = nbr * 8, sp = cpad + 4;   // staging row pitch: float4-aligned, rows shifted by 4 banks
    const bool own = tid < nblk;
    int bi = 0;
    if (own) {   // thread t owns lower block (bi, bj), t = bi (bi + 1) / 2 + bj
        bi = (int)((sqrtf(8.f * (float)tid + 1.f) - 1.f) * 0.5f);
        while ((bi + 1) * (bi + 2) / 2 <= tid) ++bi;
        while (bi * (bi + 1) / 2 > tid) --bi;
    }
    const int bj = own ? tid - bi * (bi + 1) / 2 : 0;
    const int i0 = bi * 8, j0 = bj * 8;
    const bool diag = own && bi == bj;

    for (int e = tid; e < 4 * kV; e += nt) (&ubuf[0][0][0])[e] = 0.f;
    for (int e = tid; e < kV; e += nt) {
        piv[e] = 1.f;
        deadsm[e] = 0;
    }
    if (tid == 0) {
        s_bad = 0;
        s_emax = 0.f;
    }
    // S (lower triangle, partials summed) -> registers, kGjStageRows rows at a
    // time: coalesced float4 loads into shared memory (two units of every
    // partial in flight per thread), then each owner picks up its block.  Padding rows are the identity.
    float a[8][8];
#pragma unroll
    for (int ii = 0; ii < 8; ++ii)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) a[ii][jj] = 0.f;
    if (in.lds == 0) {
        // block-major input: this thread's 8 x 8 block is 64 contiguous floats
        if (own) {
            const float4* src = reinterpret_cast<const float4*>(Sb + (size_t)tid * 64);
            float4 x[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) x[q] = __ldg(src + q);
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                a[ii][0] = x[2 * ii].x; a[ii][1] = x[2 * ii].y; a[ii][2] = x[2 * ii].z; a[ii][3] = x[2 * ii].w;
                a[ii][4] = x[2 * ii + 1].x; a[ii][5] = x[2 * ii + 1].y; a[ii][6] = x[2 * ii + 1].z;
                a[ii][7] = x[2 * ii + 1].w;
            }
        }
    }
    // 4-column units: float4 loads when every row start is 16-byte aligned
    const bool vec = ((in.lds & 3) == 0) && ((in.pstride & 3) == 0) && ((in.mstride & 3) == 0) &&
                     (((uintptr_t)Sin & 15u) == 0);
    const int upr = cpad >> 2;   // units per staging row
    const int upr_round = kGjMaxParts / nparts;   // units loaded per round
    for (int c = 0; c < (in.lds == 0 ? 0 : cpad); c += kGjStageRows) {
        const int rows = min(kGjStageRows, cpad - c), tot = rows * upr;
        // kGjMaxParts float4 loads in flight per thread: upr_round units of
        // nparts partials each (slot s = unit t * nparts + partial q)
        for (int e0 = tid; e0 < tot; e0 += upr_round * nt) {
            float4 pv[kGjMaxParts];
#pragma unroll
            for (int sl = 0; sl < kGjMaxParts; ++sl) {
                const int t = sl / nparts, q = sl - t * nparts;
                const int e = e0 + t * nt, ri = e / upr, j = (e - ri * upr) * 4, i = c + ri;
                const bool ld = t < upr_round && e < tot && i < r && j <= i;   // a lower-triangle unit
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ld) {
                    const float* src = Sb + (size_t)q * in.pstride + (size_t)i * in.lds + j;
                    if (vec && j + 4 <= r) {
                        x = __ldg(reinterpret_cast<const float4*>(src));
                    } else {
                        x.x = src[0];
                        if (j + 1 < r) x.y = src[1];
                        if (j + 2 < r) x.z = src[2];
                        if (j + 3 < r) x.w = src[3];
                    }
                }
                pv[sl] = x;
            }
            for (int t = 0; t < upr_round; ++t) {
                const int e = e0 + t * nt, ri = e / upr, j = (e - ri * upr) * 4, i = c + ri;
                if (e < tot) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int sl = 0; sl < kGjMaxParts; ++sl)
                        if (sl / nparts == t) {
                            v.x += pv[sl].x; v.y += pv[sl].y; v.z += pv[sl].z; v.w += pv[sl].w;
                        }
                    if (i >= r) {   // padding rows: identity
                        v.x = (i == j) ? 1.f : 0.f;
                        v.y = (i == j + 1) ? 1.f : 0.f;
                        v.z = (i == j + 2) ? 1.f : 0.f;
                        v.w = (i == j + 3) ? 1.f : 0.f;
                    }
                    *reinterpret_cast<float4*>(stage + ri * sp + j) = v;
                }
            }
        }
        __syncthreads();
        if (own && i0 >= c && i0 < c + rows) {
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                const float4 x0 = *reinterpret_cast<const float4*>(stage + (i0 - c + ii) * sp + j0);
                const float4 x1 = *reinterpret_cast<const float4*>(stage + (i0 - c + ii) * sp + j0 + 4);
                a[ii][0] = x0.x; a[ii][1] = x0.y; a[ii][2] = x0.z; a[ii][3] = x0.w;
                a[ii][4] = x1.x; a[ii][5] = x1.y; a[ii][6] = x1.z; a[ii][7] = x1.w;
            }
            if (diag) {   // the strict upper part of a diagonal block is unused: keep it zero
#pragma unroll
                for (int ii = 0; ii < 8; ++ii)
#pragma unroll
                    for (int jj = ii + 1; jj < 8; ++jj) a[ii][jj] = 0.f;
            }
        }
        __syncthreads();
    }
    if (diag) {
#pragma unroll
        for (int ii = 0; ii < 8; ++ii)
            if (i0 + ii < r) d0[i0 + ii] = a[ii][ii];
    }
    if (in.d0) {   // reference diagonal given (a Schur complement is factored)
        __syncthreads();
        for (int k = tid; k < r; k += nt) d0[k] = in.d0[(size_t)b * in.d0stride + k];
    }
    // near-identity Gram: L^{-1} = I - strictly_lower(E) - diag(E)/2 (see chol_inv_kernel)
    float em = 0.f;
    if (own) {
#pragma unroll
        for (int ii = 0; ii < 8; ++ii)
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int i = i0 + ii, j = j0 + jj;
                if (i < r && j <= i) {
                    const float ev = a[ii][jj] - (i == j ? 1.f : 0.f);
                    em = fmaxf(em, isfinite(ev) ? fabsf(ev) : 1e30f);
                }
            }
    }
    for (int o = 16; o > 0; o >>= 1) em = fmaxf(em, __shfl_xor_sync(0xffffffffu, em, o));
    __syncthreads();
    if ((tid & 31) == 0) atomicMax((int*)&s_emax, __float_as_int(em));   // em >= 0: int order = float order
    __syncthreads();
    const bool near = s_emax <= kNearIdentityTol;

    if (!near) {
        // Two pivots per barrier.  The writers store the raw column and row of
        // pivots k and k+1 (U0, U1); every thread then forms both pivots and
        // their tests, and the vectors of step k+1 after step k:
        //     g = A(k+1, k) / d_k,  d_{k+1} = A(k+1, k+1) - g A(k+1, k),
        //     u'_j = U1_j - g u_j   (u = U0 with u_k = d_k + 1),  u'_{k+1} += 1,
        //     column k+1 below it: U1_i - g U0_i,
        // and applies both rank-1 updates to its block.  Unrolled by 8 so that
        // every register index is static; the per-row and per-column
        // predicates are fixed per group of 8 pivots.  Threads own blocks in
        // block-row order, so the warps that still hold rows of block row
        // k0/8 - 1 or later are a contiguous range [wfirst, nwo): only they take
        // part in a group, on named barrier 1.  A warp stays one group after
        // its last update, so that no buffer it read is rewritten before it
        // has passed another barrier.
        const int warp = tid >> 5, nwo = (nblk + 31) >> 5;
        const int wlast = __reduce_max_sync(0xffffffffu, own ? i0 + 7 : -1);
        for (int k0 = 0; k0 < r && warp < nwo; k0 += 8) {
            const int br = k0 >> 3, brl = br > 0 ? br - 1 : 0, wfirst = ((brl * (brl + 1)) >> 1) >> 5;
            if (warp < wfirst) break;
            const int nbar = (nwo - wfirst) * 32;
            const bool cw = own && j0 == k0, rw = own && i0 == k0;
            const bool cwb = cw && !diag;          // columns k, k+1: every row of a block below the diagonal block
            const bool below = own && i0 > k0;     // all rows of the block below this group's pivots
            const bool live = below || (own && i0 == k0);
            const bool dg = diag && j0 == k0;
            const float one_cw = cw ? 1.f : 0.f;
            // A block has at most one writer role in a group: below the
            // diagonal block in column k0/8 (writes its column), left of it in
            // row k0/8 (writes its row), or the diagonal block (column entries
            // from row k on, row entries before it).  Its 8 entries of U0 and
            // U1 are contiguous: two 16-byte stores each.
            const bool wr = cw || rw;
            const int wbase = cwb ? i0 : j0;
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
                const int k = k0 + kk, k1 = k + 1;
                if (k >= r) break;
                float* U0 = ubuf[(kk >> 1) & 1][0];
                float* U1 = ubuf[(kk >> 1) & 1][1];
                if (wr) {
                    float w0[8], w1[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        w0[t] = (t >= kk ? cw : cwb) ? a[t][kk] : a[kk][t];
                        w1[t] = (t >= kk + 1 ? cw : cwb) ? a[t][kk + 1] : a[kk + 1][t];
                    }
                    *reinterpret_cast<float4*>(U0 + wbase) = make_float4(w0[0], w0[1], w0[2], w0[3]);
                    *reinterpret_cast<float4*>(U0 + wbase + 4) = make_float4(w0[4], w0[5], w0[6], w0[7]);
                    *reinterpret_cast<float4*>(U1 + wbase) = make_float4(w1[0], w1[1], w1[2], w1[3]);
                    *reinterpret_cast<float4*>(U1 + wbase + 4) = make_float4(w1[4], w1[5], w1[6], w1[7]);
                    if (dg) piv[k] = a[kk][kk];
                }
                asm volatile("bar.sync 1, %0;" ::"r"(nbar) : "memory");
                if (k < wlast) {
                    const float dk = U0[k];
                    const bool okk = isfinite(dk) && dk > 1e-6f * d0[k];
                    const float invk = okk ? __fdividef(1.f, dk) : 0.f;
                    float g1 = 0.f, inv1 = 0.f;
                    bool ok1 = true;
                    if (k1 < r) {
                        const float ak = U0[k1];
                        g1 = ak * invk;
                        const float d1 = fmaf(-g1, ak, U1[k1]);
                        ok1 = isfinite(d1) && d1 > 1e-6f * d0[k1];
                        inv1 = ok1 ? __fdividef(1.f, d1) : 0.f;
                        if (dg) piv[k1] = d1;
                    }
                    const float s0l = live ? invk : 0.f, s0b = below ? invk : 0.f;
                    const float s1l = live ? inv1 : 0.f, s1b = below ? inv1 : 0.f;
                    float c0[8], c1[8], u0[8], u1[8];
                    {
                        const float4 x0 = *reinterpret_cast<const float4*>(U0 + i0);
                        const float4 x1 = *reinterpret_cast<const float4*>(U0 + i0 + 4);
                        const float4 y0 = *reinterpret_cast<const float4*>(U1 + i0);
                        const float4 y1 = *reinterpret_cast<const float4*>(U1 + i0 + 4);
                        const float4 p0 = *reinterpret_cast<const float4*>(U0 + j0);
                        const float4 p1 = *reinterpret_cast<const float4*>(U0 + j0 + 4);
                        const float4 q0 = *reinterpret_cast<const float4*>(U1 + j0);
                        const float4 q1 = *reinterpret_cast<const float4*>(U1 + j0 + 4);
                        c0[0] = x0.x; c0[1] = x0.y; c0[2] = x0.z; c0[3] = x0.w;
                        c0[4] = x1.x; c0[5] = x1.y; c0[6] = x1.z; c0[7] = x1.w;
                        c1[0] = y0.x; c1[1] = y0.y; c1[2] = y0.z; c1[3] = y0.w;
                        c1[4] = y1.x; c1[5] = y1.y; c1[6] = y1.z; c1[7] = y1.w;
                        u0[0] = p0.x; u0[1] = p0.y; u0[2] = p0.z; u0[3] = p0.w;
                        u0[4] = p1.x; u0[5] = p1.y; u0[6] = p1.z; u0[7] = p1.w;
                        u1[0] = q0.x; u1[1] = q0.y; u1[2] = q0.z; u1[3] = q0.w;
                        u1[4] = q1.x; u1[5] = q1.y; u1[6] = q1.z; u1[7] = q1.w;
                    }
                    u0[kk] += one_cw;   // u_k = d_k + 1
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) u1[jj] = fmaf(-g1, u0[jj], u1[jj]);
                    u1[kk + 1] += one_cw;                      // u'_{k+1} = d_{k+1} + 1
                    if (!okk) u1[kk] = cw ? 0.f : u1[kk];      // E(k+1, k) of a dependent column k is zero
#pragma unroll
                    for (int ii = 0; ii < 8; ++ii) {
                        const float gk = c0[ii] * (ii > kk ? s0l : s0b);                        // rows i > k
                        const float gk1 = fmaf(-g1, c0[ii], c1[ii]) * (ii > kk + 1 ? s1l : s1b); // rows i > k+1
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) a[ii][jj] = fmaf(-gk1, u1[jj], fmaf(-gk, u0[jj], a[ii][jj]));
                    }
                    if (!okk) {   // uniform: dependent column k, its entries of E are zero
#pragma unroll
                        for (int ii = 0; ii < 8; ++ii)
                            if (ii > kk ? cw : cwb) a[ii][kk] = 0.f;
                    }
                    if (!ok1) {   // uniform: dependent column k+1
#pragma unroll
                        for (int ii = 0; ii < 8; ++ii)
                            if (ii > kk + 1 ? cw : cwb) a[ii][kk + 1] = 0.f;
                    }
                }
            }
        }
        __syncthreads();
        for (int k = tid; k < r; k += nt) {
            const float d = piv[k];
            const bool fin = isfinite(d);
            const bool ok = fin && d > 1e-6f * d0[k];
            deadsm[k] = !ok;
            if (!ok) atomicOr(&s_bad, fin ? kStatusPivot : kStatusNonFinite);
        }
        __syncthreads();
    }
    // a <- L^{-1} (own block)
    if (own) {
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
            const int i = i0 + ii;
            const float rs = (i < r && !deadsm[i]) ? rsqrtf(piv[i]) : 0.f;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                float z;
                if (near) z = j < i ? -a[ii][jj] : (j == i ? 1.f - 0.5f * (a[ii][jj] - 1.f) : 0.f);
                else z = j < i ? (deadsm[j] ? 0.f : a[ii][jj] * rs) : (j == i ? rs : 0.f);
                a[ii][jj] = z;
            }
        }
    }
    for (int i = tid; i < r; i += nt) dead[i] = near ? 0 : deadsm[i];
    // registers -> shared staging rows -> coalesced stores of whole rows (zero
    // right of the owned blocks): W (pitch r) or the three bf16 terms (pitch ldz)
    const int ncol = W ? r : ldz;
    const size_t zs = (size_t)r * ldz;
    bf16* z0 = W ? nullptr : Z3 + (size_t)3 * b * zs;
    float* Wo = W ? W + (size_t)b * r * r : nullptr;
    if (!W && (ldz & 7) == 0) {
        // straight from registers: each owner writes its block's three bf16
        // terms (one 16-byte store per row and term); the blocks right of the
        // diagonal blocks and the columns past them are written as zero
        if (own) {
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                if (i0 + ii >= r) break;
                uint32_t w[3][4];
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    uint32_t p1 = 0, p2 = 0, p3 = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float v = a[ii][t + h];
                        const bf16 h1 = __float2bfloat16_rn(v);
                        const float r1 = v - __bfloat162float(h1);
                        const bf16 h2 = __float2bfloat16_rn(r1);
                        const bf16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
                        p1 |= (uint32_t)__bfloat16_as_ushort(h1) << (16 * h);
                        p2 |= (uint32_t)__bfloat16_as_ushort(h2) << (16 * h);
                        p3 |= (uint32_t)__bfloat16_as_ushort(h3) << (16 * h);
                    }
                    w[0][t / 2] = p1;
                    w[1][t / 2] = p2;
                    w[2][t / 2] = p3;
                }
                bf16* o = z0 + (size_t)(i0 + ii) * ldz + j0;
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    *reinterpret_cast<uint4*>(o + q * zs) = make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
            }
        }
        const int upr8 = ldz >> 3, tot = r * upr8;
        for (int e = tid; e < tot; e += nt) {
            const int i = e / upr8, jb = e - i * upr8;
            if (jb > (i >> 3)) {
                bf16* o = z0 + (size_t)i * ldz + jb * 8;
#pragma unroll
                for (int q = 0; q < 3; ++q) *reinterpret_cast<uint4*>(o + q * zs) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    for (int c = 0; c < ((!W && (ldz & 7) == 0) ? 0 : r); c += kGjStageRows) {
        const int rows = min(kGjStageRows, r - c);
        if (own && i0 >= c && i0 < c + rows) {
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                float* o = stage + (i0 - c + ii) * sp + j0;
                *reinterpret_cast<float4*>(o) = make_float4(a[ii][0], a[ii][1], a[ii][2], a[ii][3]);
                *reinterpret_cast<float4*>(o + 4) = make_float4(a[ii][4], a[ii][5], a[ii][6], a[ii][7]);
            }
        }
        __syncthreads();
        if (W ? (r & 3) == 0 : (ldz & 7) == 0) {
            // 8-column units: two float4 stores, or one uint4 store per bf16 term
            const int upr8 = (ncol + 7) >> 3, tot = rows * upr8;
            for (int e = tid; e < tot; e += nt) {
                const int ri = e / upr8, j = (e - ri * upr8) * 8, i = c + ri;
                float v[8];
                const bool inb = (j >> 3) <= (i >> 3);   // owned block (else zero)
#pragma unroll
                for (int t = 0; t < 8; ++t) v[t] = inb ? stage[ri * sp + j + t] : 0.f;
                if (W) {
                    float* o = Wo + (size_t)i * r + j;
                    *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
                    if (j + 4 < r) *reinterpret_cast<float4*>(o + 4) = make_float4(v[4], v[5], v[6], v[7]);
                } else {
                    uint32_t w[3][4];
#pragma unroll
                    for (int t = 0; t < 8; t += 2) {
                        uint32_t p1 = 0, p2 = 0, p3 = 0;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const bf16 h1 = __float2bfloat16_rn(v[t + h]);
                            const float r1 = v[t + h] - __bfloat162float(h1);
                            const bf16 h2 = __float2bfloat16_rn(r1);
                            const bf16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
                            p1 |= (uint32_t)__bfloat16_as_ushort(h1) << (16 * h);
                            p2 |= (uint32_t)__bfloat16_as_ushort(h2) << (16 * h);
                            p3 |= (uint32_t)__bfloat16_as_ushort(h3) << (16 * h);
                        }
                        w[0][t / 2] = p1;
                        w[1][t / 2] = p2;
                        w[2][t / 2] = p3;
                    }
                    bf16* o = z0 + (size_t)i * ldz + j;
#pragma unroll
                    for (int q = 0; q < 3; ++q)
                        *reinterpret_cast<uint4*>(o + q * zs) = make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
                }
            }
        } else {
            const int tot = rows * ncol;
            for (int e = tid; e < tot; e += nt) {
                const int ri = e / ncol, j = e - ri * ncol, i = c + ri;
                const float v = ((j >> 3) <= (i >> 3)) ? stage[ri * sp + j] : 0.f;
                if (W) {
                    Wo[(size_t)i * r + j] = v;
                } else {
                    const bf16 h1 = __float2bfloat16_rn(v);
                    const float r1 = v - __bfloat162float(h1);
                    const bf16 h2 = __float2bfloat16_rn(r1);
                    const size_t o = (size_t)i * ldz + j;
                    z0[o] = h1;
                    z0[zs + o] = h2;
                    z0[2 * zs + o] = __float2bfloat16_rn(r1 - __bfloat162float(h2));
                }
            }
        }
        __syncthreads();
    }
    __syncthreads();
    if (tid == 0 && s_bad) {
        atomicOr(status + (size_t)b * in.sstride, s_bad);
        if (in.any) atomicOr(in.any, 1);
    }
}

static size_t chol_smem_bytes(int r, bool in_smem)
{
    const size_t scratch = (size_t)(r > 32 ? r - 32 : 0) * 32;
    return in_smem ? ((size_t)r * (r + 1) + 3 * (size_t)r + scratch) * sizeof(float) : (size_t)3 * r * sizeof(float);
}

cudaError_t chol_inv(const char* name, int batch, int r, const float* Sin, int nparts, float* Swork, float* Wbuf, float* W, bf16* Z3,
                     int ldz, int* dead, int* status, cudaStream_t st, const int* emax_pre, long long sstride, int* any)
{
    const long long rr = (long long)r * r;
    return chol_inv_io(name, batch, r, Sin, nparts, Swork, Wbuf, W, Z3, ldz, dead, status, st, emax_pre,
                       CholIn{nparts * rr, rr, r, r, nullptr, 0, sstride, any});
}

cudaError_t chol_inv_io(const char* name, int batch, int r, const float* Sin, int nparts, float* Swork, float* Wbuf,
                        float* W, bf16* Z3, int ldz, int* dead, int* status, cudaStream_t st, const int* emax_pre,
                        CholIn in)
{
    if (in.lds == 0 && (r > kGjMaxR || nparts != 1)) return cudaErrorInvalidValue;   // block-major input
    if (r <= kGjMaxR) {
        if (nparts < 1 || nparts > kGjMaxParts) return cudaErrorInvalidValue;
        static std::atomic<unsigned long long> gj_attr{0};
        const size_t smem = (size_t)kGjStageRows * (align_up((size_t)r, 8) + 4) * sizeof(float);
        cudaError_t e = smem_attr_once((const void*)chol_gj_kernel,
                                       (int)((size_t)kGjStageRows * (kGjMaxR + 4) * sizeof(float)), gj_attr);
        if (e != cudaSuccess) return e;
        return launch(name, chol_gj_kernel, dim3(batch), dim3(512), smem, st, r, Sin, nparts, W, Z3, ldz, dead, status,
                      emax_pre, in);
    }
    // 3 r floats of dynamic shared memory: up to 48 KB at r = 4096, plus the static part
    static std::atomic<unsigned long long> gattr{0};
    cudaError_t e = smem_attr_once((const void*)chol_inv_kernel<false>, 96 * 1024, gattr);
    if (e != cudaSuccess) return e;
    if (chol_smem_bytes(r, false) > 96 * 1024) return cudaErrorInvalidValue;
    return launch(name, chol_inv_kernel<false>, dim3(batch), dim3(512), chol_smem_bytes(r, false), st, r,
                  Sin, nparts, Swork, Wbuf, W, Z3, ldz, dead, status, emax_pre, in);
}

cudaError_t qr_cholesky2(int batch, int m, int r, long long ldp, float* P, float* Ptmp, float* S, float* W,
                         int* dead, int* status, int* hard, double* S64, cudaStream_t st)
{
    const long long sp = (long long)m * ldp, ss = (long long)r * r;
    // the first pass reports unresolved pivots per matrix (hard); those
    // matrices redo it in float64 (qr64.cu) before the second pass
    const bool fb = qr64_supported(r) && ldp == r;
    if (fb) {
        cudaError_t e = cudaMemsetAsync(hard, 0, sizeof(int) * (batch + 1), st);
        if (e != cudaSuccess) return e;
    }
    float* src = P;
    float* dst = Ptmp;
    for (int pass = 0; pass < 2; ++pass) {
        cudaError_t e = gemm_simt<1>("qr_gram", batch, r, r, m, LdA<float, false>{src, sp, ldp},
                                     LdB<float, true>{src, sp, ldp}, LdB<float, true>{src, sp, ldp},
                                     EpStore{S, ss, r}, st);
        if (e != cudaSuccess) return e;
        const bool first_fb = fb && pass == 0;
        e = chol_inv(pass == 0 ? "chol_inv_pass1" : "chol_inv_pass2", batch, r, S, 1, S, W, W, nullptr, 0, dead,
                     first_fb ? hard : status, st, nullptr, first_fb ? 1 : 0, first_fb ? hard + batch : nullptr);
        if (e != cudaSuccess) return e;
        // P <- P L^{-T}: B(k, j) = L^{-1}[j][k]
        e = gemm_simt<1>("qr_apply", batch, m, r, r, LdA<float, true>{src, sp, ldp}, LdB<float, false>{W, ss, r},
                         LdB<float, false>{W, ss, r}, EpStore{dst, sp, ldp}, st);
        if (e != cudaSuccess) return e;
        if (first_fb) {
            e = qr64_first_pass(batch, m, r, r, P, 1, 0, S64, dst, nullptr, dead, status, hard, st);
            if (e != cudaSuccess) return e;
        }
        float* t = src; src = dst; dst = t;
    }
    return cudaSuccess;  // two passes: the result is back in P
}

}  // namespace dion
