// qr64.cu -- the first CholeskyQR pass in float64, for panels whose float32
// pass found a pivot it could not resolve.
//
// Dion's power iteration needs an orthonormal basis of P = B Q ("Dion: The
// distributed orthonormal update revolution is here", Dion paragraphs).  The
// float32 Gram S = P^T P only resolves columns whose part outside the span of
// the columns before it is above about 1e-3 of their norm (pivot > 1e-6 S_jj):
// a panel with a dominant direction (condition number beyond about 1e3) trips
// that test although it has full rank.  Such matrices are flagged per matrix
// by the float32 factorization (`hard`), and for them alone the first pass is
// redone here, in float64 from the stored state:
//     P = (M + G) Q  (float64, from float32 M and Q and the stored G: no bf16
//                     rounding of B or Q, whose effect on the basis grows as a
//                     column's component along the dominant direction shrinks)
//     S = P^T P (float64),  S = L L^T (float64),  P1 = P L^{-T}
// P1 is orthonormal to float32 rounding for condition numbers up to about
// 1e7, and the regular second CholeskyQR pass (float32) then finishes.  A
// column is dependent when its float64 pivot is at most kDep64 times its
// squared norm, i.e. its independent part is below 1e-6 of its norm: that is
// an order of magnitude above the rounding noise of the float32 panel itself,
// so only true rank deficiency is flagged.  Its column of P1 is zero and the
// status word records it, as in the float32 factorization.
//
// Every kernel returns at once for matrices that are not flagged (and the
// Gram and the apply at their first instruction when no matrix of the batch
// is), so the step always enqueues the same launches (graph capture sees a
// fixed sequence).
// The factorization runs one CTA per flagged matrix (O(r^3) on one SM: about
// 0.1 s at r = 1024): a fallback for rare panels, not the fast path.
#include <algorithm>

#include "internal.h"

namespace dion {

namespace {

constexpr double kDep64 = 1e-12;
constexpr int kT = 64;    // output tile (rows and columns) of the Gram and the apply
constexpr int kK = 32;    // contraction chunk

// Tiles of S = P^T P on or below the diagonal, matrices b with hard[b] only;
// P = sum of nparts float32 partials (matrix b at part + b m rp, partial q at
// + q pstride, row pitch rp).  S (r x r, pitch r) gets its lower triangle
// (and the full diagonal tiles).
__global__ void __launch_bounds__(256) qr64_gram_kernel(int m, int r, int rp, const float* __restrict__ part,
                                                        int nparts, long long pstride, double* __restrict__ S64,
                                                        const int* __restrict__ hard, int batch)
{
    __shared__ double a[kK][kT + 1], c[kK][kT + 1];
    if (!hard[batch]) return;   // no matrix flagged
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nt = (r + kT - 1) / kT, tiles = nt * (nt + 1) / 2;
    for (long long w = blockIdx.x; w < (long long)tiles * batch; w += gridDim.x) {
        const int b = (int)(w / tiles), t = (int)(w - (long long)b * tiles);
        if (!hard[b]) continue;
        int ti = (int)((sqrtf(8.f * (float)t + 1.f) - 1.f) * 0.5f);
        while ((ti + 1) * (ti + 2) / 2 <= t) ++ti;
        while (ti * (ti + 1) / 2 > t) --ti;
        const int tj = t - ti * (ti + 1) / 2, I = ti * kT, J = tj * kT;
        const float* Pb = part + (size_t)b * m * rp;
        double acc[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = 0.0;
        for (int i0 = 0; i0 < m; i0 += kK) {
            for (int e = tid; e < kK * kT; e += 256) {
                const int ri = e / kT, cc = e - ri * kT, i = i0 + ri;
                double va = 0.0, vc = 0.0;
                if (i < m) {
                    const size_t o = (size_t)i * rp;
                    for (int q = 0; q < nparts; ++q) {
                        if (I + cc < r) va += (double)Pb[q * pstride + o + I + cc];
                        if (J + cc < r) vc += (double)Pb[q * pstride + o + J + cc];
                    }
                }
                a[ri][cc] = va;
                c[ri][cc] = vc;
            }
            __syncthreads();
#pragma unroll 4
            for (int k = 0; k < kK; ++k) {
                double x[4], y[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    x[u] = a[k][ty + 16 * u];
                    y[u] = c[k][tx + 16 * u];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[u][v] = fma(x[u], y[v], acc[u][v]);
            }
            __syncthreads();
        }
        double* Sb = S64 + (size_t)b * r * r;
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int i = I + ty + 16 * u, j = J + tx + 16 * v;
                if (i < r && j < r) Sb[(size_t)i * r + j] = acc[u][v];
            }
    }
}

// One CTA per flagged matrix: right-looking Cholesky of S (the strict lower
// triangle becomes that of L in place; L's diagonal is kept only as the
// reciprocal pivots) with the dependence test, then Z = L^{-1} (lower, by
// forward substitution; rows and columns of dependent columns zero).  Shared
// memory: the original diagonal, the current column (then row) of L, the
// reciprocal pivots (r doubles each) and r flags.
__global__ void __launch_bounds__(512) qr64_chol_kernel(int r, double* __restrict__ S64, double* __restrict__ Z64,
                                                        int* __restrict__ dead_g, int* status, const int* hard)
{
    extern __shared__ double sm64[];
    double* d0 = sm64;
    double* col = d0 + r;
    double* rinv = col + r;
    int* deadsm = (int*)(rinv + r);
    __shared__ int s_bad;
    const int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = nt >> 5;
    if (!hard[gridDim.x] || !hard[b]) return;   // (one CTA per matrix: hard[gridDim.x] is the any-word)
    double* S = S64 + (size_t)b * r * r;
    double* Z = Z64 + (size_t)b * r * r;
    if (tid == 0) s_bad = 0;
    for (int i = tid; i < r; i += nt) d0[i] = S[(size_t)i * r + i];
    __syncthreads();
    for (int k = 0; k < r; ++k) {
        const double d = S[(size_t)k * r + k];
        const bool fin = isfinite(d);
        const bool ok = fin && d > kDep64 * d0[k];
        const double inv = ok ? 1.0 / sqrt(d) : 0.0;
        // column k of L below the diagonal (zero for a dependent column)
        for (int i = k + 1 + tid; i < r; i += nt) {
            const double l = S[(size_t)i * r + k] * inv;
            S[(size_t)i * r + k] = l;
            col[i] = l;
        }
        if (tid == 0) {   // (the diagonal of S is left as is: every thread has read it as the pivot)
            rinv[k] = inv;
            deadsm[k] = !ok;
            if (!ok) s_bad |= fin ? kStatusPivot : kStatusNonFinite;
        }
        __syncthreads();
        if (ok) {   // trailing lower triangle: one warp per row, lanes over columns
            for (int i = k + 1 + warp; i < r; i += nwarps) {
                const double li = col[i];
                double* Si = S + (size_t)i * r;
                for (int j = k + 1 + lane; j <= i; j += 32) Si[j] = fma(-li, col[j], Si[j]);
            }
        }
        __syncthreads();
    }
    // Z = L^{-1}, one row at a time: Z(i, c) = (delta_ic - sum_{c<=k<i} L(i, k) Z(k, c)) / L(i, i)
    for (int i = 0; i < r; ++i) {
        for (int k = tid; k < i; k += nt) col[k] = S[(size_t)i * r + k];   // row i of L
        __syncthreads();
        const double ri = rinv[i];
        for (int c = tid; c <= i; c += nt) {
            double s = (c == i) ? 1.0 : 0.0;
            for (int k = c; k < i; ++k) s = fma(-col[k], Z[(size_t)k * r + c], s);
            Z[(size_t)i * r + c] = (deadsm[i] || deadsm[c]) ? 0.0 : s * ri;
        }
        __syncthreads();
    }
    for (int i = tid; i < r; i += nt) dead_g[(size_t)b * r + i] = deadsm[i];
    if (tid == 0 && s_bad) atomicOr(status, s_bad);
}

__device__ __forceinline__ void split3_64(float v, bf16& h1, bf16& h2, bf16& h3)
{
    h1 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(h1);
    h2 = __float2bfloat16_rn(r1);
    h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
}

// P1 = P Z^T (m x r; Z lower triangular, so only k <= j contributes), flagged
// matrices only, rounded once to float32.  Writes P1 (pitch rp, columns r..rp-1
// zero) to Pf and/or its three bf16 terms to P3 (term t of matrix b at
// P3 + (3 b + t) m rp), each when given.
__global__ void __launch_bounds__(256) qr64_apply_kernel(int m, int r, int rp, const float* __restrict__ part,
                                                         int nparts, long long pstride, const double* __restrict__ Z64,
                                                         float* __restrict__ Pf, bf16* __restrict__ P3,
                                                         const int* __restrict__ hard, int batch)
{
    __shared__ double a[kK][kT + 1], z[kK][kT + 1];
    if (!hard[batch]) return;   // no matrix flagged
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int tmr = (m + kT - 1) / kT, tnr = (rp + kT - 1) / kT, tiles = tmr * tnr;
    const size_t pn = (size_t)m * rp;
    for (long long w = blockIdx.x; w < (long long)tiles * batch; w += gridDim.x) {
        const int b = (int)(w / tiles), t = (int)(w - (long long)b * tiles);
        if (!hard[b]) continue;
        const int I = (t / tnr) * kT, J = (t % tnr) * kT;
        const float* Pb = part + (size_t)b * pn;
        const double* Zb = Z64 + (size_t)b * r * r;
        double acc[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = 0.0;
        const int kend = min(r, J + kT);   // Z(j, k) = 0 for k > j
        for (int k0 = 0; k0 < kend; k0 += kK) {
            for (int e = tid; e < kK * kT; e += 256) {
                const int kk = e / kT, cc = e - kk * kT, k = k0 + kk;
                double va = 0.0, vz = 0.0;
                if (k < r) {
                    const int i = I + cc, j = J + cc;
                    if (i < m)
                        for (int q = 0; q < nparts; ++q) va += (double)Pb[q * pstride + (size_t)i * rp + k];
                    if (j < r && k <= j) vz = Zb[(size_t)j * r + k];
                }
                a[kk][cc] = va;
                z[kk][cc] = vz;
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < kK; ++kk) {
                double x[4], y[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    x[u] = a[kk][ty + 16 * u];
                    y[u] = z[kk][tx + 16 * u];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[u][v] = fma(x[u], y[v], acc[u][v]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int i = I + ty + 16 * u, j = J + tx + 16 * v;
                if (i >= m || j >= rp) continue;
                const float val = j < r ? (float)acc[u][v] : 0.f;
                const size_t o = (size_t)i * rp + j;
                if (Pf) Pf[(size_t)b * pn + o] = val;
                if (P3) {
                    bf16 h1, h2, h3;
                    split3_64(val, h1, h2, h3);
                    bf16* p = P3 + (size_t)3 * b * pn + o;
                    p[0] = h1;
                    p[pn] = h2;
                    p[2 * pn] = h3;
                }
            }
    }
}

// dynamic shared memory of the factorization: three r-double rows and r
// flags, up to 200 KB (the opt-in limit of 227 KB also covers the kernel's
// static shared memory, so the full limit cannot be requested): r <= 7314
constexpr size_t kMaxSmem64 = 200 * 1024;
size_t qr64_chol_smem(int r) { return 3 * (size_t)r * sizeof(double) + (size_t)r * sizeof(int); }

// P = (M + G) Q for the flagged matrices, in float64, rounded once to float32
// into part (matrix b at part + b m rp, pitch rp; columns r..rp-1 zero).
// M (m x n float32), G (m x n bf16), Q (n x r float32), row-major per matrix.
__global__ void __launch_bounds__(256) qr64_bq_kernel(int m, int n, int r, int rp, const float* __restrict__ M,
                                                      const bf16* __restrict__ G, const float* __restrict__ Q,
                                                      float* __restrict__ part, const int* __restrict__ hard, int batch)
{
    __shared__ double a[kK][kT + 1], q[kK][kT + 1];
    if (!hard[batch]) return;   // no matrix flagged
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int tmr = (m + kT - 1) / kT, tnr = (rp + kT - 1) / kT, tiles = tmr * tnr;
    for (long long w = blockIdx.x; w < (long long)tiles * batch; w += gridDim.x) {
        const int b = (int)(w / tiles), t = (int)(w - (long long)b * tiles);
        if (!hard[b]) continue;
        const int I = (t / tnr) * kT, J = (t % tnr) * kT;
        const float* Mb = M + (size_t)b * m * n;
        const bf16* Gb = G + (size_t)b * m * n;
        const float* Qb = Q + (size_t)b * n * r;
        double acc[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = 0.0;
        for (int k0 = 0; k0 < n; k0 += kK) {
            for (int e = tid; e < kK * kT; e += 256) {
                const int rr = e / kK, kk = e - rr * kK, i = I + rr, k = k0 + kk;   // a: row i, column k
                a[kk][rr] = (i < m && k < n)
                                ? (double)Mb[(size_t)i * n + k] + (double)__bfloat162float(Gb[(size_t)i * n + k])
                                : 0.0;
                const int kq = e / kT, c = e - kq * kT, kr = k0 + kq, j = J + c;  // q: row kr, column j
                q[kq][c] = (kr < n && j < r) ? (double)Qb[(size_t)kr * r + j] : 0.0;
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < kK; ++kk) {
                double x[4], y[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    x[u] = a[kk][ty + 16 * u];
                    y[u] = q[kk][tx + 16 * u];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[u][v] = fma(x[u], y[v], acc[u][v]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int i = I + ty + 16 * u, j = J + tx + 16 * v;
                if (i < m && j < rp) part[(size_t)b * m * rp + (size_t)i * rp + j] = j < r ? (float)acc[u][v] : 0.f;
            }
    }
}

}  // namespace

bool qr64_supported(int r) { return qr64_chol_smem(r) <= kMaxSmem64; }

cudaError_t qr64_first_pass(int batch, int m, int r, int rp, float* part, int nparts, long long pstride,
                            double* S64, float* Pf, bf16* P3, int* dead, int* status, const int* hard,
                            cudaStream_t st, int n, const float* M, const bf16* G, const float* Q)
{
    const int grid_cap = 2 * num_sms();
    if (M) {   // P = (M + G) Q again in float64 for the flagged matrices, into the first partial
        const long long btiles = cdiv(m, kT) * cdiv(rp, kT) * batch;
        cudaError_t e = launch("qr64_bq", qr64_bq_kernel, dim3((unsigned)std::min<long long>(btiles, grid_cap)),
                               dim3(256), 0, st, m, n, r, rp, M, G, Q, part, hard, batch);
        if (e != cudaSuccess) return e;
        nparts = 1;
    }
    const int nt = (r + kT - 1) / kT;
    const long long gtiles = (long long)nt * (nt + 1) / 2 * batch;
    cudaError_t e = launch("qr64_gram", qr64_gram_kernel, dim3((unsigned)std::min<long long>(gtiles, grid_cap)),
                           dim3(256), 0, st, m, r, rp, part, nparts, pstride, S64, hard, batch);
    if (e != cudaSuccess) return e;
    double* Z64 = S64 + (size_t)batch * r * r;
    const size_t smem = qr64_chol_smem(r);
    static std::atomic<unsigned long long> attr{0};
    e = smem_attr_once((const void*)qr64_chol_kernel, (int)kMaxSmem64, attr);
    if (e != cudaSuccess) return e;
    if (smem > kMaxSmem64) return cudaErrorInvalidValue;
    e = launch("qr64_chol", qr64_chol_kernel, dim3(batch), dim3(512), smem, st, r, S64, Z64, dead, status, hard);
    if (e != cudaSuccess) return e;
    const long long atiles = cdiv(m, kT) * cdiv(rp, kT) * batch;
    return launch("qr64_apply", qr64_apply_kernel, dim3((unsigned)std::min<long long>(atiles, grid_cap)), dim3(256),
                  0, st, m, r, rp, part, nparts, pstride, (const double*)Z64, Pf, P3, hard, batch);
}

}  // namespace dion
