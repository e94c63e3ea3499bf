// simt.cu -- the float32 CUDA-core path of the Dion step and of Newton-Schulz.
//
// Used for float32 storage (DION_F32), where the parity bound of 1e-4 relative
// error rules out bf16 or tf32 tensor-core operands.  Every product is the
// batched SIMT GEMM of simt_gemm.cuh; B = M + G is formed inside the operand
// loader and never stored.
#include "internal.h"
#include "simt_gemm.cuh"
#include "ns_common.cuh"

namespace dion {

// ------------------------------------------------------------------ Dion ----

// Q_j <- R_j / max(||R_j||, floor), column norms over the n rows of R (n x r).
__global__ void __launch_bounds__(256) colnorm_kernel(int n, int r, long long ldr, const float* R, float* Q,
                                                     float* inv_out, float floor_nrm, int* status)
{
    __shared__ float red[8][33];
    __shared__ float s_inv[32];
    const int b = blockIdx.y, tx = threadIdx.x, ty = threadIdx.y;
    const int j = blockIdx.x * 32 + tx;
    const float* Rb = R + (size_t)b * n * ldr;
    float s = 0.f;
    if (j < r)
        for (int i = ty; i < n; i += 8) {
            const float v = Rb[(size_t)i * ldr + j];
            s = fmaf(v, v, s);
        }
    red[ty][tx] = s;
    __syncthreads();
    if (ty == 0) {
        float t = 0.f;
        for (int k = 0; k < 8; ++k) t += red[k][tx];
        const float nrm = fmaxf(sqrtf(t), floor_nrm);
        const float inv = 1.f / nrm;
        s_inv[tx] = inv;
        if (j < r) {
            if (inv_out) inv_out[(size_t)b * r + j] = inv;
            if (!isfinite(t)) atomicOr(status, kStatusNonFinite);
        }
    }
    __syncthreads();
    if (j < r && Q) {
        float* Qb = Q + (size_t)b * n * r;
        for (int i = ty; i < n; i += 8) Qb[(size_t)i * r + j] = Rb[(size_t)i * ldr + j] * s_inv[tx];
    }
}

// Fused error-feedback and weight update over the m x n grid:
//   M <- M + G - (1 - mu) * (P R^T)          (acc0)
//   X <- (1 - lr wd) X - lr sqrt(m/n) * (P Q^T)   (acc1)
template <typename T>
struct EpDionUpdate {
    T* X; const T* G; float* M; long long sb; long long ld;
    StepHyper hp;
    __device__ __forceinline__ void operator()(int b, int i, int j, float prt, float pqt) const {
        float one_minus_mu, decay, scale;
        hp.get(one_minus_mu, decay, scale);
        const long long o = b * sb + i * ld + j;
        M[o] = M[o] + to_f(G[o]) - one_minus_mu * prt;
        X[o] = from_f<T>(decay * to_f(X[o]) - scale * pqt);
    }
};

// Non-finite device-side hyperparameters set the status word.
__global__ void hyper_check_kernel(const float* hyper, int* status)
{
    if (threadIdx.x == 0 && !(isfinite(hyper[0]) && isfinite(hyper[1]) && isfinite(hyper[2])))
        atomicOr(status, kStatusNonFinite);
}

template <typename T>
static dion_status dion_simt_t(int batch, int m, int n, int r, T* X, const T* G, float* M, float* Q, float mu,
                               float lr, float wd, const float* hyper, char* ws, const DionLayout& L, cudaStream_t st)
{
    int* status = (int*)(ws + L.status);
    float* P0 = (float*)(ws + L.P0);
    float* P1 = (float*)(ws + L.P1);
    float* R = (float*)(ws + L.R);
    float* S = (float*)(ws + L.S);
    float* W = (float*)(ws + L.W);
    int* dead = (int*)(ws + L.dead);
    float* inv = (float*)(ws + L.inv);
    const long long mn = (long long)m * n, mr = (long long)m * r, nr = (long long)n * r;

    DION_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
    // P = (M + G) Q
    DION_TRY((gemm_simt<1>("dion_bq_simt", batch, m, r, n, LdSum<float, T, true>{M, G, mn, n},
                           LdB<float, true>{Q, nr, r}, LdB<float, true>{Q, nr, r}, EpStore{P0, mr, r}, st)));
    // P <- orthonormalize(P)
    DION_TRY(qr_cholesky2(batch, m, r, r, P0, P1, S, W, dead, status, (int*)(ws + L.hard), (double*)(ws + L.S64),
                          st));
    // R = B^T P
    DION_TRY((gemm_simt<1>("dion_btp_simt", batch, n, r, m, LdSum<float, T, false>{M, G, mn, n},
                           LdB<float, true>{P0, mr, r}, LdB<float, true>{P0, mr, r}, EpStore{R, nr, r}, st)));
    // Q <- column-normalized R
    DION_TRY(launch("dion_colnorm", colnorm_kernel, dim3((unsigned)cdiv(r, 32), batch), dim3(32, 8), 0, st, n, r,
                    (long long)r, (const float*)R, Q, inv, 1e-12f * sqrtf((float)n), status));
    // M, X updates
    EpDionUpdate<T> ep{X, G, M, mn, n, StepHyper{mu, lr, wd, sqrtf((float)m / (float)n), hyper}};
    if (hyper) DION_TRY(launch("dion_hyper_check", hyper_check_kernel, dim3(1), dim3(32), 0, st, hyper, status));
    DION_TRY((gemm_simt<2>("dion_update_simt", batch, m, n, r, LdA<float, true>{P0, mr, r},
                           LdB<float, false>{R, nr, r}, LdB<float, false>{Q, nr, r}, ep, st)));
    return DION_OK;
}

dion_status dion_step_simt(int batch, int m, int n, int r, dion_dtype dt, void* X, const void* G, float* M,
                           float* Q, float mu, float lr, float wd, const float* hyper, char* ws, const DionLayout& L,
                           cudaStream_t st)
{
    if (dt == DION_F32)
        return dion_simt_t<float>(batch, m, n, r, (float*)X, (const float*)G, M, Q, mu, lr, wd, hyper, ws, L, st);
    return dion_simt_t<bf16>(batch, m, n, r, (bf16*)X, (const bf16*)G, M, Q, mu, lr, wd, hyper, ws, L, st);
}

// ---------------------------------------------------------- Newton-Schulz ----

// X0[bh] (s x l) = y / (||y||_F + eps), transposed when the block is taller
// than wide (tr): X0[p][q] = y[q][p].
template <typename T>
__global__ void __launch_bounds__(256) ns_load_kernel(int m, int n, int hd, int heads, int s, int l, int tr, const T* G,
                                                      const float* M, const float* nrm, float eps, float* X0)
{
    const int bh = blockIdx.y, b = bh / heads, h = bh % heads;
    const float inv = 1.f / (sqrtf(nrm[bh]) + eps);
    const long long cnt = (long long)s * l;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < cnt; e += (long long)gridDim.x * blockDim.x) {
        const int p = (int)(e / l), q = (int)(e % l);
        const int i = tr ? q : p, c = tr ? p : q;        // row in [0, m), column in the block
        const long long o = (long long)b * m * n + (long long)i * n + (long long)h * hd + c;
        const float y = M ? M[o] : to_f(G[o]);
        X0[(long long)bh * cnt + e] = y * inv;
    }
}

// Scatter the final iterate back: O = Xf (transposed back), optional store of
// O and the weight update X <- decay X - scale O.
template <typename T>
__global__ void __launch_bounds__(256) ns_finish_kernel(int batch, int m, int n, int hd, int heads, int s, int l, int tr,
                                                        const float* Xf, T* O, T* X, float decay, float scale)
{
    const long long total = (long long)batch * m * n;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(e / ((long long)m * n));
        const long long rem = e % ((long long)m * n);
        const int i = (int)(rem / n), col = (int)(rem % n);
        const int h = col / hd, c = col % hd;
        const long long bh = (long long)b * heads + h;
        const float o = tr ? Xf[bh * s * l + (long long)c * l + i] : Xf[bh * s * l + (long long)i * l + c];
        if (O) O[e] = from_f<T>(o);
        if (X) X[e] = from_f<T>(decay * to_f(X[e]) - scale * o);
    }
}

struct EpNsPoly {   // Bm = b*A + c*(A A)
    const float* A; float* Bm; long long sb; long long ld; float bc, cc;
    __device__ __forceinline__ void operator()(int b, int i, int j, float v, float) const {
        const long long o = b * sb + i * ld + j;
        Bm[o] = bc * A[o] + cc * v;
    }
};
struct EpNsAxpy {   // Xn = a*X + Bm X
    const float* X; float* Xn; long long sb; long long ld; float a;
    __device__ __forceinline__ void operator()(int b, int i, int j, float v, float) const {
        const long long o = b * sb + i * ld + j;
        Xn[o] = a * X[o] + v;
    }
};

template <typename T>
static dion_status muon_simt_t(int batch, int m, int n, T* X, const T* G, float* M, T* O, int steps,
                               const float* coeff, float mu, float lr, float wd, char* ws, const MuonLayout& L,
                               cudaStream_t st)
{
    int* status = (int*)(ws + L.status);
    float* nrm = (float*)(ws + L.nrm);
    float* Xa = (float*)(ws + L.Xa);
    float* Xb = (float*)(ws + L.Xb);
    float* A = (float*)(ws + L.A);
    float* Bm = (float*)(ws + L.Bm);
    const int s = L.s, l = L.l, nb = L.nb;
    const long long sl = (long long)s * l, ss = (long long)s * s;

    DION_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
    DION_TRY(cudaMemsetAsync(nrm, 0, sizeof(float) * nb, st));
    const unsigned chunks = (unsigned)std::min<long long>(cdiv((long long)m * L.hd, 256 * 8), 64);
    DION_TRY(launch("ns_prep", ns_prep_kernel<T>, dim3(chunks, nb), dim3(256), 0, st, m, n, L.hd, L.heads, G, M, mu,
                    nrm));
    const unsigned lchunks = (unsigned)std::min<long long>(cdiv(sl, 256 * 4), 1024);
    DION_TRY(launch("ns_load", ns_load_kernel<T>, dim3(lchunks, nb), dim3(256), 0, st, m, n, L.hd, L.heads, s, l,
                    (int)L.tr, G, (const float*)M, (const float*)nrm, 1e-7f, Xa));
    for (int k = 0; k < steps; ++k) {
        // A = X X^T
        DION_TRY((gemm_simt<1>("ns_gram_simt", nb, s, s, l, LdA<float, true>{Xa, sl, l}, LdB<float, false>{Xa, sl, l},
                               LdB<float, false>{Xa, sl, l}, EpStore{A, ss, s}, st)));
        // Bm = b A + c A A
        DION_TRY((gemm_simt<1>("ns_poly_simt", nb, s, s, s, LdA<float, true>{A, ss, s}, LdB<float, true>{A, ss, s},
                               LdB<float, true>{A, ss, s}, EpNsPoly{A, Bm, ss, s, coeff[1], coeff[2]}, st)));
        // Xb = a Xa + Bm Xa
        DION_TRY((gemm_simt<1>("ns_axpy_simt", nb, s, l, s, LdA<float, true>{Bm, ss, s}, LdB<float, true>{Xa, sl, l},
                               LdB<float, true>{Xa, sl, l}, EpNsAxpy{Xa, Xb, sl, l, coeff[0]}, st)));
        float* t = Xa; Xa = Xb; Xb = t;
    }
    const long long total = (long long)batch * m * n;
    const unsigned fchunks = (unsigned)std::min<long long>(cdiv(total, 256 * 4), 65535);
    DION_TRY(launch("ns_finish", ns_finish_kernel<T>, dim3(fchunks), dim3(256), 0, st, batch, m, n, L.hd, L.heads, s,
                    l, (int)L.tr, (const float*)Xa, O, X, 1.f - lr * wd, lr * sqrtf((float)m / (float)n)));
    return DION_OK;
}

dion_status muon_simt(int batch, int m, int n, dion_dtype dt, void* X, const void* G, float* M, void* O, int steps,
                      const float* coeff, float mu, float lr, float wd, char* ws, const MuonLayout& L, cudaStream_t st)
{
    if (dt == DION_F32)
        return muon_simt_t<float>(batch, m, n, (float*)X, (const float*)G, M, (float*)O, steps, coeff, mu, lr, wd,
                                  ws, L, st);
    return muon_simt_t<bf16>(batch, m, n, (bf16*)X, (const bf16*)G, M, (bf16*)O, steps, coeff, mu, lr, wd, ws, L,
                             st);
}

}  // namespace dion
