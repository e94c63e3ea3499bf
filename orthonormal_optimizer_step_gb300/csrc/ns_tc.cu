// ns_tc.cu -- Newton-Schulz on the tensor cores (bf16 operands, fp32
// accumulation), the Muon comparison path for bf16 storage.
//
// Per block (a whole matrix, or one m x head_dim column block in per-head
// mode), with Y of shape s x l (s = the smaller side, Y transposed when the
// block is taller than wide):
//   Y <- Y / (||Y||_F + 1e-7)
//   repeat: A = Y Y^T ; Bm = b A + c A A ; Y <- a Y + Bm Y
// The three products are the persistent tcgen05 GEMM of tc_gemm.cuh.  Y is
// kept in bf16 as s x l only: A = Y Y^T and Bm = b A + c A A read K-major
// operands, and Bm Y reads both operands MN-major (Y row-major with K = s
// rows, and Bm, which is symmetric, as its own transpose), so no transposed
// copy of Y is ever written.
#include "internal.h"
#include "ns_common.cuh"
#include "tc_gemm.cuh"
#include "tmap.h"

namespace dion {

// SM count of the current device, cached per device (thread-safe: a race
// only repeats the query).
int num_sms()
{
    static std::atomic<int> cache[64];
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) cur = 0;
    if (cur >= 0 && cur < 64) {
        const int c = cache[cur].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, cur) != cudaSuccess || n <= 0) n = 1;
    if (cur >= 0 && cur < 64) cache[cur].store(n, std::memory_order_relaxed);
    return n;
}

// Scaled bf16 copy of each block as s x l (pitch ldy).  Source block bh =
// (b, h): y(i, c) = M or G at row i, column h*hd + c.  With tr (m > hd) the
// block is transposed: Y[p][q] = y(q, p), written through the shared tile.
template <typename T>
__global__ void __launch_bounds__(256) ns_load_tc_kernel(int m, int n, int hd, int heads, int tr, const T* G,
                                                         const float* M, const float* nrm, float eps, bf16* Y,
                                                         long long ldy, long long sy)
{
    __shared__ float tile[32][33];
    const int bh = blockIdx.z, b = bh / heads, h = bh % heads;
    const int i0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const float inv = 1.f / (sqrtf(nrm[bh]) + eps);
    const long long base = (long long)b * m * n + (long long)h * hd;
    for (int ii = threadIdx.y; ii < 32; ii += 8) {
        const int i = i0 + ii, c = c0 + threadIdx.x;
        float v = 0.f;
        if (i < m && c < hd) {
            const long long o = base + (long long)i * n + c;
            v = (M ? M[o] : to_f(G[o])) * inv;
        }
        tile[ii][threadIdx.x] = v;
    }
    __syncthreads();
    bf16* Yb = Y + bh * sy;
    if (!tr) {
        for (int ii = threadIdx.y; ii < 32; ii += 8) {
            const int i = i0 + ii, c = c0 + threadIdx.x;
            if (i < m && c < hd) Yb[(long long)i * ldy + c] = __float2bfloat16_rn(tile[ii][threadIdx.x]);
        }
    } else {
        for (int cc = threadIdx.y; cc < 32; cc += 8) {
            const int c = c0 + cc, i = i0 + threadIdx.x;
            if (i < m && c < hd) Yb[(long long)c * ldy + i] = __float2bfloat16_rn(tile[threadIdx.x][cc]);
        }
    }
}

// O = final iterate in the parameter's layout; optional store of O and the
// weight update X <- decay X - scale O.  src is the block in the source
// orientation (rows i < m, columns c < hd), pitch lds, block pitch sbs.
template <typename T>
__global__ void __launch_bounds__(256) ns_finish_tc_kernel(int batch, int m, int n, int hd, int heads,
                                                           const bf16* src, long long lds, long long sbs, T* O, T* X,
                                                           float decay, float scale)
{
    const long long total = (long long)batch * m * n;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long mn = (long long)m * n;
        const int b = (int)(e / mn);
        const long long rem = e % mn;
        const int i = (int)(rem / n), col = (int)(rem % n);
        const int h = col / hd, c = col % hd;
        const float o = __bfloat162float(src[((long long)b * heads + h) * sbs + (long long)i * lds + c]);
        if (O) O[e] = from_f<T>(o);
        if (X) X[e] = from_f<T>(decay * to_f(X[e]) - scale * o);
    }
}

// ns_finish_tc_kernel with eight columns per thread (n % 8 == 0, hd % 8 == 0).
template <typename T>
__global__ void __launch_bounds__(256) ns_finish_vec_kernel(int batch, int m, int n, int hd, int heads,
                                                            const bf16* src, long long lds, long long sbs, T* O, T* X,
                                                            float decay, float scale)
{
    const int upr = n >> 3;
    const long long total = (long long)batch * m * upr;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long row = e / upr;                 // b * m + i
        const int col = (int)(e - row * upr) * 8;
        const int b = (int)(row / m), i = (int)(row - (long long)b * m);
        const int h = col / hd, c = col - h * hd;
        float o[8];
        ld8(src + ((long long)b * heads + h) * sbs + (long long)i * lds + c, o);
        const long long eo = row * n + col;
        if (O) st8(O + eo, o);
        if (X) {
            float x[8];
            ld8(X + eo, x);
#pragma unroll
            for (int t = 0; t < 8; ++t) x[t] = decay * x[t] - scale * o[t];
            st8(X + eo, x);
        }
    }
}

// ns_finish_tc_kernel for transposed blocks (m > hd): Y[bh] is hd x m, so
// O(i, c) = Y[c][i]; 32 x 32 tiles through shared memory keep both sides
// coalesced.
template <typename T>
__global__ void __launch_bounds__(256) ns_finish_tr_kernel(int m, int n, int hd, int heads, const bf16* Y,
                                                           long long ldy, long long sy, T* O, T* X, float decay,
                                                           float scale)
{
    __shared__ float tile[32][33];
    const int bh = blockIdx.z, b = bh / heads, h = bh % heads;
    const int i0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    const bf16* Yb = Y + bh * sy;
    for (int cc = threadIdx.y; cc < 32; cc += 8) {
        const int c = c0 + cc, i = i0 + threadIdx.x;
        tile[cc][threadIdx.x] = (c < hd && i < m) ? __bfloat162float(Yb[(long long)c * ldy + i]) : 0.f;
    }
    __syncthreads();
    for (int ii = threadIdx.y; ii < 32; ii += 8) {
        const int i = i0 + ii, c = c0 + threadIdx.x;
        if (i < m && c < hd) {
            const long long e = ((long long)b * m + i) * n + (long long)h * hd + c;
            const float o = tile[threadIdx.x][ii];
            if (O) O[e] = from_f<T>(o);
            if (X) X[e] = from_f<T>(decay * to_f(X[e]) - scale * o);
        }
    }
}

// Row-tile bands of the Newton-Schulz GEMMs (see TcGemmEpi::band_m): with
// 152 CTAs in flight, 16 row tiles by about 9 column tiles of 256 share their
// operand panels in L2 (about 4.5k panel rows against 17k for a whole row of
// column tiles).
constexpr int kNsBand = 16;

static int pick_bn(int n) { return n <= 64 ? 64 : (n <= 128 ? 128 : 256); }

static cudaError_t gemm_bn_mn(int bn, const char* name, const CUtensorMap& ta, const CUtensorMap& tb, int K,
                              const TcGemmEpi& ep, cudaStream_t st)
{
    if (bn == 64) return tc_gemm<64, true>(name, ta, tb, K, ep, st);
    if (bn == 128) return tc_gemm<128, true>(name, ta, tb, K, ep, st);
    return tc_gemm<256, true>(name, ta, tb, K, ep, st);
}

static cudaError_t gemm_bn(int bn, const char* name, const CUtensorMap& ta, const CUtensorMap& tb, int K,
                           const TcGemmEpi& ep, cudaStream_t st)
{
    if (bn == 64) return tc_gemm<64>(name, ta, tb, K, ep, st);
    if (bn == 128) return tc_gemm<128>(name, ta, tb, K, ep, st);
    return tc_gemm<256>(name, ta, tb, K, ep, st);
}

dion_status muon_tc(int batch, int m, int n, dion_dtype dt, void* X, const void* G, float* M, void* O, int steps,
                    const float* coeff, float mu, float lr, float wd, char* ws, const MuonLayout& L,
                    cudaStream_t st)
{
    int* status = (int*)(ws + L.status);
    float* nrm = (float*)(ws + L.nrm);
    bf16* Ya = (bf16*)(ws + L.Xa);
    bf16* Yb = (bf16*)(ws + L.Xb);
    bf16* A = (bf16*)(ws + L.A);
    bf16* Bm = (bf16*)(ws + L.Bm);
    const int s = L.s, l = L.l, nb = L.nb;
    const long long lp = L.lp, sp = L.sp;
    const long long sy = (long long)s * lp, sa = (long long)s * sp;

    DION_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
    DION_TRY(cudaMemsetAsync(nrm, 0, sizeof(float) * nb, st));
    const unsigned chunks = (unsigned)std::min<long long>(cdiv((long long)m * L.hd, 256 * 8), 64);
    const bool vec8 = (L.hd % 8) == 0 && (n % 8) == 0;
    if (vec8) {
        const unsigned vchunks = (unsigned)std::min<long long>(cdiv((long long)m * (L.hd / 8), 256 * 4), 64);
        if (dt == DION_F32)
            DION_TRY(launch("ns_prep", ns_prep_vec_kernel<float>, dim3(vchunks, nb), dim3(256), 0, st, m, n, L.hd,
                            L.heads, (const float*)G, M, mu, nrm));
        else
            DION_TRY(launch("ns_prep", ns_prep_vec_kernel<bf16>, dim3(vchunks, nb), dim3(256), 0, st, m, n, L.hd,
                            L.heads, (const bf16*)G, M, mu, nrm));
    } else if (dt == DION_F32)
        DION_TRY(launch("ns_prep", ns_prep_kernel<float>, dim3(chunks, nb), dim3(256), 0, st, m, n, L.hd, L.heads,
                        (const float*)G, M, mu, nrm));
    else
        DION_TRY(launch("ns_prep", ns_prep_kernel<bf16>, dim3(chunks, nb), dim3(256), 0, st, m, n, L.hd, L.heads,
                        (const bf16*)G, M, mu, nrm));
    dim3 lgrid((unsigned)cdiv(L.hd, 32), (unsigned)cdiv(m, 32), (unsigned)nb);
    if (dt == DION_F32)
        DION_TRY(launch("ns_load_tc", ns_load_tc_kernel<float>, lgrid, dim3(32, 8), 0, st, m, n, L.hd, L.heads,
                        (int)L.tr, (const float*)G, (const float*)M, (const float*)nrm, 1e-7f, Ya, lp, sy));
    else
        DION_TRY(launch("ns_load_tc", ns_load_tc_kernel<bf16>, lgrid, dim3(32, 8), 0, st, m, n, L.hd, L.heads,
                        (int)L.tr, (const bf16*)G, (const float*)M, (const float*)nrm, 1e-7f, Ya, lp, sy));

    const int bn_s = pick_bn(s), bn_l = pick_bn(l);
    const int tm = (int)cdiv(s, 128);
    for (int k = 0; k < steps; ++k) {
        CUtensorMap tYa_a, tYa_b, tA_a, tA_b, tBm_mn, tYa_mn;
        bool ok = make_tmap_3d(&tYa_a, Ya, TmapType::BF16, l, s, nb, lp * 2, sy * 2, 64, 128) &&
                  make_tmap_3d(&tYa_b, Ya, TmapType::BF16, l, s, nb, lp * 2, sy * 2, 64, bn_s) &&
                  make_tmap_3d(&tA_a, A, TmapType::BF16, s, s, nb, sp * 2, sa * 2, 64, 128) &&
                  make_tmap_3d(&tA_b, A, TmapType::BF16, s, s, nb, sp * 2, sa * 2, 64, bn_s) &&
                  make_tmap_3d(&tBm_mn, Bm, TmapType::BF16, s, s, nb, sp * 2, sa * 2, 64, 64) &&
                  make_tmap_3d(&tYa_mn, Ya, TmapType::BF16, l, s, nb, lp * 2, sy * 2, 64, 64);
        if (!ok) return DION_ERR_CUDA;
        // A = Y Y^T
        TcGemmEpi e1{s, s, tm, (int)cdiv(s, bn_s), nb, A, sp, sa, nullptr, 0, 0, nullptr, 0, 0, 0.f, 1.f, status, nullptr, 1, 1, 0, 0u, 0u};
        e1.band_m = kNsBand;
        DION_TRY(gemm_bn(bn_s, "ns_gram_tc", tYa_a, tYa_b, l, e1, st));
        // Bm = b A + c A A   (A symmetric: A A = A A^T)
        TcGemmEpi e2{s, s, tm, (int)cdiv(s, bn_s), nb, Bm, sp, sa, A, sp, sa, nullptr, 0, 0, coeff[1], coeff[2],
                     status, nullptr, 1, 1, 0, 0u, 0u};
        e2.band_m = kNsBand;
        DION_TRY(gemm_bn(bn_s, "ns_poly_tc", tA_a, tA_b, s, e2, st));
        // Y' = a Y + Bm Y: both operands MN-major (Bm symmetric, Y row-major with K = s rows)
        TcGemmEpi e3{s, l, tm, (int)cdiv(l, bn_l), nb, Yb, lp, sy, Ya, lp, sy, nullptr, 0, 0, coeff[0], 1.f, status,
                     nullptr, 1, 1, 0, 0u, 0u};
        e3.band_m = kNsBand;
        DION_TRY(gemm_bn_mn(bn_l, "ns_axpy_tc", tBm_mn, tYa_mn, s, e3, st));
        std::swap(Ya, Yb);
    }
    const float decay = 1.f - lr * wd, scale = lr * sqrtf((float)m / (float)n);
    if (L.tr) {
        const dim3 fgrid((unsigned)cdiv(m, 32), (unsigned)cdiv(L.hd, 32), (unsigned)nb);
        if (dt == DION_F32)
            DION_TRY(launch("ns_finish_tc", ns_finish_tr_kernel<float>, fgrid, dim3(32, 8), 0, st, m, n, L.hd,
                            L.heads, (const bf16*)Ya, lp, sy, (float*)O, (float*)X, decay, scale));
        else
            DION_TRY(launch("ns_finish_tc", ns_finish_tr_kernel<bf16>, fgrid, dim3(32, 8), 0, st, m, n, L.hd,
                            L.heads, (const bf16*)Ya, lp, sy, (bf16*)O, (bf16*)X, decay, scale));
        return DION_OK;
    }
    const long long total = (long long)batch * m * n;
    if (vec8) {
        const unsigned vchunks = (unsigned)std::min<long long>(cdiv(total / 8, 256 * 2), 65535);
        if (dt == DION_F32)
            DION_TRY(launch("ns_finish_tc", ns_finish_vec_kernel<float>, dim3(vchunks), dim3(256), 0, st, batch, m, n,
                            L.hd, L.heads, (const bf16*)Ya, lp, sy, (float*)O, (float*)X, decay, scale));
        else
            DION_TRY(launch("ns_finish_tc", ns_finish_vec_kernel<bf16>, dim3(vchunks), dim3(256), 0, st, batch, m, n,
                            L.hd, L.heads, (const bf16*)Ya, lp, sy, (bf16*)O, (bf16*)X, decay, scale));
        return DION_OK;
    }
    const unsigned fchunks = (unsigned)std::min<long long>(cdiv(total, 256 * 4), 65535);
    if (dt == DION_F32)
        DION_TRY(launch("ns_finish_tc", ns_finish_tc_kernel<float>, dim3(fchunks), dim3(256), 0, st, batch, m, n, L.hd,
                        L.heads, (const bf16*)Ya, lp, sy, (float*)O, (float*)X, decay, scale));
    else
        DION_TRY(launch("ns_finish_tc", ns_finish_tc_kernel<bf16>, dim3(fchunks), dim3(256), 0, st, batch, m, n,
                        L.hd, L.heads, (const bf16*)Ya, lp, sy, (bf16*)O, (bf16*)X, decay, scale));
    return DION_OK;
}

}  // namespace dion
