// ns_tc.cu -- Newton-Schulz on the tensor cores (bf16 operands, fp32
// accumulation), the Muon comparison path for bf16 storage.
//
// Per block (a whole matrix, or one m x head_dim column block in per-head
// mode), with Y of shape s x l (s = the smaller side, Y transposed when the
// block is taller than wide):
//   Y <- Y / (||Y||_F + 1e-7)
//   repeat: A = Y Y^T ; Bm = b A + c A A ; Y <- a Y + Bm Y
// The three products are the persistent tcgen05 GEMM of tc_gemm.cuh.  Y is
// kept in bf16 in both layouts (Y: s x l and Y^T: l x s) so that every product
// reads K-major operands: A = Y Y^T contracts over l (rows of Y), and
// Bm Y = Bm (Y^T)^T contracts over s (rows of Y^T).  The last product writes
// both layouts from its epilogue.
#include "internal.h"
#include "ns_common.cuh"
#include "tc_gemm.cuh"
#include "tmap.h"

namespace dion {

int num_sms()
{
    static int dev = -1, n = 0;
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != dev || n == 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, cur);
        dev = cur;
        if (n <= 0) n = 1;
    }
    return n;
}

// Scaled bf16 copies of each block in both layouts.  Source block bh = (b, h):
// y(i, c) = M or G at row i, column h*hd + c.  With tr (m > hd) the block is
// transposed: Y[p][q] = y(q, p).  Writes Y (s x lp pitch) and YT (l x sp).
template <typename T>
__global__ void __launch_bounds__(256) ns_load_tc_kernel(int m, int n, int hd, int heads, int tr, const T* G,
                                                         const float* M, const float* nrm, float eps, bf16* Y,
                                                         long long ldy, long long sy, bf16* YT, long long ldyt,
                                                         long long syt)
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
    // same orientation as the source: row i, column c
    bf16* same = tr ? YT + bh * syt : Y + bh * sy;
    const long long lds = tr ? ldyt : ldy;
    bf16* other = tr ? Y + bh * sy : YT + bh * syt;
    const long long ldo = tr ? ldy : ldyt;
    for (int ii = threadIdx.y; ii < 32; ii += 8) {
        const int i = i0 + ii, c = c0 + threadIdx.x;
        if (i < m && c < hd) same[(long long)i * lds + c] = __float2bfloat16_rn(tile[ii][threadIdx.x]);
    }
    for (int cc = threadIdx.y; cc < 32; cc += 8) {
        const int c = c0 + cc, i = i0 + threadIdx.x;
        if (i < m && c < hd) other[(long long)c * ldo + i] = __float2bfloat16_rn(tile[threadIdx.x][cc]);
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

static int pick_bn(int n) { return n <= 64 ? 64 : (n <= 128 ? 128 : 256); }

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
    bf16* YTa = (bf16*)(ws + L.XTa);
    bf16* YTb = (bf16*)(ws + L.XTb);
    bf16* A = (bf16*)(ws + L.A);
    bf16* Bm = (bf16*)(ws + L.Bm);
    const int s = L.s, l = L.l, nb = L.nb;
    const long long lp = L.lp, sp = L.sp;
    const long long sy = (long long)s * lp, syt = (long long)l * sp, sa = (long long)s * sp;

    DION_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
    DION_TRY(cudaMemsetAsync(nrm, 0, sizeof(float) * nb, st));
    const unsigned chunks = (unsigned)std::min<long long>(cdiv((long long)m * L.hd, 256 * 8), 64);
    if (dt == DION_F32)
        DION_TRY(launch("ns_prep", ns_prep_kernel<float>, dim3(chunks, nb), dim3(256), 0, st, m, n, L.hd, L.heads,
                        (const float*)G, M, mu, nrm));
    else
        DION_TRY(launch("ns_prep", ns_prep_kernel<bf16>, dim3(chunks, nb), dim3(256), 0, st, m, n, L.hd, L.heads,
                        (const bf16*)G, M, mu, nrm));
    dim3 lgrid((unsigned)cdiv(L.hd, 32), (unsigned)cdiv(m, 32), (unsigned)nb);
    if (dt == DION_F32)
        DION_TRY(launch("ns_load_tc", ns_load_tc_kernel<float>, lgrid, dim3(32, 8), 0, st, m, n, L.hd, L.heads,
                        (int)L.tr, (const float*)G, (const float*)M, (const float*)nrm, 1e-7f, Ya, lp, sy, YTa, sp,
                        syt));
    else
        DION_TRY(launch("ns_load_tc", ns_load_tc_kernel<bf16>, lgrid, dim3(32, 8), 0, st, m, n, L.hd, L.heads,
                        (int)L.tr, (const bf16*)G, (const float*)M, (const float*)nrm, 1e-7f, Ya, lp, sy, YTa, sp,
                        syt));

    const int bn_s = pick_bn(s), bn_l = pick_bn(l);
    const int tm = (int)cdiv(s, 128);
    for (int k = 0; k < steps; ++k) {
        CUtensorMap tYa_a, tYa_b, tA_a, tA_b, tBm_a, tYTa_b;
        bool ok = make_tmap_3d(&tYa_a, Ya, TmapType::BF16, l, s, nb, lp * 2, sy * 2, 64, 128) &&
                  make_tmap_3d(&tYa_b, Ya, TmapType::BF16, l, s, nb, lp * 2, sy * 2, 64, bn_s) &&
                  make_tmap_3d(&tA_a, A, TmapType::BF16, s, s, nb, sp * 2, sa * 2, 64, 128) &&
                  make_tmap_3d(&tA_b, A, TmapType::BF16, s, s, nb, sp * 2, sa * 2, 64, bn_s) &&
                  make_tmap_3d(&tBm_a, Bm, TmapType::BF16, s, s, nb, sp * 2, sa * 2, 64, 128) &&
                  make_tmap_3d(&tYTa_b, YTa, TmapType::BF16, s, l, nb, sp * 2, syt * 2, 64, bn_l);
        if (!ok) return DION_ERR_CUDA;
        // A = Y Y^T
        TcGemmEpi e1{s, s, tm, (int)cdiv(s, bn_s), nb, A, sp, sa, nullptr, 0, 0, nullptr, 0, 0, 0.f, 1.f, status, nullptr, 1, 1, 0, 0u, 0u};
        DION_TRY(gemm_bn(bn_s, "ns_gram_tc", tYa_a, tYa_b, l, e1, st));
        // Bm = b A + c A A   (A symmetric: A A = A A^T)
        TcGemmEpi e2{s, s, tm, (int)cdiv(s, bn_s), nb, Bm, sp, sa, A, sp, sa, nullptr, 0, 0, coeff[1], coeff[2],
                     status, nullptr, 1, 1, 0, 0u, 0u};
        DION_TRY(gemm_bn(bn_s, "ns_poly_tc", tA_a, tA_b, s, e2, st));
        // Y' = a Y + Bm Y, written as Y' and Y'^T
        TcGemmEpi e3{s, l, tm, (int)cdiv(l, bn_l), nb, Yb, lp, sy, Ya, lp, sy, YTb, sp, syt, coeff[0], 1.f, status, nullptr, 1, 1, 0, 0u, 0u};
        DION_TRY(gemm_bn(bn_l, "ns_axpy_tc", tBm_a, tYTa_b, s, e3, st));
        std::swap(Ya, Yb);
        std::swap(YTa, YTb);
    }
    const bf16* src = L.tr ? YTa : Ya;
    const long long lds = L.tr ? sp : lp, sbs = L.tr ? syt : sy;
    const long long total = (long long)batch * m * n;
    const unsigned fchunks = (unsigned)std::min<long long>(cdiv(total, 256 * 4), 65535);
    const float decay = 1.f - lr * wd, scale = lr * sqrtf((float)m / (float)n);
    if (dt == DION_F32)
        DION_TRY(launch("ns_finish_tc", ns_finish_tc_kernel<float>, dim3(fchunks), dim3(256), 0, st, batch, m, n, L.hd,
                        L.heads, src, lds, sbs, (float*)O, (float*)X, decay, scale));
    else
        DION_TRY(launch("ns_finish_tc", ns_finish_tc_kernel<bf16>, dim3(fchunks), dim3(256), 0, st, batch, m, n,
                        L.hd, L.heads, src, lds, sbs, (bf16*)O, (bf16*)X, decay, scale));
    return DION_OK;
}

}  // namespace dion
