// qr_tc.cu -- CholeskyQR2 of the m x r panels on the tensor cores.
//
// Each pass is S = P^T P, S = L L^T, P <- P L^{-T} (see qr.cu for the r x r
// factorization).  The two products run on the tcgen05 GEMM with float32
// accuracy from bf16 operands: every operand X is split into three bf16 terms
// X = X1 + X2 + X3 (X1 = bf16(X), X2 = bf16(X - X1), X3 = bf16(X - X1 - X2),
// together 24 significant bits), and the product keeps the six cross terms
// whose weight is at least 2^-16:
//     X Y ~ X1Y1 + X1Y2 + X1Y3 + X2Y1 + X2Y2 + X3Y1
// The GEMM walks these as six K segments that pick the split of each operand.
// The Gram runs the segments as six separate partial products (more CTAs on
// the small r x r output); the factorization kernel sums them on load.
#include "internal.h"
#include "tc_gemm.cuh"
#include "tmap.h"

namespace dion {

namespace {

// Six cross terms (A split, B split): (0,0) (0,1) (0,2) (1,0) (1,1) (2,0)
constexpr uint32_t kSelA = 0u | (0u << 4) | (0u << 8) | (1u << 12) | (1u << 16) | (2u << 20);
constexpr uint32_t kSelB = 0u | (1u << 4) | (2u << 8) | (0u << 12) | (1u << 16) | (0u << 20);

__device__ __forceinline__ void split3(float v, bf16& h1, bf16& h2, bf16& h3)
{
    h1 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(h1);
    h2 = __float2bfloat16_rn(r1);
    h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
}

// P (m x rp fp32, pitch rp) -> P3[3b + t] (m x rp, natural) and T3[3b + t]
// (rp x mp, transposed), t = 0, 1, 2 the three bf16 terms.
// P may be given as nparts split partials (summed here, pitch pstride).
__global__ void __launch_bounds__(256) qr_split_kernel(int m, int rp, int mp, const float* P, int nparts,
                                                       long long pstride, bf16* P3, bf16* T3)
{
    __shared__ float tile[32][33];
    const int b = blockIdx.z, c0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    const size_t pn = (size_t)m * rp, tn = (size_t)rp * mp;
    for (int ii = threadIdx.y; ii < 32; ii += 8) {
        const int i = i0 + ii, c = c0 + threadIdx.x;
        float v = 0.f;
        if (i < m && c < rp) {
            const size_t o = (size_t)b * pn + (size_t)i * rp + c;
            v = P[o];
            for (int q = 1; q < nparts; ++q) v += P[o + q * pstride];
            bf16 h1, h2, h3;
            split3(v, h1, h2, h3);
            bf16* po = P3 + (size_t)3 * b * pn + (size_t)i * rp + c;
            po[0] = h1;
            po[pn] = h2;
            po[2 * pn] = h3;
        }
        tile[ii][threadIdx.x] = v;
    }
    __syncthreads();
    for (int cc = threadIdx.y; cc < 32; cc += 8) {
        const int c = c0 + cc, i = i0 + threadIdx.x;
        if (i < m && c < rp) {
            bf16 h1, h2, h3;
            split3(tile[threadIdx.x][cc], h1, h2, h3);
            bf16* o = T3 + (size_t)3 * b * tn + (size_t)c * mp + i;
            o[0] = h1;
            o[tn] = h2;
            o[2 * tn] = h3;
        }
    }
}

// Second CholeskyQR pass of a well-conditioned panel: the summed Gram is
// S = I + E.  Writes the first-order inverse L^{-1} = I - F, F = strictly
// lower(E) + diag(E)/2 (error O(E^2)), as three bf16 terms, and max|E| per
// matrix; the factorization kernel then skips matrices with max|E| <= 1e-4 and
// factors the others in full (overwriting these terms).
__global__ void __launch_bounds__(256) qr_near_identity_kernel(int r, int ldz, const float* __restrict__ S6,
                                                               bf16* __restrict__ Z3, int* emax)
{
    const int b = blockIdx.y;
    const size_t rr = (size_t)r * r, zs = (size_t)r * ldz;
    const float* Sb = S6 + (size_t)b * 6 * rr;
    bf16* z0 = Z3 + (size_t)3 * b * zs;
    float em = 0.f;
    const long long total = (long long)r * ldz;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(e / ldz), k = (int)(e % ldz);
        float v = 0.f;
        if (k < r) {
            const size_t o = (size_t)i * r + k;
            float sv = Sb[o];
#pragma unroll
            for (int q = 1; q < 6; ++q) sv += Sb[q * rr + o];
            const float ev = sv - (i == k ? 1.f : 0.f);
            em = fmaxf(em, isfinite(ev) ? fabsf(ev) : 1e30f);
            v = (k < i) ? -sv : (k == i ? 1.f - 0.5f * ev : 0.f);
        }
        bf16 h1, h2, h3;
        split3(v, h1, h2, h3);
        z0[e] = h1;
        z0[zs + e] = h2;
        z0[2 * zs + e] = h3;
    }
    for (int o = 16; o > 0; o >>= 1) em = fmaxf(em, __shfl_xor_sync(0xffffffffu, em, o));
    if ((threadIdx.x & 31) == 0) atomicMax(&emax[b], __float_as_int(em));   // em >= 0: int order = float order
}

int pick_bn_qr(int n) { return n <= 64 ? 64 : (n <= 128 ? 128 : 256); }

cudaError_t gemm_any(int bn, const char* name, const CUtensorMap& ta, const CUtensorMap& tb, int K, const TcGemmEpi& ep,
                     cudaStream_t st)
{
    if (bn == 64) return tc_gemm<64>(name, ta, tb, K, ep, st);
    if (bn == 128) return tc_gemm<128>(name, ta, tb, K, ep, st);
    return tc_gemm<256>(name, ta, tb, K, ep, st);
}

}  // namespace

cudaError_t qr_cholesky2_tc(int batch, int m, int r, int rp, const float* Pin, int nparts, float* P, float* Ptmp,
                            bf16* P16, char* ws, const DionLayout& L, int* status, cudaStream_t st)
{
    bf16* T3 = (bf16*)(ws + L.T3);
    bf16* P3 = (bf16*)(ws + L.P3);
    bf16* Z3 = (bf16*)(ws + L.Z3);
    float* S6 = (float*)(ws + L.S6);
    float* S = (float*)(ws + L.S);
    float* W = (float*)(ws + L.W);
    int* dead = (int*)(ws + L.dead);
    int* emax = (int*)(ws + L.emax);
    const long long mp = (long long)align_up((size_t)m, 8);
    const int bn = pick_bn_qr(r), bna = pick_bn_qr(rp);

    CUtensorMap tTa, tTb, tPa, tZb;
    if (!make_tmap_3d(&tTa, T3, TmapType::BF16, m, rp, 3ll * batch, mp * 2, (long long)rp * mp * 2, 64, 128) ||
        !make_tmap_3d(&tTb, T3, TmapType::BF16, m, rp, 3ll * batch, mp * 2, (long long)rp * mp * 2, 64, bn) ||
        !make_tmap_3d(&tPa, P3, TmapType::BF16, rp, m, 3ll * batch, (long long)rp * 2, (long long)m * rp * 2, 64, 128) ||
        !make_tmap_3d(&tZb, Z3, TmapType::BF16, rp, r, 3ll * batch, (long long)rp * 2, (long long)r * rp * 2, 64, bna))
        return cudaErrorInvalidValue;

    // pass 1: split partials of P -> Ptmp;  pass 2: Ptmp -> P (and P16)
    for (int pass = 0; pass < 2; ++pass) {
        const float* src = pass == 0 ? Pin : Ptmp;
        float* dst = pass == 0 ? Ptmp : P;
        const int np_ = pass == 0 ? nparts : 1;
        cudaError_t e = launch("qr_split", qr_split_kernel, dim3((unsigned)cdiv(rp, 32), (unsigned)cdiv(m, 32), batch),
                               dim3(32, 8), 0, st, m, rp, (int)mp, src, np_, (long long)batch * m * rp, P3, T3);
        if (e != cudaSuccess) return e;
        // six partial Grams S6[6b + q] = T_a(q) T_b(q)^T  (r x r)
        TcGemmEpi eg{r, r, (int)cdiv(r, 128), (int)cdiv(r, bn), 6 * batch, nullptr, r, (long long)r * r,
                     nullptr, 0, 0, nullptr, 0, 0, 0.f, 1.f, status, S6, 6, 3, 1, kSelA, kSelB};
        e = gemm_any(bn, "qr_gram_tc", tTa, tTb, m, eg, st);
        if (e != cudaSuccess) return e;
        if (pass == 1) {
            // near-identity inverse on all SMs; the factorization runs only where it does not apply
            e = cudaMemsetAsync(emax, 0, sizeof(int) * batch, st);
            if (e != cudaSuccess) return e;
            const long long tot = (long long)r * rp;
            e = launch("qr_near_identity", qr_near_identity_kernel,
                       dim3((unsigned)std::min<long long>(cdiv(tot, 1024), 1024), batch), dim3(256), 0, st, r, rp,
                       (const float*)S6, Z3, emax);
            if (e != cudaSuccess) return e;
        }
        e = chol_inv(pass == 0 ? "chol_inv_pass1" : "chol_inv_pass2", batch, r, S6, 6, S, W, nullptr, Z3, rp, dead,
                     status, st, pass == 1 ? emax : nullptr);
        if (e != cudaSuccess) return e;
        // dst = P L^{-T}: all six cross terms accumulated; columns r..rp-1 come out zero
        TcGemmEpi ea{m, rp, (int)cdiv(m, 128), (int)cdiv(rp, bna), batch, pass == 1 ? P16 : nullptr, rp,
                     (long long)m * rp, nullptr, 0, 0, nullptr, 0, 0, 0.f, 1.f, status, dst, 6, 3, 0, kSelA, kSelB};
        e = gemm_any(bna, "qr_apply_tc", tPa, tZb, rp, ea, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dion
