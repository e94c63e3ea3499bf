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
// The Gram reads the terms of the row-major m x r panel MN-major (no
// transposed copy) and runs the segments as six separate partial products
// (more CTAs on the small r x r output), summed afterwards.  Only the first
// pass splits a float32 panel: its apply writes the terms of its result
// directly for the second pass.
#include <algorithm>

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

// P (m x rp fp32, pitch rp) -> P3[3b + t] (m x rp), t = 0, 1, 2 the three
// bf16 terms; columns r..rp-1 are written as zero.  P may be given as nparts
// split partials (summed here, pitch pstride); Pf, if set, receives the
// float32 sum (pitch rp).  One thread per 4 columns.
__global__ void __launch_bounds__(256) qr_split_kernel(int m, int r, int rp, const float* P, int nparts,
                                                       long long pstride, bf16* P3, float* Pf, long long total4)
{
    const int b = blockIdx.y;
    const size_t pn = (size_t)m * rp;
    const int upr = rp >> 2;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < (int)total4; e += gridDim.x * blockDim.x) {
        const int i = e / upr, c = (e - i * upr) * 4;
        const size_t o = (size_t)b * pn + (size_t)i * rp + c;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < r) {
            v = *reinterpret_cast<const float4*>(P + o);
            for (int q = 1; q < nparts; ++q) {
                const float4 u = *reinterpret_cast<const float4*>(P + o + q * pstride);
                v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
            }
            if (c + 1 >= r) v.y = 0.f;
            if (c + 2 >= r) v.z = 0.f;
            if (c + 3 >= r) v.w = 0.f;
        }
        if (Pf) *reinterpret_cast<float4*>(Pf + o) = v;
        const float x[4] = {v.x, v.y, v.z, v.w};
        uint32_t w[3][2];
#pragma unroll
        for (int t = 0; t < 4; t += 2) {
            uint32_t p1 = 0, p2 = 0, p3 = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                bf16 h1, h2, h3;
                split3(x[t + h], h1, h2, h3);
                p1 |= (uint32_t)__bfloat16_as_ushort(h1) << (16 * h);
                p2 |= (uint32_t)__bfloat16_as_ushort(h2) << (16 * h);
                p3 |= (uint32_t)__bfloat16_as_ushort(h3) << (16 * h);
            }
            w[0][t / 2] = p1;
            w[1][t / 2] = p2;
            w[2][t / 2] = p3;
        }
        bf16* po = P3 + (size_t)3 * b * pn + (size_t)i * rp + c;
#pragma unroll
        for (int t = 0; t < 3; ++t) *reinterpret_cast<uint2*>(po + t * pn) = make_uint2(w[t][0], w[t][1]);
    }
}

// Second CholeskyQR pass of a well-conditioned panel: the summed Gram is
// S = I + E.  Writes the first-order inverse L^{-1} = I - F, F = strictly
// lower(E) + diag(E)/2 (error O(E^2)), as three bf16 terms, and max|E| per
// matrix; the factorization then runs only for matrices with max|E| above
// kNearIdentityTol (overwriting these terms).  Only the lower triangle of S is
// read (S is symmetric; the blocked path computes only that half).
template <bool V4>
__global__ void __launch_bounds__(256) qr_near_identity_kernel(int r, int ldz, const float* __restrict__ S6,
                                                               int nparts, bf16* __restrict__ Z3, int* emax)
{
    // V4: four consecutive columns per thread (r and ldz multiples of 4): one
    // 16-byte load per partial and one 8-byte store per term
    constexpr int kW = V4 ? 4 : 1;
    const int b = blockIdx.y;
    const size_t rr = (size_t)r * r, zs = (size_t)r * ldz;
    const float* Sb = S6 + (size_t)b * nparts * rr;
    bf16* z0 = Z3 + (size_t)3 * b * zs;
    float em = 0.f;
    const int upr = ldz / kW, total = r * upr;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int i = e / upr, k0 = (e - i * upr) * kW;
        float sv[kW];
#pragma unroll
        for (int t = 0; t < kW; ++t) sv[t] = 0.f;
        if (k0 <= i) {
            const size_t o = (size_t)i * r + k0;
            if constexpr (V4) {
#pragma unroll
                for (int q = 0; q < 6; ++q)
                    if (q < nparts) {
                        const float4 x = __ldg(reinterpret_cast<const float4*>(Sb + q * rr + o));
                        sv[0] += x.x; sv[1] += x.y; sv[2] += x.z; sv[3] += x.w;
                    }
            } else {
#pragma unroll
                for (int q = 0; q < 6; ++q)
                    if (q < nparts) sv[0] += Sb[q * rr + o];
            }
        }
        float v[kW];
#pragma unroll
        for (int t = 0; t < kW; ++t) {
            const int k = k0 + t;
            v[t] = 0.f;
            if (k <= i) {
                const float ev = sv[t] - (i == k ? 1.f : 0.f);
                em = fmaxf(em, isfinite(ev) ? fabsf(ev) : 1e30f);
                v[t] = (k < i) ? -sv[t] : 1.f - 0.5f * ev;
            }
        }
        const size_t zo = (size_t)i * ldz + k0;
        if constexpr (V4) {
            uint32_t w[3][2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                bf16 a1, a2, a3, c1, c2, c3;
                split3(v[2 * h], a1, a2, a3);
                split3(v[2 * h + 1], c1, c2, c3);
                w[0][h] = (uint32_t)__bfloat16_as_ushort(a1) | ((uint32_t)__bfloat16_as_ushort(c1) << 16);
                w[1][h] = (uint32_t)__bfloat16_as_ushort(a2) | ((uint32_t)__bfloat16_as_ushort(c2) << 16);
                w[2][h] = (uint32_t)__bfloat16_as_ushort(a3) | ((uint32_t)__bfloat16_as_ushort(c3) << 16);
            }
#pragma unroll
            for (int q = 0; q < 3; ++q) *reinterpret_cast<uint2*>(z0 + q * zs + zo) = make_uint2(w[q][0], w[q][1]);
        } else {
            bf16 h1, h2, h3;
            split3(v[0], h1, h2, h3);
            z0[zo] = h1;
            z0[zs + zo] = h2;
            z0[2 * zs + zo] = h3;
        }
    }
    for (int o = 16; o > 0; o >>= 1) em = fmaxf(em, __shfl_xor_sync(0xffffffffu, em, o));
    if ((threadIdx.x & 31) == 0) atomicMax(&emax[b], __float_as_int(em));   // em >= 0: int order = float order
}

__device__ __forceinline__ bool gated_off(const int* gate, int b)
{
    return gate && __int_as_float(gate[b]) <= kNearIdentityTol;
}

// S[b] = sum of the nparts partial Grams S6[nparts * b + q] (r x r each).
__global__ void __launch_bounds__(256) qr_sum_kernel(long long rr, int nparts, const float* __restrict__ S6,
                                                     float* __restrict__ S, const int* gate)
{
    const int b = blockIdx.y;
    if (gated_off(gate, b)) return;
    const float* src = S6 + (size_t)b * nparts * rr;
    float* dst = S + (size_t)b * rr;
    const long long stride = (long long)gridDim.x * blockDim.x;
    if ((rr & 3) == 0) {
        for (long long e = 4 * ((long long)blockIdx.x * blockDim.x + threadIdx.x); e < rr; e += 4 * stride) {
            float4 v = *reinterpret_cast<const float4*>(src + e);
            for (int q = 1; q < nparts; ++q) {
                const float4 u = *reinterpret_cast<const float4*>(src + q * rr + e);
                v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
            }
            *reinterpret_cast<float4*>(dst + e) = v;
        }
    } else {
        for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < rr; e += stride) {
            float v = src[e];
            for (int q = 1; q < nparts; ++q) v += src[q * rr + e];
            dst[e] = v;
        }
    }
}

// S[b] = sum of the nparts partial Grams, written block-major for the
// one-CTA factorization: the lower triangle in 8 x 8 blocks t = bi (bi + 1)/2
// + bj, 64 contiguous floats each (row-major inside the block); the strict
// upper part of a diagonal block is zero and rows beyond r are the identity.
__global__ void __launch_bounds__(256) qr_sum_blocks_kernel(int r, int nparts, const float* __restrict__ S6,
                                                            float* __restrict__ Sblk, long long sblk)
{
    const int b = blockIdx.y;
    const int nbr = (r + 7) >> 3;
    const long long tot4 = (long long)nbr * (nbr + 1) / 2 * 16;   // float4 units
    const size_t rr = (size_t)r * r;
    const float* src = S6 + (size_t)b * nparts * rr;
    float* dst = Sblk + (size_t)b * sblk;
    const bool vec = (r % 4) == 0 && ((uintptr_t)S6 & 15u) == 0;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < tot4;
         e += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(e >> 4), q = (int)(e & 15), ii = q >> 1, j0 = (q & 1) * 4;
        int bi = (int)((sqrtf(8.f * (float)t + 1.f) - 1.f) * 0.5f);
        while ((bi + 1) * (bi + 2) / 2 <= t) ++bi;
        while (bi * (bi + 1) / 2 > t) --bi;
        const int bj = t - bi * (bi + 1) / 2;
        const int i = bi * 8 + ii, j = bj * 8 + j0;
        float v[4];
        if (vec && i < r && j + 3 <= i) {   // whole quad in the lower triangle: one 16-byte load per partial
            const size_t o = (size_t)i * r + j;
            float4 x[6];
#pragma unroll
            for (int p = 0; p < 6; ++p)
                if (p < nparts) x[p] = __ldg(reinterpret_cast<const float4*>(src + p * rr + o));
            v[0] = x[0].x; v[1] = x[0].y; v[2] = x[0].z; v[3] = x[0].w;
#pragma unroll
            for (int p = 1; p < 6; ++p)
                if (p < nparts) {
                    v[0] += x[p].x; v[1] += x[p].y; v[2] += x[p].z; v[3] += x[p].w;
                }
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int jj = j + u;
                float x = (i == jj && i >= r) ? 1.f : 0.f;
                if (i < r && jj <= i) {
                    const size_t o = (size_t)i * r + jj;
                    x = src[o];
#pragma unroll
                    for (int p = 1; p < 6; ++p)
                        if (p < nparts) x += src[p * rr + o];
                }
                v[u] = x;
            }
        }
        reinterpret_cast<float4*>(dst)[e] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// dg[b][i] = S[b](i, i): the original diagonal, the reference of the
// dependent-column test in every diagonal block of the blocked factorization.
__global__ void __launch_bounds__(256) qr_diag_kernel(int r, const float* __restrict__ S, float* __restrict__ dg)
{
    const int b = blockIdx.y;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < r; i += gridDim.x * blockDim.x)
        dg[(size_t)b * r + i] = S[(size_t)b * r * r + (size_t)i * r + i];
}

// Panel of the blocked factorization: rows x w block of S (pitch r, matrix
// pitch r*r) -> three bf16 terms A3[3b + t] (rows x nb, pitch nb, term pitch
// r*nb), columns w..nb-1 zero.
__global__ void __launch_bounds__(256) qr_panel_split_kernel(int r, int rows, int w, int nb, const float* __restrict__ S,
                                                             bf16* __restrict__ A3, const int* gate)
{
    const int b = blockIdx.y;
    if (gated_off(gate, b)) return;
    const float* Sb = S + (size_t)b * r * r;
    const size_t ts = (size_t)r * nb;
    bf16* a0 = A3 + (size_t)3 * b * ts;
    const int total = rows * nb;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int i = e / nb, c = e - i * nb;
        const float v = c < w ? Sb[(size_t)i * r + c] : 0.f;
        bf16 h1, h2, h3;
        split3(v, h1, h2, h3);
        a0[e] = h1;
        a0[ts + e] = h2;
        a0[2 * ts + e] = h3;
    }
}

// Panels up to this rank are factored by one CTA per matrix (the matrix held
// in shared memory); wider ones by the blocked path with blocks of kCholBlock.
constexpr int kCholOneCtaMaxR = 248;
constexpr int kCholBlock = 128;

int pick_bn_qr(int n) { return n <= 64 ? 64 : (n <= 128 ? 128 : (n <= 192 ? 192 : 256)); }

// Both operands MN-major (the Gram of a row-major panel).
cudaError_t gemm_mn(int bn, const char* name, const CUtensorMap& ta, const CUtensorMap& tb, int K, const TcGemmEpi& ep,
                    cudaStream_t st)
{
    if (bn == 64) return tc_gemm<64, true>(name, ta, tb, K, ep, st);
    if (bn == 128) return tc_gemm<128, true>(name, ta, tb, K, ep, st);
    if (bn == 192) return tc_gemm<192, true>(name, ta, tb, K, ep, st);
    return tc_gemm<256, true>(name, ta, tb, K, ep, st);
}

// Both operands K-major: the applies, the blocked factorization's panel,
// trailing update and solve.  Their K ranges are short (a 128-column block,
// or rp), so the epilogue (float32, bf16 and three-term outputs, 12 bytes per
// element for an apply) is a large part of each tile: eight epilogue warps
// with the coalesced (shared-memory transposed) epilogue.
cudaError_t gemm_any(int bn, const char* name, const CUtensorMap& ta, const CUtensorMap& tb, int K, const TcGemmEpi& ep,
                     cudaStream_t st)
{
    if (bn == 64) return tc_gemm<64, false, 8, 1>(name, ta, tb, K, ep, st);
    if (bn == 128) return tc_gemm<128, false, 8, 1>(name, ta, tb, K, ep, st);
    if (bn == 192) return tc_gemm<192, false, 8, 1>(name, ta, tb, K, ep, st);
    return tc_gemm<256, false, 8, 1>(name, ta, tb, K, ep, st);
}

bool tmap_bf16(CUtensorMap* t, const bf16* base, long long inner, long long rows, long long nz, long long ld,
               long long zs, int box_rows)
{
    return make_tmap_3d(t, base, TmapType::BF16, inner, rows, nz, ld * 2, zs * 2, 64, box_rows);
}

TcGemmEpi six_term_epi(int M, int N, int bn, int batch, int* status, const int* gate)
{
    TcGemmEpi ep{};
    ep.M = M;
    ep.N = N;
    ep.tiles_m = (int)cdiv(M, 128);
    ep.tiles_n = (int)cdiv(N, bn);
    ep.batch = batch;
    ep.alpha = 0.f;
    ep.beta = 1.f;
    ep.status = status;
    ep.nseg = 6;
    ep.zmul = 3;
    ep.seg_batch = 0;
    ep.asel = kSelA;
    ep.bsel = kSelB;
    ep.gate = gate;
    return ep;
}

// Blocked Cholesky S = L L^T (block size nb; the lower triangle of S is read
// and overwritten) fused with the triangular solve dst = Psrc L^{-T}, for
// panels too wide for one CTA.  Per block column J (columns j0 .. j0 + w):
//   Z_JJ = L_JJ^{-1}                 one CTA per matrix (chol_inv, in shared memory)
//   L_PJ = S_PJ Z_JJ^T               panel below the diagonal block
//   S_T -= L_PJ L_PJ^T               trailing lower triangle
//   Y_J  = P_J - X_{<J} L_{J,<J}^T   forward substitution ...
//   X_J  = Y_J Z_JJ^T                ... and the diagonal block
// All products are six-term split GEMMs (float32 accuracy).  L lives only as
// its three bf16 terms in L3 (r x rp, pitch rp); the terms of X and Y replace
// those of P in P3 column block by column block (with keep_terms, P3 ends as
// the terms of X).  Matrices whose gate entry is at most kNearIdentityTol are
// skipped by every kernel.
cudaError_t chol_blocked_apply(int batch, int m, int r, int rp, int nb, const float* Psrc, float* dst, bf16* P16,
                               float* S, float* W, bf16* ZJ, bf16* A3, bf16* L3, bf16* P3, int* dead, int* status,
                               int* fac_status, long long fac_sstride, int* fac_any, const int* gate,
                               bool keep_terms, cudaStream_t st)
{
    const int nblk = (int)cdiv(r, nb);
    const long long z3 = 3ll * batch, rr = (long long)r * r, mrp = (long long)m * rp, rrp = (long long)r * rp;
    float* dg = W;   // batch x r original diagonal (W is otherwise unused here)
    {
        cudaError_t e = launch("chol_blk_diag0", qr_diag_kernel, dim3((unsigned)cdiv(r, 256), batch), dim3(256), 0, st, r,
                               (const float*)S, dg);
        if (e != cudaSuccess) return e;
    }
    for (int J = 0; J < nblk; ++J) {
        const int j0 = J * nb, w = std::min(nb, r - j0), rest = r - j0 - w;
        const int bnw = pick_bn_qr(w);
        cudaError_t e = chol_inv_io("chol_blk_diag", batch, w, S + (size_t)j0 * r + j0, 1, S, W, nullptr, ZJ, nb,
                                    dead + j0, fac_status, st, gate,
                                    CholIn{rr, 0, r, r, dg + j0, r, fac_sstride, fac_any});
        if (e != cudaSuccess) return e;
        CUtensorMap tZ;
        if (!tmap_bf16(&tZ, ZJ, nb, w, z3, nb, (long long)w * nb, bnw)) return cudaErrorInvalidValue;
        if (rest > 0) {
            const long long tot = (long long)rest * nb;
            e = launch("chol_blk_split", qr_panel_split_kernel,
                       dim3((unsigned)std::min<long long>(cdiv(tot, 256), 2048), batch), dim3(256), 0, st, r, rest,
                       w, nb, (const float*)(S + (size_t)(j0 + w) * r + j0), A3, gate);
            if (e != cudaSuccess) return e;
            CUtensorMap tA;
            if (!tmap_bf16(&tA, A3, nb, rest, z3, nb, (long long)r * nb, 128)) return cudaErrorInvalidValue;
            TcGemmEpi ep = six_term_epi(rest, w, bnw, batch, status, gate);
            ep.Cs3 = L3 + (size_t)(j0 + w) * rp + j0;
            ep.ldcs3 = rp;
            ep.scs3 = rrp;
            e = gemm_any(bnw, "chol_blk_panel", tA, tZ, w, ep, st);
            if (e != cudaSuccess) return e;
            const int bnt = pick_bn_qr(rest);
            const bf16* lp = L3 + (size_t)(j0 + w) * rp + j0;
            CUtensorMap tLa, tLb;
            if (!tmap_bf16(&tLa, lp, w, rest, z3, rp, rrp, 128) || !tmap_bf16(&tLb, lp, w, rest, z3, rp, rrp, bnt))
                return cudaErrorInvalidValue;
            TcGemmEpi et = six_term_epi(rest, rest, bnt, batch, status, gate);
            et.Cf = S + (size_t)(j0 + w) * r + j0 + w;
            et.ldc = r;
            et.sc = rr;
            et.auxf = et.Cf;
            et.ldauxf = r;
            et.sauxf = rr;
            et.alpha = 1.f;
            et.beta = -1.f;
            et.lower = 1;
            e = gemm_any(bnt, "chol_blk_trail", tLa, tLb, w, et, st);
            if (e != cudaSuccess) return e;
        }
        if (J > 0) {
            CUtensorMap tX, tL;
            if (!tmap_bf16(&tX, P3, j0, m, z3, rp, mrp, 128) ||
                !tmap_bf16(&tL, L3 + (size_t)j0 * rp, j0, w, z3, rp, rrp, bnw))
                return cudaErrorInvalidValue;
            TcGemmEpi e1 = six_term_epi(m, w, bnw, batch, status, gate);
            e1.auxf = Psrc + j0;
            e1.ldauxf = rp;
            e1.sauxf = mrp;
            e1.alpha = 1.f;
            e1.beta = -1.f;
            e1.Cs3 = P3 + j0;
            e1.ldcs3 = rp;
            e1.scs3 = mrp;
            e = gemm_any(bnw, "chol_blk_solve", tX, tL, j0, e1, st);
            if (e != cudaSuccess) return e;
        }
        CUtensorMap tY;
        if (!tmap_bf16(&tY, P3 + j0, w, m, z3, rp, mrp, 128)) return cudaErrorInvalidValue;
        TcGemmEpi e2 = six_term_epi(m, w, bnw, batch, status, gate);
        e2.Cf = dst + j0;
        e2.C = P16 ? P16 + j0 : nullptr;
        e2.ldc = rp;
        e2.sc = mrp;
        if (J + 1 < nblk || keep_terms) {   // the terms of X feed later blocks (and the second pass)
            e2.Cs3 = P3 + j0;
            e2.ldcs3 = rp;
            e2.scs3 = mrp;
        }
        e = gemm_any(bnw, "chol_blk_apply", tY, tZ, w, e2, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

int chol_block_size(int r) { return r > kCholOneCtaMaxR ? kCholBlock : 0; }

cudaError_t qr_cholesky2_tc(int batch, int m, int r, int rp, float* Pin, int nparts, float* P, float* Ptmp,
                            bf16* P16, char* ws, const DionLayout& L, int* status, cudaStream_t st, int n,
                            const float* M, const bf16* G, const float* Q, bool terms_ready)
{
    bf16* P3 = (bf16*)(ws + L.P3);
    bf16* P3b = (bf16*)(ws + L.P3b);
    bf16* Z3 = (bf16*)(ws + L.Z3);
    float* S6 = (float*)(ws + L.S6);
    float* S = (float*)(ws + L.S);
    float* W = (float*)(ws + L.W);
    int* dead = (int*)(ws + L.dead);
    int* emax = (int*)(ws + L.emax);
    int* hard = (int*)(ws + L.hard);
    // the first pass's factorization reports unresolved pivots per matrix
    // (hard); those matrices redo the first pass in float64 (qr64.cu)
    const bool fb = qr64_supported(r);
    if (fb) {
        cudaError_t e = cudaMemsetAsync(hard, 0, sizeof(int) * (batch + 1), st);
        if (e != cudaSuccess) return e;
    }
    int* fac1 = fb ? hard : status;
    int* any1 = fb ? hard + batch : nullptr;
    const long long fac1_stride = fb ? 1 : 0;
    const int bn = pick_bn_qr(r), bna = pick_bn_qr(rp);
    const bool blocked = L.nbc > 0;
    // blocked: the Gram's lower half, accumulated straight into S when that
    // alone fills the SMs, else as six partials summed afterwards
    const bool direct = blocked && cdiv(r, 128) * cdiv(r, bn) * batch / 2 >= num_sms();

    // The bf16 terms of the panel: P3 holds those of the first pass's input;
    // the second pass reads those of its input from P3b (written by the
    // first apply) or, on the blocked path, from P3 (rewritten in place by the
    // blocked solve).  The Gram reads them MN-major (64 x 64 boxes), the apply
    // K-major (64 x 128).
    const long long pz = (long long)m * rp * 2;
    CUtensorMap tG[2], tPa[2], tZb;
    for (int t = 0; t < 2; ++t) {
        bf16* base = t == 0 ? P3 : P3b;
        if (!make_tmap_3d(&tG[t], base, TmapType::BF16, rp, m, 3ll * batch, (long long)rp * 2, pz, 64, 64) ||
            !make_tmap_3d(&tPa[t], base, TmapType::BF16, rp, m, 3ll * batch, (long long)rp * 2, pz, 64, 128))
            return cudaErrorInvalidValue;
    }
    if (!make_tmap_3d(&tZb, Z3, TmapType::BF16, rp, r, 3ll * batch, (long long)rp * 2, (long long)r * rp * 2, 64, bna))
        return cudaErrorInvalidValue;

    // pass 1: split partials of P -> Ptmp;  pass 2: Ptmp -> P (and P16)
    for (int pass = 0; pass < 2; ++pass) {
        const float* src = pass == 0 ? Pin : Ptmp;
        float* dst = pass == 0 ? Ptmp : P;
        const int ti = (pass == 1 && !blocked) ? 1 : 0;   // which terms hold this pass's input
        cudaError_t e = cudaSuccess;
        if (pass == 0 && !terms_ready) {
            const long long total4 = (long long)m * (rp / 4);
            e = launch("qr_split", qr_split_kernel, dim3((unsigned)std::min<long long>(cdiv(total4, 256), 2048), batch),
                       dim3(256), 0, st, m, r, rp, src, nparts, (long long)batch * m * rp, P3,
                       blocked ? dst : (float*)nullptr, total4);
            if (e != cudaSuccess) return e;
        }
        if (direct) {
            TcGemmEpi eg = six_term_epi(r, r, bn, batch, status, nullptr);
            eg.Cf = S;
            eg.ldc = r;
            eg.sc = (long long)r * r;
            eg.lower = 1;
            e = gemm_mn(bn, "qr_gram_tc", tG[ti], tG[ti], m, eg, st);
        } else {
            // six partial Grams S6[6b + q] = T_a(q) T_b(q)^T  (r x r)
            TcGemmEpi eg{r, r, (int)cdiv(r, 128), (int)cdiv(r, bn), 6 * batch, nullptr, r, (long long)r * r,
                         nullptr, 0, 0, nullptr, 0, 0, 0.f, 1.f, status, S6, 6, 3, 1, kSelA, kSelB};
            eg.lower = blocked ? 1 : 0;
            e = gemm_mn(bn, "qr_gram_tc", tG[ti], tG[ti], m, eg, st);
        }
        if (e != cudaSuccess) return e;
        if (pass == 1) {
            // near-identity inverse on all SMs; the factorization runs only where it does not apply
            e = cudaMemsetAsync(emax, 0, sizeof(int) * batch, st);
            if (e != cudaSuccess) return e;
            const float* Sn = direct ? S : S6;
            const bool v4 = (r % 4) == 0 && (rp % 4) == 0 && ((uintptr_t)Sn & 15u) == 0;
            const long long units = (long long)r * rp / (v4 ? 4 : 1);
            e = launch("qr_near_identity", v4 ? qr_near_identity_kernel<true> : qr_near_identity_kernel<false>,
                       dim3((unsigned)std::min<long long>(cdiv(units, 256), 1024), batch), dim3(256), 0, st, r, rp, Sn,
                       direct ? 1 : 6, Z3, emax);
            if (e != cudaSuccess) return e;
        }
        const int* gate = pass == 1 ? emax : nullptr;
        if (!blocked) {
            // first pass: the six partials summed on all SMs, so the one-CTA
            // factorization reads one matrix; the second pass factors only
            // matrices that failed the near-identity test and reads the partials
            if (pass == 0) {
                const long long nb8 = (r + 7) / 8, sblk = nb8 * (nb8 + 1) / 2 * 64;
                e = launch("qr_gram_sum", qr_sum_blocks_kernel,
                           dim3((unsigned)std::min<long long>(cdiv(sblk / 4, 256), 1024), batch), dim3(256), 0, st, r, 6,
                           (const float*)S6, S, sblk);
                if (e != cudaSuccess) return e;
                e = chol_inv_io("chol_inv_pass1", batch, r, S, 1, S, W, nullptr, Z3, rp, dead, fac1, st, nullptr,
                                CholIn{sblk, 0, 0, r, nullptr, 0, fac1_stride, any1});
            } else {
                e = chol_inv("chol_inv_pass2", batch, r, S6, 6, S, W, nullptr, Z3, rp, dead, status, st, gate);
            }
            if (e != cudaSuccess) return e;
        }
        if (!blocked || pass == 1) {
            // P L^{-T}: all six cross terms accumulated; columns r..rp-1 come out
            // zero.  First pass: only its bf16 terms (P3b) for the second pass;
            // second pass: P (float32) and P16.
            TcGemmEpi ea{m, rp, (int)cdiv(m, 128), (int)cdiv(rp, bna), batch, pass == 1 ? P16 : nullptr, rp,
                         (long long)m * rp, nullptr, 0, 0, nullptr, 0, 0, 0.f, 1.f, status, pass == 1 ? dst : nullptr,
                         6, 3, 0, kSelA, kSelB};
            if (pass == 0) {
                ea.Cs3 = P3b;
                ea.ldcs3 = rp;
                ea.scs3 = (long long)m * rp;
            }
            e = gemm_any(bna, "qr_apply_tc", tPa[ti], tZb, rp, ea, st);
            if (e != cudaSuccess) return e;
        }
        if (blocked) {
            if (!direct) {
                const long long rr = (long long)r * r;
                e = launch("qr_gram_sum", qr_sum_kernel, dim3((unsigned)std::min<long long>(cdiv(rr, 1024), 1024), batch),
                           dim3(256), 0, st, rr, 6, (const float*)S6, S, gate);
                if (e != cudaSuccess) return e;
            }
            e = chol_blocked_apply(batch, m, r, rp, L.nbc, pass == 0 ? dst : src, dst, pass == 1 ? P16 : nullptr, S, W,
                                   (bf16*)(ws + L.ZJ), (bf16*)(ws + L.A3), Z3, P3, dead, status,
                                   pass == 0 ? fac1 : status, pass == 0 ? fac1_stride : 0, pass == 0 ? any1 : nullptr,
                                   gate, pass == 0, st);
            if (e != cudaSuccess) return e;
        }
        if (pass == 0 && fb) {
            // flagged matrices: B Q and the first pass again in float64 from the step's inputs,
            // written where the second pass reads its input (blocked: P3 and the float32 panel; else P3b)
            e = qr64_first_pass(batch, m, r, rp, Pin, nparts, (long long)batch * m * rp, (double*)(ws + L.S64),
                                blocked ? dst : nullptr, blocked ? P3 : P3b, dead, status, hard, st, n, M, G, Q);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace dion
