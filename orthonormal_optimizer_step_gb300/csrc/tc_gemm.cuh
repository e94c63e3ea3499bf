// tc_gemm.cuh -- persistent batched bf16 GEMM on the 5th-generation tensor
// cores (tcgen05.mma, accumulator in tensor memory), fed by TMA.
//
//   C[b] (M x N) = alpha * aux[b] + beta * (A[b] (M x K) . B[b] (N x K)^T)
//
// Both operands are K-major (row-major with K contiguous).  One CTA per SM
// walks the output tiles (BM = 128 rows, BN = 64/128/192/256 columns) of every
// matrix of the batch.  Warp 0 issues TMA loads into a ring of shared-memory
// stages, warp 1 issues tcgen05.mma from one thread into a double-buffered
// TMEM accumulator, warps 2..2+EW-1 drain the accumulator (tcgen05.ld), apply
// the epilogue and store the results (optionally also the transpose), so the
// epilogue of one tile overlaps the MMAs of the next.  EW = 4 gives one warp
// per TMEM lane quarter; EW = 8 or 12 split each quarter's columns between
// two or three warps, for epilogues that read float32 addends from HBM and
// need more loads in flight than four warps keep.  COAL routes each warp's
// 32 x 32 accumulator block through a padded shared-memory tile, so that its
// global loads and stores cover four whole 128-byte row segments per
// instruction instead of 32 rows (one per lane): the form for epilogues that
// stream their addends and outputs from and to HBM.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace dion {

struct TcGemmEpi {
    int M, N;                       // valid output extent of one matrix
    int tiles_m, tiles_n, batch;
    bf16* C; long long ldc, sc;     // output, row pitch and matrix pitch (elements)
    const bf16* aux; long long ldaux, saux;   // optional addend (same shape as C)
    bf16* CT; long long ldct, sct;  // optional transposed copy of the output (N x M)
    float alpha, beta;
    int* status;
    float* Cf;                      // if set: float32 output (row pitch ldc, matrix pitch sc); C, if also
                                    // set, receives a bf16 copy
    // K segments: the contraction runs over nseg segments of K each; segment q
    // reads operand matrices zmul*b + asel[q] (A) and zmul*b + bsel[q] (B),
    // 4-bit entries packed in asel/bsel; with K-major operands walked chunk by
    // chunk (every segment's chunk kc before chunk kc + 1), with MN-major ones
    // segment by segment.  seg_batch = 1: each segment is its own output
    // matrix (index nseg*b + q) instead of being accumulated.
    int nseg, zmul, seg_batch;
    uint32_t asel, bsel;
    // float32 addend (used instead of aux when set): C = alpha * auxf + beta * acc
    const float* auxf; long long ldauxf, sauxf;
    // three-term bf16 split of the result (X = X1 + X2 + X3), term t of matrix b
    // at Cs3 + (3b + t) * scs3 + row * ldcs3 + col
    bf16* Cs3; long long ldcs3, scs3;
    // tiles that run: with `gate`, only those of matrices b whose gate[b]
    // (a float max|S - I| stored as int bits) exceeds kNearIdentityTol; with
    // `lower`, only tiles holding an element on or below the diagonal
    const int* gate;
    int lower;
    // second addend (bf16), added after the float32 one: C += alpha2 * aux2
    const bf16* aux2; long long ldaux2, saux2; float alpha2;
    // hp_mode != 0: the step scalars come from hp (see StepHyper), formed in
    // the epilogue: 1 -> beta = -(1 - mu); 2 -> alpha = 1 - lr wd,
    // beta = -lr sqrt(m/n).  Non-finite device values set the status word.
    StepHyper hp;
    int hp_mode;
    // tile order within a matrix: 0 walks the column tiles fastest, 1 the row
    // tiles (pick the shorter direction, so the operand tiles that cycle stay
    // small enough for L2 while the other operand is reused by consecutive tiles)
    int m_fast;
    // band_m > 0 (overrides m_fast): bands of band_m row tiles, row tiles
    // fastest inside a band.  The CTAs in flight then cover a few row tiles
    // by a few column tiles, so both operand panels they stream are shared in
    // L2 (for long K, where no single panel order keeps one operand resident)
    int band_m;
};

__device__ __forceinline__ void tc_tile_mn(const TcGemmEpi& ep, int rem, int& tm, int& tn)
{
    if (ep.band_m > 0) {
        const int per_band = ep.band_m * ep.tiles_n;
        const int band = rem / per_band, in = rem - band * per_band;
        const int m0 = band * ep.band_m, bm = min(ep.band_m, ep.tiles_m - m0);
        tm = m0 + in % bm;
        tn = in / bm;
    } else if (ep.m_fast) {
        tm = rem % ep.tiles_m;
        tn = rem / ep.tiles_m;
    } else {
        tm = rem / ep.tiles_n;
        tn = rem % ep.tiles_n;
    }
}

template <int BN>
struct TcGemmCfg {
    static constexpr int BM = 128, BK = 64;
    static constexpr int STAGES = BN == 256 ? 4 : (BN == 192 ? 5 : (BN == 128 ? 6 : 8));
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BYTES = BN * BK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = BN == 192 ? 512 : 2 * BN;   // a power of two >= 2 BN
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 256;
};

// Operand stages of a GEMM whose epilogue stages through EW blocks of 32 x 33
// floats (COAL != 0): as many of the configuration's stages as fit beside
// them in the 227 KB a CTA may use.
template <int BN, int EW, int COAL>
constexpr int tc_stages()
{
    using Cfg = TcGemmCfg<BN>;
    if (!COAL) return Cfg::STAGES;
    const int fit = (int)((232448 - 1024 - 256 - (size_t)EW * 32 * 33 * 4) / Cfg::STAGE_BYTES);
    return fit < Cfg::STAGES ? fit : Cfg::STAGES;
}

template <int BN, int EW, int COAL>
constexpr size_t tc_smem()
{
    return (size_t)tc_stages<BN, EW, COAL>() * TcGemmCfg<BN>::STAGE_BYTES + 1024 + 256 +
           (COAL ? (size_t)EW * 32 * 33 * 4 : 0);
}

int num_sms();

// Kernels defined in this header get internal linkage: every translation unit
// that includes it owns its own copy (and its own one-time attribute setup).
namespace {

__device__ __forceinline__ bool tc_tile_on(const TcGemmEpi& ep, int b, int tm, int tn, int bm_rows, int bn_cols)
{
    if (ep.lower && tn * bn_cols > tm * bm_rows + bm_rows - 1) return false;
    if (ep.gate) {
        const int bm = ep.seg_batch ? b / ep.nseg : b;
        if (__int_as_float(ep.gate[bm]) <= kNearIdentityTol) return false;
    }
    return true;
}

__device__ __forceinline__ void tc_epi_store(const TcGemmEpi& ep, int b, int row, int col0, const uint32_t (&v)[32],
                                             float alpha, float beta)
{
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = beta * __uint_as_float(v[i]);
    const int ncol = min(32, ep.N - col0);
    if (ep.auxf) {
        const float* ap = ep.auxf + b * ep.sauxf + (long long)row * ep.ldauxf + col0;
        if (ncol == 32 && ((uintptr_t)ap & 15u) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 u = *reinterpret_cast<const float4*>(ap + j);
                acc[j] = fmaf(alpha, u.x, acc[j]);
                acc[j + 1] = fmaf(alpha, u.y, acc[j + 1]);
                acc[j + 2] = fmaf(alpha, u.z, acc[j + 2]);
                acc[j + 3] = fmaf(alpha, u.w, acc[j + 3]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncol) acc[i] = fmaf(alpha, ap[i], acc[i]);
        }
    } else if (ep.aux) {
        const bf16* ap = ep.aux + b * ep.saux + (long long)row * ep.ldaux + col0;
        if (ncol == 32) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 u = *reinterpret_cast<const uint4*>(ap + 8 * j);
                const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[8 * j + e] = fmaf(alpha, __bfloat162float(h[e]), acc[8 * j + e]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncol) acc[i] = fmaf(alpha, __bfloat162float(ap[i]), acc[i]);
        }
    }
    if (ep.aux2) {
        const bf16* ap = ep.aux2 + b * ep.saux2 + (long long)row * ep.ldaux2 + col0;
        if (ncol == 32 && ((uintptr_t)ap & 15u) == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 u = *reinterpret_cast<const uint4*>(ap + 8 * j);
                const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[8 * j + e] = fmaf(ep.alpha2, __bfloat162float(h[e]), acc[8 * j + e]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncol) acc[i] = fmaf(ep.alpha2, __bfloat162float(ap[i]), acc[i]);
        }
    }
    if (ep.Cs3) {
        bf16* sp = ep.Cs3 + (long long)3 * b * ep.scs3 + (long long)row * ep.ldcs3 + col0;
        if (ncol == 32 && ((uintptr_t)sp & 15u) == 0 && (ep.scs3 & 7) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                uint32_t t1[4], t2[4], t3[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    uint32_t w1 = 0, w2 = 0, w3 = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float v = acc[j + e + h];
                        const bf16 h1 = __float2bfloat16_rn(v);
                        const float r1 = v - __bfloat162float(h1);
                        const bf16 h2 = __float2bfloat16_rn(r1);
                        const bf16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
                        w1 |= (uint32_t)__bfloat16_as_ushort(h1) << (16 * h);
                        w2 |= (uint32_t)__bfloat16_as_ushort(h2) << (16 * h);
                        w3 |= (uint32_t)__bfloat16_as_ushort(h3) << (16 * h);
                    }
                    t1[e / 2] = w1;
                    t2[e / 2] = w2;
                    t3[e / 2] = w3;
                }
                *reinterpret_cast<uint4*>(sp + j) = make_uint4(t1[0], t1[1], t1[2], t1[3]);
                *reinterpret_cast<uint4*>(sp + ep.scs3 + j) = make_uint4(t2[0], t2[1], t2[2], t2[3]);
                *reinterpret_cast<uint4*>(sp + 2 * ep.scs3 + j) = make_uint4(t3[0], t3[1], t3[2], t3[3]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (i >= ncol) break;
                const bf16 h1 = __float2bfloat16_rn(acc[i]);
                const float r1 = acc[i] - __bfloat162float(h1);
                const bf16 h2 = __float2bfloat16_rn(r1);
                sp[i] = h1;
                sp[ep.scs3 + i] = h2;
                sp[2 * ep.scs3 + i] = __float2bfloat16_rn(r1 - __bfloat162float(h2));
            }
        }
    }
    if (ep.Cf) {
        float* fp = ep.Cf + b * ep.sc + (long long)row * ep.ldc + col0;
        if (ncol == 32 && ((uintptr_t)fp & 15u) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(fp + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncol) fp[i] = acc[i];
        }
        if (!ep.C) return;             // else also a bf16 copy with the same pitches
    }
    if (!ep.C) return;
    bf16* cp = ep.C + b * ep.sc + (long long)row * ep.ldc + col0;
    if (ncol == 32) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 u;
            u.x = tc::pack_bf16x2(acc[8 * j + 0], acc[8 * j + 1]);
            u.y = tc::pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]);
            u.z = tc::pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]);
            u.w = tc::pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]);
            *reinterpret_cast<uint4*>(cp + 8 * j) = u;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < ncol) cp[i] = __float2bfloat16_rn(acc[i]);
    }
    if (ep.CT) {
        bf16* tp = ep.CT + b * ep.sct + (long long)col0 * ep.ldct + row;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < ncol) tp[(long long)i * ep.ldct] = __float2bfloat16_rn(acc[i]);
    }
}

// Coalesced epilogue of one 32 x 32 block: tb holds the block (row i at
// tb[33 i]), rows row0.. and columns col0.. of the output.  Lane l handles
// columns col0 + 4 (l % 8) .. +3 of rows 4p + l / 8, p = 0..7, so each
// instruction moves four whole row segments.  Supports the float32 and bf16
// addends (auxf or aux, then aux2) and the float32, bf16 and three-term bf16
// outputs (Cf, C, Cs3).
// Interior blocks with aligned rows ("fast") load all of a lane's addends
// into a TcCoalPref, branch-free, before any arithmetic (so their latencies
// overlap); edge blocks go element by element.
__device__ __forceinline__ bool tc_coal_aligned(const void* p, long long ld, long long sm, unsigned bytes)
{
    return p == nullptr || (((uintptr_t)p & (bytes - 1)) == 0 && (ld & 3) == 0 && (sm & 3) == 0);
}

__device__ __forceinline__ bool tc_coal_rows_aligned(const TcGemmEpi& ep)
{
    return tc_coal_aligned(ep.auxf, ep.ldauxf, ep.sauxf, 16) && tc_coal_aligned(ep.aux, ep.ldaux, ep.saux, 8) &&
           tc_coal_aligned(ep.aux2, ep.ldaux2, ep.saux2, 8) && tc_coal_aligned(ep.Cf, ep.ldc, ep.sc, 16) &&
           tc_coal_aligned(ep.C, ep.ldc, ep.sc, 8) && tc_coal_aligned(ep.Cs3, ep.ldcs3, ep.scs3, 8);
}

// one lane's addends of a fast block: a = auxf (float4) or aux (bf16 x 4 in
// the first two words), a2 = aux2 (bf16 x 4)
struct TcCoalPref {
    float4 a[8];
    uint2 a2[8];
};

__device__ __forceinline__ void tc_coal_prefetch(const TcGemmEpi& ep, int b, int row0, int col0, int lane,
                                                 TcCoalPref& pf)
{
    const long long r = (long long)(row0 + (lane >> 3));
    const int gc = col0 + 4 * (lane & 7);
    if (ep.auxf) {
        const float* ap = ep.auxf + b * ep.sauxf + r * ep.ldauxf + gc;
#pragma unroll
        for (int p = 0; p < 8; ++p) pf.a[p] = *reinterpret_cast<const float4*>(ap + 4 * p * ep.ldauxf);
    } else if (ep.aux) {
        const bf16* ap = ep.aux + b * ep.saux + r * ep.ldaux + gc;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const uint2 u = *reinterpret_cast<const uint2*>(ap + 4 * p * ep.ldaux);
            pf.a[p].x = __uint_as_float(u.x);
            pf.a[p].y = __uint_as_float(u.y);
        }
    }
    if (ep.aux2) {
        const bf16* ap = ep.aux2 + b * ep.saux2 + r * ep.ldaux2 + gc;
#pragma unroll
        for (int p = 0; p < 8; ++p) pf.a2[p] = *reinterpret_cast<const uint2*>(ap + 4 * p * ep.ldaux2);
    }
}

__device__ __forceinline__ void tc_coal_add_bf16x4(float (&o)[4], uint32_t lo, uint32_t hi, float w)
{
    o[0] = fmaf(w, __uint_as_float(lo << 16), o[0]);
    o[1] = fmaf(w, __uint_as_float(lo & 0xffff0000u), o[1]);
    o[2] = fmaf(w, __uint_as_float(hi << 16), o[2]);
    o[3] = fmaf(w, __uint_as_float(hi & 0xffff0000u), o[3]);
}

__device__ __forceinline__ void tc_coal_finish(const TcGemmEpi& ep, int b, int row0, int col0, const float* tb,
                                               int lane, float alpha, float beta, const TcCoalPref& pf)
{
    const int cl = 4 * (lane & 7), r8 = lane >> 3;
    const long long r = (long long)(row0 + r8);
    const int gc = col0 + cl;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = beta * tb[(4 * p + r8) * 33 + cl + e];
        if (ep.auxf) {
            o[0] = fmaf(alpha, pf.a[p].x, o[0]);
            o[1] = fmaf(alpha, pf.a[p].y, o[1]);
            o[2] = fmaf(alpha, pf.a[p].z, o[2]);
            o[3] = fmaf(alpha, pf.a[p].w, o[3]);
        } else if (ep.aux) {
            tc_coal_add_bf16x4(o, __float_as_uint(pf.a[p].x), __float_as_uint(pf.a[p].y), alpha);
        }
        if (ep.aux2) tc_coal_add_bf16x4(o, pf.a2[p].x, pf.a2[p].y, ep.alpha2);
        const long long off = (r + 4 * p) * ep.ldc + gc;
        if (ep.Cf) *reinterpret_cast<float4*>(ep.Cf + b * ep.sc + off) = make_float4(o[0], o[1], o[2], o[3]);
        if (ep.C)
            *reinterpret_cast<uint2*>(ep.C + b * ep.sc + off) =
                make_uint2(tc::pack_bf16x2(o[0], o[1]), tc::pack_bf16x2(o[2], o[3]));
        if (ep.Cs3) {   // the three bf16 terms of each value (term t at + t scs3)
            uint32_t w[3][2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t p1 = 0, p2 = 0, p3 = 0;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float x = o[2 * hh + e];
                    const bf16 h1 = __float2bfloat16_rn(x);
                    const float r1 = x - __bfloat162float(h1);
                    const bf16 h2 = __float2bfloat16_rn(r1);
                    const bf16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
                    p1 |= (uint32_t)__bfloat16_as_ushort(h1) << (16 * e);
                    p2 |= (uint32_t)__bfloat16_as_ushort(h2) << (16 * e);
                    p3 |= (uint32_t)__bfloat16_as_ushort(h3) << (16 * e);
                }
                w[0][hh] = p1;
                w[1][hh] = p2;
                w[2][hh] = p3;
            }
            bf16* sp = ep.Cs3 + 3ll * b * ep.scs3 + (r + 4 * p) * ep.ldcs3 + gc;
#pragma unroll
            for (int t = 0; t < 3; ++t) *reinterpret_cast<uint2*>(sp + t * ep.scs3) = make_uint2(w[t][0], w[t][1]);
        }
    }
}

// this warp's 32 x 32 accumulator block (TMEM address tq: its lane quarter,
// first column) into tb, row `lane` at tb[33 lane], 16 columns at a time
__device__ __forceinline__ void tc_coal_stage(uint32_t tq, float* tb, int lane)
{
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t v[16];
        tc::tmem_ld16(tq + 16 * half, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) tb[lane * 33 + 16 * half + j] = __uint_as_float(v[j]);
    }
    __syncwarp();
}

// edge blocks: element by element, every access guarded
__device__ __forceinline__ void tc_coal_slow(const TcGemmEpi& ep, int b, int row0, int col0, const float* tb, int lane,
                                             float alpha, float beta)
{
    const int cl = 4 * (lane & 7), r8 = lane >> 3, gc = col0 + cl;
#pragma unroll 1
    for (int p = 0; p < 8; ++p) {
        const int gr = row0 + 4 * p + r8;
#pragma unroll 1
        for (int e = 0; e < 4; ++e) {
            const int c = gc + e;
            if (gr >= ep.M || c >= ep.N) continue;
            float v = beta * tb[(4 * p + r8) * 33 + cl + e];
            if (ep.auxf) v = fmaf(alpha, ep.auxf[b * ep.sauxf + (long long)gr * ep.ldauxf + c], v);
            else if (ep.aux) v = fmaf(alpha, __bfloat162float(ep.aux[b * ep.saux + (long long)gr * ep.ldaux + c]), v);
            if (ep.aux2) v = fmaf(ep.alpha2, __bfloat162float(ep.aux2[b * ep.saux2 + (long long)gr * ep.ldaux2 + c]), v);
            if (ep.Cf) ep.Cf[b * ep.sc + (long long)gr * ep.ldc + c] = v;
            if (ep.C) ep.C[b * ep.sc + (long long)gr * ep.ldc + c] = __float2bfloat16_rn(v);
            if (ep.Cs3) {
                bf16* sp = ep.Cs3 + 3ll * b * ep.scs3 + (long long)gr * ep.ldcs3 + c;
                const bf16 h1 = __float2bfloat16_rn(v);
                const float r1 = v - __bfloat162float(h1);
                const bf16 h2 = __float2bfloat16_rn(r1);
                sp[0] = h1;
                sp[ep.scs3] = h2;
                sp[2 * ep.scs3] = __float2bfloat16_rn(r1 - __bfloat162float(h2));
            }
        }
    }
}

// MN = true: both operands are MN-major (the M or N index contiguous, K
// rows): tmA and tmB have 64 x 64 boxes (MN x K) landing as 64-wide MN blocks
// of the 128-byte swizzle (8 KB apart), so a row-major m x r panel serves as
// the operand of its own Gram matrix without a transposed copy.
template <int BN, bool MN = false, int EW = 4, int COAL = 0>
__global__ void __launch_bounds__(64 + 32 * EW, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int K, TcGemmEpi ep)
{
    static_assert(EW % 4 == 0 && EW >= 4 && EW <= 12, "epilogue warps: 4, 8 or 12");
    constexpr int STAGES = tc_stages<BN, EW, COAL>();
    static_assert(STAGES >= 3, "operand stages");
    using Cfg = TcGemmCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = (uint32_t*)(acc_empty + 2);
    int* abort_flag = (int*)(tmem_slot + 1);
    volatile int* abrt = abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&acc_full[b], 1);
            tc::mbar_init(&acc_empty[b], EW);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int per_mat = ep.tiles_m * ep.tiles_n;
    const int tiles = ep.batch * per_mat;
    const int kchunks = (K + Cfg::BK - 1) / Cfg::BK;

    if (warp == 0) {
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmA);
            tc::tma_prefetch_desc(&tmB);
            int stage = 0;
            uint32_t ph = 0;
            for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x) {
                const int b = t / per_mat, rem = t % per_mat;
                int tm, tn;
                tc_tile_mn(ep, rem, tm, tn);
                if (!tc_tile_on(ep, b, tm, tn, Cfg::BM, BN)) continue;
                const int q0 = ep.seg_batch ? b % ep.nseg : 0, q1 = ep.seg_batch ? q0 + 1 : ep.nseg;
                const int bm = ep.seg_batch ? b / ep.nseg : b;
                // One stage: operand chunk kc of segment q.  K-major operands
                // walk the segments chunk-major (for each K chunk, every
                // segment in turn), so the operand chunks that several
                // segments share (the split terms) are reused from L2 within a
                // few stages instead of being fetched again per segment.
                // MN-major operands (the Grams) walk them segment-major, so
                // consecutive stages read consecutive rows of one term.
                auto issue = [&](int q, int kc) -> bool {
                    const int za = bm * ep.zmul + (int)((ep.asel >> (4 * q)) & 15u);
                    const int zb = bm * ep.zmul + (int)((ep.bsel >> (4 * q)) & 15u);
                    if (!tc::mbar_wait(&empty[stage], ph ^ 1, abrt, ep.status)) return false;
                    uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
                    tc::mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
                    if (MN) {
#pragma unroll
                        for (int blk = 0; blk < Cfg::BM / 64; ++blk)
                            tc::tma_load_3d(sa + blk * 8192, &tmA, &full[stage], tm * Cfg::BM + blk * 64,
                                            kc * Cfg::BK, za);
#pragma unroll
                        for (int blk = 0; blk < BN / 64; ++blk)
                            tc::tma_load_3d(sa + Cfg::A_BYTES + blk * 8192, &tmB, &full[stage], tn * BN + blk * 64,
                                            kc * Cfg::BK, zb);
                    } else {
                        tc::tma_load_3d(sa, &tmA, &full[stage], kc * Cfg::BK, tm * Cfg::BM, za);
                        tc::tma_load_3d(sa + Cfg::A_BYTES, &tmB, &full[stage], kc * Cfg::BK, tn * BN, zb);
                    }
                    if (++stage == STAGES) { stage = 0; ph ^= 1; }
                    return true;
                };
                bool ok = true;
                if (MN) {
                    for (int q = q0; q < q1 && ok; ++q)
                        for (int kc = 0; kc < kchunks && ok; ++kc) ok = issue(q, kc);
                } else {
                    for (int kc = 0; kc < kchunks && ok; ++kc)
                        for (int q = q0; q < q1 && ok; ++q) ok = issue(q, kc);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = tc::make_idesc(Cfg::BM, BN, 1, MN, MN);
            int stage = 0;
            uint32_t ph = 0;
            int it = 0;
            for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x) {
                {
                    const int b = t / per_mat, rem = t % per_mat;
                    int tm, tn;
                    tc_tile_mn(ep, rem, tm, tn);
                    if (!tc_tile_on(ep, b, tm, tn, Cfg::BM, BN)) continue;
                }
                const int buf = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!tc::mbar_wait(&acc_empty[buf], aph ^ 1, abrt, ep.status)) break;
                tc::tc_fence_after();
                const uint32_t d = tmem + buf * BN;
                bool ok = true;
                const int nchunks = kchunks * (ep.seg_batch ? 1 : ep.nseg);
                for (int kc = 0; kc < nchunks; ++kc) {
                    if (!tc::mbar_wait(&full[stage], ph, abrt, ep.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(smem + stage * Cfg::STAGE_BYTES);
                    const uint32_t b0 = a0 + Cfg::A_BYTES;
#pragma unroll
                    for (int k = 0; k < Cfg::BK / 16; ++k) {
                        if (MN)
                            tc::mma_bf16(d, tc::make_sdesc(a0 + k * 2048, 8192, 1024),
                                         tc::make_sdesc(b0 + k * 2048, 8192, 1024), idesc, (kc | k) != 0);
                        else
                            tc::mma_bf16(d, tc::make_sdesc(a0 + k * 32, 16, 1024), tc::make_sdesc(b0 + k * 32, 16, 1024),
                                         idesc, (kc | k) != 0);
                    }
                    tc::mma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; ph ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&acc_full[buf]);
                ++it;
            }
        }
    } else {
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int h = (warp - 2) >> 2;   // which of the quarter's EW / 4 column slices
        float alpha = ep.alpha, beta = ep.beta;
        if (ep.hp_mode) {
            float one_minus_mu, decay, scale;
            ep.hp.get(one_minus_mu, decay, scale);
            if (ep.hp_mode == 1) {
                beta = -one_minus_mu;
            } else {
                alpha = decay;
                beta = -scale;
            }
            if (blockIdx.x == 0 && warp == 2 && lane == 0 && !ep.hp.finite()) atomicOr(ep.status, kStatusNonFinite);
        }
        int it = 0;
        if constexpr (COAL == 2) {
            // bf16 addend (aux) to bf16 output (C): a lane's addends for all
            // NCH blocks of the tile (8 x 4 bf16 each) are loaded before the
            // accumulator wait, so they arrive under the tile's MMAs
            constexpr int STEP = 32 * (EW / 4), NCH = BN / STEP;
            static_assert(BN % STEP == 0, "whole 32-column blocks per epilogue warp");
            float* tb = reinterpret_cast<float*>(smem + STAGES * Cfg::STAGE_BYTES + 256) + (warp - 2) * (32 * 33);
            const bool rows_aligned = tc_coal_rows_aligned(ep);
            const int cl = 4 * (lane & 7), r8 = lane >> 3;
            for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x) {
                const int b = t / per_mat, rem = t % per_mat;
                int tm, tn;
                tc_tile_mn(ep, rem, tm, tn);
                if (!tc_tile_on(ep, b, tm, tn, Cfg::BM, BN)) continue;
                const int buf = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                ++it;
                const int row0 = tm * Cfg::BM + q * 32, colw = tn * BN + h * 32;
                const bool fast = rows_aligned && row0 + 32 <= ep.M && colw + (NCH - 1) * STEP + 32 <= ep.N;
                const long long off0 = b * ep.saux + (long long)(row0 + r8) * ep.ldaux + colw + cl;
                uint2 xs[NCH][8];
                if (fast) {
#pragma unroll
                    for (int k = 0; k < NCH; ++k)
#pragma unroll
                        for (int p = 0; p < 8; ++p)
                            xs[k][p] = *reinterpret_cast<const uint2*>(ep.aux + off0 + 4 * p * ep.ldaux + k * STEP);
                }
                if (!tc::mbar_wait(&acc_full[buf], aph, abrt, ep.status)) break;
                tc::tc_fence_after();
                const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * 32);
#pragma unroll
                for (int k = 0; k < NCH; ++k) {
                    const int col0 = colw + k * STEP;
                    tc_coal_stage(tq + k * STEP, tb, lane);
                    if (fast) {
                        const long long offc = b * ep.sc + (long long)(row0 + r8) * ep.ldc + col0 + cl;
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            float o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) o[e] = beta * tb[(4 * p + r8) * 33 + cl + e];
                            tc_coal_add_bf16x4(o, xs[k][p].x, xs[k][p].y, alpha);
                            *reinterpret_cast<uint2*>(ep.C + offc + 4 * p * ep.ldc) =
                                make_uint2(tc::pack_bf16x2(o[0], o[1]), tc::pack_bf16x2(o[2], o[3]));
                        }
                    } else if (row0 < ep.M && col0 < ep.N) {
                        tc_coal_slow(ep, b, row0, col0, tb, lane, alpha, beta);
                    }
                    __syncwarp();
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
            }
        } else if constexpr (COAL == 1) {
            // per tile, this warp's NCH blocks of 32 x 32 (columns h * 32 +
            // k * STEP), one after another: stage the block, load its
            // addends (all of a lane's loads issued together), finish it.
            // (Loading the next block's addends ahead, in a second register
            // set, measured slower: the extra loads in flight throttled the
            // load/store unit.)  tb: this warp's block, row `lane` at
            // tb[33 lane] (the padding makes both the row writes and the
            // four-rows-at-a-time reads conflict-free).
            constexpr int STEP = 32 * (EW / 4), NCH = BN / STEP;
            static_assert(BN % STEP == 0, "whole 32-column blocks per epilogue warp");
            float* tb = reinterpret_cast<float*>(smem + STAGES * Cfg::STAGE_BYTES + 256) + (warp - 2) * (32 * 33);
            const bool rows_aligned = tc_coal_rows_aligned(ep);
            for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x) {
                const int b = t / per_mat, rem = t % per_mat;
                int tm, tn;
                tc_tile_mn(ep, rem, tm, tn);
                if (!tc_tile_on(ep, b, tm, tn, Cfg::BM, BN)) continue;
                const int buf = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                ++it;
                if (!tc::mbar_wait(&acc_full[buf], aph, abrt, ep.status)) break;
                tc::tc_fence_after();
                const int row0 = tm * Cfg::BM + q * 32, colw = tn * BN + h * 32;
                const bool rows_in = rows_aligned && row0 + 32 <= ep.M;
                const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * 32);
#pragma unroll 1
                for (int k = 0; k < NCH; ++k) {
                    const int col0 = colw + k * STEP;
                    tc_coal_stage(tq + k * STEP, tb, lane);
                    if (rows_in && col0 + 32 <= ep.N) {
                        TcCoalPref pf;
                        tc_coal_prefetch(ep, b, row0, col0, lane, pf);
                        tc_coal_finish(ep, b, row0, col0, tb, lane, alpha, beta, pf);
                    } else if (row0 < ep.M && col0 < ep.N) {
                        tc_coal_slow(ep, b, row0, col0, tb, lane, alpha, beta);
                    }
                    __syncwarp();
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
            }
        } else {
        for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x) {
            const int b = t / per_mat, rem = t % per_mat;
            int tm, tn;
            tc_tile_mn(ep, rem, tm, tn);
            if (!tc_tile_on(ep, b, tm, tn, Cfg::BM, BN)) continue;
            const int buf = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            ++it;
            if (!tc::mbar_wait(&acc_full[buf], aph, abrt, ep.status)) break;
            tc::tc_fence_after();
            const int row = tm * Cfg::BM + q * 32 + lane;
#pragma unroll 1
            for (int c0 = h * 32; c0 < BN; c0 += 32 * (EW / 4)) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c0), v);
                tc::tmem_ld_wait();
                const int col0 = tn * BN + c0;
                if (row < ep.M && col0 < ep.N) tc_epi_store(ep, b, row, col0, v, alpha, beta);
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
        }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

// Launches the GEMM; tmA has boxes of 64 x 128 (K x rows), tmB of 64 x BN
// (MN: both 64 x 64, MN x K).
// COAL (1 or 2): the epilogue transposes through EW blocks of 32 x 33 floats
// placed after the stages and barriers (tc_stages() keeps as many operand
// stages as fit beside them); it serves the addends and the float32, bf16
// and three-term outputs (not CT).  COAL = 2 is the bf16 addend to bf16 output
// form (aux and C only), which loads a whole tile's addends ahead.
template <int BN, bool MN = false, int EW = 4, int COAL = 0>
cudaError_t tc_gemm(const char* name, const CUtensorMap& tmA, const CUtensorMap& tmB, int K, const TcGemmEpi& ep,
                    cudaStream_t st)
{
    using Cfg = TcGemmCfg<BN>;
    constexpr size_t smem = tc_smem<BN, EW, COAL>();
    static_assert(smem <= 232448, "shared memory per CTA");
    if (COAL && ep.CT) return cudaErrorInvalidValue;
    if (COAL == 2 && (!ep.aux || !ep.C || ep.auxf || ep.aux2 || ep.Cf || ep.Cs3)) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> attr{0};
    cudaError_t e = smem_attr_once((const void*)tc_gemm_kernel<BN, MN, EW, COAL>, (int)smem, attr);
    if (e != cudaSuccess) return e;
    const int tiles = ep.batch * ep.tiles_m * ep.tiles_n;
    const int grid = tiles < num_sms() ? tiles : num_sms();
    return launch(name, tc_gemm_kernel<BN, MN, EW, COAL>, dim3(grid), dim3(64 + 32 * EW), smem, st, tmA, tmB, K, ep);
}

}  // namespace

}  // namespace dion
