// simt_gemm.cuh -- a batched float32 CUDA-core GEMM with pluggable operand
// loaders and epilogues.  It serves the float32 storage path, where the 1e-4
// relative tolerance rules out bf16/tf32 tensor-core operands, and the small
// r x r products of the orthonormalization.
//
//   C[b](i, j) = sum_k A[b](i, k) * B[b](k, j)      (and a second product
//                                                    with B2 when NACC == 2)
// A loader: float operator()(b, i, k); kKContig says whether k is the
// contiguous index in memory (chooses the coalesced load order).
// B loader: float operator()(b, k, j); kJContig likewise for j.
// Epilogue: void operator()(b, i, j, acc0, acc1), called once per output.
#pragma once

#include "common.cuh"

namespace dion {

// A(i, k) = p[b*sb + i*ld + k]  (KC) or p[b*sb + k*ld + i]  (!KC)
template <typename T, bool KC>
struct LdA {
    const T* p; long long sb; long long ld;
    static constexpr bool kKContig = KC;
    __device__ __forceinline__ float operator()(int b, int i, int k) const {
        return to_f(KC ? p[b * sb + i * ld + k] : p[b * sb + k * ld + i]);
    }
};

// A(i, k) = p1[...] + p2[...], same indexing as LdA (forms B = M + G on the fly)
template <typename T1, typename T2, bool KC>
struct LdSum {
    const T1* p1; const T2* p2; long long sb; long long ld;
    static constexpr bool kKContig = KC;
    __device__ __forceinline__ float operator()(int b, int i, int k) const {
        const long long o = KC ? b * sb + i * ld + k : b * sb + k * ld + i;
        return to_f(p1[o]) + to_f(p2[o]);
    }
};

// B(k, j) = p[b*sb + k*ld + j]  (JC) or p[b*sb + j*ld + k]  (!JC)
template <typename T, bool JC>
struct LdB {
    const T* p; long long sb; long long ld;
    static constexpr bool kJContig = JC;
    __device__ __forceinline__ float operator()(int b, int k, int j) const {
        return to_f(JC ? p[b * sb + k * ld + j] : p[b * sb + j * ld + k]);
    }
};

struct EpStore {
    float* c; long long sb; long long ld;
    __device__ __forceinline__ void operator()(int b, int i, int j, float v, float) const {
        c[b * sb + i * ld + j] = v;
    }
};

// Kernels defined in this header get internal linkage (one copy per
// translation unit).
namespace {

template <int NACC, class AL, class BL, class BL2, class EP>
__global__ void __launch_bounds__(256) gemm_simt_kernel(int Md, int Nd, int Kd, AL al, BL bl, BL2 bl2, EP ep)
{
    constexpr int TM = 64, TN = 64, TK = 16;
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs[NACC][TK][TN + 4];
    const int b = blockIdx.z;
    const int i0 = blockIdx.y * TM, j0 = blockIdx.x * TN;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float acc[NACC][4][4];
#pragma unroll
    for (int a = 0; a < NACC; ++a)
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[a][p][q] = 0.f;

    for (int k0 = 0; k0 < Kd; k0 += TK) {
#pragma unroll
        for (int e = tid; e < TM * TK; e += 256) {
            int ii, kk;
            if (AL::kKContig) { kk = e % TK; ii = e / TK; } else { ii = e % TM; kk = e / TM; }
            const int i = i0 + ii, k = k0 + kk;
            As[kk][ii] = (i < Md && k < Kd) ? al(b, i, k) : 0.f;
        }
#pragma unroll
        for (int e = tid; e < TN * TK; e += 256) {
            int jj, kk;
            if (BL::kJContig) { jj = e % TN; kk = e / TN; } else { kk = e % TK; jj = e / TK; }
            const int j = j0 + jj, k = k0 + kk;
            const bool in = (j < Nd && k < Kd);
            Bs[0][kk][jj] = in ? bl(b, k, j) : 0.f;
            if constexpr (NACC == 2) Bs[NACC - 1][kk][jj] = in ? bl2(b, k, j) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            float av[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) av[p] = As[kk][ty * 4 + p];
#pragma unroll
            for (int a = 0; a < NACC; ++a) {
                float bv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) bv[q] = Bs[a][kk][tx * 4 + q];
#pragma unroll
                for (int p = 0; p < 4; ++p)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][p][q] = fmaf(av[p], bv[q], acc[a][p][q]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = i0 + ty * 4 + p, j = j0 + tx * 4 + q;
            if (i < Md && j < Nd) ep(b, i, j, acc[0][p][q], acc[NACC - 1][p][q]);
        }
}

template <int NACC, class AL, class BL, class BL2, class EP>
cudaError_t gemm_simt(const char* name, int batch, int Md, int Nd, int Kd, AL al, BL bl, BL2 bl2, EP ep,
                      cudaStream_t st)
{
    dim3 grid((unsigned)cdiv(Nd, 64), (unsigned)cdiv(Md, 64), (unsigned)batch);
    return launch(name, gemm_simt_kernel<NACC, AL, BL, BL2, EP>, grid, dim3(256), 0, st, Md, Nd, Kd, al, bl, bl2, ep);
}

}  // namespace

}  // namespace dion
