// internal.h -- host-side interfaces shared by libdion's translation units.
#pragma once

#include "common.cuh"

namespace dion {

// Workspace layout of dion_step_batched (byte offsets, each 256-aligned).
struct DionLayout {
    int rp;                 // r rounded up to 64 on the tensor-core path (== r on the fp32 path)
    bool tc;                // tensor-core (bf16) path
    int ksplit;             // splits of the B Q contraction over n (partials in Ppart)
    int ksplit_r;           // splits of the B^T P contraction over m
    size_t status, P0, P1, R, S, W, dead, inv, Ppart, Qt16, P16, R16, Q16;
    size_t P3, P3b, Z3, S6; // CholeskyQR2 operands of the tensor-core path (P3, P3b: bf16 terms of the panel)
    size_t normp;           // per-chunk column sums of squares of R
    size_t rcount;          // per matrix arrival counter of the column-norm reduction
    size_t emax;            // per matrix max|S - I| of the second CholeskyQR Gram
    int nbc;                // block size of the blocked Cholesky (0: one CTA per matrix)
    size_t ZJ, A3;          // its diagonal-block inverse and panel terms
    bool wide;              // rp > 256: B formed once in bf16 for both products
    size_t B16, B16T, P16T; // bf16 B [m][round8(n)], B^T [n][round8(m)], P^T [rp][round8(m)]
    size_t total;
};
DionLayout dion_layout(int batch, int m, int n, int r, dion_dtype dt);

// Workspace layout of muon_ns_batched.
struct MuonLayout {
    int heads, hd, s, l, nb;   // blocks per matrix, block width, Gram side, long side, total blocks
    bool tr, tc;               // blocks transposed (m > hd); tensor-core path
    int lp, sp;                // row pitches (elements) of the bf16 s x l and s x s buffers
    size_t status, nrm, Xa, Xb, XTa, XTb, A, Bm, total;
};
MuonLayout muon_layout(int batch, int m, int n, int head_dim, dion_dtype dt);

// CholeskyQR2 of `batch` m x r float panels, in place in P (Ptmp is scratch of
// the same size).  S, W: batch*r*r floats; dead: batch*r ints.
cudaError_t qr_cholesky2(int batch, int m, int r, long long ldp, float* P, float* Ptmp, float* S, float* W,
                         int* dead, int* status, cudaStream_t st);

// Where the Gram matrices of chol_inv_io are read: matrix b starts at
// Sin + b * mstride, its partial q at + q * pstride, row i at + i * lds;
// dependent-column flags of matrix b at dead + b * dstride.
struct CholIn {
    long long mstride, pstride;
    int lds;
    long long dstride;
    // lds == 0 (factorization kernel for r <= 248, one partial only): the
    // lower triangle is stored block-major, 8 x 8 block t = bi (bi + 1) / 2 + bj
    // at Sin + b * mstride + 64 t, row-major inside the block (as written by
    // qr_gram_sum_blocks)
    // d0 (optional): the reference diagonal of the dependent-column test,
    // d0[b * d0stride + j], when the matrix factored is a Schur complement
    // (a diagonal block of the blocked factorization): a column is dependent
    // when its pivot is at most 1e-6 of its original squared norm
    const float* d0;
    long long d0stride;
};
// Cholesky + inverse of batch r x r Gram matrices (one CTA each); see qr.cu.
cudaError_t chol_inv(const char* name, int batch, int r, const float* Sin, int nparts, float* Swork, float* Wbuf, float* W, bf16* Z3,
                     int ldz, int* dead, int* status, cudaStream_t st, const int* emax_pre = nullptr);
cudaError_t chol_inv_io(const char* name, int batch, int r, const float* Sin, int nparts, float* Swork, float* Wbuf,
                        float* W, bf16* Z3, int ldz, int* dead, int* status, cudaStream_t st, const int* emax_pre,
                        CholIn in);
// Block size of the tensor-core CholeskyQR2's factorization for rank r
// (0: one CTA per matrix, no blocking).
int chol_block_size(int r);
// CholeskyQR2 on the tensor cores (3-term bf16 splits, fp32 accuracy); see qr_tc.cu.
cudaError_t qr_cholesky2_tc(int batch, int m, int r, int rp, const float* Pin, int nparts, float* P, float* Ptmp,
                            bf16* P16, char* ws, const struct DionLayout& L, int* status, cudaStream_t st);

dion_status dion_step_simt(int batch, int m, int n, int r, dion_dtype dt, void* X, const void* G, float* M,
                           float* Q, float mu, float lr, float wd, const float* hyper, char* ws, const DionLayout& L,
                           cudaStream_t st);
dion_status dion_step_tc(int batch, int m, int n, int r, void* X, const void* G, float* M, float* Q, float mu,
                         float lr, float wd, const float* hyper, char* ws, const DionLayout& L, cudaStream_t st);
dion_status muon_tc(int batch, int m, int n, dion_dtype dt, void* X, const void* G, float* M, void* O, int steps,
                    const float* coeff, float mu, float lr, float wd, char* ws, const MuonLayout& L,
                    cudaStream_t st);
dion_status muon_simt(int batch, int m, int n, dion_dtype dt, void* X, const void* G, float* M, void* O,
                      int steps, const float* coeff, float mu, float lr, float wd, char* ws,
                      const MuonLayout& L, cudaStream_t st);

}  // namespace dion
