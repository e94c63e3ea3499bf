// internal.h -- host-side interfaces shared by libdion's translation units.
#pragma once

#include "common.cuh"

namespace dion {

// SM count of the current device (cached per device).
int num_sms();

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
    size_t hard;            // per matrix (batch + 1 ints): the float32 first pass found an unresolved
                            // pivot; entry batch: any matrix did
    size_t S64;             // float64 Gram and inverse factor of the fallback first pass (2 batch r r doubles)
    bool wide;              // rp > 256: B formed once in bf16 (B16) for both products
    bool b16_narrow;        // rp <= 256, n % 8 == 0: the B Q pass stores bf16 B (B16) for a TMA B^T P
    size_t B16;             // bf16 B [m][round8(n)] (wide ranks), [m][n] (narrow, n % 8 == 0)
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
                         int* dead, int* status, int* hard, double* S64, cudaStream_t st);

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
    // status word of matrix b at status + b * sstride (0: one word for all)
    long long sstride;
    // if set: also raised (to 1) when any matrix reports a numeric event
    int* any;
};
// Cholesky + inverse of batch r x r Gram matrices (one CTA each); see qr.cu.
cudaError_t chol_inv(const char* name, int batch, int r, const float* Sin, int nparts, float* Swork, float* Wbuf, float* W, bf16* Z3,
                     int ldz, int* dead, int* status, cudaStream_t st, const int* emax_pre = nullptr,
                     long long sstride = 0, int* any = nullptr);
cudaError_t chol_inv_io(const char* name, int batch, int r, const float* Sin, int nparts, float* Swork, float* Wbuf,
                        float* W, bf16* Z3, int ldz, int* dead, int* status, cudaStream_t st, const int* emax_pre,
                        CholIn in);
// First CholeskyQR pass in float64 for the matrices b with hard[b] != 0 (see
// qr64.cu): P from nparts float32 partials at part (pitch rp, partial stride
// pstride); writes P L^{-T} to Pf (float32, pitch rp) and/or its three bf16
// terms to P3, the dependent-column flags to dead, and numeric events to
// status.  S64 holds 2 batch r r doubles of scratch.  hard[batch] is the
// "any matrix flagged" word: with it zero every kernel returns at once.
// With M set (tensor-core path: B Q was formed from bf16 operands), P is
// first recomputed as (M + G) Q in float64 from M, G (bf16) and Q (n x r
// float32) into the first partial of part, which the pass then reads.
bool qr64_supported(int r);
cudaError_t qr64_first_pass(int batch, int m, int r, int rp, float* part, int nparts, long long pstride,
                            double* S64, float* Pf, bf16* P3, int* dead, int* status, const int* hard,
                            cudaStream_t st, int n = 0, const float* M = nullptr, const bf16* G = nullptr,
                            const float* Q = nullptr);
// Block size of the tensor-core CholeskyQR2's factorization for rank r
// (0: one CTA per matrix, no blocking).
int chol_block_size(int r);
// CholeskyQR2 on the tensor cores (3-term bf16 splits, fp32 accuracy); see qr_tc.cu.
// M, G, Q, n: the step's inputs (B = M + G is m x n), for the float64 first
// pass of flagged matrices; Pin (the B Q partials) may be overwritten there.
// terms_ready: the B Q pass already wrote the three bf16 terms of P to P3
// (and, for the blocked factorization, P as float32 to Ptmp); Pin is unused.
cudaError_t qr_cholesky2_tc(int batch, int m, int r, int rp, float* Pin, int nparts, float* P, float* Ptmp,
                            bf16* P16, char* ws, const struct DionLayout& L, int* status, cudaStream_t st,
                            int n, const float* M, const bf16* G, const float* Q, bool terms_ready = false);

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
