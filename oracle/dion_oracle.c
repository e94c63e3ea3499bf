/*
 * dion_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU statement of the orthonormalized
 * optimizer step: the legacy Dion update (amortized power iteration with error
 * feedback at a low-rank fraction) and Muon's Newton-Schulz orthogonalization
 * (whole matrix or per attention head).  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may call it; the library's product path
 * never does.  It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (page titles; sections):
 *   [talk]  "Dion: The distributed orthonormal update revolution is here"
 *           - orthonormal update paragraph: the update direction is U V^T from
 *             the SVD G = U S V^T; Muon reaches it by Newton-Schulz iteration.
 *           - "Dion precisely answers this question" paragraph: Dion replaces
 *             Newton-Schulz by amortized power iteration, with a low-rank
 *             fraction lever and error feedback (low-rank fraction paragraph).
 *   [paper] "Dion: Distributed Orthonormalized Updates" (abstract): low-rank
 *           approximation with decoupled momentum buffers.
 *   [card]  "microsoft/dion" project card, "How it works": Dion uses power
 *           iteration for a low-rank approximation with error feedback;
 *           "Highlights": per-head Newton-Schulz for attention projections.
 *
 * The pages name the steps but print no equations.  The update written out
 * below is the legacy Dion rule for one m x n matrix at rank r:
 *     B = M + G
 *     P = orthonormalize(B Q)                (m x r, here Householder QR)
 *     R = B^T P                              (n x r)
 *     M <- B - (1 - mu) P R^T                (error feedback)
 *     Q <- R with unit-norm columns
 *     X <- (1 - lr*wd) X - lr*sqrt(m/n) P Q^T
 * Readings taken where the pages are silent (each also listed in the design
 * notes): Householder QR with diag(R_qr) >= 0; column norm floor
 * 1e-12*sqrt(n); Newton-Schulz normalizes by (||Y||_F + eps); Muon momentum is
 * heavy-ball M <- mu M + G; the per-head scale is that of the whole parameter.
 *
 * Every routine is written as the definition reads: a library-free triple loop
 * for each product, no blocking, no fusion, no reordering.  OpenMP splits the
 * outer row loop of each product only.
 *
 * All matrices are row-major, contiguous, double precision.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define AT(A, i, j, ld) ((A)[(size_t)(i) * (size_t)(ld) + (size_t)(j)])

/* C (p x q) = A (p x k) * B (k x q) */
static void mm_nn(int p, int k, int q, const double* A, const double* B, double* C)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < p; ++i) {
        for (int j = 0; j < q; ++j) AT(C, i, j, q) = 0.0;
        for (int t = 0; t < k; ++t) {
            const double a = AT(A, i, t, k);
            for (int j = 0; j < q; ++j) AT(C, i, j, q) += a * AT(B, t, j, q);
        }
    }
}

/* C (p x q) = A^T * B, with A (k x p) and B (k x q) */
static void mm_tn(int p, int k, int q, const double* A, const double* B, double* C)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < p; ++i) {
        for (int j = 0; j < q; ++j) AT(C, i, j, q) = 0.0;
        for (int t = 0; t < k; ++t) {
            const double a = AT(A, t, i, p);
            for (int j = 0; j < q; ++j) AT(C, i, j, q) += a * AT(B, t, j, q);
        }
    }
}

/* C (p x q) = A * B^T, with A (p x k) and B (q x k) */
static void mm_nt(int p, int k, int q, const double* A, const double* B, double* C)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < p; ++i) {
        for (int j = 0; j < q; ++j) {
            double s = 0.0;
            for (int t = 0; t < k; ++t) s += AT(A, i, t, k) * AT(B, j, t, k);
            AT(C, i, j, q) = s;
        }
    }
}

/*
 * Householder QR of A (m x r, m >= r).  On return A holds the thin factor Qf
 * (m x r, orthonormal columns) and, if Rq is not NULL, Rq holds the r x r upper
 * triangular factor, with A_in = Qf * Rq and diag(Rq) >= 0.  A zero column
 * (rank deficiency) gives a zero reflector, a zero diagonal entry of Rq and
 * still an orthonormal column of Qf.  Returns 0, or -1 on bad arguments.
 */
int oracle_householder_qr(int m, int r, double* A, double* Rq)
{
    if (m <= 0 || r <= 0 || r > m || !A) return -1;
    double* W = (double*)malloc(sizeof(double) * (size_t)m * r);   /* becomes R */
    double* V = (double*)calloc((size_t)m * r, sizeof(double));     /* reflectors */
    double* tau = (double*)calloc((size_t)r, sizeof(double));
    double* E = (double*)calloc((size_t)m * r, sizeof(double));     /* becomes Qf */
    if (!W || !V || !tau || !E) { free(W); free(V); free(tau); free(E); return -1; }
    memcpy(W, A, sizeof(double) * (size_t)m * r);

    for (int k = 0; k < r; ++k) {
        double nrm2 = 0.0;
        for (int i = k; i < m; ++i) nrm2 += AT(W, i, k, r) * AT(W, i, k, r);
        const double nrm = sqrt(nrm2);
        if (nrm == 0.0) { tau[k] = 0.0; continue; }          /* H_k = I */
        const double alpha = (AT(W, k, k, r) >= 0.0) ? -nrm : nrm;
        double vv = 0.0;
        for (int i = k; i < m; ++i) {
            double v = AT(W, i, k, r) - (i == k ? alpha : 0.0);
            AT(V, i, k, r) = v;
            vv += v * v;
        }
        tau[k] = (vv > 0.0) ? 2.0 / vv : 0.0;
        /* W[k:, k:] <- (I - tau v v^T) W[k:, k:] */
        for (int j = k; j < r; ++j) {
            double s = 0.0;
            for (int i = k; i < m; ++i) s += AT(V, i, k, r) * AT(W, i, j, r);
            s *= tau[k];
            for (int i = k; i < m; ++i) AT(W, i, j, r) -= s * AT(V, i, k, r);
        }
    }

    /* Qf = H_0 H_1 ... H_{r-1} [I_r; 0] */
    for (int i = 0; i < r; ++i) AT(E, i, i, r) = 1.0;
    for (int k = r - 1; k >= 0; --k) {
        if (tau[k] == 0.0) continue;
        for (int j = 0; j < r; ++j) {
            double s = 0.0;
            for (int i = k; i < m; ++i) s += AT(V, i, k, r) * AT(E, i, j, r);
            s *= tau[k];
            for (int i = k; i < m; ++i) AT(E, i, j, r) -= s * AT(V, i, k, r);
        }
    }

    /* Sign convention: diag(Rq) >= 0.  Flip column k of Qf and row k of R. */
    for (int k = 0; k < r; ++k) {
        if (AT(W, k, k, r) < 0.0) {
            for (int i = 0; i < m; ++i) AT(E, i, k, r) = -AT(E, i, k, r);
            for (int j = k; j < r; ++j) AT(W, k, j, r) = -AT(W, k, j, r);
        }
    }
    memcpy(A, E, sizeof(double) * (size_t)m * r);
    if (Rq) {
        for (int i = 0; i < r; ++i)
            for (int j = 0; j < r; ++j) AT(Rq, i, j, r) = (j >= i) ? AT(W, i, j, r) : 0.0;
    }
    free(W); free(V); free(tau); free(E);
    return 0;
}

/*
 * One Dion step on one m x n matrix at rank r (1 <= r <= min(m, n)).
 *   X (m x n, in/out)  weights             G (m x n, in)   gradient
 *   M (m x n, in/out)  momentum buffer     Q (n x r, in/out) right factor
 *   P_out (m x r) and R_out (n x r): optional copies of this step's P and R.
 * The steps follow the order of the power-iteration update ([talk], Dion
 * paragraphs; [card], "How it works").  Returns 0, or -1 on bad arguments.
 */
int oracle_dion_step(int m, int n, int r, double* X, const double* G, double* M, double* Q,
                     double mu, double lr, double wd, double* P_out, double* R_out)
{
    if (m <= 0 || n <= 0 || r <= 0 || r > m || r > n || !X || !G || !M || !Q) return -1;
    const size_t mn = (size_t)m * n;
    double* B = (double*)malloc(sizeof(double) * mn);
    double* P = (double*)malloc(sizeof(double) * (size_t)m * r);
    double* R = (double*)malloc(sizeof(double) * (size_t)n * r);
    double* PRt = (double*)malloc(sizeof(double) * mn);
    double* PQt = (double*)malloc(sizeof(double) * mn);
    if (!B || !P || !R || !PRt || !PQt) { free(B); free(P); free(R); free(PRt); free(PQt); return -1; }

    /* B = M + G */
    for (size_t e = 0; e < mn; ++e) B[e] = M[e] + G[e];
    /* P = B Q, then orthonormalize P */
    mm_nn(m, n, r, B, Q, P);
    oracle_householder_qr(m, r, P, NULL);
    /* R = B^T P */
    mm_tn(n, m, r, B, P, R);
    /* M <- B - (1 - mu) P R^T */
    mm_nt(m, r, n, P, R, PRt);
    for (size_t e = 0; e < mn; ++e) M[e] = B[e] - (1.0 - mu) * PRt[e];
    /* Q <- column-normalized R */
    const double floor_nrm = 1e-12 * sqrt((double)n);
    for (int j = 0; j < r; ++j) {
        double s = 0.0;
        for (int i = 0; i < n; ++i) s += AT(R, i, j, r) * AT(R, i, j, r);
        double nrm = sqrt(s);
        if (nrm < floor_nrm) nrm = floor_nrm;
        for (int i = 0; i < n; ++i) AT(Q, i, j, r) = AT(R, i, j, r) / nrm;
    }
    /* X <- (1 - lr wd) X - lr sqrt(m/n) P Q^T */
    mm_nt(m, r, n, P, Q, PQt);
    const double decay = 1.0 - lr * wd;
    const double scale = lr * sqrt((double)m / (double)n);
    for (size_t e = 0; e < mn; ++e) X[e] = decay * X[e] - scale * PQt[e];

    if (P_out) memcpy(P_out, P, sizeof(double) * (size_t)m * r);
    if (R_out) memcpy(R_out, R, sizeof(double) * (size_t)n * r);
    free(B); free(P); free(R); free(PRt); free(PQt);
    return 0;
}

/*
 * Newton-Schulz orthogonalization of one m x n matrix ([talk], orthonormal
 * update paragraph: Muon approximates U V^T by iterated matrix products).
 *   Y = Yin, transposed first when m > n so that the Gram matrix is the
 *   smaller one; Y <- Y / (||Y||_F + eps); then `steps` times
 *       A = Y Y^T,  Y <- a Y + (b A + c A A) Y;
 *   O = Y, transposed back.  O and Yin are m x n.  Returns 0 or -1.
 */
int oracle_newton_schulz(int m, int n, int steps, double a, double b, double c, double eps,
                         const double* Yin, double* O)
{
    if (m <= 0 || n <= 0 || steps < 0 || !Yin || !O) return -1;
    const int tr = m > n;
    const int s = tr ? n : m, l = tr ? m : n;
    double* Y = (double*)malloc(sizeof(double) * (size_t)s * l);
    double* Yn = (double*)malloc(sizeof(double) * (size_t)s * l);
    double* A = (double*)malloc(sizeof(double) * (size_t)s * s);
    double* AA = (double*)malloc(sizeof(double) * (size_t)s * s);
    double* Bm = (double*)malloc(sizeof(double) * (size_t)s * s);
    if (!Y || !Yn || !A || !AA || !Bm) { free(Y); free(Yn); free(A); free(AA); free(Bm); return -1; }

    for (int i = 0; i < s; ++i)
        for (int j = 0; j < l; ++j) AT(Y, i, j, l) = tr ? AT(Yin, j, i, n) : AT(Yin, i, j, n);
    double fro2 = 0.0;
    for (size_t e = 0; e < (size_t)s * l; ++e) fro2 += Y[e] * Y[e];
    const double inv = 1.0 / (sqrt(fro2) + eps);
    for (size_t e = 0; e < (size_t)s * l; ++e) Y[e] *= inv;

    for (int k = 0; k < steps; ++k) {
        mm_nt(s, l, s, Y, Y, A);                 /* A = Y Y^T */
        mm_nn(s, s, s, A, A, AA);                /* A A */
        for (size_t e = 0; e < (size_t)s * s; ++e) Bm[e] = b * A[e] + c * AA[e];
        mm_nn(s, s, l, Bm, Y, Yn);               /* (b A + c A A) Y */
        for (size_t e = 0; e < (size_t)s * l; ++e) Y[e] = a * Y[e] + Yn[e];
    }
    for (int i = 0; i < m; ++i)
        for (int j = 0; j < n; ++j) AT(O, i, j, n) = tr ? AT(Y, j, i, l) : AT(Y, i, j, l);
    free(Y); free(Yn); free(A); free(AA); free(Bm);
    return 0;
}

/*
 * One Muon step on one m x n parameter.
 *   M (nullable): heavy-ball momentum, M <- mu M + G, and Y = M; else Y = G.
 *   head_dim = 0: Newton-Schulz on the whole Y.  head_dim > 0 (n % head_dim
 *   == 0): Newton-Schulz on each m x head_dim column block separately, so
 *   that heads are not blended ([card], "Highlights", per-head handling).
 *   O (nullable): receives the orthogonalized m x n update.
 *   X (nullable): X <- (1 - lr wd) X - lr sqrt(m/n) O, with m, n the
 *   parameter's own shape.
 * Returns 0 or -1.
 */
int oracle_muon_step(int m, int n, int head_dim, int steps, double a, double b, double c,
                     double eps, double* X, const double* G, double* M, double* O,
                     double mu, double lr, double wd)
{
    if (m <= 0 || n <= 0 || !G || head_dim < 0) return -1;
    if (head_dim > 0 && n % head_dim != 0) return -1;
    const size_t mn = (size_t)m * n;
    double* Y = (double*)malloc(sizeof(double) * mn);
    double* U = (double*)malloc(sizeof(double) * mn);
    if (!Y || !U) { free(Y); free(U); return -1; }
    if (M) {
        for (size_t e = 0; e < mn; ++e) M[e] = mu * M[e] + G[e];
        memcpy(Y, M, sizeof(double) * mn);
    } else {
        memcpy(Y, G, sizeof(double) * mn);
    }
    int rc = 0;
    if (head_dim == 0) {
        rc = oracle_newton_schulz(m, n, steps, a, b, c, eps, Y, U);
    } else {
        const int hd = head_dim;
        double* blk = (double*)malloc(sizeof(double) * (size_t)m * hd);
        double* out = (double*)malloc(sizeof(double) * (size_t)m * hd);
        if (!blk || !out) { free(blk); free(out); free(Y); free(U); return -1; }
        for (int h = 0; h < n / hd && rc == 0; ++h) {
            for (int i = 0; i < m; ++i)
                for (int j = 0; j < hd; ++j) AT(blk, i, j, hd) = AT(Y, i, h * hd + j, n);
            rc = oracle_newton_schulz(m, hd, steps, a, b, c, eps, blk, out);
            for (int i = 0; i < m; ++i)
                for (int j = 0; j < hd; ++j) AT(U, i, h * hd + j, n) = AT(out, i, j, hd);
        }
        free(blk); free(out);
    }
    if (rc == 0 && O) memcpy(O, U, sizeof(double) * mn);
    if (rc == 0 && X) {
        const double decay = 1.0 - lr * wd;
        const double scale = lr * sqrt((double)m / (double)n);
        for (size_t e = 0; e < mn; ++e) X[e] = decay * X[e] - scale * U[e];
    }
    free(Y); free(U);
    return rc;
}
