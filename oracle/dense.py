"""Dense-library form of the oracle -- TEST INFRASTRUCTURE ONLY.

The same update rules as ``dion_oracle.c``, in float64, with two library
primitives as steps: numpy's matrix product and LAPACK's Householder QR
(``numpy.linalg.qr``).  Nothing is blocked, fused or reordered beyond what the
rules state; each line below is one step of the rule.  This form exists so
that the full-size workloads (matrices up to 53248 x 16384) can be checked
against the oracle in seconds, where the triple loops of the C form take hours.
Both forms are pinned by the same tests (``tests/test_oracle.py``), and a
test checks that they agree with each other.

Only ``tests/``, the smoke check and the benchmark's CPU-baseline leg may
import this module.  It imports nothing from the CUDA library.

Sources: "Dion: The distributed orthonormal update revolution is here" (talk
page, orthonormal-update and Dion paragraphs), "Dion: Distributed
Orthonormalized Updates" (abstract), "microsoft/dion" project card ("How it
works", "Highlights").  The step order and the readings where the pages are
silent (Householder QR with diag(R_qr) >= 0, column-norm floor
1e-12 sqrt(n), Newton-Schulz normalization by ||Y||_F + eps, heavy-ball Muon
momentum, whole-parameter scale in per-head mode) are those of the C form.
"""
from __future__ import annotations

import numpy as np

QUINTIC = (3.4445, -4.7750, 2.0315)
NS_EPS = 1e-7


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def householder_qr(A):
    """Thin QR by Householder reflections (LAPACK), signs fixed so that
    diag(Rq) >= 0: returns (Qf, Rq) with A = Qf Rq."""
    Qf, Rq = np.linalg.qr(_f64(A), mode="reduced")
    s = np.where(np.diag(Rq) < 0.0, -1.0, 1.0)
    return Qf * s, Rq * s[:, None]


def dion_step(X, G, M, Q, mu, lr, wd):
    """One Dion step on one m x n matrix at rank r = Q.shape[1] (float64).
    Returns a dict with the new X, M, Q and this step's P (m x r) and
    R (n x r); the inputs are not modified."""
    X, G, M, Q = _f64(X), _f64(G), _f64(M), _f64(Q)
    m, n = X.shape
    r = Q.shape[1]
    if not (1 <= r <= min(m, n)) or G.shape != (m, n) or M.shape != (m, n) or Q.shape[0] != n:
        raise ValueError("dense.dion_step: bad shapes")
    B = M + G                                    # B = M + G
    P, _ = householder_qr(B @ Q)                 # P = orthonormalize(B Q)
    R = B.T @ P                                  # R = B^T P
    M_new = B - (1.0 - mu) * (P @ R.T)           # M <- B - (1 - mu) P R^T
    nrm = np.maximum(np.linalg.norm(R, axis=0), 1e-12 * np.sqrt(n))
    Q_new = R / nrm                              # Q <- R with unit-norm columns
    X_new = (1.0 - lr * wd) * X - (lr * np.sqrt(m / n)) * (P @ Q_new.T)
    return {"X": X_new, "M": M_new, "Q": Q_new, "P": P, "R": R}


def newton_schulz(Y, steps=5, coeff=QUINTIC, eps=NS_EPS):
    """Newton-Schulz orthogonalization of one matrix (float64): transposed
    when taller than wide, Y <- Y / (||Y||_F + eps), then `steps` times
    A = Y Y^T, Y <- a Y + (b A + c A A) Y; transposed back."""
    Y = _f64(Y)
    tr = Y.shape[0] > Y.shape[1]
    if tr:
        Y = Y.T
    Y = Y / (np.linalg.norm(Y) + eps)
    a, b, c = coeff
    for _ in range(int(steps)):
        A = Y @ Y.T
        Bm = b * A + c * (A @ A)
        Y = a * Y + Bm @ Y
    return np.ascontiguousarray(Y.T if tr else Y)


def muon_step(X, G, M, *, head_dim=0, steps=5, coeff=QUINTIC, eps=NS_EPS, mu=0.95, lr=0.02, wd=0.0):
    """One Muon step on one m x n parameter (float64).  M (nullable):
    heavy-ball momentum M <- mu M + G, and Newton-Schulz acts on it; else on G.
    head_dim > 0: each m x head_dim column block separately.  X (nullable):
    X <- (1 - lr wd) X - lr sqrt(m/n) O.  Returns a dict with O and the new X
    and M (None where the input was None)."""
    G = _f64(G)
    m, n = G.shape
    if head_dim < 0 or (head_dim > 0 and n % head_dim != 0):
        raise ValueError("dense.muon_step: bad head_dim")
    M_new = None if M is None else mu * _f64(M) + G
    Y = G if M_new is None else M_new
    if head_dim == 0:
        O = newton_schulz(Y, steps, coeff, eps)
    else:
        O = np.concatenate([newton_schulz(Y[:, h:h + head_dim], steps, coeff, eps)
                            for h in range(0, n, head_dim)], axis=1)
    X_new = None if X is None else (1.0 - lr * wd) * _f64(X) - (lr * np.sqrt(m / n)) * O
    return {"O": O, "X": X_new, "M": M_new}


def newton_schulz_rows(Y, rows, steps=5, coeff=QUINTIC, eps=NS_EPS):
    """Rows `rows` of newton_schulz(Y), computed without forming the other rows.

    With Y0 the normalized short-side matrix (s x l) and A_k = Y_k Y_k^T, each
    step is Y_{k+1} = p(A_k) Y_k with p(x) = a + b x + c x^2, so
    A_{k+1} = A_k p(A_k)^2, every A_k is a polynomial in A_0 (they commute),
    and the result is p(A_{K-1}) ... p(A_0) Y0.  A product with A_k is
    evaluated through that recursion (one product with A_k costs five with
    A_{k-1}), on a few vectors at a time: each step of the iteration applied
    as written, to the sampled rows (short side) or columns (long side) only.
    Cost: one s x s Gram matrix plus 2 (1 + 5 + ... + 5^(K-1)) products of it
    with a thin block."""
    Y = _f64(Y)
    m, n = Y.shape
    rows = np.asarray(rows, dtype=np.int64)
    tr = m > n
    Y0 = Y.T if tr else Y                       # s x l, s = min(m, n)
    Y0 = Y0 / (np.linalg.norm(Y0) + eps)
    A0 = Y0 @ Y0.T
    a, b, c = coeff

    def apply_A(k, V):                          # A_k V
        if k == 0:
            return A0 @ V
        return apply_A(k - 1, apply_p(k - 1, apply_p(k - 1, V)))

    def apply_p(k, V):                          # p(A_k) V
        AV = apply_A(k, V)
        return a * V + b * AV + c * apply_A(k, AV)

    if tr:
        # rows of O are columns of the final s x l iterate: p-chain on Y0's columns
        V = np.ascontiguousarray(Y0[:, rows])
        for k in range(int(steps)):
            V = apply_p(k, V)
        return np.ascontiguousarray(V.T)
    # rows of O are rows of the final iterate: (p-chain e_i)^T Y0 (symmetric, commuting factors)
    E = np.zeros((Y0.shape[0], rows.size))
    E[rows, np.arange(rows.size)] = 1.0
    for k in range(int(steps)):
        E = apply_p(k, E)
    return np.ascontiguousarray(E.T @ Y0)
