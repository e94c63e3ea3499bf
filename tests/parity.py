"""Helpers for GPU-vs-oracle parity: teacher-forced steps and comparisons.

Tolerances (relative Frobenius error per step): 1e-4 for float32 storage,
2e-2 for bfloat16 storage; orthonormality ||P^T P - I||_max <= 1e-3.
"""
import numpy as np
import torch

import oracle
import orthonormal_optimizer_step_gb300 as od

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
ORTH_TOL = 1e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def rel(a, b) -> float:
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def sign_align(A, B):
    """Flip the columns of A to agree in sign with B (columns are unique only
    up to sign)."""
    s = np.sign(np.sum(A * B, axis=0))
    s[s == 0] = 1.0
    return A * s


def storage_round(x, dtype):
    return oracle.round_bf16(x) if dtype == torch.bfloat16 else oracle.round_f32(x)


def rel_outer(A, B, C, D) -> float:
    """||A B^T - C D^T||_F / ||C D^T||_F from r x r products only:
    ||A B^T - C D^T||_F^2 = <A^T A, B^T B> - 2 <A^T C, B^T D> + <C^T C, D^T D>."""
    aa, bb, cc, dd = A.T @ A, B.T @ B, C.T @ C, D.T @ D
    num = np.sum(aa * bb) - 2.0 * np.sum((A.T @ C) * (B.T @ D)) + np.sum(cc * dd)
    den = np.sum(cc * dd)
    return float(np.sqrt(max(num, 0.0) / (den if den > 0 else 1.0)))


def dion_snapshot(X, G, M, Q, samples=None):
    """float64 host copies of the state of the sampled matrices (default: all)."""
    idx = list(range(X.shape[0])) if samples is None else list(samples)
    return idx, {k: f64(t[idx]) for k, t in (("X", X), ("G", G), ("M", M), ("Q", Q))}


def dion_pair(X, G, M, Q, mu, lr, wd, samples=None, form=oracle):
    """Run one GPU Dion step (in place on X, M, Q) and the oracle on copies of
    the same state for the matrices in `samples` (default: all).  `form` is
    the oracle form (the C triple loops, or oracle.dense for full-size
    matrices).  Returns a dict of per-quantity worst relative errors and the
    GPU status."""
    idx, host = dion_snapshot(X, G, M, Q, samples)
    ws = od.dion_step_batched(X, G, M, Q, mu=mu, lr=lr, weight_decay=wd)
    torch.cuda.synchronize()
    return dion_compare(idx, host, X, M, Q, ws, mu, lr, wd, form)


def dion_compare(idx, host, X, M, Q, ws, mu, lr, wd, form=oracle):
    """Compares the GPU state after a completed step (X, M, Q and the panels P,
    R left in the workspace ws) with the oracle run from the snapshot `host`."""
    batch, m, n = X.shape
    r = Q.shape[-1]
    dt = X.dtype
    status = od.dion_get_status(ws)
    P_gpu, R_gpu = od.dion_panels(ws, batch, m, n, r, od.DION_BF16 if dt == torch.bfloat16 else od.DION_F32)
    out = {"M": 0.0, "Q": 0.0, "X": 0.0, "PQt": 0.0, "orth": 0.0, "R": 0.0, "x_ulps": 0.0, "qcol": 0.0}
    for k, b in enumerate(idx):
        o = form.dion_step(host["X"][k], host["G"][k], host["M"][k], host["Q"][k], mu, lr, wd)
        Pg, Rg, Qg = f64(P_gpu[b]), f64(R_gpu[b]), f64(Q[b])
        out["M"] = max(out["M"], rel(f64(M[b]), o["M"]))
        out["Q"] = max(out["Q"], rel(sign_align(Qg, o["Q"]), o["Q"]))
        out["R"] = max(out["R"], rel(sign_align(Rg, o["R"]), o["R"]))
        out["PQt"] = max(out["PQt"], rel_outer(Pg, Qg, o["P"], o["Q"]))
        out["orth"] = max(out["orth"], float(np.abs(Pg.T @ Pg - np.eye(r)).max()))
        # the GPU's own Q' is its own R with unit-norm columns (zero columns stay zero)
        nr = np.linalg.norm(Rg, axis=0)
        out["qcol"] = max(out["qcol"], float(np.abs(Qg - Rg / np.where(nr > 0, nr, 1.0)).max()))
        x0 = host["X"][k]
        Xg = f64(X[b])
        dX_exact_max = float(np.abs(o["X"] - x0).max())
        Xo = storage_round(o["X"], dt)
        del o
        out["X"] = max(out["X"], rel(Xg - x0, Xo - x0))
        if dt == torch.bfloat16:
            out["x_ulps"] = max(out["x_ulps"], max_ulps(Xg, Xo, TOL[dt] * dX_exact_max))
        del Xg, Xo
    out["status"] = status
    return out


def max_ulps(Xg, Xo, slack, rows=4096):
    """max |Xg - Xo| / (ulp + slack) over all elements, in row blocks.  ulp is
    one bfloat16 unit in the last place of the larger of the two stored
    values; slack is the tolerated error of the unrounded update (the
    relative tolerance times the largest update entry): two fp32 values that
    differ by d round to bf16 values at most d plus one unit apart."""
    worst = 0.0
    for i in range(0, Xg.shape[0], rows):
        g, o = Xg[i:i + rows], Xo[i:i + rows]
        mag = np.maximum(np.maximum(np.abs(o), np.abs(g)), 1e-30)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
        worst = max(worst, float(np.max(np.abs(g - o) / (ulp + slack))))
    return worst


def muon_pair(G, M, X, head_dim, steps, coeff, mu, lr, wd, samples=None, form=oracle):
    """One GPU Newton-Schulz step on the whole megabatch and the oracle (`form`)
    on the sampled matrices; worst relative errors of O, M and the change of X."""
    batch, m, n = G.shape
    dt = G.dtype
    idx = list(range(batch)) if samples is None else list(samples)
    hG = f64(G[idx])
    hM = None if M is None else f64(M[idx])
    hX = None if X is None else f64(X[idx])
    O = torch.empty_like(G)
    ws = od.muon_ns_batched(G, X=X, M=M, O=O, head_dim=head_dim, steps=steps, coeff=coeff, mu=mu, lr=lr,
                            weight_decay=wd)
    torch.cuda.synchronize()
    out = {"O": 0.0, "M": 0.0, "X": 0.0}
    for k, b in enumerate(idx):
        o = form.muon_step(None if hX is None else hX[k], hG[k], None if hM is None else hM[k],
                             head_dim=head_dim, steps=steps, coeff=coeff, mu=mu, lr=lr, wd=wd)
        out["O"] = max(out["O"], rel(f64(O[b]), o["O"]))
        if M is not None:
            out["M"] = max(out["M"], rel(f64(M[b]), o["M"]))
        if X is not None:
            dX_o = storage_round(o["X"], dt) - hX[k]
            out["X"] = max(out["X"], rel(f64(X[b]) - hX[k], dX_o))
    out["status"] = od.dion_get_status(ws)
    return out
