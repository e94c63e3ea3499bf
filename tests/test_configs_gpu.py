"""Full-size Dion and Newton-Schulz steps on the large workloads: the square
sweep (8 x n x n, n up to 16384, rank fractions 1/4 and 1/16), the
Llama-3-8B stack and the Llama-3-405B layer.  The oracle cannot run these
sizes, so each step is checked through properties that hold at any size,
evaluated in float64 from the GPU's own panels P and R on sampled rows and
columns:

  P^T P = I                                   (orthonormal P)
  ||Q'_j|| = 1                                (unit-norm columns of the new Q)
  Q'_j = R_j / ||R_j||                        (the new Q is R column-normalized)
  R[j, :] = sum_i B[i, j] P[i, :]             (R = B^T P, sampled columns j)
  M'[i, :] = B[i, :] - (1 - mu) P[i, :] R^T   (error feedback, sampled rows i)
  (B Q)[i, :] = P[i, :] (R^T Q)               (B Q lies in span(P); P^T B Q = R^T Q)
  X'[i, :] = (1 - lr wd) X[i, :] - lr sqrt(m/n) P[i, :] Q'^T   (sampled rows)

plus, for Newton-Schulz, that O G^T is symmetric (k steps of the iteration act
on singular values only: O = U p_k(S) V^T, so O G^T = U p_k(S) S U^T).
The same shapes are compared with the oracle itself in test_full_size_gpu.py.
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
import orthonormal_optimizer_step_gb300 as od

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2e-2


def _rel(a, b):
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


def _sample(n, k, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randperm(n, generator=g)[:min(k, n)].to(DEV)


def _check_dion_group(g, r, dtype, mu, lr, wd, g_std, seed, bi=0):
    """One full-size Dion step on group g; properties on matrix bi."""
    X, M, Q = wl.make_state(g, r, dtype, DEV, seed)
    M = wl.make_momentum(g, g_std, DEV, seed)
    G = wl.make_grad(g, g_std, dtype, DEV, seed, step=1)
    return _check_dion_tensors(g, r, dtype, X, G, M, Q, mu, lr, wd, seed, bi)


def _check_dion_tensors(g, r, dtype, X, G, M, Q, mu, lr, wd, seed, bi):
    X0, M0, Q0 = X[bi].double(), M[bi].double(), Q[bi].double()
    B = M0 + G[bi].double()
    ws = od.dion_step_batched(X, G, M, Q, mu=mu, lr=lr, weight_decay=wd)
    torch.cuda.synchronize()
    assert od.dion_get_status(ws) == 0
    dt = od.DION_BF16 if dtype == torch.bfloat16 else od.DION_F32
    Pv, Rv = od.dion_panels(ws, g.batch, g.m, g.n, r, dt)
    P, R = Pv[bi].double(), Rv[bi].double()
    out = {}
    out["orth"] = float((P.T @ P - torch.eye(r, device=DEV, dtype=torch.float64)).abs().max())
    out["qnorm"] = float((Q[bi].double().norm(dim=0) - 1).abs().max())
    out["qcol"] = float((Q[bi].double() - R / R.norm(dim=0).clamp_min(1e-30)).abs().max())
    cols = _sample(g.n, 64, seed + 1)
    rows = _sample(g.m, 64, seed + 2)
    out["R"] = _rel(R[cols], B[:, cols].T @ P)
    out["M"] = _rel(M[bi].double()[rows] - B[rows], -(1 - mu) * (P[rows] @ R.T))
    out["span"] = _rel(P[rows] @ (R.T @ Q0), B[rows] @ Q0)
    dX = X[bi].double()[rows] - (1 - lr * wd) * X0[rows]
    expect = -lr * math.sqrt(g.m / g.n) * (P[rows] @ Q[bi].double().T)
    # bf16 weights: one unit in the last place of the stored value, plus the tolerance on the update
    ulp = 2.0 ** (torch.floor(torch.log2(X[bi].double()[rows].abs().clamp_min(1e-30))) - 7)
    slack = TOL * expect.abs().max()
    out["x_ulps"] = float(((dX - expect).abs() / (ulp + slack)).max()) if dtype == torch.bfloat16 else _rel(dX, expect)
    del X, M, Q, G, ws
    torch.cuda.empty_cache()
    return out


def _assert_dion(out, dtype):
    assert out["orth"] <= 1e-3, out
    assert out["qnorm"] <= 1e-4, out
    assert out["qcol"] <= 1e-5, out
    for k in ("R", "M", "span"):
        assert out[k] <= TOL, (k, out)
    if dtype == torch.bfloat16:
        assert out["x_ulps"] <= 1.0 + 1e-9, out


@pytest.mark.parametrize("gi", [0, 1, 2, 3])
def test_llama3_8b_megabatch(gi):
    """32 layers x {4096x4096 (Q, O), 4096x1024 (K, V), 4096x14336 (gate, up),
    14336x4096 (down)}, bf16, rank fraction 1/16 (ranks 256, 64, 256, 256)."""
    w = wl.llama3_8b()
    g = w.groups[gi]
    out = _check_dion_group(g, g.rank(w.fraction), w.dtype, w.mu, w.lr, w.wd, w.g_std, seed=4000 + gi, bi=g.batch - 1)
    _assert_dion(out, w.dtype)


@pytest.mark.parametrize("gi", [0, 1, 2, 3])
def test_llama3_405b_layer(gi):
    """{16384x16384 x2, 16384x1024 x2, 16384x53248 x2, 53248x16384}, bf16,
    rank fraction 1/16 (ranks 1024, 64, 1024, 1024), Gaussian G."""
    w = wl.llama3_405b_layer()
    g = w.groups[gi]
    out = _check_dion_group(g, g.rank(w.fraction), w.dtype, w.mu, w.lr, w.wd, w.g_std, seed=5000 + gi, bi=0)
    _assert_dion(out, w.dtype)


@pytest.mark.parametrize("n", [1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("frac", [0.25, 1.0 / 16])
def test_square_sweep_dion(n, frac):
    """8 x n x n, bf16, Gaussian G and X, rank n/4 or n/16."""
    w = wl.square(n)
    g = w.groups[0]
    out = _check_dion_group(g, g.rank(frac), w.dtype, w.mu, w.lr, w.wd, w.g_std, seed=6000 + n, bi=3)
    _assert_dion(out, w.dtype)


@pytest.mark.parametrize("r", [96, 320])
def test_ill_conditioned_panel_takes_full_second_pass(r):
    """B = G with singular values 1 .. 1e-6 (geometric) and M = 0: B Q has a
    condition number in the hundreds, so after the first CholeskyQR pass
    P^T P - I is far above the near-identity threshold and the second pass
    factors in full (one CTA per matrix at rank 96, blocked at rank 320).
    P must still come out orthonormal, spanning B Q."""
    g = wl.Group(2, 1024, 768)
    gen = torch.Generator(device="cpu").manual_seed(91)
    Gs = []
    for _ in range(g.batch):
        U, _ = torch.linalg.qr(torch.randn(g.m, g.n, generator=gen, dtype=torch.float64))
        V, _ = torch.linalg.qr(torch.randn(g.n, g.n, generator=gen, dtype=torch.float64))
        s = torch.logspace(0, -6, g.n, dtype=torch.float64)
        Gs.append((U * s) @ V.T * 30.0)
    G = torch.stack(Gs).to(torch.bfloat16).to(DEV)
    X, _, Q = wl.make_state(g, r, torch.bfloat16, DEV, 91)
    M = torch.zeros(g.batch, g.m, g.n, dtype=torch.float32, device=DEV)
    out = _check_dion_tensors(g, r, torch.bfloat16, X, G, M, Q, 0.9, 0.01, 0.0, 91, 1)
    _assert_dion(out, torch.bfloat16)


def _check_ns_group(g, dtype, seed, bi=0, steps=5):
    G = wl.make_grad(g, 1.0, dtype, DEV, seed, step=0)
    O = torch.empty_like(G)
    od.muon_ns_batched(G, O=O, head_dim=g.head_dim, steps=steps)
    torch.cuda.synchronize()
    o, gg = O[bi].float(), G[bi].float()
    C = o @ gg.T if g.m <= g.n else gg.T @ o        # the smaller Gram-like product
    sym = _rel(C, C.T)
    finite = bool(torch.isfinite(O).all())
    del G, O
    torch.cuda.empty_cache()
    return sym, finite


@pytest.mark.parametrize("n", [1024, 4096, 16384])
def test_square_sweep_newton_schulz(n):
    g = wl.square(n).groups[0]
    sym, finite = _check_ns_group(g, torch.bfloat16, seed=7000 + n, bi=2)
    assert finite and sym <= TOL, sym


@pytest.mark.parametrize("gi", [0, 1, 2, 3])
def test_llama3_405b_newton_schulz(gi):
    g = wl.llama3_405b_layer().groups[gi]
    sym, finite = _check_ns_group(g, torch.bfloat16, seed=7100 + gi, bi=0)
    assert finite and sym <= TOL, sym
