"""Oracle parity at full size, teacher-forced.

Every shape of the large workloads -- the square-matrix sweep (8 x n x n,
n = 1024 ... 16384, rank fractions 1/4 and 1/16), the Llama-3-8B stack and
the Llama-3-405B layer ("Dion: The distributed orthonormal update revolution
is here": the square-matrix microbenchmark at fractions 1/4 and 1/16 and the
Llama 3 405B configuration) -- takes one Dion step on the GPU over its whole
megabatch, one call per shape group exactly as the benchmark times it.  One
sampled matrix of each group is then compared with the dense-library form of
the oracle (numpy products, LAPACK Householder QR, float64) run from the same
stored state: M, Q (sign-aligned), R (sign-aligned), P Q^T, the change of X
and the stored X, plus ||P^T P - I||.

The learning rate here is set per shape so that the weight change has rms
0.01 (half that of X ~ N(0, 0.02^2), about 80 bf16 units): lr = 0.01 n / sqrt(r),
since rms(P Q^T) = sqrt(r / (m n)).  It does not change the launch
configuration (the workloads use 0.01), and with the change spanning many
units the relative error of the stored change measures the update, not the
bf16 rounding of X: at a change of a few units, rounding-boundary flips alone
make a few percent.

Newton-Schulz (Muon, 5 quintic steps, with momentum and the weight step) is
compared with the oracle in full where the oracle's 5 dense steps take
seconds (n <= 4096, and the 405B layer's 16384 x 1024), and on 16 sampled
rows elsewhere (the rows computed by the oracle's step recursion, see
oracle.dense.newton_schulz_rows).
"""
import gc
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.dense
import workloads as wl
import orthonormal_optimizer_step_gb300 as od
from parity import ORTH_TOL, TOL, dion_pair, f64, muon_pair, rel

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


def lr_for(g, r):
    return 0.01 * g.n / math.sqrt(r)


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _dion(g, r, w, seed, bi):
    X, _, Q = wl.make_state(g, r, w.dtype, DEV, seed)
    M = wl.make_momentum(g, w.g_std, DEV, seed)
    G = wl.make_grad(g, w.g_std, w.dtype, DEV, seed, step=1)
    out = dion_pair(X, G, M, Q, w.mu, lr_for(g, r), w.wd, samples=[bi], form=oracle.dense)
    del X, M, Q, G
    _free()
    tol = TOL[w.dtype]
    assert out["status"] == 0, out
    assert out["orth"] <= ORTH_TOL, out
    assert out["qcol"] <= 1e-5, out
    for key in ("M", "Q", "R", "PQt", "X"):
        assert out[key] <= tol, (key, out)
    assert out["x_ulps"] <= 1.0 + 1e-9, out
    return out


@pytest.mark.parametrize("gi", [0, 1, 2, 3])
def test_llama3_8b_megabatch_oracle(gi):
    """32 layers x {4096x4096 (Q, O), 4096x1024 (K, V), 4096x14336 (gate, up),
    14336x4096 (down)}, bf16, rank fraction 1/16 (ranks 256, 64, 256, 256);
    the last matrix of each group is checked."""
    w = wl.llama3_8b()
    g = w.groups[gi]
    _dion(g, g.rank(w.fraction), w, seed=4000 + gi, bi=g.batch - 1)


@pytest.mark.parametrize("gi", [0, 1, 2, 3])
def test_llama3_405b_layer_oracle(gi):
    """{16384x16384 x2, 16384x1024 x2, 16384x53248 x2, 53248x16384}, bf16,
    rank fraction 1/16 (ranks 1024, 64, 1024, 1024), Gaussian G."""
    w = wl.llama3_405b_layer()
    g = w.groups[gi]
    _dion(g, g.rank(w.fraction), w, seed=5000 + gi, bi=0)


@pytest.mark.parametrize("n", [1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("frac", [0.25, 1.0 / 16])
def test_square_sweep_oracle(n, frac):
    """8 x n x n, bf16, Gaussian G and X, rank n/4 or n/16; matrix 3 checked."""
    w = wl.square(n)
    g = w.groups[0]
    _dion(g, g.rank(frac), w, seed=6000 + n + int(1 / frac), bi=3)


# ------------------------------------------------------------ Newton-Schulz

def _muon_full(g, seed, bi):
    G = wl.make_grad(g, 1.0, BF, DEV, seed, step=0)
    M = wl.make_momentum(g, 1.0, DEV, seed)
    X = wl.randn((g.batch, g.m, g.n), 0.02, BF, DEV, seed + 1)
    out = muon_pair(G, M, X, g.head_dim, 5, oracle.QUINTIC, 0.95, 0.5, 0.01, samples=[bi], form=oracle.dense)
    del G, M, X
    _free()
    for key in ("O", "M", "X"):
        assert out[key] <= TOL[BF], (key, out)


def _muon_rows(g, seed, bi, nrows=16):
    """Whole-megabatch Newton-Schulz on the GPU; 16 sampled rows of matrix bi
    against the oracle's rows, and the momentum update in full."""
    G = wl.make_grad(g, 1.0, BF, DEV, seed, step=0)
    M = wl.make_momentum(g, 1.0, DEV, seed)
    hG, hM = f64(G[bi]), f64(M[bi])
    O = torch.empty_like(G)
    od.muon_ns_batched(G, M=M, O=O, head_dim=0, steps=5, mu=0.95)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(seed).choice(g.m, size=min(nrows, g.m), replace=False))
    Y = 0.95 * hM + hG                                  # the oracle's momentum step
    e_m = rel(f64(M[bi]), Y)
    want = oracle.dense.newton_schulz_rows(Y, rows, 5, oracle.QUINTIC, oracle.NS_EPS)
    got = f64(O[bi][torch.as_tensor(rows, device=DEV)])
    e_o = rel(got, want)
    del G, M, O, hG, hM, Y
    _free()
    assert e_m <= TOL[torch.float32], e_m
    assert e_o <= TOL[BF], e_o


@pytest.mark.parametrize("n", [1024, 2048, 4096])
def test_square_sweep_newton_schulz_oracle(n):
    _muon_full(wl.square(n).groups[0], seed=7000 + n, bi=2)


@pytest.mark.parametrize("n", [8192, 16384])
def test_square_sweep_newton_schulz_oracle_rows(n):
    _muon_rows(wl.square(n).groups[0], seed=7000 + n, bi=2)


def test_llama3_405b_newton_schulz_oracle_kv():
    _muon_full(wl.llama3_405b_layer().groups[1], seed=7101, bi=1)


@pytest.mark.parametrize("gi", [2, 3])
def test_llama3_405b_newton_schulz_oracle_rows(gi):
    """16384 x 53248 (the Gram over the long side) and 53248 x 16384 (the
    transposed block); the 16384 x 16384 group is the square sweep's shape."""
    _muon_rows(wl.llama3_405b_layer().groups[gi], seed=7100 + gi, bi=0)
