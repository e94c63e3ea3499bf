"""GPU parity of muon_ns_batched (Newton-Schulz, whole matrix and per head)
against the oracle, through the C ABI."""
import pytest
import torch

import oracle
import workloads as wl
from parity import TOL, muon_pair

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_single_256_fp32_five_steps():
    """Five quintic Newton-Schulz steps on the 256 x 256 float32 gradient."""
    w = wl.single_256()
    g = w.groups[0]
    G = wl.make_grad(g, 1.0, torch.float32, DEV, seed=1001, step=0)
    X = wl.randn((1, 256, 256), 0.02, torch.float32, DEV, seed=3)
    out = muon_pair(G, None, X, 0, 5, oracle.QUINTIC, 0.95, 0.01, 0.01)
    assert out["O"] <= TOL[torch.float32], out
    assert out["X"] <= TOL[torch.float32], out


@pytest.mark.parametrize("batch,m,n,hd,dtype", [
    (2, 200, 136, 0, torch.float32),
    (2, 136, 200, 0, torch.bfloat16),
    (2, 96, 128, 32, torch.bfloat16),
    (1, 64, 64, 0, torch.bfloat16),
    (3, 130, 70, 0, torch.float32),
    (1, 8, 300, 0, torch.bfloat16),
])
def test_ragged_shapes(batch, m, n, hd, dtype):
    g = wl.Group(batch, m, n)
    G = wl.make_grad(g, 1.0, dtype, DEV, seed=m + n, step=0)
    M = wl.make_momentum(g, 1.0, DEV, seed=m + n)
    out = muon_pair(G, M, None, hd, 5, oracle.QUINTIC, 0.9, 0.0, 0.0)
    assert out["O"] <= TOL[dtype], out
    assert out["M"] <= TOL[dtype], out


def test_gpt_small_megabatch_sampled():
    """GPT-small megabatch in bf16 with momentum; QKV per head (12 heads of
    64 for each of Q, K, V); one sampled matrix per group is checked."""
    w = wl.gpt_small()
    for gi, g in enumerate(w.groups):
        G = wl.make_grad(g, w.g_std, w.dtype, DEV, seed=3000 + gi, step=1)
        M = wl.make_momentum(g, w.g_std, DEV, seed=3000 + gi)
        X = wl.randn((g.batch, g.m, g.n), 0.02, w.dtype, DEV, seed=3100 + gi)
        out = muon_pair(G, M, X, g.head_dim, 5, oracle.QUINTIC, w.mu, 0.02, w.wd, samples=[7])
        assert out["O"] <= TOL[w.dtype], (gi, out)
        assert out["M"] <= TOL[w.dtype], (gi, out)
