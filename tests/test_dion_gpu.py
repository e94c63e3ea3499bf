"""GPU parity of dion_step_batched against the oracle (teacher-forced: both
sides start every step from the same stored state).  Calls go through the C
ABI (ctypes binding)."""
import numpy as np
import pytest
import torch

import workloads as wl
import orthonormal_optimizer_step_gb300 as od
from parity import ORTH_TOL, TOL, dion_compare, dion_pair, dion_snapshot, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(out, dtype, x_rel=True):
    tol = TOL[dtype]
    assert out["orth"] <= ORTH_TOL, out
    assert out["qcol"] <= 1e-5, out
    for key in ("M", "Q", "R", "PQt"):
        assert out[key] <= tol, (key, out)
    if x_rel:
        assert out["X"] <= tol, ("X", out)
    if dtype == torch.bfloat16:
        assert out["x_ulps"] <= 1.0 + 1e-9, out


def test_single_256_fp32_ten_steps():
    """256 x 256 float32, rank 64, mu = 0.95, lr = wd = 0.01, ten steps with a
    fresh N(0, 1) gradient each step; every step is compared."""
    w = wl.single_256()
    g = w.groups[0]
    r = g.rank(w.fraction)
    assert r == 64
    X, M, Q = wl.make_state(g, r, w.dtype, DEV, seed=1001)
    for step in range(w.steps):
        G = wl.make_grad(g, w.g_std, w.dtype, DEV, seed=1001, step=step)
        out = dion_pair(X, G, M, Q, w.mu, w.lr, w.wd)
        assert out["status"] == 0
        _check(out, w.dtype)


RAGGED = [
    (3, 200, 136, 24, torch.float32),
    (2, 136, 200, 136, torch.float32),     # r = m = min(m, n)
    (2, 200, 136, 136, torch.bfloat16),    # r = n = min(m, n)
    (1, 97, 131, 1, torch.float32),        # r = 1, odd sizes
    (2, 130, 260, 17, torch.bfloat16),
    (1, 64, 64, 16, torch.bfloat16),
    (1, 1024, 1024, 288, torch.bfloat16),  # r > 256: two 256-column chunks of the rank
    (2, 700, 600, 300, torch.bfloat16),    # blocked factorization: blocks of 128, 128, 44
    (1, 1100, 1300, 520, torch.bfloat16),  # blocked factorization: four blocks and a ragged 8
    (1, 700, 1000, 600, torch.bfloat16),   # rp > 512: the M update as a 128 x 256 GEMM, ragged edge blocks
    (1, 8, 520, 3, torch.bfloat16),        # very wide
    (2, 520, 8, 8, torch.float32),         # very tall, full rank
]


@pytest.mark.parametrize("batch,m,n,r,dtype", RAGGED)
def test_ragged_shapes(batch, m, n, r, dtype):
    g = wl.Group(batch, m, n)
    seed = 7 + m + n + r
    X, _, Q = wl.make_state(g, r, dtype, DEV, seed)
    M = wl.make_momentum(g, 0.5, DEV, seed)
    G = wl.make_grad(g, 1.0, dtype, DEV, seed, step=3)
    # lr = 0.5 makes the weight change span many bf16 units, so its direction is checked too
    out = dion_pair(X, G, M, Q, 0.9, 0.5, 0.02)
    assert out["status"] == 0
    _check(out, dtype)


@pytest.mark.parametrize("lr", [0.01, 0.5])
def test_gpt_small_megabatch_sampled(lr):
    """Full GPT-small megabatch (12 matrices per shape group), bf16, rank 192;
    the oracle checks one sampled matrix of every group (matrices of a batch
    are independent).  At the workload's lr = 0.01 the weight change
    (about 6e-5) is below half a bf16 unit of X (about 0.02), so only the
    stored X is compared there; lr = 0.5 makes the change span many units,
    and its relative error is checked too."""
    w = wl.gpt_small()
    for gi, g in enumerate(w.groups):
        r = g.rank(w.fraction)
        X, _, Q = wl.make_state(g, r, w.dtype, DEV, seed=2000 + gi)
        M = wl.make_momentum(g, w.g_std, DEV, seed=2000 + gi)
        G = wl.make_grad(g, w.g_std, w.dtype, DEV, seed=2000 + gi, step=1)
        out = dion_pair(X, G, M, Q, w.mu, lr, w.wd, samples=[5])
        assert out["status"] == 0
        _check(out, w.dtype, x_rel=lr >= 0.5)


def test_zero_gradient_reports_breakdown_and_stays_finite():
    g = wl.Group(2, 64, 96)
    X, M, Q = wl.make_state(g, 8, torch.bfloat16, DEV, seed=5)
    G = torch.zeros_like(X)
    X0 = X.clone()
    ws = od.dion_step_batched(X, G, M, Q, mu=0.95, lr=0.01, weight_decay=0.1)
    torch.cuda.synchronize()
    st = od.dion_get_status(ws)
    assert st & 1
    assert torch.isfinite(Q).all() and torch.isfinite(M).all() and torch.isfinite(X.float()).all()
    assert torch.count_nonzero(M) == 0
    # B = 0: only the decay acts on X (computed in float32 as the kernel does)
    decay = np.float32(1.0) - np.float32(0.01) * np.float32(0.1)
    ref = (X0.float() * float(decay)).to(torch.bfloat16)
    assert torch.equal(X, ref)


def test_rank_deficient_gradient():
    """G of rank 2 with r = 6: dependent columns of P are zeroed and flagged;
    the rest stay orthonormal."""
    g = wl.Group(1, 48, 40)
    gen = torch.Generator(device="cpu").manual_seed(3)
    u = torch.randn(48, 2, generator=gen, dtype=torch.float64)
    v = torch.randn(2, 40, generator=gen, dtype=torch.float64)
    G = (u @ v).to(torch.float32).unsqueeze(0).to(DEV)
    X, M, Q = wl.make_state(g, 6, torch.float32, DEV, seed=9)
    ws = od.dion_step_batched(X, G, M, Q, mu=0.9, lr=0.01, weight_decay=0.0)
    torch.cuda.synchronize()
    assert od.dion_get_status(ws) & 1
    P, _ = od.dion_panels(ws, 1, 48, 40, 6, od.DION_F32)
    P = f64(P[0])
    live = np.linalg.norm(P, axis=0) > 0.5
    assert 1 <= live.sum() <= 2 + 1
    np.testing.assert_allclose(P[:, live].T @ P[:, live], np.eye(live.sum()), atol=1e-3)
    assert np.all(np.abs(P[:, ~live]) == 0)
    assert torch.isfinite(X).all() and torch.isfinite(M).all() and torch.isfinite(Q).all()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_checkpoint_resume_is_bitwise(dtype):
    """The optimizer state is (X, M, Q): saving it, reloading it and stepping
    gives exactly the uninterrupted run."""
    g = wl.Group(3, 192, 320)
    r = 48
    X, M, Q = wl.make_state(g, r, dtype, DEV, seed=77)
    grads = [wl.make_grad(g, 1.0, dtype, DEV, 77, s) for s in range(5)]
    for s in range(3):
        od.dion_step_batched(X, grads[s], M, Q, mu=0.9, lr=0.02, weight_decay=0.01)
    saved = [t.clone() for t in (X, M, Q)]
    for s in range(3, 5):
        od.dion_step_batched(X, grads[s], M, Q, mu=0.9, lr=0.02, weight_decay=0.01)
    X2, M2, Q2 = [t.clone() for t in saved]
    for s in range(3, 5):
        od.dion_step_batched(X2, grads[s], M2, Q2, mu=0.9, lr=0.02, weight_decay=0.01)
    torch.cuda.synchronize()
    assert torch.equal(X, X2) and torch.equal(M, M2) and torch.equal(Q, Q2)


def test_streams_and_reused_workspace():
    """A caller stream and a reused workspace give the same result as the
    default stream with a fresh one."""
    g = wl.Group(2, 128, 256)
    X, M, Q = wl.make_state(g, 32, torch.bfloat16, DEV, seed=4)
    G = wl.make_grad(g, 1.0, torch.bfloat16, DEV, 4, 0)
    A = [t.clone() for t in (X, M, Q)]
    od.dion_step_batched(*A[:1], G, *A[1:], mu=0.9, lr=0.1, weight_decay=0.0)
    s = torch.cuda.Stream()
    ws = od.new_workspace(od.dion_workspace_size(2, 128, 256, 32, od.DION_BF16), DEV)
    ws.fill_(0xAB)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        od.dion_step_batched(X, G, M, Q, mu=0.9, lr=0.1, weight_decay=0.0, workspace=ws, stream=s)
    s.synchronize()
    assert torch.equal(X, A[0]) and torch.equal(M, A[1]) and torch.equal(Q, A[2])


def test_blocked_factorization_reads_no_stale_workspace():
    """Rank 300 takes the blocked factorization, which computes only the lower
    half of each Gram matrix: a workspace full of NaN bit patterns gives the
    same bits as a zeroed one."""
    g = wl.Group(2, 640, 512)
    r = 300
    X, M, Q = wl.make_state(g, r, torch.bfloat16, DEV, seed=31)
    G = wl.make_grad(g, 1.0, torch.bfloat16, DEV, 31, 0)
    n_ws = od.dion_workspace_size(2, 640, 512, r, od.DION_BF16)
    outs = []
    for fill in (0x00, 0xFF):
        A = [t.clone() for t in (X, M, Q)]
        ws = od.new_workspace(n_ws, DEV)
        ws.fill_(fill)
        od.dion_step_batched(A[0], G, A[1], A[2], mu=0.9, lr=0.1, weight_decay=0.0, workspace=ws)
        torch.cuda.synchronize()
        assert od.dion_get_status(ws) == 0
        outs.append(A)
    for a, b in zip(*outs):
        assert torch.isfinite(a.float()).all()
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,m,n,r", [(torch.float32, 192, 320, 48), (torch.bfloat16, 192, 320, 48),
                                         (torch.bfloat16, 640, 512, 300)])
def test_device_scalars_follow_schedule_under_graph_replay(dtype, m, n, r):
    """dion_step_batched_dev captured once in a CUDA graph and replayed while
    the caller writes a new (mu, lr, weight_decay) into device memory: every
    replayed step matches the oracle at that schedule entry, and the run gives
    the same bits as direct calls with those values passed by value (rank 300:
    the wide path, whose update runs in GEMM epilogues).  The learning rates
    of the schedule move X by less than a bf16 unit, so the stored X is
    compared within one unit and the update itself through M, Q and P Q^T."""
    g = wl.Group(2, m, n)
    X, M, Q = wl.make_state(g, r, dtype, DEV, seed=41)
    grads = [wl.make_grad(g, 1.0, dtype, DEV, 41, s) for s in range(4)]
    schedule = [(0.9, 0.02, 0.01), (0.9, 0.01, 0.01), (0.8, 0.005, 0.0), (0.95, 0.03, 0.1)]
    ref = [t.clone() for t in (X, M, Q)]
    ws_ref = od.new_workspace(od.dion_workspace_size(2, m, n, r, od.DION_BF16 if dtype == torch.bfloat16
                                                     else od.DION_F32), DEV)
    for (mu, lr, wd), Gs in zip(schedule, grads):
        od.dion_step_batched(ref[0], Gs, ref[1], ref[2], mu=mu, lr=lr, weight_decay=wd, workspace=ws_ref)
    # graph: static input buffer for G, device scalars
    Gbuf = grads[0].clone()
    hyper = torch.tensor(schedule[0], dtype=torch.float32, device=DEV)
    ws = od.new_workspace(ws_ref.numel(), DEV)
    cur = [t.clone() for t in (X, M, Q)]
    warm = [t.clone() for t in (X, M, Q)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # first call outside the capture (launch attributes)
        od.dion_step_batched(warm[0], Gbuf, warm[1], warm[2], hyper=hyper, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        od.dion_step_batched(cur[0], Gbuf, cur[1], cur[2], hyper=hyper, workspace=ws)
    for (mu, lr, wd), Gs in zip(schedule, grads):
        Gbuf.copy_(Gs)
        hyper.copy_(torch.tensor([mu, lr, wd], dtype=torch.float32))
        idx, host = dion_snapshot(cur[0], Gbuf, cur[1], cur[2], samples=[1])
        graph.replay()
        torch.cuda.synchronize()
        # each replayed step against the oracle at that step's schedule entry
        out = dion_compare(idx, host, cur[0], cur[1], cur[2], ws, mu, lr, wd)
        assert out["status"] == 0
        _check(out, dtype, x_rel=dtype == torch.float32)
    torch.cuda.synchronize()
    assert od.dion_get_status(ws) == 0
    for a, b in zip(cur, ref):
        assert torch.equal(a, b)


def test_device_scalars_non_finite_sets_status():
    g = wl.Group(1, 64, 96)
    X, M, Q = wl.make_state(g, 8, torch.bfloat16, DEV, seed=43)
    G = wl.make_grad(g, 1.0, torch.bfloat16, DEV, 43, 0)
    hyper = torch.tensor([0.9, float("nan"), 0.0], dtype=torch.float32, device=DEV)
    ws = od.dion_step_batched(X, G, M, Q, hyper=hyper)
    torch.cuda.synchronize()
    assert od.dion_get_status(ws) & 2


def test_rank_deficient_gradient_blocked_factorization():
    """Rank 300 (blocked factorization) on B = G of rank 20: the dependent
    columns found inside the 128-column diagonal blocks are zeroed and
    flagged, and the remaining columns are orthonormal.  G is built from +-1
    factors, so its entries are small integers, exact in bf16, and G has
    rank 20 exactly (a rounded real low-rank G would not be)."""
    g = wl.Group(1, 512, 640)
    r = 300
    gen = torch.Generator(device="cpu").manual_seed(5)
    u = torch.randint(0, 2, (512, 20), generator=gen).to(torch.float64) * 2 - 1
    v = torch.randint(0, 2, (20, 640), generator=gen).to(torch.float64) * 2 - 1
    G = (u @ v).to(torch.bfloat16).unsqueeze(0).to(DEV)
    X, M, Q = wl.make_state(g, r, torch.bfloat16, DEV, seed=11)
    M.zero_()
    ws = od.dion_step_batched(X, G, M, Q, mu=0.9, lr=0.01, weight_decay=0.0)
    torch.cuda.synchronize()
    assert od.dion_get_status(ws) & 1
    P, _ = od.dion_panels(ws, 1, 512, 640, r, od.DION_BF16)
    P = f64(P[0])
    live = np.linalg.norm(P, axis=0) > 0.5
    assert 1 <= live.sum() <= 20 + 1
    np.testing.assert_allclose(P[:, live].T @ P[:, live], np.eye(live.sum()), atol=1e-3)
    assert np.all(np.abs(P[:, ~live]) == 0)
    assert torch.isfinite(X.float()).all() and torch.isfinite(M).all() and torch.isfinite(Q).all()


def _dominant_gradient(m, n, scale, seed, blk=64):
    """bf16 gradient with one dominant direction, stored exactly: rows and
    columns of block-diag(scale u v^T, C) permuted at random, with u, v in
    {-1, +1}^blk (scale u v^T has singular value scale*blk, exact in bf16 for a
    bf16-exact scale) and C = (m-blk) x (n-blk) with orthonormal columns
    (singular values 1, up to bf16 rounding).  sigma_1 / sigma_2 = scale*blk."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    u = torch.randint(0, 2, (blk,), generator=gen).double() * 2 - 1
    v = torch.randint(0, 2, (blk,), generator=gen).double() * 2 - 1
    C, _ = torch.linalg.qr(torch.randn(m - blk, n - blk, generator=gen, dtype=torch.float64))
    G = torch.zeros(m, n, dtype=torch.float64)
    G[:blk, :blk] = scale * torch.outer(u, v)
    G[blk:, blk:] = C
    G = G[torch.randperm(m, generator=gen)][:, torch.randperm(n, generator=gen)]
    return G.to(torch.bfloat16)


@pytest.mark.parametrize("r", [64, 300])
@pytest.mark.parametrize("scale", [16.0, 160.0, 1536.0])
def test_ill_conditioned_full_rank_matches_oracle(r, scale):
    """B = G with sigma_1 / sigma_2 = 1.0e3, 1.0e4, 9.8e4 (M = 0, random Q0),
    full rank: the float32 Gram of B Q cannot resolve its small directions, so
    the first CholeskyQR pass is redone in float64 for these matrices.  Every
    column must stay live (no status bit) and the step must match the oracle
    (one-CTA factorization at rank 64, blocked at rank 300)."""
    m, n = 1024, 768
    g = wl.Group(2, m, n)
    G = torch.stack([_dominant_gradient(m, n, scale, 17 + k + int(scale)) for k in range(2)]).to(DEV)
    X, _, Q = wl.make_state(g, r, torch.bfloat16, DEV, seed=23 + r)
    M = torch.zeros(2, m, n, dtype=torch.float32, device=DEV)
    out = dion_pair(X, G, M, Q, 0.9, 0.5, 0.0)
    assert out["status"] == 0, out
    _check(out, torch.bfloat16)


def test_ill_conditioned_and_healthy_matrices_in_one_batch():
    """The float64 first pass runs only for the flagged matrix of a batch; the
    healthy one takes the float32 path, and both match the oracle."""
    m, n, r = 512, 384, 48
    g = wl.Group(2, m, n)
    G = torch.stack([_dominant_gradient(m, n, 1536.0, 3),
                     wl.make_grad(wl.Group(1, m, n), 1.0, torch.bfloat16, "cpu", 5, 0)[0]]).to(DEV)
    X, _, Q = wl.make_state(g, r, torch.bfloat16, DEV, seed=29)
    M = torch.zeros(2, m, n, dtype=torch.float32, device=DEV)
    out = dion_pair(X, G, M, Q, 0.9, 0.5, 0.0)
    assert out["status"] == 0, out
    _check(out, torch.bfloat16)
