"""Pins for the oracle: every routine is checked against something other than
itself -- hand-derived worked examples, closed forms, special cases of the
update rule, LAPACK's QR and SVD (numpy), and brute-force convergence to the
exact U V^T.  CPU only.

A plausible slip in the oracle (a dropped M, a transposed operand, sqrt(n/m)
for sqrt(m/n), mu for 1-mu, the wrong Newton-Schulz coefficient order) fails at
least one test here.
"""
import os

import numpy as np
import pytest

import oracle
import oracle.dense

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dion_hand_examples.txt")


def _parse_golden(path):
    cases, cur = {}, None
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        if line.startswith("case "):
            cur = {}
            cases[line.split()[1]] = cur
            continue
        key, rest = line.split(":", 1)
        key = key.strip()
        if key in ("params", "ns"):
            cur[key] = {kv.split("=")[0]: float(kv.split("=")[1]) for kv in rest.split()}
            continue
        shape, vals = rest.split(":", 1)
        r, c = (int(v) for v in shape.strip().split("x"))
        cur[key] = np.array([float(v) for v in vals.split()]).reshape(r, c)
    return cases


# Both forms of the oracle: the C triple loops and the dense-library form
# (numpy products, LAPACK QR).  Every pin below runs on each of them.
FORMS = {"c": oracle, "dense": oracle.dense}


@pytest.fixture(params=sorted(FORMS))
def form(request):
    return FORMS[request.param]


def _svd(A):
    U, s, Vt = np.linalg.svd(A, full_matrices=False)
    return U, s, Vt


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- Householder

@pytest.mark.parametrize("m,r", [(50, 12), (7, 7), (30, 1), (9, 4)])
def test_householder_matches_lapack(form, m, r):
    rng = np.random.default_rng(m * 100 + r)
    A = _rand(rng, m, r)
    Qf, Rq = form.householder_qr(A)
    Qn, Rn = np.linalg.qr(A)
    d = np.sign(np.diag(Rn))
    d[d == 0] = 1
    Qn, Rn = Qn * d, (Rn.T * d).T
    np.testing.assert_allclose(Qf, Qn, atol=1e-12)
    np.testing.assert_allclose(Rq, Rn, atol=1e-12)
    np.testing.assert_allclose(Qf.T @ Qf, np.eye(r), atol=1e-13)
    np.testing.assert_allclose(Qf @ Rq, A, atol=1e-12)
    assert np.all(np.diag(Rq) >= 0) and np.allclose(np.tril(Rq, -1), 0)


def test_householder_rank_deficient_still_orthonormal(form):
    rng = np.random.default_rng(3)
    A = _rand(rng, 10, 4)
    A[:, 2] = 0.0
    Qf, Rq = form.householder_qr(A)
    np.testing.assert_allclose(Qf.T @ Qf, np.eye(4), atol=1e-13)
    np.testing.assert_allclose(Qf @ Rq, A, atol=1e-12)
    assert abs(Rq[2, 2]) < 1e-12


# ---------------------------------------------------------- worked examples

@pytest.mark.parametrize("name", ["A", "B", "C"])
def test_dion_hand_examples(form, name):
    c = _parse_golden(GOLDEN)[name]
    p = c["params"]
    out = form.dion_step(c["X"], c["G"], c["M"], c["Q"], p["mu"], p["lr"], p["wd"])
    for key in ("P", "R", "Q", "M", "X"):
        np.testing.assert_allclose(out[key], c[key + "_out"], atol=1e-13, err_msg=key)


def test_newton_schulz_hand_example(form):
    c = _parse_golden(GOLDEN)["NS1"]
    ns = c["ns"]
    O = form.newton_schulz(c["Y"], int(ns["steps"]), (ns["a"], ns["b"], ns["c"]), ns["eps"])
    np.testing.assert_allclose(O, c["O_out"], atol=1e-14)


# ------------------------------------------------------------- Dion step

SHAPES = [(12, 7, 3), (7, 12, 3), (9, 9, 1), (6, 10, 6), (10, 6, 6), (16, 16, 4)]


def _state(rng, m, n, r):
    X = 0.02 * _rand(rng, m, n)
    G = _rand(rng, m, n)
    M = 0.5 * _rand(rng, m, n)
    Q = _rand(rng, n, r)
    Q /= np.linalg.norm(Q, axis=0)
    return X, G, M, Q


@pytest.mark.parametrize("m,n,r", SHAPES)
def test_dion_invariants(form, m, n, r):
    rng = np.random.default_rng(m * 31 + n * 7 + r)
    X, G, M, Q = _state(rng, m, n, r)
    mu, lr, wd = 0.95, 0.01, 0.01
    out = form.dion_step(X, G, M, Q, mu, lr, wd)
    B = M + G
    P = out["P"]
    # P has orthonormal columns spanning B Q (LAPACK QR as the independent basis).
    np.testing.assert_allclose(P.T @ P, np.eye(r), atol=1e-12)
    Qb, _ = np.linalg.qr(B @ Q)
    np.testing.assert_allclose(P @ P.T, Qb @ Qb.T, atol=1e-12)
    # Unit-norm columns of the new Q.
    np.testing.assert_allclose(np.linalg.norm(out["Q"], axis=0), np.ones(r), atol=1e-12)
    # Closed form of the error feedback: M' = (I - (1 - mu) P P^T) B.
    M_closed = (np.eye(m) - (1 - mu) * (P @ P.T)) @ B
    np.testing.assert_allclose(out["M"], M_closed, atol=1e-12)
    # The step sees M and G only through B = M + G.
    out2 = form.dion_step(X, B, np.zeros_like(M), Q, mu, lr, wd)
    for key in ("X", "M", "Q", "P", "R"):
        np.testing.assert_allclose(out[key], out2[key], atol=1e-12, err_msg=key)


@pytest.mark.parametrize("m,n,r", SHAPES)
def test_dion_special_cases(form, m, n, r):
    rng = np.random.default_rng(m + 5 * n + 11 * r)
    X, G, M, Q = _state(rng, m, n, r)
    B = M + G
    # mu = 1: no error feedback removed, M' = B.
    out = form.dion_step(X, G, M, Q, 1.0, 0.01, 0.0)
    np.testing.assert_allclose(out["M"], B, atol=1e-12)
    # lr = 0: the weights do not move.
    out = form.dion_step(X, G, M, Q, 0.9, 0.0, 0.3)
    np.testing.assert_allclose(out["X"], X, atol=0)
    # Full rank r = m <= n: P P^T = I, so M' = mu B exactly.
    if r == m <= n:
        out = form.dion_step(X, G, M, Q, 0.8, 0.01, 0.0)
        np.testing.assert_allclose(out["M"], 0.8 * B, atol=1e-12)


def _fixed_B(rng, m, n, sig):
    U, _ = np.linalg.qr(_rand(rng, m, m))
    V, _ = np.linalg.qr(_rand(rng, n, n))
    k = min(m, n)
    S = np.zeros((m, n))
    S[np.arange(k), np.arange(k)] = sig[:k]
    return U @ S @ V.T


@pytest.mark.parametrize("m,n,r", [(8, 12, 8), (12, 8, 8), (8, 12, 3), (12, 8, 2)])
def test_dion_power_iteration_reaches_svd(form, m, n, r):
    """With mu = 1 and no new gradient after the first step, B stays fixed and
    Dion is orthogonal iteration on B: P Q^T -> U_r V_r^T of the exact SVD, and
    the weight step is -lr sqrt(m/n) U_r V_r^T."""
    rng = np.random.default_rng(m * 13 + r)
    sig = np.array([10, 6, 3.5, 2, 1.2, 0.7, 0.4, 0.24])
    B = _fixed_B(rng, m, n, sig)
    Q = _rand(rng, n, r)
    Q /= np.linalg.norm(Q, axis=0)
    X = np.zeros((m, n))
    M = np.zeros((m, n))
    G = B
    lr = 0.1
    for _ in range(60):
        out = form.dion_step(X, G, M, Q, 1.0, lr, 0.0)
        M, Q, G = out["M"], out["Q"], np.zeros((m, n))
        Xprev, X = X, out["X"]
    U, s, Vt = _svd(B)
    target = U[:, :r] @ Vt[:r, :]
    np.testing.assert_allclose(out["P"] @ out["Q"].T, target, atol=1e-9)
    np.testing.assert_allclose(X - Xprev, -lr * np.sqrt(m / n) * target, atol=1e-9)
    # The columns themselves converge to the singular vectors, up to sign.
    sgn = np.sign(np.sum(out["P"] * U[:, :r], axis=0))
    np.testing.assert_allclose(out["P"] * sgn, U[:, :r], atol=1e-8)
    np.testing.assert_allclose(out["Q"] * sgn, Vt[:r, :].T, atol=1e-8)
    np.testing.assert_allclose(np.linalg.norm(out["R"], axis=0), s[:r], rtol=1e-9)


# ------------------------------------------------------------ Newton-Schulz

def _ns_closed_form(Y, steps, coeff, eps):
    a, b, c = coeff
    U, s, Vt = _svd(Y)
    x = s / (np.linalg.norm(Y) + eps)
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return (U * x) @ Vt


@pytest.mark.parametrize("m,n", [(6, 9), (9, 6), (8, 8), (1, 5)])
@pytest.mark.parametrize("steps", [1, 5])
def test_newton_schulz_closed_form(form, m, n, steps):
    """k steps of NS act on singular values only: U p_k(S/(||Y||_F+eps)) V^T."""
    rng = np.random.default_rng(m * 17 + n + steps)
    Y = _rand(rng, m, n)
    O = form.newton_schulz(Y, steps, oracle.QUINTIC, oracle.NS_EPS)
    np.testing.assert_allclose(O, _ns_closed_form(Y, steps, oracle.QUINTIC, oracle.NS_EPS), atol=1e-12)


@pytest.mark.parametrize("m,n", [(6, 10), (10, 6)])
def test_cubic_newton_schulz_reaches_polar_factor(form, m, n):
    """The textbook cubic iteration converges to U V^T (Higham)."""
    rng = np.random.default_rng(m + n)
    k = min(m, n)
    sig = np.linspace(1.0, 0.3, k)
    Y = _fixed_B(rng, m, n, sig)
    O = form.newton_schulz(Y, 40, oracle.CUBIC, oracle.NS_EPS)
    U, s, Vt = _svd(Y)
    np.testing.assert_allclose(O, U @ Vt, atol=1e-10)


def test_muon_per_head_and_update(form):
    rng = np.random.default_rng(7)
    m, n, hd = 12, 16, 4
    G = _rand(rng, m, n)
    M = _rand(rng, m, n)
    X = _rand(rng, m, n)
    mu, lr, wd = 0.9, 0.05, 0.1
    out = form.muon_step(X, G, M, head_dim=hd, steps=5, mu=mu, lr=lr, wd=wd)
    Y = mu * M + G
    O_ref = np.concatenate([_ns_closed_form(Y[:, h * hd:(h + 1) * hd], 5, oracle.QUINTIC, oracle.NS_EPS)
                            for h in range(n // hd)], axis=1)
    np.testing.assert_allclose(out["O"], O_ref, atol=1e-12)
    np.testing.assert_allclose(out["X"], (1 - lr * wd) * X - lr * np.sqrt(m / n) * O_ref, atol=1e-12)
    # Whole-matrix mode differs from per-head mode (heads are blended).
    whole = form.muon_step(None, G, M, head_dim=0, steps=5, mu=mu)
    np.testing.assert_allclose(whole["O"], _ns_closed_form(Y, 5, oracle.QUINTIC, oracle.NS_EPS), atol=1e-12)
    assert np.abs(whole["O"] - out["O"]).max() > 1e-3
    # mu = 0 with a momentum buffer equals no momentum at all.
    a = form.muon_step(None, G, M, mu=0.0)["O"]
    b = form.muon_step(None, G, None)["O"]
    np.testing.assert_allclose(a, b, atol=1e-14)


# -------------------------------------------------------- storage rounding

def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000) * 10.0 ** rng.integers(-8, 8, 10000),
                        [0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 65504.0, 3e38]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), ref)
    np.testing.assert_array_equal(oracle.round_f32(x), x.astype(np.float32).astype(np.float64))


# ------------------------------------------------------ the two forms agree

@pytest.mark.parametrize("m,n,r", [(40, 30, 7), (30, 40, 30), (25, 25, 1)])
def test_forms_agree_on_dion_step(m, n, r):
    rng = np.random.default_rng(m + n + r)
    X, G, M, Q = _state(rng, m, n, r)
    a = oracle.dion_step(X, G, M, Q, 0.9, 0.05, 0.1)
    b = oracle.dense.dion_step(X, G, M, Q, 0.9, 0.05, 0.1)
    for key in ("X", "M", "Q", "P", "R"):
        np.testing.assert_allclose(a[key], b[key], atol=1e-11, err_msg=key)


@pytest.mark.parametrize("hd", [0, 8])
def test_forms_agree_on_muon_step(hd):
    rng = np.random.default_rng(hd + 1)
    G, M, X = _rand(rng, 20, 32), _rand(rng, 20, 32), _rand(rng, 20, 32)
    a = oracle.muon_step(X, G, M, head_dim=hd, steps=5, mu=0.9, lr=0.1, wd=0.1)
    b = oracle.dense.muon_step(X, G, M, head_dim=hd, steps=5, mu=0.9, lr=0.1, wd=0.1)
    for key in ("O", "X", "M"):
        np.testing.assert_allclose(a[key], b[key], atol=1e-11, err_msg=key)


@pytest.mark.parametrize("m,n", [(6, 9), (9, 6), (8, 8), (1, 5), (5, 1)])
@pytest.mark.parametrize("steps", [1, 3, 5])
def test_newton_schulz_rows_closed_form(m, n, steps):
    """Sampled rows of Newton-Schulz through the step recursion equal the
    same rows of U p_k(S / (||Y||_F + eps)) V^T from the exact SVD."""
    rng = np.random.default_rng(m * 7 + n + 3 * steps)
    Y = _rand(rng, m, n)
    rows = np.arange(m)[::2] if m > 1 else np.array([0])
    got = oracle.dense.newton_schulz_rows(Y, rows, steps, oracle.QUINTIC, oracle.NS_EPS)
    want = _ns_closed_form(Y, steps, oracle.QUINTIC, oracle.NS_EPS)[rows]
    np.testing.assert_allclose(got, want, atol=1e-12)
    # and with the cubic coefficients (a different polynomial: pins the coefficient order)
    got = oracle.dense.newton_schulz_rows(Y, rows, steps, oracle.CUBIC, oracle.NS_EPS)
    np.testing.assert_allclose(got, _ns_closed_form(Y, steps, oracle.CUBIC, oracle.NS_EPS)[rows], atol=1e-12)
