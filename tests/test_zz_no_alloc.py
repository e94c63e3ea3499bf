"""dion_step_batched_static: the Dion step for callers that cannot allocate
device memory (their device memory is owned by another allocator, or an
allocation's possible device synchronization is not acceptable on their
path).  Its scratch is a fixed array inside libdion.  This file is collected
last on purpose, so that a run stopping at the first failure has already run
every other test; it also passes when run alone in a fresh process, where
its first call is the one that sets the array up."""
import ctypes

import pytest
import torch

import workloads as wl
import orthonormal_optimizer_step_gb300 as od
from parity import TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _raw_static(X, G, M, Q, mu, lr, wd, dt):
    """Calls the C entry point directly (no binding-level checks)."""
    b, m, n = X.shape
    r = Q.shape[-1]
    return od.lib().dion_step_batched_static(b, m, n, r, dt, X.data_ptr(), G.data_ptr(), M.data_ptr(), Q.data_ptr(),
                                             ctypes.c_float(mu), ctypes.c_float(lr), ctypes.c_float(wd),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype,shape", [(torch.float32, (1, 256, 256, 64)), (torch.bfloat16, (3, 256, 384, 48))])
def test_static_scratch_matches_workspace_entry(dtype, shape):
    batch, m, n, r = shape
    g = wl.Group(batch, m, n)
    dt = od.DION_BF16 if dtype == torch.bfloat16 else od.DION_F32
    X, M, Q = wl.make_state(g, r, dtype, DEV, seed=31)
    M = wl.make_momentum(g, 0.5, DEV, seed=31)
    A = [t.clone() for t in (X, M, Q)]      # driven by dion_step_batched (caller workspace)
    B = [t.clone() for t in (X, M, Q)]      # driven by dion_step_batched_static
    for step in range(2):                   # two calls in a row: the shared scratch is reused
        G = wl.make_grad(g, 1.0, dtype, DEV, seed=31, step=step)
        od.dion_step_batched(A[0], G, A[1], A[2], mu=0.95, lr=0.05, weight_decay=0.01)
        code = _raw_static(B[0], G, B[1], B[2], 0.95, 0.05, 0.01, dt)
        assert code == od.DION_OK, od.status_string(code)
        torch.cuda.synchronize()
        tol = TOL[dtype]
        for a, b in zip(A, B):
            err = (a.double() - b.double()).norm() / a.double().norm()
            assert err <= tol, (step, float(err))


def test_static_scratch_rejects_shapes_beyond_its_size():
    # 12 x 768 x 2304 at rank 192 (bf16) needs more than the fixed scratch holds
    need = od.dion_workspace_size(12, 768, 2304, 192, od.DION_BF16)
    assert need > od.STATIC_SCRATCH_BYTES
    X = torch.zeros((12, 768, 2304), dtype=torch.bfloat16, device=DEV)
    M = torch.zeros((12, 768, 2304), dtype=torch.float32, device=DEV)
    Q = torch.zeros((12, 2304, 192), dtype=torch.float32, device=DEV)
    with pytest.raises(od.DionError) as ei:
        od.dion_step_batched_static(X, X, M, Q, mu=0.9, lr=0.01)
    assert ei.value.code == od.DION_ERR_WORKSPACE
