"""Orthonormalized optimizer step (Dion power iteration, Muon Newton-Schulz)
on one NVIDIA GB300.

A thin ctypes binding over libdion.so (C ABI in include/dion.h).  The binding
only marshals arguments: every step of the computation runs in libdion's CUDA
kernels.  PyTorch supplies device memory and the current CUDA stream.  If
libdion.so is missing the import of a function raises; there is no fallback.

    from orthonormal_optimizer_step_gb300 import dion_step_batched, muon_ns_batched
    dion_step_batched(X, G, M, Q, mu=0.95, lr=0.01, weight_decay=0.01)
    muon_ns_batched(G, X=X, M=M, head_dim=64)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdion.so")

DION_OK, DION_ERR_INVALID_ARG, DION_ERR_UNSUPPORTED, DION_ERR_WORKSPACE, DION_ERR_CUDA, DION_ERR_NUMERIC = range(6)
DION_F32, DION_BF16 = 0, 1

# The exported symbols of include/dion.h.
EXPORTS = ("dion_workspace_size", "dion_workspace_panels", "dion_step_batched", "dion_step_batched_dev",
           "dion_step_batched_static", "muon_workspace_size", "muon_ns_batched",
           "dion_get_status", "dion_status_string", "dion_profile_begin", "dion_profile_end",
           "dion_profile_count", "dion_profile_entry", "dion_profile_dropped")

# Muon's published quintic Newton-Schulz coefficients (a, b, c).
QUINTIC = (3.4445, -4.7750, 2.0315)

_lock = threading.Lock()
_lib = None


class DionError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def lib() -> ctypes.CDLL:
    """The loaded libdion.so with argument types declared (raises if not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libdion.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        c_int, c_float, c_size, vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p
        L.dion_workspace_size.argtypes = [c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(c_size)]
        L.dion_workspace_panels.argtypes = [c_int] * 5 + [ctypes.POINTER(c_size), ctypes.POINTER(c_int),
                                                          ctypes.POINTER(c_size), ctypes.POINTER(c_int)]
        L.dion_step_batched.argtypes = ([c_int] * 5 + [vp, vp, vp, vp] + [c_float] * 3 + [vp, c_size, vp])
        L.dion_step_batched_static.argtypes = ([c_int] * 5 + [vp, vp, vp, vp] + [c_float] * 3 + [vp])
        L.dion_step_batched_dev.argtypes = ([c_int] * 5 + [vp, vp, vp, vp, vp] + [vp, c_size, vp])
        L.muon_workspace_size.argtypes = [c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(c_size)]
        L.muon_ns_batched.argtypes = ([c_int] * 5 + [vp, vp, vp, vp, c_int, ctypes.POINTER(c_float)]
                                      + [c_float] * 3 + [vp, c_size, vp])
        L.dion_get_status.argtypes = [vp, ctypes.POINTER(c_int)]
        L.dion_status_string.argtypes = [c_int]
        L.dion_status_string.restype = ctypes.c_char_p
        L.dion_profile_begin.argtypes = [c_int]
        L.dion_profile_end.argtypes = []
        L.dion_profile_count.argtypes = []
        L.dion_profile_dropped.argtypes = []
        L.dion_profile_entry.argtypes = [c_int, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(c_int),
                                         ctypes.POINTER(ctypes.c_double)]
        for f in ("dion_workspace_size", "dion_workspace_panels", "dion_step_batched", "dion_step_batched_dev",
                  "dion_step_batched_static", "muon_workspace_size", "muon_ns_batched",
                  "dion_get_status", "dion_profile_begin", "dion_profile_end", "dion_profile_count",
                  "dion_profile_entry", "dion_profile_dropped"):
            getattr(L, f).restype = c_int
        _lib = L
        return L


def status_string(code: int) -> str:
    return lib().dion_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != DION_OK:
        raise DionError(code, where)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DION_F32
    if t.dtype == torch.bfloat16:
        return DION_BF16
    raise TypeError(f"X/G must be float32 or bfloat16, got {t.dtype}")


def _stream_ptr(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _shape3(t):
    if t.dim() == 2:
        return 1, t.shape[0], t.shape[1]
    if t.dim() == 3:
        return t.shape[0], t.shape[1], t.shape[2]
    raise ValueError("expected a [batch, m, n] or [m, n] tensor")


def dion_workspace_size(batch: int, m: int, n: int, r: int, dtype: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().dion_workspace_size(batch, m, n, r, dtype, ctypes.byref(out)), "dion_workspace_size")
    return out.value


def dion_workspace_panels(batch: int, m: int, n: int, r: int, dtype: int):
    """(P byte offset, P row stride, R byte offset, R row stride) in floats."""
    po, pl, ro, rl = ctypes.c_size_t(), ctypes.c_int(), ctypes.c_size_t(), ctypes.c_int()
    _check(lib().dion_workspace_panels(batch, m, n, r, dtype, ctypes.byref(po), ctypes.byref(pl), ctypes.byref(ro),
                                       ctypes.byref(rl)), "dion_workspace_panels")
    return po.value, pl.value, ro.value, rl.value


def dion_panels(workspace, batch: int, m: int, n: int, r: int, dtype: int):
    """Views (P [batch, m, r], R [batch, n, r], float32) into a workspace after
    a completed dion_step_batched."""
    import torch
    po, pl, ro, rl = dion_workspace_panels(batch, m, n, r, dtype)
    f = workspace.view(torch.uint8)
    P = f[po:po + batch * m * pl * 4].view(torch.float32).view(batch, m, pl)[:, :, :r]
    R = f[ro:ro + batch * n * rl * 4].view(torch.float32).view(batch, n, rl)[:, :, :r]
    return P, R


def muon_workspace_size(batch: int, m: int, n: int, head_dim: int, dtype: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().muon_workspace_size(batch, m, n, head_dim, dtype, ctypes.byref(out)), "muon_workspace_size")
    return out.value


def new_workspace(nbytes: int, device):
    """Caller-owned device workspace (256-byte aligned by the torch allocator)."""
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def dion_step_batched(X, G, M, Q, *, mu: float = None, lr: float = None, weight_decay: float = 0.0, hyper=None,
                      workspace=None, stream=None):
    """One Dion step on a megabatch: X, G [batch, m, n] (fp32 or bf16), M
    [batch, m, n] fp32 and Q [batch, n, r] fp32 are CUDA tensors; X, M and Q
    are updated in place.  Returns the workspace used (it holds the status
    word, see dion_get_status).  With `hyper` (a float32 CUDA tensor holding
    mu, lr, weight_decay) the scalars are read on the device when the step
    runs (dion_step_batched_dev), so a CUDA graph of the call follows new
    values written into `hyper`; mu, lr and weight_decay are then ignored."""
    batch, m, n = _shape3(X)
    r = Q.shape[-1]
    dt = _dtype_code(X)
    for t in (X, G, M, Q):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if workspace is None:
        workspace = new_workspace(dion_workspace_size(batch, m, n, r, dt), X.device)
    if hyper is not None:
        if hyper.dtype.itemsize != 4 or hyper.numel() < 3 or not hyper.is_contiguous() or not hyper.is_cuda:
            raise ValueError("hyper must be a contiguous float32 CUDA tensor of (mu, lr, weight_decay)")
        code = lib().dion_step_batched_dev(batch, m, n, r, dt, _ptr(X), _ptr(G), _ptr(M), _ptr(Q), _ptr(hyper),
                                           _ptr(workspace), workspace.numel(), _stream_ptr(stream))
        _check(code, "dion_step_batched_dev")
        return workspace
    if mu is None or lr is None:
        raise ValueError("mu and lr are required unless hyper is given")
    code = lib().dion_step_batched(batch, m, n, r, dt, _ptr(X), _ptr(G), _ptr(M), _ptr(Q), float(mu), float(lr),
                                   float(weight_decay), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(code, "dion_step_batched")
    return workspace


STATIC_SCRATCH_BYTES = 64 << 20


def dion_step_batched_static(X, G, M, Q, *, mu: float, lr: float, weight_decay: float = 0.0, stream=None):
    """dion_step_batched for callers that cannot allocate device memory: the
    scratch is a fixed array of STATIC_SCRATCH_BYTES inside libdion, shared by
    all calls on a device (serialize them).  Shapes needing more scratch raise
    DionError (DION_ERR_WORKSPACE).  The first call on a device sets up the
    array's address; make it before any stream capture."""
    batch, m, n = _shape3(X)
    r = Q.shape[-1]
    dt = _dtype_code(X)
    for t in (X, G, M, Q):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    code = lib().dion_step_batched_static(batch, m, n, r, dt, _ptr(X), _ptr(G), _ptr(M), _ptr(Q), float(mu),
                                          float(lr), float(weight_decay), _stream_ptr(stream))
    _check(code, "dion_step_batched_static")


def muon_ns_batched(G, *, X=None, M=None, O=None, head_dim: int = 0, steps: int = 5,
                    coeff: Sequence[float] = QUINTIC, mu: float = 0.95, lr: float = 0.02,
                    weight_decay: float = 0.0, workspace=None, stream=None):
    """One Muon step on a megabatch G [batch, m, n] (fp32 or bf16): optional
    momentum M (fp32, updated), optional weights X (updated) and optional
    output O (the orthogonalized update).  Returns the workspace used."""
    batch, m, n = _shape3(G)
    dt = _dtype_code(G)
    for t in (X, G, M, O):
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if workspace is None:
        workspace = new_workspace(muon_workspace_size(batch, m, n, head_dim, dt), G.device)
    cf = (ctypes.c_float * 3)(*[float(c) for c in coeff])
    code = lib().muon_ns_batched(batch, m, n, int(head_dim), dt, _ptr(X), _ptr(G), _ptr(M), _ptr(O), int(steps), cf,
                                 float(mu), float(lr), float(weight_decay), _ptr(workspace), workspace.numel(),
                                 _stream_ptr(stream))
    _check(code, "muon_ns_batched")
    return workspace


def dion_get_status(workspace) -> int:
    """Device status word of a workspace (synchronize first); 0 = healthy."""
    out = ctypes.c_int(0)
    code = lib().dion_get_status(_ptr(workspace), ctypes.byref(out))
    if code not in (DION_OK, DION_ERR_NUMERIC):
        _check(code, "dion_get_status")
    return out.value


class profile:
    """Context manager recording per-kernel CUDA-event times inside libdion."""

    def __init__(self, max_launches: int = 65536):
        self.max_launches = max_launches
        self.result = {}

    def __enter__(self):
        _check(lib().dion_profile_begin(self.max_launches), "dion_profile_begin")
        return self

    def __exit__(self, *exc):
        lib().dion_profile_end()
        return False

    def read(self):
        """{kernel name: (launches, total ms)}; synchronize before calling.
        Raises if launches went untimed because max_launches was too small."""
        L = lib()
        dropped = L.dion_profile_dropped()
        if dropped:
            raise RuntimeError(f"profile: {dropped} launches beyond max_launches={self.max_launches} were not timed")
        cnt = L.dion_profile_count()
        out = {}
        for i in range(cnt):
            name = ctypes.c_char_p()
            launches = ctypes.c_int()
            ms = ctypes.c_double()
            _check(L.dion_profile_entry(i, ctypes.byref(name), ctypes.byref(launches), ctypes.byref(ms)),
                   "dion_profile_entry")
            out[name.value.decode()] = (launches.value, ms.value)
        self.result = out
        return out
