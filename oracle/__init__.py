"""Oracle for the orthonormalized optimizer step -- TEST INFRASTRUCTURE ONLY.

A plain double-precision CPU statement of the legacy Dion step (amortized
power iteration with error feedback) and of Muon's Newton-Schulz
orthogonalization, in ``dion_oracle.c``.  Only ``tests/``, the smoke check and
the benchmark's CPU-baseline leg may import this package.  The library's
product path never does, and the two share no code: this package imports
nothing from the CUDA library, and the CUDA library knows nothing of it.

Sources: "Dion: The distributed orthonormal update revolution is here" (talk
page, orthonormal-update and Dion paragraphs), "Dion: Distributed
Orthonormalized Updates" (abstract), "microsoft/dion" project card ("How it
works", "Highlights").

Every routine here has a pin in ``tests/test_oracle.py`` (closed forms, special
cases, brute force against an exact SVD from numpy, hand-derived golden
values).  Storage rounding (fp32, bf16 round-to-nearest-even) is emulated by
``round_f32`` / ``round_bf16``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dion_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Newton-Schulz coefficient sets.  The pages name Newton-Schulz but print no
# coefficients.  QUINTIC is the quintic published with Muon itself (the Keller
# Jordan blog post, which the project review page names as Muon's source; the
# numbers are not on the pages).  CUBIC is the textbook Newton-Schulz polar
# iteration, which converges to U V^T for ||Y||_2 < sqrt(3).
QUINTIC = (3.4445, -4.7750, 2.0315)
CUBIC = (1.5, -0.5, 0.0)
NS_EPS = 1e-7


def build(force: bool = False) -> str:
    """Compile dion_oracle.c into liboracle.so with gcc (OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_householder_qr.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp]
            lib.oracle_dion_step.argtypes = [ctypes.c_int] * 3 + [dp] * 4 + [ctypes.c_double] * 3 + [dp, dp]
            lib.oracle_newton_schulz.argtypes = [ctypes.c_int] * 3 + [ctypes.c_double] * 4 + [dp, dp]
            lib.oracle_muon_step.argtypes = ([ctypes.c_int] * 4 + [ctypes.c_double] * 4
                                             + [dp] * 4 + [ctypes.c_double] * 3)
            for f in (lib.oracle_householder_qr, lib.oracle_dion_step,
                      lib.oracle_newton_schulz, lib.oracle_muon_step):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def householder_qr(A):
    """Thin QR by Householder reflections: returns (Qf, Rq), diag(Rq) >= 0."""
    Qf = _f64(A).copy()
    m, r = Qf.shape
    Rq = np.zeros((r, r))
    rc = _load().oracle_householder_qr(m, r, _ptr(Qf), _ptr(Rq))
    if rc != 0:
        raise ValueError("oracle_householder_qr: bad arguments")
    return Qf, Rq


def dion_step(X, G, M, Q, mu, lr, wd):
    """One Dion step on one matrix (all float64).  Returns a dict with the new
    X, M, Q and this step's P (m x r) and R (n x r); the inputs are not
    modified."""
    X = _f64(X).copy(); M = _f64(M).copy(); Q = _f64(Q).copy(); G = _f64(G)
    m, n = X.shape
    r = Q.shape[1]
    P = np.zeros((m, r)); R = np.zeros((n, r))
    rc = _load().oracle_dion_step(m, n, r, _ptr(X), _ptr(G), _ptr(M), _ptr(Q),
                                  float(mu), float(lr), float(wd), _ptr(P), _ptr(R))
    if rc != 0:
        raise ValueError("oracle_dion_step: bad arguments")
    return {"X": X, "M": M, "Q": Q, "P": P, "R": R}


def newton_schulz(Y, steps=5, coeff=QUINTIC, eps=NS_EPS):
    """Newton-Schulz orthogonalization of one matrix (float64)."""
    Y = _f64(Y)
    m, n = Y.shape
    O = np.zeros((m, n))
    a, b, c = coeff
    rc = _load().oracle_newton_schulz(m, n, int(steps), a, b, c, eps, _ptr(Y), _ptr(O))
    if rc != 0:
        raise ValueError("oracle_newton_schulz: bad arguments")
    return O


def muon_step(X, G, M, *, head_dim=0, steps=5, coeff=QUINTIC, eps=NS_EPS,
              mu=0.95, lr=0.02, wd=0.0):
    """One Muon step on one parameter.  X and M may be None.  Returns a dict
    with O (the orthogonalized update) and the new X and M (None where the
    input was None); the inputs are not modified."""
    G = _f64(G)
    m, n = G.shape
    Xc = None if X is None else _f64(X).copy()
    Mc = None if M is None else _f64(M).copy()
    O = np.zeros((m, n))
    a, b, c = coeff
    rc = _load().oracle_muon_step(m, n, int(head_dim), int(steps), a, b, c, eps,
                                  _ptr(Xc), _ptr(G), _ptr(Mc), _ptr(O),
                                  float(mu), float(lr), float(wd))
    if rc != 0:
        raise ValueError("oracle_muon_step: bad arguments")
    return {"O": O, "X": Xc, "M": Mc}


def round_f32(x):
    """Storage emulation: round to fp32 (nearest-even), returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_bf16(x):
    """Storage emulation: round to bfloat16 (nearest-even from the fp32 value,
    the precision the kernels compute in), returned as float64."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = ((u + 0x7FFF + lsb) >> 16) & 0xFFFF
    nan = np.isnan(f)
    rounded = np.where(nan, (u >> 16) | 0x40, rounded).astype(np.uint32)
    out = (rounded << 16).astype(np.uint32).view(np.float32)
    return out.astype(np.float64)
