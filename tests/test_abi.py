"""CPU-only checks of the C ABI: the library builds, loads and exports every
symbol include/*.h declares; host-side argument validation rejects bad calls
before anything touches the device."""
import ctypes
import glob
import os
import re

import pytest

import orthonormal_optimizer_step_gb300 as od
from orthonormal_optimizer_step_gb300 import build as odbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    odbuild.build()
    return od.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"dion_step_batched", "muon_ns_batched", "dion_workspace_size", "dion_get_status"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(od.EXPORTS)


def test_status_strings(lib):
    for code in range(6):
        assert od.status_string(code)
    assert od.status_string(5) == "numeric breakdown on the device"


def test_workspace_size_validation(lib):
    out = ctypes.c_size_t()
    assert lib.dion_workspace_size(1, 256, 256, 64, 0, ctypes.byref(out)) == 0 and out.value > 0
    assert lib.dion_workspace_size(1, 256, 256, 0, 0, ctypes.byref(out)) == od.DION_ERR_INVALID_ARG
    assert lib.dion_workspace_size(1, 256, 100, 101, 1, ctypes.byref(out)) == od.DION_ERR_INVALID_ARG
    assert lib.dion_workspace_size(0, 256, 256, 64, 1, ctypes.byref(out)) == od.DION_ERR_INVALID_ARG
    assert lib.dion_workspace_size(1, 256, 256, 64, 7, ctypes.byref(out)) == od.DION_ERR_INVALID_ARG
    assert lib.dion_workspace_size(1, 256, 256, 64, 0, None) == od.DION_ERR_INVALID_ARG
    assert lib.muon_workspace_size(12, 768, 2304, 64, 1, ctypes.byref(out)) == 0 and out.value > 0
    assert lib.muon_workspace_size(12, 768, 2304, 100, 1, ctypes.byref(out)) == od.DION_ERR_INVALID_ARG
    # bigger rank never needs less workspace
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    lib.dion_workspace_size(2, 512, 384, 16, 1, ctypes.byref(a))
    lib.dion_workspace_size(2, 512, 384, 128, 1, ctypes.byref(b))
    assert b.value > a.value


def test_step_rejects_bad_arguments_before_launch(lib):
    """All of these fail on the host; no CUDA call is made (works without a GPU)."""
    big = ctypes.c_size_t(1 << 40)
    fake = ctypes.c_void_p(1 << 20)        # never dereferenced: validation fails first
    ws = ctypes.c_void_p(1 << 24)
    # empty megabatch or empty matrices
    for (b, m, n) in [(0, 64, 64), (1, 0, 64), (1, 64, 0), (-1, 64, 64)]:
        assert lib.dion_step_batched(b, m, n, 1, 0, fake, fake, fake, fake, 0.9, 0.01, 0.0, ws, big, None) \
            == od.DION_ERR_INVALID_ARG
        assert lib.muon_ns_batched(b, m, n, 0, 1, fake, fake, None, None, 5,
                                   (ctypes.c_float * 3)(3.4445, -4.775, 2.0315), 0.9, 0.01, 0.0, ws, big, None) \
            == od.DION_ERR_INVALID_ARG
    # null pointers
    assert lib.dion_step_batched(1, 64, 64, 8, 0, None, fake, fake, fake, 0.9, 0.01, 0.0, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    # rank out of range
    assert lib.dion_step_batched(1, 64, 32, 33, 0, fake, fake, fake, fake, 0.9, 0.01, 0.0, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    # misaligned pointer
    assert lib.dion_step_batched(1, 64, 64, 8, 0, ctypes.c_void_p((1 << 20) + 4), fake, fake, fake, 0.9, 0.01, 0.0,
                                 ws, big, None) == od.DION_ERR_INVALID_ARG
    # non-finite hyper-parameter
    assert lib.dion_step_batched(1, 64, 64, 8, 0, fake, fake, fake, fake, float("nan"), 0.01, 0.0, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    # workspace missing / too small / misaligned
    assert lib.dion_step_batched(1, 64, 64, 8, 0, fake, fake, fake, fake, 0.9, 0.01, 0.0, None, big, None) \
        == od.DION_ERR_WORKSPACE
    assert lib.dion_step_batched(1, 64, 64, 8, 0, fake, fake, fake, fake, 0.9, 0.01, 0.0, ws, 16, None) \
        == od.DION_ERR_WORKSPACE
    assert lib.dion_step_batched(1, 64, 64, 8, 0, fake, fake, fake, fake, 0.9, 0.01, 0.0,
                                 ctypes.c_void_p((1 << 24) + 16), big, None) == od.DION_ERR_WORKSPACE
    # device-scalar variant: missing or misaligned hyper, and the shape checks of dion_step_batched
    assert lib.dion_step_batched_dev(1, 64, 64, 8, 0, fake, fake, fake, fake, None, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    assert lib.dion_step_batched_dev(1, 64, 64, 8, 0, fake, fake, fake, fake, ctypes.c_void_p((1 << 20) + 2), ws, big,
                                     None) == od.DION_ERR_INVALID_ARG
    assert lib.dion_step_batched_dev(1, 64, 32, 33, 0, fake, fake, fake, fake, fake, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    assert lib.dion_step_batched_dev(1, 64, 64, 8, 0, fake, fake, fake, fake, fake, ws, 16, None) \
        == od.DION_ERR_WORKSPACE
    coeff = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    # Muon: neither X nor O
    assert lib.muon_ns_batched(1, 64, 64, 0, 1, None, fake, None, None, 5, coeff, 0.9, 0.01, 0.0, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    # Muon: head_dim does not divide n
    assert lib.muon_ns_batched(1, 64, 60, 16, 1, fake, fake, None, None, 5, coeff, 0.9, 0.01, 0.0, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    # Muon: negative steps, missing coefficients
    assert lib.muon_ns_batched(1, 64, 64, 0, 1, fake, fake, None, None, -1, coeff, 0.9, 0.01, 0.0, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    assert lib.muon_ns_batched(1, 64, 64, 0, 1, fake, fake, None, None, 5, None, 0.9, 0.01, 0.0, ws, big, None) \
        == od.DION_ERR_INVALID_ARG
    assert lib.dion_get_status(None, None) == od.DION_ERR_INVALID_ARG


def test_panels_lie_inside_workspace(lib):
    for (b, m, n, r, dt) in [(1, 256, 256, 64, 0), (12, 768, 2304, 192, 1), (3, 200, 136, 24, 1)]:
        size = od.dion_workspace_size(b, m, n, r, dt)
        po, pl, ro, rl = od.dion_workspace_panels(b, m, n, r, dt)
        assert pl >= r and rl >= r
        assert po % 16 == 0 and ro % 16 == 0
        assert po + b * m * pl * 4 <= size and ro + b * n * rl * 4 <= size
