"""Argument errors that need a device to detect, through the C ABI: a host
pointer where device memory is required (MRI_ERR_NOT_DEVICE), a device
pointer off the 4-byte grid (MRI_ERR_ALIGN), and that a rejected call leaves
the outputs, the device error word and the next call untouched.  Every
entry point that takes device arrays is tried, each argument in turn."""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

OK, NULL, SIZE, ALIGN, NOT_DEVICE, MODE = 0, 1, 2, 3, 4, 5
P = ctypes.c_void_p
I64 = ctypes.c_int64
I = ctypes.c_int


@pytest.fixture(scope="module")
def mri():
    from non_cartesian_mri_gb300 import build
    build.build()
    import non_cartesian_mri_gb300 as m
    return m


@pytest.fixture(scope="module")
def lib(mri):
    return mri.load()


def ptr(t):
    return P(t.data_ptr())


def calls(lib, M, nx, ny, nz):
    """(name, function taking a list of pointers, number of pointers)."""
    N = nx * ny * nz

    def fhd(p):
        f = lib.mri_fhd
        f.argtypes = [P] * 10 + [I64, I64, P, P, I, I, P]
        return f(*p[:10], M, N, p[10], p[11], 1, 0, None)

    def q(p):
        f = lib.mri_q
        f.argtypes = [P] * 8 + [I64, I64, P, P, I, I, P]
        return f(*p[:8], M, N, p[8], p[9], 1, 0, None)

    def fhd_grid(p):
        f = lib.mri_fhd_grid
        f.argtypes = [P, P, P, P, I, P, I, P, I, P, P, P, P, I64, P, P, I, I, P]
        return f(p[0], p[1], p[2], p[3], nx, p[4], ny, p[5], nz, p[6], p[7], p[8], p[9], M,
                 p[10], p[11], 1, 0, None)

    def forward_grid(p):
        f = lib.mri_forward_grid
        f.argtypes = [P, P, P, P, I, P, I, P, I, P, P, I64, P, P, I, I, P]
        return f(p[0], p[1], p[2], p[3], nx, p[4], ny, p[5], nz, p[6], p[7], M, p[8], p[9],
                 1, 0, None)

    def fhd_noalloc(p):
        f = lib.mri_fhd_noalloc
        f.argtypes = [P] * 10 + [I64, I64, P, P, I, I, P]
        return f(*p[:10], M, N, p[10], p[11], 1, 0, None)

    return [("mri_fhd", fhd, 12), ("mri_q", q, 10), ("mri_fhd_grid", fhd_grid, 12),
            ("mri_forward_grid", forward_grid, 10), ("mri_fhd_noalloc", fhd_noalloc, 12)]


def test_host_and_misaligned_pointers(mri, lib):
    M, nx, ny, nz = 300, 16, 4, 3
    n = max(M, nx * ny * nz, 64)
    dev = [torch.full((n + 1,), 0.5, device="cuda") for _ in range(12)]
    host = np.zeros(n + 1, np.float32)
    for name, fn, k in calls(lib, M, nx, ny, nz):
        good = [ptr(t) for t in dev[:k]]
        assert fn(good) == OK, name
        torch.cuda.synchronize()
        outs = [t.clone() for t in dev[k - 2:k]]
        for i in range(k):
            bad = list(good)
            bad[i] = P(host.ctypes.data)
            assert fn(bad) == NOT_DEVICE, f"{name}: host pointer in slot {i}"
            bad[i] = P(dev[i].data_ptr() + 2)
            assert fn(bad) == ALIGN, f"{name}: misaligned slot {i}"
        torch.cuda.synchronize()
        # rejected calls launched nothing: the outputs are as the good call left them
        for a, b in zip(outs, dev[k - 2:k]):
            assert torch.equal(a, b), name
    assert mri.device_errors(clear=True) == 0
    # and the library still works
    assert calls(lib, M, nx, ny, nz)[2][1]([ptr(t) for t in dev[:12]]) == OK
    torch.cuda.synchronize()
    assert mri.device_errors(clear=True) == 0


def test_pinned_host_memory_is_not_device_memory(mri, lib):
    """Page-locked host memory is mapped for the device but is not device
    memory of the current device: rejected, not read through PCIe/C2C."""
    M, nx, ny, nz = 100, 16, 2, 2
    dev = [torch.zeros(256, device="cuda") for _ in range(12)]
    pinned = torch.zeros(256).pin_memory()
    for name, fn, k in (calls(lib, M, nx, ny, nz)[2], calls(lib, M, nx, ny, nz)[4]):
        for slot in (0, k - 1):
            p = [ptr(t) for t in dev[:k]]
            p[slot] = ptr(pinned)
            assert fn(p) == NOT_DEVICE, f"{name}: pinned host memory in slot {slot}"
