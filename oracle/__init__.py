"""fp64 CPU oracle for F^H D, Q, batched F^H D, the forward model, (in
``oracle.toeplitz``) the Toeplitz F^H F product and the CG solve, and (in
``oracle.gridding``) the gridding / inverse-DFT reconstruction.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path (the CUDA library and
its Python binding) never imports this package, and this package imports
nothing from the product path.

The arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP over
independent voxels); this module builds it with gcc and wraps it with ctypes.
The PSNR metric is here in numpy.

Every function is pinned by CPU tests against closed forms; none is
"parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, OpenMP, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _idx(idx, N):
    if idx is None:
        return None, N, None
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= N):
        raise IndexError("voxel index out of range")
    return idx, int(idx.size), idx.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes wrapper around one build of oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_threads.argtypes = [ctypes.c_int]
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_mu.argtypes = [_i64, _f32p, _f32p, _f32p, _f32p, _f64p, _f64p]
        lib.oracle_mu.restype = None
        idxp = ctypes.c_void_p
        lib.oracle_fhd.argtypes = ([_i64] + [_f32p] * 3 + [_f32p] * 4 + [_f32p] * 3
                                   + [_i64, idxp, _f64p, _f64p, _f64p, _f64p, ctypes.c_int])
        lib.oracle_fhd.restype = None
        lib.oracle_q.argtypes = ([_i64] + [_f32p] * 3 + [_f32p] * 2 + [_f32p] * 3
                                 + [_i64, idxp, _f64p, _f64p, _f64p, ctypes.c_int])
        lib.oracle_q.restype = None
        lib.oracle_fhd_batched.argtypes = ([_i64, _i64] + [_f32p] * 3 + [_f32p] * 4
                                           + [_f32p] * 3
                                           + [_i64, idxp, _f64p, _f64p, _f64p, _f64p,
                                              ctypes.c_int])
        lib.oracle_fhd_batched.restype = None
        lib.oracle_forward.argtypes = ([_i64] + [_f32p] * 3 + [_i64] + [_f32p] * 3
                                       + [_f64p, _f64p, _f64p, _f64p, ctypes.c_int])
        lib.oracle_forward.restype = None
        self.lib = lib
        self.path = path

    def threads(self, n: int = 0) -> int:
        """Set (n > 0) and return the OpenMP thread count the oracle will use."""
        return int(self.lib.oracle_threads(int(n)))

    def mu(self, rPhi, iPhi, rD, iD):
        """cmpMu: Mu = conj(Phi) * D, returned as complex128 [M]."""
        rPhi, iPhi, rD, iD = map(_f32, (rPhi, iPhi, rD, iD))
        M = rPhi.size
        rMu = np.empty(M, np.float64)
        iMu = np.empty(M, np.float64)
        self.lib.oracle_mu(M, rPhi, iPhi, rD, iD, rMu, iMu)
        return rMu + 1j * iMu

    def fhd(self, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD, idx=None, threads: int = 0):
        """F^H D[n] = sum_m conj(Phi_m) D_m e^{+i 2 pi k_m . x_n}, complex128.

        ``idx`` selects a voxel subset (output j is voxel idx[j]).
        """
        kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD = map(
            _f32, (kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD))
        M, N = kx.size, x.size
        idx, nout, idxp = _idx(idx, N)
        re = np.empty(nout, np.float64)
        im = np.empty(nout, np.float64)
        mr = np.empty(max(M, 1), np.float64)
        mi = np.empty(max(M, 1), np.float64)
        self.lib.oracle_fhd(M, kx, ky, kz, rPhi, iPhi, rD, iD, x, y, z, nout, idxp,
                            re, im, mr, mi, int(threads))
        return re + 1j * im

    def q(self, kx, ky, kz, x, y, z, rPhi, iPhi, idx=None, threads: int = 0):
        """Q[n] = sum_m |Phi_m|^2 e^{+i 2 pi k_m . x_n}, complex128."""
        kx, ky, kz, x, y, z, rPhi, iPhi = map(_f32, (kx, ky, kz, x, y, z, rPhi, iPhi))
        M, N = kx.size, x.size
        idx, nout, idxp = _idx(idx, N)
        re = np.empty(nout, np.float64)
        im = np.empty(nout, np.float64)
        w = np.empty(max(M, 1), np.float64)
        self.lib.oracle_q(M, kx, ky, kz, rPhi, iPhi, x, y, z, nout, idxp, re, im, w,
                          int(threads))
        return re + 1j * im

    def fhd_batched(self, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD, idx=None,
                    threads: int = 0):
        """Batched F^H D: rD, iD are [B, M] (coil-major); returns complex128 [B, nout]."""
        kx, ky, kz, x, y, z, rPhi, iPhi = map(_f32, (kx, ky, kz, x, y, z, rPhi, iPhi))
        rD, iD = _f32(rD), _f32(iD)
        B, M = rD.shape
        N = x.size
        idx, nout, idxp = _idx(idx, N)
        re = np.empty(B * nout, np.float64)
        im = np.empty(B * nout, np.float64)
        mr = np.empty(max(M, 1), np.float64)
        mi = np.empty(max(M, 1), np.float64)
        self.lib.oracle_fhd_batched(B, M, kx, ky, kz, rPhi, iPhi, rD.reshape(-1),
                                    iD.reshape(-1), x, y, z, nout, idxp, re, im, mr, mi,
                                    int(threads))
        return (re + 1j * im).reshape(B, nout)

    def forward(self, kx, ky, kz, x, y, z, rho, threads: int = 0):
        """Forward model D[m] = sum_n rho[n] e^{-i 2 pi k_m . x_n}, complex128 [M]."""
        kx, ky, kz, x, y, z = map(_f32, (kx, ky, kz, x, y, z))
        rho = np.asarray(rho)
        rr = np.ascontiguousarray(rho.real, dtype=np.float64)
        ri = np.ascontiguousarray(np.imag(rho), dtype=np.float64)
        M, N = kx.size, x.size
        rD = np.empty(M, np.float64)
        iD = np.empty(M, np.float64)
        self.lib.oracle_forward(M, kx, ky, kz, N, x, y, z, rr, ri, rD, iD, int(threads))
        return rD + 1j * iD


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
        return _lib


def use(instance: Oracle | None) -> Oracle | None:
    """Route the module-level functions to another build (None: the default).

    Returns the previous instance.  Used by the mutation test, which swaps in
    deliberately broken builds to show the pins reject them.
    """
    global _lib
    with _lock:
        prev, _lib = _lib, instance
        return prev


def threads(n: int = 0) -> int:
    return _default().threads(n)


def mu(*a, **k):
    return _default().mu(*a, **k)


def fhd(*a, **k):
    return _default().fhd(*a, **k)


def q(*a, **k):
    return _default().q(*a, **k)


def fhd_batched(*a, **k):
    return _default().fhd_batched(*a, **k)


def forward(*a, **k):
    return _default().forward(*a, **k)


threads.__doc__ = Oracle.threads.__doc__
mu.__doc__ = Oracle.mu.__doc__
fhd.__doc__ = Oracle.fhd.__doc__
q.__doc__ = Oracle.q.__doc__
fhd_batched.__doc__ = Oracle.fhd_batched.__doc__
forward.__doc__ = Oracle.forward.__doc__


def psnr(ideal, image) -> float:
    """Peak signal-to-noise ratio, 20*log10(max|I0| / sqrt(MSE)) in dB.

    The practice page on the chapter states this form for the accuracy metric
    of Fig. 17.18; for complex images the peak is max |I0| and the MSE is the
    mean over voxels of |I - I0|^2.
    """
    ideal = np.asarray(ideal)
    image = np.asarray(image)
    mse = float(np.mean(np.abs(image - ideal) ** 2))
    peak = float(np.max(np.abs(ideal)))
    if mse == 0.0:
        return float("inf")
    return 20.0 * np.log10(peak / np.sqrt(mse))


def rel_l2(test, ref) -> float:
    """||test - ref||_2 / ||ref||_2 over real and imaginary parts."""
    test = np.asarray(test, dtype=np.complex128)
    ref = np.asarray(ref, dtype=np.complex128)
    den = float(np.sqrt(np.sum(np.abs(ref) ** 2)))
    num = float(np.sqrt(np.sum(np.abs(test - ref) ** 2)))
    return num / den if den > 0 else num
