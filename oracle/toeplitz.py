"""fp64 oracle of the "find rho" step: F^H F as a Toeplitz operator built
from Q, and the conjugate-gradient solve.

TEST INFRASTRUCTURE ONLY (as the rest of this package).

The chapter "Iterative MRI reconstruction" (background section, Fig. 17.3)
states the reconstruction as rho = (F^H F + lambda W^H W)^{-1} F^H D, solved
by conjugate gradients, whose cost per iteration is the product of
F^H F + lambda W^H W with the current rho; F^H F is a Toeplitz matrix, so
that product goes through FFTs, and Q (Stone et al. 2008) is the data that
lets it be formed without F^H F itself.  Readings taken here:

- F[m][n] = Phi_m e^{-i 2 pi k_m . x_n} (the sensitivity Phi inside F, so that
  F^H D is the F^H D of the chapter and (F^H F)[n][n'] = Q(x_n - x_n') with
  Q(d) = sum_m |Phi_m|^2 e^{+i 2 pi k_m . d}, the chapter's Q);
- the voxels are a regular grid x = (ix hx, iy hy, iz hz), so every
  difference x_n - x_n' is a grid vector and Q is needed on the differences
  -(n-1) .. n-1 per axis;
- W is not on the pages (it comes from the patient's scans): W = I, with
  lambda given by the caller (lambda = 0 allowed).

Functions: q_difference_grid (Q on the circular grid of differences, from
the oracle's own Q), fhf_direct (the definition: a sum over every voxel
pair), fhf_fft (the same product through numpy's FFT, the library
primitive the pages name), zero_unused_planes / toeplitz_spectrum /
fhf_spectrum (the real spectrum the product multiplies by, and the product
through it), cg (the conjugate-gradient iteration).  Pinned in
tests/test_oracle_toeplitz.py: fhf_direct against F^H (F rho) formed from
the oracle's forward model and F^H D, fhf_fft and fhf_spectrum against
fhf_direct, the spectrum's imaginary part against rounding (and the grid
without the zeroed planes against a large one), cg against a dense solve and
its own residuals.
"""

from __future__ import annotations

import numpy as np


def difference_axis(n: int, h: float) -> np.ndarray:
    """The 2n grid differences of one axis in circular order: i h for
    i < n, (i - 2n) h for i >= n (float32, as the device receives them)."""
    i = np.arange(2 * n)
    return (np.where(i < n, i, i - 2 * n) * h).astype(np.float32)


def q_difference_grid(kx, ky, kz, rPhi, iPhi, shape, spacing=(1.0, 1.0, 1.0), threads=0):
    """Q on the circular grid of voxel differences of a grid of shape
    (nz, ny, nx): complex128 array [2nz, 2ny, 2nx] whose element
    (jz, jy, jx) is Q(d) for d = (dx[jx], dy[jy], dz[jz]) of difference_axis."""
    from . import q
    nz, ny, nx = shape
    hx, hy, hz = spacing
    dx, dy, dz = difference_axis(nx, hx), difference_axis(ny, hy), difference_axis(nz, hz)
    z, y, x = np.meshgrid(dz, dy, dx, indexing="ij")
    Q = q(kx, ky, kz, x.reshape(-1), y.reshape(-1), z.reshape(-1), rPhi, iPhi, threads=threads)
    return Q.reshape(2 * nz, 2 * ny, 2 * nx)


def zero_unused_planes(Qc):
    """Qc with the planes at index n of every axis set to zero.  Those hold
    Q at the difference -n h, which no pair of voxels of an n grid has
    (differences stay within -(n-1) .. n-1), so the product is unchanged; with
    them gone the grid is Hermitian-symmetric, Qc[-j mod 2n] = conj(Qc[j])
    (Q(-d) is the conjugate of Q(d)), and its spectrum is real."""
    Z = np.array(Qc, dtype=np.complex128)
    nz, ny, nx = (s // 2 for s in Z.shape)
    Z[nz, :, :] = 0
    Z[:, ny, :] = 0
    Z[:, :, nx] = 0
    return Z


def toeplitz_spectrum(Qc):
    """The spectrum the product multiplies by: the real part of the FFT of
    zero_unused_planes(Qc), and the largest imaginary part dropped relative
    to the largest real one (rounding only: the pins check it)."""
    S = np.fft.fftn(zero_unused_planes(Qc))
    return S.real.copy(), float(np.abs(S.imag).max() / max(np.abs(S.real).max(), 1e-300))


def fhf_spectrum(Kr, rho):
    """F^H F rho through a real spectrum Kr of the doubled grid:
    crop(IFFT(Kr * FFT(zero-padded rho)))."""
    rho = np.asarray(rho, dtype=np.complex128)
    nz, ny, nx = rho.shape
    pad = np.zeros(Kr.shape, np.complex128)
    pad[:nz, :ny, :nx] = rho
    return np.fft.ifftn(Kr * np.fft.fftn(pad))[:nz, :ny, :nx]


def fhf_direct(Qc, rho):
    """(F^H F rho)[n] = sum_{n'} Q(x_n - x_n') rho[n'] over every voxel pair,
    rho and the result [nz, ny, nx] complex128 (O(N^2): small grids)."""
    rho = np.asarray(rho, dtype=np.complex128)
    nz, ny, nx = rho.shape
    out = np.zeros(rho.shape, np.complex128)
    for jz in range(nz):
        for jy in range(ny):
            for jx in range(nx):
                v = rho[jz, jy, jx]
                if v == 0:
                    continue
                # element i of the rolled array is Q at grid difference i - j
                shifted = np.roll(Qc, (jz, jy, jx), axis=(0, 1, 2))
                out += v * shifted[:nz, :ny, :nx]
    return out


def fhf_fft(Qc, rho):
    """The same product as a circular convolution on the doubled grid:
    crop(IFFT(FFT(Qc) * FFT(zero-padded rho))).  Differences stay inside
    (-n, n) per axis, so nothing wraps into the cropped corner."""
    rho = np.asarray(rho, dtype=np.complex128)
    nz, ny, nx = rho.shape
    pad = np.zeros(Qc.shape, np.complex128)
    pad[:nz, :ny, :nx] = rho
    y = np.fft.ifftn(np.fft.fftn(Qc) * np.fft.fftn(pad))
    return y[:nz, :ny, :nx]


def cg(apply, b, x0, lam: float, iters: int):
    """Conjugate gradients for (A + lam I) x = b, A Hermitian positive
    semi-definite given by apply(v): the iteration of the textbook method
    (residual r, direction p, step alpha = r.r / p.Ap, beta = new r.r / old
    r.r).  Returns the iterate after `iters` steps and the residual norms
    ||r_0|| .. ||r_iters||; stops early (norms padded with 0) once r = 0."""
    b = np.asarray(b, dtype=np.complex128)
    x = np.array(x0, dtype=np.complex128)

    def op(v):
        return apply(v) + lam * v

    r = b - op(x)
    p = r.copy()
    rr = float(np.vdot(r, r).real)
    norms = [np.sqrt(rr)]
    for _ in range(iters):
        if rr == 0.0:
            norms.append(0.0)
            continue
        Ap = op(p)
        pAp = float(np.vdot(p, Ap).real)
        alpha = rr / pAp
        x = x + alpha * p
        r = r - alpha * Ap
        rr_new = float(np.vdot(r, r).real)
        norms.append(np.sqrt(rr_new))
        p = r + (rr_new / rr) * p
        rr = rr_new
    return x, np.array(norms)
