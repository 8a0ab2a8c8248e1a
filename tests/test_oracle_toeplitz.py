"""Pins of the "find rho" oracle (oracle/toeplitz.py), no GPU.

- fhf_direct (F^H F as the convolution of Q over voxel differences) equals
  F^H (F rho) formed from the oracle's forward model and F^H D -- a different
  route through the definition of F -- on non-cubic grids with unequal
  spacings per axis (an axis or sign mix-up in Q's difference grid fails);
- fhf_fft equals fhf_direct (the circular embedding does not wrap);
- zeroing the index-n planes of the difference grid leaves the product
  unchanged and makes the spectrum real (imaginary part at rounding level,
  while the unzeroed grid's is not);
- the operator is Hermitian and positive semi-definite;
- cg after N steps on an N-voxel problem equals the dense solve of
  (A + lambda I) x = b, and its reported residual norms are those of its
  iterates.
"""

import numpy as np
import pytest

import oracle
from oracle import toeplitz as T


def problem(shape, spacing, M, seed):
    rng = np.random.default_rng(seed)
    nz, ny, nx = shape
    hx, hy, hz = spacing
    k = rng.uniform(-0.5, 0.5, (3, M)).astype(np.float32)
    rPhi = rng.standard_normal(M).astype(np.float32)
    iPhi = rng.standard_normal(M).astype(np.float32)
    xs = (np.arange(nx) * hx - 3.0).astype(np.float32)
    ys = (np.arange(ny) * hy + 1.0).astype(np.float32)
    zs = (np.arange(nz) * hz - 0.5).astype(np.float32)
    z, y, x = np.meshgrid(zs, ys, xs, indexing="ij")
    rho = rng.standard_normal(shape) + 1j * rng.standard_normal(shape)
    return k, rPhi, iPhi, (x.reshape(-1), y.reshape(-1), z.reshape(-1)), rho


def fhf_by_definition(k, rPhi, iPhi, xyz, rho):
    """F^H (F rho) with F[m][n] = Phi_m e^{-i2pi k_m.x_n}, through the oracle's
    forward model and F^H D (the intermediate rounded to float32 on entry)."""
    phi = rPhi.astype(np.float64) + 1j * iPhi
    v = phi * oracle.forward(k[0], k[1], k[2], *xyz, rho.reshape(-1))
    return oracle.fhd(k[0], k[1], k[2], *xyz, rPhi, iPhi, v.real, v.imag)


def test_difference_axis():
    assert list(T.difference_axis(3, 0.5)) == [0.0, 0.5, 1.0, -1.5, -1.0, -0.5]


@pytest.mark.parametrize("shape,spacing", [((2, 3, 4), (1.0, 0.75, 1.5)),
                                           ((3, 1, 5), (0.5, 1.0, 2.0)),
                                           ((1, 4, 2), (1.25, 1.0, 1.0))])
def test_fhf_direct_is_fh_of_f(shape, spacing):
    k, rPhi, iPhi, xyz, rho = problem(shape, spacing, 257, sum(shape))
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing)
    got = T.fhf_direct(Qc, rho).reshape(-1)
    ref = fhf_by_definition(k, rPhi, iPhi, xyz, rho)
    assert oracle.rel_l2(got, ref) < 1e-6


def test_fhf_fft_equals_direct_and_is_hermitian():
    shape, spacing = (3, 4, 5), (1.0, 1.0, 0.5)
    k, rPhi, iPhi, xyz, rho = problem(shape, spacing, 300, 3)
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing)
    a = T.fhf_direct(Qc, rho)
    assert oracle.rel_l2(T.fhf_fft(Qc, rho), a) < 1e-12
    rng = np.random.default_rng(4)
    u = rng.standard_normal(shape) + 1j * rng.standard_normal(shape)
    lhs = np.vdot(u, T.fhf_direct(Qc, rho))
    rhs = np.vdot(T.fhf_direct(Qc, u), rho)
    assert abs(lhs - rhs) < 1e-10 * abs(lhs)
    assert np.vdot(rho, a).real > 0 and abs(np.vdot(rho, a).imag) < 1e-9 * abs(np.vdot(rho, a))


@pytest.mark.parametrize("shape,spacing", [((3, 4, 5), (1.0, 1.0, 0.5)),
                                           ((2, 1, 4), (0.5, 1.0, 2.0))])
def test_real_spectrum_gives_the_same_product(shape, spacing):
    """Zeroing the index-n planes leaves F^H F unchanged and makes the
    spectrum real: a wrong difference axis (a sign, an off-by-one in the
    wrap) or a zeroed plane that is used fails one of the three checks."""
    k, rPhi, iPhi, xyz, rho = problem(shape, spacing, 300, 7 + shape[2])
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing)
    Kr, imag = T.toeplitz_spectrum(Qc)
    assert imag < 1e-12
    ref = T.fhf_direct(Qc, rho)
    assert oracle.rel_l2(T.fhf_spectrum(Kr, rho), ref) < 1e-12
    # the planes are needed for the symmetry: without the zeroing the
    # spectrum is complex
    full = np.fft.fftn(Qc)
    assert np.abs(full.imag).max() > 1e-3 * np.abs(full.real).max()


def test_cg_reaches_the_dense_solution():
    shape, spacing = (2, 3, 4), (1.0, 1.0, 1.0)
    k, rPhi, iPhi, xyz, rho = problem(shape, spacing, 400, 5)
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing)
    N = int(np.prod(shape))
    A = np.zeros((N, N), np.complex128)
    for j in range(N):
        e = np.zeros(N, np.complex128)
        e[j] = 1.0
        A[:, j] = T.fhf_direct(Qc, e.reshape(shape)).reshape(-1)
    lam = 0.3
    b = rho.reshape(-1)
    ref = np.linalg.solve(A + lam * np.eye(N), b)
    apply = lambda v: T.fhf_direct(Qc, v.reshape(shape)).reshape(-1)   # noqa: E731
    x, norms = T.cg(apply, b, np.zeros(N), lam, 3 * N)
    assert np.abs(x - ref).max() < 1e-8 * np.abs(ref).max()
    # the reported norms are the residuals of the iterates
    assert norms[0] == pytest.approx(np.linalg.norm(b))
    assert norms[-1] <= 1e-8 * norms[0]
    x4, n4 = T.cg(apply, b, np.zeros(N), lam, 4)
    assert n4[-1] == pytest.approx(np.linalg.norm(b - (A + lam * np.eye(N)) @ x4), rel=1e-9)
