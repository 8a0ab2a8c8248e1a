"""The find-rho step on the GPU against the oracle (oracle/toeplitz.py).

- mri_fft3 against numpy's FFT (fp64) on power-of-two shapes, forward and
  inverse, contiguous and strided axes, a one-point axis;
- mri_toeplitz_kernel against the oracle's real spectrum (the FFT of Q on
  the circular difference grid with the unused index-n planes zeroed);
- mri_toeplitz_apply against the oracle's F^H F by its definition (plus
  lambda I), non-cubic grids with unequal spacings, both trig paths,
  accumulate and in place;
- mri_cg_solve against the oracle's CG (same iterations, fp64 operator):
  iterates and residual norms, and a reconstruction of a seeded image from
  its own samples (D = F rho, b = F^H D) whose error falls with the
  iterations;
- at the benchmarked size (128^3, radial trajectory): the product against
  F^H (Phi F v) from the grid forward model and F^H D, Hermitian symmetry,
  positivity and the lambda term; CG lowering its energy functional at every
  step and reporting the residual of its iterate;
- argument errors.

Tolerances: one Toeplitz product is Q (accurate path, ~2e-6) through two
fp32 FFTs of the doubled grid (~1e-7 log2 per transform): 1e-5 accurate,
2e-4 fast.  CG amplifies the per-iteration error by the conditioning of the
operator; after a few iterations on these well-sampled problems 1e-4 holds
for the iterate and the residual norms.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import toeplitz as T

pytestmark = pytest.mark.gpu

TOL = {"accurate": 1e-5, "fast": 2e-4}


@pytest.fixture(scope="module")
def mri():
    from non_cartesian_mri_gb300 import build
    build.build()
    import non_cartesian_mri_gb300 as m
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def cplx(r, i):
    return r.cpu().numpy().astype(np.float64) + 1j * i.cpu().numpy()


def samples(M, seed, kmax=0.5):
    rng = np.random.default_rng(seed)
    k = rng.uniform(-kmax, kmax, (3, M)).astype(np.float32)
    rPhi = rng.standard_normal(M).astype(np.float32)
    iPhi = rng.standard_normal(M).astype(np.float32)
    return k, rPhi, iPhi


@pytest.mark.parametrize("shape", [(4, 8, 16), (2, 1, 32), (1, 1, 1024), (16, 16, 16),
                                   (8, 2, 512), (1, 1, 1)])
def test_fft3_matches_numpy(mri, shape):
    rng = np.random.default_rng(sum(shape))
    x = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    got = mri.fft3(dev(x).clone()).cpu().numpy()
    ref = np.fft.fftn(x.astype(np.complex128))
    assert oracle.rel_l2(got, ref) < 1e-6
    back = mri.fft3(dev(x).clone(), inverse=True).cpu().numpy()
    assert oracle.rel_l2(back, np.fft.ifftn(x.astype(np.complex128)) * x.size) < 1e-6


@pytest.mark.parametrize("shape,spacing", [((2, 4, 8), (1.0, 0.75, 1.5)),
                                           ((4, 4, 4), (1.0, 1.0, 1.0)),
                                           ((1, 2, 16), (0.5, 2.0, 1.0))])
def test_toeplitz_kernel_is_the_spectrum_of_q(mri, shape, spacing):
    k, rPhi, iPhi = samples(700, 11)
    K = mri.toeplitz_kernel(dev(k[0]), dev(k[1]), dev(k[2]), dev(rPhi), dev(iPhi), shape,
                            spacing).cpu().numpy()
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing)
    Kr, _ = T.toeplitz_spectrum(Qc)
    assert K.dtype == np.float32
    assert oracle.rel_l2(K, Kr) < 1e-5


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("shape,spacing,lam", [((2, 4, 8), (1.0, 0.75, 1.5), 0.0),
                                               ((4, 4, 4), (1.0, 1.0, 1.0), 0.7),
                                               ((1, 2, 16), (0.5, 2.0, 1.0), 2.5),
                                               ((8, 8, 8), (1.0, 1.0, 1.0), 0.1)])
def test_toeplitz_apply_matches_fhf(mri, shape, spacing, lam, trig):
    k, rPhi, iPhi = samples(900, 12 + shape[2])
    K = mri.toeplitz_kernel(dev(k[0]), dev(k[1]), dev(k[2]), dev(rPhi), dev(iPhi), shape,
                            spacing, trig=trig)
    rng = np.random.default_rng(13)
    v = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    r, i = mri.toeplitz_apply(K, dev(v.real.reshape(-1)), dev(v.imag.reshape(-1)), lam=lam)
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing)
    ref = (T.fhf_direct(Qc, v) + lam * v).reshape(-1)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]
    # accumulate adds onto what is there; in place reads before it writes
    out = (torch.full_like(r, 0.5), torch.full_like(i, -1.0))
    mri.toeplitz_apply(K, dev(v.real.reshape(-1)), dev(v.imag.reshape(-1)), lam=lam,
                       accumulate=True, out=out)
    assert oracle.rel_l2(cplx(out[0] - 0.5, out[1] + 1.0), ref) <= TOL[trig]
    vr, vi = dev(v.real.reshape(-1)), dev(v.imag.reshape(-1))
    mri.toeplitz_apply(K, vr, vi, lam=lam, out=(vr, vi))
    assert oracle.rel_l2(cplx(vr, vi), ref) <= TOL[trig]
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("shape,spacing", [((8, 4, 2), (1.0, 0.5, 1.0)),
                                           ((4, 2, 1), (1.0, 1.0, 1.0)),
                                           ((1, 1, 512), (1.0, 1.0, 1.0)),
                                           ((2, 512, 1), (1.0, 0.25, 1.0)),
                                           ((16, 32, 64), (1.0, 1.0, 1.0)),
                                           ((512, 1, 1), (1.0, 1.0, 1.0)),
                                           ((256, 2, 2), (1.0, 1.0, 0.5)),
                                           ((64, 4, 2), (1.0, 1.0, 1.0)),
                                           ((32, 2, 16), (0.5, 1.0, 1.0))])
def test_toeplitz_apply_shapes(mri, shape, spacing):
    """Narrow x (a CTA's 16 strided lines span several outer slabs), one-voxel
    axes, the longest lines (2 n = 1024) on every axis including z (whose
    stage keeps a forward transform's registers for the inverse one: the
    512- and 1024-long plans with an odd radix), and a grid of 32768 voxels,
    checked through the oracle's FFT route (fhf_fft, pinned to the
    definition)."""
    k, rPhi, iPhi = samples(600, 40 + shape[2])
    K = mri.toeplitz_kernel(dev(k[0]), dev(k[1]), dev(k[2]), dev(rPhi), dev(iPhi), shape,
                            spacing, trig="accurate")
    rng = np.random.default_rng(41)
    v = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    r, i = mri.toeplitz_apply(K, dev(v.real.reshape(-1)), dev(v.imag.reshape(-1)), lam=0.3)
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing, threads=0)
    ref = (T.fhf_fft(Qc, v) + 0.3 * v).reshape(-1)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL["accurate"]
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("lam", [0.05, 1.0])
def test_cg_matches_the_oracle(mri, lam):
    shape, spacing = (4, 8, 8), (1.0, 1.0, 1.0)
    k, rPhi, iPhi = samples(3000, 21)
    K = mri.toeplitz_kernel(dev(k[0]), dev(k[1]), dev(k[2]), dev(rPhi), dev(iPhi), shape,
                            spacing)
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing)
    rng = np.random.default_rng(22)
    b = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    x0 = (0.1 * rng.standard_normal(shape)).astype(np.complex64)
    iters = 6
    xr, xi, norms = mri.cg_solve(K, dev(b.real.reshape(-1)), dev(b.imag.reshape(-1)), lam=lam,
                                 iters=iters, x0=(dev(x0.real.reshape(-1)),
                                                  dev(x0.imag.reshape(-1))))
    apply = lambda v: T.fhf_fft(Qc, v.reshape(shape)).reshape(-1)   # noqa: E731
    ref_x, ref_n = T.cg(apply, b.reshape(-1), x0.reshape(-1), lam, iters)
    assert oracle.rel_l2(cplx(xr, xi), ref_x) < 1e-4
    assert np.abs(norms.cpu().numpy() - ref_n).max() < 1e-4 * ref_n[0]
    assert mri.device_errors(clear=True) == 0


def test_cg_reconstructs_an_image_from_its_samples(mri):
    """D = F rho_true (the forward model with the sensitivity), b = F^H D;
    CG on (F^H F + lam I) x = b approaches rho_true."""
    shape = (8, 16, 16)
    nz, ny, nx = shape
    M = 6 * nx * ny * nz
    k, _, _ = samples(M, 31)
    rPhi = np.ones(M, np.float32)
    iPhi = np.zeros(M, np.float32)
    xs = np.arange(nx, dtype=np.float32)
    ys = np.arange(ny, dtype=np.float32)
    zs = np.arange(nz, dtype=np.float32)
    z, y, x = np.meshgrid(zs, ys, xs, indexing="ij")
    rho = (np.exp(-((x - 7.5) ** 2 + (y - 6.0) ** 2) / 20.0 - (z - 3.5) ** 2 / 6.0)
           * (1.0 + 0.5j)).astype(np.complex64)
    kk = [dev(a) for a in k]
    ax = [dev(xs), dev(ys), dev(zs)]
    dr, di = mri.forward_grid(*kk, *ax, dev(rho.real.reshape(-1)), dev(rho.imag.reshape(-1)),
                              trig="accurate")
    br, bi = mri.fhd_grid(*kk, *ax, dev(rPhi), dev(iPhi), dr, di, trig="accurate")
    K = mri.toeplitz_kernel(*kk, dev(rPhi), dev(iPhi), shape)
    errs = []
    for iters in (2, 8, 30):
        xr, xi, norms = mri.cg_solve(K, br, bi, lam=1e-3, iters=iters)
        errs.append(oracle.rel_l2(cplx(xr, xi), rho.reshape(-1)))
    assert errs[0] > errs[1] > errs[2]
    assert errs[2] < 1e-2
    n = norms.cpu().numpy()
    assert n[-1] < 1e-3 * n[0]
    assert mri.device_errors(clear=True) == 0


def test_toeplitz_argument_errors(mri):
    lib = mri.load()
    K = torch.zeros((8, 8, 8), dtype=torch.float32, device="cuda")
    v = torch.zeros(64, device="cuda")
    P = ctypes.c_void_p
    for nx, ny, nz in ((3, 4, 4), (4, 4, 1024), (0, 4, 4)):
        assert lib.mri_toeplitz_apply(P(K.data_ptr()), nx, ny, nz, 0.0, P(v.data_ptr()),
                                      P(v.data_ptr()), P(v.data_ptr()), P(v.data_ptr()), 0,
                                      None) == 2   # MRI_ERR_SIZE
    assert lib.mri_toeplitz_apply(P(K.data_ptr() + 4), 4, 4, 4, 0.0, P(v.data_ptr()),
                                  P(v.data_ptr()), P(v.data_ptr()), P(v.data_ptr()), 0,
                                  None) == 3       # MRI_ERR_ALIGN
    C = torch.zeros((8, 8, 8), dtype=torch.complex64, device="cuda")
    assert lib.mri_fft3(P(C.data_ptr()), 6, 8, 8, 0, None) == 2
    assert lib.mri_fft3(P(C.data_ptr()), 8, 8, 8, 2, None) == 5   # MRI_ERR_MODE
    with pytest.raises(ValueError):
        mri.toeplitz_apply(C, v[:64], v[:64])


@pytest.fixture(scope="module")
def radial_128(mri):
    """The 128^3 radial workload (the benchmarked find-rho configuration):
    its trajectory and weights on the device, the spectrum with accurate trig,
    and a seeded complex vector."""
    from non_cartesian_mri_gb300 import workloads as wl
    w = wl.make_workload("fhd_128_radial")
    k = [dev(w.kx), dev(w.ky), dev(w.kz)]
    phi = [dev(w.rPhi), dev(w.iPhi)]
    ax = [dev(a) for a in w.axes()]
    K = mri.toeplitz_kernel(*k, *phi, (w.L, w.L, w.L), trig="accurate")
    rng = np.random.default_rng(123)
    v = [dev(rng.standard_normal(w.N).astype(np.float32)) for _ in range(2)]
    return w, k, phi, ax, K, v


def test_toeplitz_apply_full_size_matches_forward_then_adjoint(mri, radial_128):
    """At the benchmarked size the oracle cannot form F^H F v, so the product
    is checked against the other route through the definition: F^H (Phi F v)
    with the grid forward model and F^H D (both checked against the oracle at
    this size), accurate trig on every side.  Each side carries ~2e-6."""
    w, k, phi, ax, K, v = radial_128
    r, i = mri.toeplitz_apply(K, *v, lam=0.0)
    fr, fi = mri.forward_grid(*k, *ax, *v, trig="accurate")
    pr = phi[0] * fr - phi[1] * fi
    pi = phi[0] * fi + phi[1] * fr
    dr, di = mri.fhd_grid(*k, *ax, *phi, pr, pi, trig="accurate")
    assert oracle.rel_l2(cplx(r, i), cplx(dr, di)) < 2e-5
    assert mri.device_errors(clear=True) == 0


def test_toeplitz_apply_full_size_is_hermitian_and_linear(mri, radial_128):
    """<u, A v> = conj <v, A u>, <v, A v> real and positive, and
    A(a v) = a A(v) with lambda I added exactly."""
    w, k, phi, ax, K, v = radial_128
    rng = np.random.default_rng(124)
    u = [dev(rng.standard_normal(w.N).astype(np.float32)) for _ in range(2)]
    Av = cplx(*mri.toeplitz_apply(K, *v))
    Au = cplx(*mri.toeplitz_apply(K, *u))
    vv, uu = cplx(*v), cplx(*u)
    lhs = np.vdot(uu, Av)
    rhs = np.conj(np.vdot(vv, Au))
    assert abs(lhs - rhs) < 1e-5 * np.linalg.norm(uu) * np.linalg.norm(Av)
    q = np.vdot(vv, Av)
    assert q.real > 0 and abs(q.imag) < 1e-5 * abs(q)
    lam = 0.75
    Avl = cplx(*mri.toeplitz_apply(K, *v, lam=lam))
    assert oracle.rel_l2(Avl, Av + lam * vv) < 1e-6


def test_cg_full_size_descends_and_reports_its_residuals(mri, radial_128):
    """CG at the benchmarked size.  Without density compensation F^H F has a
    very wide spectrum (the radial centre of k-space is sampled densely), so
    the residual norm need not fall; what CG guarantees is that every step
    lowers phi(x) = x^H (A + lambda I) x / 2 - Re b^H x (the energy norm of
    the error).  Checked over the iterates, plus: the last reported norm is
    that of b - (A + lambda I) x recomputed from the returned iterate."""
    w, k, phi, ax, K, v = radial_128
    lam = 0.01
    b = cplx(*v)

    def energy(x_r, x_i):
        x = cplx(x_r, x_i)
        Ax = cplx(*mri.toeplitz_apply(K, x_r, x_i, lam=lam))
        return 0.5 * np.vdot(x, Ax).real - np.vdot(b, x).real, Ax

    phis = [0.0]
    for iters in (1, 2, 5, 10):
        xr, xi, norms = mri.cg_solve(K, *v, lam=lam, iters=iters)
        e, Ax = energy(xr, xi)
        phis.append(e)
    assert all(b_ < a_ for a_, b_ in zip(phis, phis[1:])), phis
    n = norms.cpu().numpy()
    assert np.all(np.isfinite(n))
    assert abs(np.linalg.norm(b - Ax) - n[-1]) < 1e-3 * n.max()
    assert mri.device_errors(clear=True) == 0
