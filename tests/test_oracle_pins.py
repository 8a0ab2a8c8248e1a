"""Pins for the fp64 CPU oracle.

Each test fixes the oracle to something other than itself: hand-derived
values, a library routine the problem reduces to, or a closed form.  Together
they catch a wrong exponent sign, a missing conjugate, a swapped or dropped
coordinate term, a wrong Q weight, and coil-indexing mistakes.
"""

import math

import numpy as np
import pytest

import oracle
from non_cartesian_mri_gb300 import workloads as wl


# ----------------------------------------------------------------------------
# hand-derived worked example (tests/golden/quarter_turn.txt)
# ----------------------------------------------------------------------------

def _quarter(golden):
    g = golden("quarter_turn.txt")
    s = g["sample"].astype(np.float32)
    v = g["voxel"]
    return g, s, v


def test_golden_mu(golden):
    g, s, _ = _quarter(golden)
    mu = oracle.mu(s[:, 4], s[:, 5], s[:, 6], s[:, 7])
    np.testing.assert_allclose(mu.real, g["mu"][:, 1], atol=1e-14)
    np.testing.assert_allclose(mu.imag, g["mu"][:, 2], atol=1e-14)


def test_golden_fhd_and_q(golden):
    _, s, v = _quarter(golden)
    x, y, z = (v[:, i].astype(np.float32) for i in (1, 2, 3))
    f = oracle.fhd(s[:, 1], s[:, 2], s[:, 3], x, y, z, s[:, 4], s[:, 5], s[:, 6], s[:, 7])
    np.testing.assert_allclose(f.real, v[:, 4], atol=1e-12)
    np.testing.assert_allclose(f.imag, v[:, 5], atol=1e-12)
    qq = oracle.q(s[:, 1], s[:, 2], s[:, 3], x, y, z, s[:, 4], s[:, 5])
    np.testing.assert_allclose(qq.real, v[:, 6], atol=1e-12)
    np.testing.assert_allclose(qq.imag, v[:, 7], atol=1e-12)


def test_golden_batched(golden):
    _, s, v = _quarter(golden)
    x, y, z = (v[:, i].astype(np.float32) for i in (1, 2, 3))
    rD = np.stack([s[:, 6], s[:, 8]])
    iD = np.stack([s[:, 7], s[:, 9]])
    fb = oracle.fhd_batched(s[:, 1], s[:, 2], s[:, 3], x, y, z, s[:, 4], s[:, 5], rD, iD)
    assert fb.shape == (2, 4)
    np.testing.assert_allclose(fb[0].real, v[:, 4], atol=1e-12)
    np.testing.assert_allclose(fb[0].imag, v[:, 5], atol=1e-12)
    np.testing.assert_allclose(fb[1].real, v[:, 8], atol=1e-12)
    np.testing.assert_allclose(fb[1].imag, v[:, 9], atol=1e-12)


def test_golden_psnr(golden):
    g = golden("psnr.txt")
    got = oracle.psnr(g["ideal"][0], g["image"][0])
    assert got == pytest.approx(g["psnr_db"][0][0], rel=1e-14)
    assert oracle.psnr(g["ideal"][0], g["ideal"][0]) == float("inf")


# ----------------------------------------------------------------------------
# special cases with a closed form
# ----------------------------------------------------------------------------

def test_single_sample_at_k0_gives_constant_image():
    """One sample at k = 0: every voxel equals Mu[0] (phase 0, cos 1, sin 0)."""
    rng = np.random.default_rng(11)
    x, y, z = wl.voxel_grid(6, 5, 4)
    z0 = np.zeros(1, np.float32)
    rPhi, iPhi, rD, iD = (rng.standard_normal(1).astype(np.float32) for _ in range(4))
    f = oracle.fhd(z0, z0, z0, x, y, z, rPhi, iPhi, rD, iD)
    mu0 = (float(rPhi[0]) - 1j * float(iPhi[0])) * (float(rD[0]) + 1j * float(iD[0]))
    np.testing.assert_allclose(f, np.full(x.size, mu0), rtol=0, atol=1e-15)


@pytest.mark.parametrize("shape", [(4, 8, 2), (8, 4, 16), (2, 16, 4)])
def test_cartesian_grid_is_inverse_dft(shape):
    """On a uniform Cartesian k-grid (section 17.1, Fig. 17.1A) the sum is an
    inverse DFT: F^H D on the integer voxel grid equals Lx*Ly*Lz * ifftn of the
    k-grid-arranged Mu, with the centred index shifts.  Non-cubic grids make a
    swapped or dropped axis fail; power-of-two edges keep k = j/L exact in
    float32."""
    Lx, Ly, Lz = shape
    rng = np.random.default_rng(sum(shape))
    kx, ky, kz = wl.traj_cartesian(Lx, Ly, Lz)
    M = kx.size
    rPhi, iPhi, rD, iD = (rng.standard_normal(M).astype(np.float32) for _ in range(4))
    x, y, z = wl.voxel_grid(Lx, Ly, Lz)
    f = oracle.fhd(kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD)
    mu = (rPhi.astype(np.float64) - 1j * iPhi) * (rD.astype(np.float64) + 1j * iD)
    grid = mu.reshape(Lz, Ly, Lx)
    # centred index j lives at array position j + L//2; ifftshift moves j to j mod L
    ref = np.fft.fftshift(Lx * Ly * Lz * np.fft.ifftn(np.fft.ifftshift(grid)))
    np.testing.assert_allclose(f.reshape(Lz, Ly, Lx), ref, rtol=0,
                               atol=1e-11 * np.abs(ref).max())


def test_cartesian_q_is_inverse_dft_of_weights():
    Lx, Ly, Lz = 8, 4, 2
    rng = np.random.default_rng(5)
    kx, ky, kz = wl.traj_cartesian(Lx, Ly, Lz)
    M = kx.size
    rPhi, iPhi = (rng.standard_normal(M).astype(np.float32) for _ in range(2))
    x, y, z = wl.voxel_grid(Lx, Ly, Lz)
    qq = oracle.q(kx, ky, kz, x, y, z, rPhi, iPhi)
    w = rPhi.astype(np.float64) ** 2 + iPhi.astype(np.float64) ** 2
    ref = np.fft.fftshift(Lx * Ly * Lz * np.fft.ifftn(np.fft.ifftshift(w.reshape(Lz, Ly, Lx))))
    np.testing.assert_allclose(qq.reshape(Lz, Ly, Lx), ref, rtol=0,
                               atol=1e-11 * np.abs(ref).max())


def test_point_source_recovered_at_its_voxel():
    """rho = delta(x0), D_m = e^{-i 2 pi k_m.x0}, Phi = 1: F^H D[x0] = M and
    |F^H D[n]| <= M elsewhere, for any trajectory (section 17.3 step 3's
    phantom -> synthetic data -> reconstruction loop with a one-voxel phantom)."""
    w = wl.make_workload("fhd_64", L=8)
    x0 = np.array([2.0, -3.0, 1.0])
    t = w.kx.astype(np.float64) * x0[0] + w.ky * x0[1] + w.kz * x0[2]
    D = np.exp(-2j * np.pi * t)
    rD, iD = D.real.astype(np.float32), D.imag.astype(np.float32)
    one = np.ones(w.M, np.float32)
    zero = np.zeros(w.M, np.float32)
    f = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, one, zero, rD, iD)
    n0 = int(np.nonzero((w.x == x0[0]) & (w.y == x0[1]) & (w.z == x0[2]))[0][0])
    # D was rounded to float32: |fl(D_m)| = 1 + O(6e-8)
    assert f[n0].real == pytest.approx(w.M, rel=2e-7)
    assert abs(f[n0].imag) < 1e-3
    assert np.all(np.abs(f) <= w.M * (1 + 2e-7))


def test_point_source_on_cartesian_grid_is_a_delta():
    Lx, Ly, Lz = 8, 16, 4
    kx, ky, kz = wl.traj_cartesian(Lx, Ly, Lz)
    x, y, z = wl.voxel_grid(Lx, Ly, Lz)
    x0 = (-3.0, 5.0, 1.0)
    t = kx.astype(np.float64) * x0[0] + ky * x0[1] + kz * x0[2]
    D = np.exp(-2j * np.pi * t)
    one = np.ones(kx.size, np.float32)
    zero = np.zeros(kx.size, np.float32)
    f = oracle.fhd(kx, ky, kz, x, y, z, one, zero, D.real.astype(np.float32),
                   D.imag.astype(np.float32))
    ref = np.zeros(x.size)
    ref[(x == x0[0]) & (y == x0[1]) & (z == x0[2])] = kx.size
    np.testing.assert_allclose(f, ref, rtol=0, atol=1e-5)


def test_linear_in_D():
    rng = np.random.default_rng(3)
    M, L = 257, 5
    kx, ky, kz = wl.traj_uniform_random(M, rng)
    x, y, z = wl.voxel_grid(L)
    rPhi, iPhi = (rng.standard_normal(M).astype(np.float32) for _ in range(2))
    # dyadic values keep 2*D1 + 0.5*D2 exact in float32
    d = [(rng.integers(-64, 64, M) / 16.0).astype(np.float32) for _ in range(4)]
    f1 = oracle.fhd(kx, ky, kz, x, y, z, rPhi, iPhi, d[0], d[1])
    f2 = oracle.fhd(kx, ky, kz, x, y, z, rPhi, iPhi, d[2], d[3])
    f12 = oracle.fhd(kx, ky, kz, x, y, z, rPhi, iPhi,
                     (2 * d[0] + 0.5 * d[2]).astype(np.float32),
                     (2 * d[1] + 0.5 * d[3]).astype(np.float32))
    np.testing.assert_allclose(f12, 2 * f1 + 0.5 * f2, rtol=0,
                               atol=1e-11 * np.abs(f12).max())


def test_q_at_origin_is_sum_of_weights_and_hermitian():
    """Q[x=0] = sum |Phi|^2 (real) and Q(-x) = conj(Q(x))."""
    rng = np.random.default_rng(9)
    M = 999
    kx, ky, kz = wl.traj_uniform_random(M, rng)
    rPhi, iPhi = (rng.standard_normal(M).astype(np.float32) for _ in range(2))
    x = np.array([0, 3, -3, 1.5, -1.5], np.float32)
    y = np.array([0, -2, 2, 4.25, -4.25], np.float32)
    z = np.array([0, 7, -7, -0.5, 0.5], np.float32)
    qq = oracle.q(kx, ky, kz, x, y, z, rPhi, iPhi)
    wsum = float(np.sum(rPhi.astype(np.float64) ** 2 + iPhi.astype(np.float64) ** 2))
    assert qq[0].real == pytest.approx(wsum, rel=1e-14)
    assert qq[0].imag == 0.0
    np.testing.assert_allclose(qq[2], np.conj(qq[1]), rtol=1e-12)
    np.testing.assert_allclose(qq[4], np.conj(qq[3]), rtol=1e-12)


@pytest.mark.parametrize("traj", ["spiral", "radial"])
def test_q_real_for_point_symmetric_trajectory(traj):
    """Trajectories closed under k -> -k with a weight even in k give Im Q = 0."""
    if traj == "spiral":
        kx, ky, kz = wl.traj_stack_of_spirals(8, 4, 64, turns=2.0)
    else:
        kx, ky, kz = wl.traj_radial_fibonacci(32, 64)
    kabs = np.sqrt(kx.astype(np.float64) ** 2 + ky.astype(np.float64) ** 2 + kz.astype(np.float64) ** 2)
    phi = (1.0 + kabs).astype(np.float32)          # real, even in k
    zero = np.zeros_like(phi)
    x, y, z = wl.voxel_grid(6)
    qq = oracle.q(kx, ky, kz, x, y, z, phi, zero)
    assert np.abs(qq.imag).max() < 1e-9 * np.abs(qq.real).max()


def test_box_phantom_forward_matches_dirichlet_kernel():
    """Forward synthesis of a uniform integer box equals the product over axes
    of the geometric sums sum_{x=a}^{b} e^{-i 2 pi k x} (closed form)."""
    rng = np.random.default_rng(21)
    kx, ky, kz = wl.traj_uniform_random(300, rng)
    x, y, z = wl.voxel_grid(8)
    box = ((-2, 1), (0, 3), (-4, -1))
    rho = ((x >= box[0][0]) & (x <= box[0][1]) & (y >= box[1][0]) & (y <= box[1][1])
           & (z >= box[2][0]) & (z <= box[2][1])).astype(np.float64)
    D = oracle.forward(kx, ky, kz, x, y, z, rho)

    def geo(k, a, b):
        k = k.astype(np.float64)
        n = b - a + 1
        out = np.empty(k.shape, np.complex128)
        small = np.abs(np.sin(np.pi * k)) < 1e-12
        ks = k[~small]
        out[~small] = np.exp(-1j * np.pi * ks * (a + b)) * np.sin(np.pi * ks * n) / np.sin(np.pi * ks)
        out[small] = n
        return out

    ref = geo(kx, *box[0]) * geo(ky, *box[1]) * geo(kz, *box[2])
    np.testing.assert_allclose(D, ref, rtol=0, atol=1e-10 * np.abs(ref).max())


def test_forward_and_fhd_are_adjoint():
    """<F rho, D> = <rho, F^H D> with Phi = 1 (F^H is F's conjugate transpose,
    section 17.2)."""
    rng = np.random.default_rng(4)
    M = 211
    kx, ky, kz = wl.traj_uniform_random(M, rng)
    x, y, z = wl.voxel_grid(5, 4, 3)
    rho = rng.standard_normal(x.size) + 1j * rng.standard_normal(x.size)
    rD, iD = (rng.standard_normal(M).astype(np.float32) for _ in range(2))
    D = rD.astype(np.float64) + 1j * iD
    Frho = oracle.forward(kx, ky, kz, x, y, z, rho)
    one, zero = np.ones(M, np.float32), np.zeros(M, np.float32)
    FhD = oracle.fhd(kx, ky, kz, x, y, z, one, zero, rD, iD)
    lhs = np.vdot(Frho, D)
    rhs = np.vdot(rho, FhD)
    assert abs(lhs - rhs) < 1e-10 * abs(lhs)


# ----------------------------------------------------------------------------
# consistency of the oracle's own plumbing
# ----------------------------------------------------------------------------

def test_voxel_subset_matches_full():
    w = wl.make_workload("fhd_tiny")
    full = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD)
    idx = wl.voxel_subset(w.N, 37, 1)
    sub = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=idx)
    np.testing.assert_array_equal(sub, full[idx])


def test_thread_count_does_not_change_results():
    w = wl.make_workload("fhd_tiny")
    idx = wl.voxel_subset(w.N, 64, 2)
    a = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=idx, threads=1)
    b = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=idx, threads=4)
    np.testing.assert_array_equal(a, b)
    oracle.threads(0)


def test_empty_inputs():
    e = np.zeros(0, np.float32)
    x, y, z = wl.voxel_grid(2)
    f = oracle.fhd(e, e, e, x, y, z, e, e, e, e)
    np.testing.assert_array_equal(f, np.zeros(x.size))
    f0 = oracle.fhd(e, e, e, e, e, e, e, e, e, e)
    assert f0.size == 0


def test_brute_force_numpy_cross_check():
    """Independent numpy evaluation of the same sum on a tiny case (a sanity
    check of the C plumbing rather than a pin)."""
    rng = np.random.default_rng(8)
    M, L = 64, 3
    kx, ky, kz = wl.traj_uniform_random(M, rng)
    x, y, z = wl.voxel_grid(L)
    rPhi, iPhi, rD, iD = (rng.standard_normal(M).astype(np.float32) for _ in range(4))
    k = np.stack([kx, ky, kz]).astype(np.float64)
    r = np.stack([x, y, z]).astype(np.float64)
    E = np.exp(2j * math.pi * (r.T @ k))
    mu = (rPhi - 1j * iPhi.astype(np.float64)) * (rD + 1j * iD.astype(np.float64))
    np.testing.assert_allclose(oracle.fhd(kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD),
                               E @ mu, rtol=1e-12, atol=1e-12)
