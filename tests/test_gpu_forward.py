"""The forward model D = F rho (mri_forward) against the oracle, and the
adjoint pair on the GPU: <F rho, D> = <rho, F^H D> with Phi = 1."""

import numpy as np
import pytest
import torch

import oracle
from non_cartesian_mri_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"accurate": 1e-5, "fast": 2e-4, "fast_rr": 2e-4}


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


def rho_for(w, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(w.N) + 1j * rng.standard_normal(w.N)).astype(np.complex64)


@pytest.mark.parametrize("trig", ["accurate", "fast", "fast_rr"])
def test_forward_tiny(mri, trig):
    w = wl.make_workload("fhd_tiny")
    rho = rho_for(w, 1)
    r, i = mri.forward(dev(w.kx), dev(w.ky), dev(w.kz), dev(w.x), dev(w.y), dev(w.z),
                       dev(rho.real), dev(rho.imag), trig=trig)
    ref = oracle.forward(w.kx, w.ky, w.kz, w.x, w.y, w.z, rho)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]


@pytest.mark.parametrize("trig", ["accurate", "fast"])
def test_forward_64_sampled(mri, trig):
    """64^3 voxels, the 32,768-sample spiral; the oracle checks 384 samples."""
    w = wl.make_workload("fhd_64")
    rho = rho_for(w, 2)
    r, i = mri.forward(dev(w.kx), dev(w.ky), dev(w.kz), dev(w.x), dev(w.y), dev(w.z),
                       dev(rho.real), dev(rho.imag), trig=trig)
    idx = np.sort(np.random.default_rng(3).choice(w.M, 384, replace=False))
    ref = oracle.forward(w.kx[idx], w.ky[idx], w.kz[idx], w.x, w.y, w.z, rho)
    assert oracle.rel_l2(cplx(r, i)[idx], ref) <= TOL[trig]


def test_forward_and_fhd_are_adjoint(mri):
    w = wl.make_workload("fhd_tiny")
    rho = rho_for(w, 4)
    rng = np.random.default_rng(5)
    d = (rng.standard_normal(w.M) + 1j * rng.standard_normal(w.M)).astype(np.complex64)
    k = [dev(w.kx), dev(w.ky), dev(w.kz)]
    x = [dev(w.x), dev(w.y), dev(w.z)]
    fr, fi = mri.forward(*k, *x, dev(rho.real), dev(rho.imag), trig="accurate")
    one, zero = dev(np.ones(w.M, np.float32)), dev(np.zeros(w.M, np.float32))
    hr, hi = mri.fhd(*k, *x, one, zero, dev(d.real), dev(d.imag), trig="accurate")
    lhs = np.vdot(d.astype(np.complex128), cplx(fr, fi))        # <D, F rho>
    rhs = np.vdot(cplx(hr, hi), rho.astype(np.complex128))      # <F^H D, rho>
    assert abs(lhs - rhs) <= 1e-5 * abs(lhs)


def test_forward_accumulate_and_empty(mri):
    w = wl.make_workload("fhd_tiny")
    rho = rho_for(w, 6)
    k = [dev(w.kx), dev(w.ky), dev(w.kz)]
    x = [dev(w.x), dev(w.y), dev(w.z)]
    r, i = mri.forward(*k, *x, dev(rho.real), dev(rho.imag), trig="accurate")
    out = (torch.full_like(r, 3.0), torch.full_like(i, -1.0))
    mri.forward(*k, *x, dev(rho.real), dev(rho.imag), trig="accurate", accumulate=True, out=out)
    assert oracle.rel_l2(cplx(out[0] - 3.0, out[1] + 1.0), cplx(r, i)) <= 1e-6
    e = torch.empty(0, device="cuda")
    rz, iz = mri.forward(*k, e, e, e, e, e)                       # no voxels: D = 0
    assert rz.numel() == w.M and torch.count_nonzero(rz) == 0 and torch.count_nonzero(iz) == 0
    re_, ie_ = mri.forward(e, e, e, *x, dev(rho.real), dev(rho.imag))   # no samples
    assert re_.numel() == 0
    assert mri.device_errors(clear=True) == 0


def expand(xs, ys, zs):
    z, y, x = np.meshgrid(zs, ys, xs, indexing="ij")
    return x.reshape(-1), y.reshape(-1), z.reshape(-1)


def grid_case(ny, nz, M, seed):
    w = wl.make_workload("fhd_128_radial")
    xs = (np.arange(128) - 64).astype(np.float32)
    rng = np.random.default_rng(seed)
    pop = np.arange(-128, 128) * 0.5
    ys = np.sort(rng.choice(pop, ny, replace=False)).astype(np.float32)
    zs = np.sort(rng.choice(pop, nz, replace=False)).astype(np.float32)
    n = 128 * ny * nz
    rho = (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)
    return w, xs, ys, zs, rho


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("ny,nz,M", [(3, 7, 1000), (256, 2, 3001)])
def test_forward_grid_tensor_cores(mri, trig, ny, nz, M):
    """nx = 128: ragged row blocks (21 rows) and several row blocks (512
    rows), ragged sample counts."""
    w, xs, ys, zs, rho = grid_case(ny, nz, M, 11 + ny)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    r, i = mri.forward_grid(*k, dev(xs), dev(ys), dev(zs), dev(rho.real), dev(rho.imag), trig=trig)
    x, y, z = expand(xs, ys, zs)
    ref = oracle.forward(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, rho)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]
    assert mri.device_errors(clear=True) == 0


def test_forward_grid_128_sampled_and_accumulate(mri):
    """The full 128^3 grid, the radial trajectory; the oracle checks 256 samples."""
    w = wl.make_workload("fhd_128_radial")
    rng = np.random.default_rng(21)
    rho = (rng.standard_normal(w.N) + 1j * rng.standard_normal(w.N)).astype(np.complex64)
    xs, ys, zs = w.axes()
    k = [dev(w.kx), dev(w.ky), dev(w.kz)]
    axes = [dev(xs), dev(ys), dev(zs)]
    for trig in ("accurate", "fast"):
        r, i = mri.forward_grid(*k, *axes, dev(rho.real), dev(rho.imag), trig=trig)
        idx = np.sort(rng.choice(w.M, 256, replace=False))
        ref = oracle.forward(w.kx[idx], w.ky[idx], w.kz[idx], w.x, w.y, w.z, rho)
        assert oracle.rel_l2(cplx(r, i)[idx], ref) <= TOL[trig], trig
    out = (torch.full_like(r, 0.25), torch.full_like(i, 4.0))
    mri.forward_grid(*k, *axes, dev(rho.real), dev(rho.imag), trig="fast", accumulate=True,
                     out=out)
    assert oracle.rel_l2(cplx(out[0] - 0.25, out[1] - 4.0), cplx(r, i)) <= 1e-6


def test_forward_grid_adjoint_of_fhd_grid(mri):
    w, xs, ys, zs, rho = grid_case(8, 4, 2000, 31)
    M = 2000
    rng = np.random.default_rng(32)
    d = (rng.standard_normal(M) + 1j * rng.standard_normal(M)).astype(np.complex64)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    axes = [dev(xs), dev(ys), dev(zs)]
    fr, fi = mri.forward_grid(*k, *axes, dev(rho.real), dev(rho.imag), trig="accurate")
    one, zero = dev(np.ones(M, np.float32)), dev(np.zeros(M, np.float32))
    hr, hi = mri.fhd_grid(*k, *axes, one, zero, dev(d.real), dev(d.imag), trig="accurate")
    lhs = np.vdot(d.astype(np.complex128), cplx(fr, fi))
    rhs = np.vdot(cplx(hr, hi), rho.astype(np.complex128))
    assert abs(lhs - rhs) <= 1e-5 * abs(lhs)


@pytest.mark.parametrize("k", [-90, 70])
def test_forward_grid_scale_is_exact(mri, k):
    """rho is scaled by a power of two from its largest value: multiplying rho
    by 2^k multiplies D by exactly 2^k."""
    w, xs, ys, zs, rho = grid_case(4, 2, 777, 41)
    kk = [dev(a[:777]) for a in (w.kx, w.ky, w.kz)]
    axes = [dev(xs), dev(ys), dev(zs)]
    r0, i0 = mri.forward_grid(*kk, *axes, dev(rho.real), dev(rho.imag), trig="fast")
    s = float(2.0 ** k)
    r1, i1 = mri.forward_grid(*kk, *axes, dev(rho.real) * s, dev(rho.imag) * s, trig="fast")
    assert torch.equal(r1, r0 * s) and torch.equal(i1, i0 * s)


def test_forward_grid_fallback_and_empty(mri):
    """nx = 6 goes through expanded coordinates and mri_forward."""
    w = wl.make_workload("fhd_64")
    M = 1500
    xs = np.array([-30.0, -7.5, 0.0, 2.0, 19.0, 31.0], np.float32)
    ys = np.array([-5.0, 9.0], np.float32)
    zs = np.array([3.0, -8.0, 12.0], np.float32)
    rng = np.random.default_rng(51)
    rho = (rng.standard_normal(6 * 6) + 1j * rng.standard_normal(6 * 6)).astype(np.complex64)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    r, i = mri.forward_grid(*k, dev(xs), dev(ys), dev(zs), dev(rho.real), dev(rho.imag),
                            trig="accurate")
    x, y, z = expand(xs, ys, zs)
    ref = oracle.forward(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, rho)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL["accurate"]
    e = torch.empty(0, device="cuda")
    rz, iz = mri.forward_grid(*k, e, dev(ys), dev(zs), e, e)      # nx = 0: no voxels
    assert torch.count_nonzero(rz) == 0 and torch.count_nonzero(iz) == 0


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("ys_kind,ny,nz", [("even", 12, 5), ("even", 16, 3), ("mixed", 24, 2),
                                          ("even", 1, 9)])
def test_forward_grid_evenly_spaced_rows(mri, trig, ys_kind, ny, nz):
    """Row factors by rotation: evenly spaced y (step 0.75, offset), groups of
    8 rows that straddle two z planes (ny = 12), a y axis that is even only
    in places (mixed), and ny = 1 (every group straddles planes)."""
    M = 1500
    w = wl.make_workload("fhd_128_radial")
    xs = (np.arange(128) - 64).astype(np.float32)
    if ys_kind == "even":
        ys = (np.arange(ny) * 0.75 - 3.0).astype(np.float32)
    else:
        ys = np.concatenate([np.arange(8) * 0.5, 10.0 + np.array([0.0, 0.3, 1.1, 1.2, 2.0, 2.5,
                                                                   4.0, 4.25]),
                             30.0 + np.arange(8) * 1.5]).astype(np.float32)
    zs = (np.arange(nz) * 2.0 - 5.0).astype(np.float32)
    rng = np.random.default_rng(ny * 100 + nz)
    n = 128 * ny * nz
    rho = (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    r, i = mri.forward_grid(*k, dev(xs), dev(ys), dev(zs), dev(rho.real), dev(rho.imag),
                            trig=trig)
    x, y, z = expand(xs, ys, zs)
    ref = oracle.forward(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, rho)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]
    assert mri.device_errors(clear=True) == 0
