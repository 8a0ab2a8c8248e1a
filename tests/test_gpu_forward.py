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
