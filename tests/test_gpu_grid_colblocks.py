"""Tensor-core grid paths at other widths than nx = 128, against the oracle.

nx = 64 runs as one block of 128 columns padded with zeros; nx a multiple of
128 runs in column blocks of 128 (a third grid dimension for F^H D, Q and the
batched form; an outer loop inside each CTA for the forward model).  The
oracle gets the expanded voxel coordinates; tolerances as everywhere (1e-5
accurate, 2e-4 fast).  Also: outputs that are not 16-byte aligned (the scalar
store path), accumulate, ragged rows and samples, and the accurate y-factor
table (ny a multiple of 128) together with several column blocks.
"""

import functools

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


def expand(xs, ys, zs):
    z, y, x = np.meshgrid(zs, ys, xs, indexing="ij")
    return x.reshape(-1), y.reshape(-1), z.reshape(-1)


def axes(nx, ny, nz, seed):
    """Non-uniform columns inside the field of view of the 128^3 workload
    (|x| < 64), so that the phases span the same range as there and the
    tolerances of that workload hold."""
    rng = np.random.default_rng(seed)
    xs = np.sort(rng.uniform(-64.0, 64.0, nx)).astype(np.float32)
    ys = (np.arange(ny) - ny // 2).astype(np.float32)
    zs = (np.arange(nz) * 2.0 - nz).astype(np.float32)
    return xs, ys, zs


@functools.lru_cache(maxsize=1)
def radial():
    return wl.make_workload("fhd_128_radial")


def samples(M, seed):
    """M samples of the radial trajectory of the 128^3 workload (|k| up to
    the edge of k-space), with its Phi and D."""
    w = radial()
    rng = np.random.default_rng(seed)
    pick = np.sort(rng.choice(w.M, M, replace=False))
    a = {n: getattr(w, n)[pick] for n in ("kx", "ky", "kz", "rPhi", "iPhi", "rD", "iD")}
    return a


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("nx,ny,nz,M", [(64, 5, 3, 3001), (256, 3, 7, 2777),
                                        (384, 2, 3, 1500), (256, 128, 1, 700)])
def test_fhd_and_q_column_blocks(mri, nx, ny, nz, M, trig):
    xs, ys, zs = axes(nx, ny, nz, nx + ny + M)
    a = samples(M, nx + M)
    k = [dev(a[n]) for n in ("kx", "ky", "kz")]
    wts = [dev(a[n]) for n in ("rPhi", "iPhi", "rD", "iD")]
    ax = [dev(xs), dev(ys), dev(zs)]
    plan = mri.plan_grid("fhd", M, nx, ny, nz)
    assert plan["tensor_cores"] == 1
    x, y, z = expand(xs, ys, zs)
    N = x.size
    idx = None if N <= 4096 else wl.voxel_subset(N, 1024, 7)
    r, i = mri.fhd_grid(*k, *ax, *wts, trig=trig)
    ref = oracle.fhd(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"], a["rD"], a["iD"],
                     idx=idx)
    got = cplx(r, i) if idx is None else cplx(r, i)[idx]
    assert oracle.rel_l2(got, ref) <= TOL[trig]
    qr, qi = mri.q_grid(*k, *ax, wts[0], wts[1], trig=trig)
    qref = oracle.q(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"], idx=idx)
    got = cplx(qr, qi) if idx is None else cplx(qr, qi)[idx]
    assert oracle.rel_l2(got, qref) <= TOL[trig]
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("nx", [64, 256])
def test_misaligned_outputs_accumulate(mri, nx):
    """Outputs one float past a 16-byte boundary take the scalar stores;
    accumulate adds onto what is there."""
    ny, nz, M = 3, 5, 1200
    xs, ys, zs = axes(nx, ny, nz, 5 * nx)
    a = samples(M, 11 * nx)
    k = [dev(a[n]) for n in ("kx", "ky", "kz")]
    wts = [dev(a[n]) for n in ("rPhi", "iPhi", "rD", "iD")]
    ax = [dev(xs), dev(ys), dev(zs)]
    N = nx * ny * nz
    base_r = torch.full((N + 1,), 0.25, device="cuda")
    base_i = torch.full((N + 1,), -0.75, device="cuda")
    out = (base_r[1:], base_i[1:])
    mri.fhd_grid(*k, *ax, *wts, trig="accurate", accumulate=True, out=out)
    x, y, z = expand(xs, ys, zs)
    ref = oracle.fhd(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"], a["rD"], a["iD"])
    assert oracle.rel_l2(cplx(out[0] - 0.25, out[1] + 0.75), ref) <= TOL["accurate"]
    assert float(base_r[0]) == 0.25 and float(base_i[0]) == -0.75     # nothing before
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("nx,B", [(64, 3), (256, 9), (384, 1)])
def test_batched_column_blocks(mri, nx, B, trig):
    ny, nz, M = 3, 4, 1800
    xs, ys, zs = axes(nx, ny, nz, 3 * nx + B)
    a = samples(M, 13 * nx + B)
    rng = np.random.default_rng(nx + B)
    g = rng.standard_normal(B) + 1j * rng.standard_normal(B)
    d = a["rD"] + 1j * a["iD"]
    dc = g[:, None] * d[None, :] + 0.1 * (rng.standard_normal((B, M))
                                          + 1j * rng.standard_normal((B, M)))
    rD, iD = dc.real.astype(np.float32), dc.imag.astype(np.float32)
    assert mri.plan_grid_batched(B, M, nx, ny, nz)["tensor_cores"] == 1
    k = [dev(a[n]) for n in ("kx", "ky", "kz")]
    r, i = mri.fhd_batched_grid(*k, dev(xs), dev(ys), dev(zs), dev(a["rPhi"]), dev(a["iPhi"]),
                                dev(rD), dev(iD), trig=trig)
    x, y, z = expand(xs, ys, zs)
    idx = wl.voxel_subset(x.size, 256, 17)
    ref = oracle.fhd_batched(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"], rD, iD,
                             idx=idx)
    got = cplx(r, i)[:, idx]
    for b in range(B):
        assert oracle.rel_l2(got[b], ref[b]) <= TOL[trig], f"coil {b}"
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("nx,ny,nz,M", [(64, 5, 3, 3001), (256, 3, 50, 777),
                                        (384, 2, 3, 1500)])
def test_forward_column_blocks(mri, nx, ny, nz, M, trig):
    xs, ys, zs = axes(nx, ny, nz, 7 * nx + M)
    a = samples(M, 17 * nx + M)
    rng = np.random.default_rng(nx * 3 + M)
    N = nx * ny * nz
    rho = (rng.standard_normal(N) + 1j * rng.standard_normal(N)).astype(np.complex64)
    k = [dev(a[n]) for n in ("kx", "ky", "kz")]
    ax = [dev(xs), dev(ys), dev(zs)]
    r, i = mri.forward_grid(*k, *ax, dev(rho.real), dev(rho.imag), trig=trig)
    x, y, z = expand(xs, ys, zs)
    ref = oracle.forward(a["kx"], a["ky"], a["kz"], x, y, z, rho)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]
    out = (torch.full_like(r, 1.5), torch.full_like(i, -2.0))
    mri.forward_grid(*k, *ax, dev(rho.real), dev(rho.imag), trig=trig, accumulate=True, out=out)
    assert oracle.rel_l2(cplx(out[0] - 1.5, out[1] + 2.0), ref) <= TOL[trig]
    assert mri.device_errors(clear=True) == 0


def test_forward_adjoint_at_256(mri):
    """<F rho, D> = <rho, F^H D> with both sides on the tensor cores at nx = 256."""
    nx, ny, nz, M = 256, 4, 3, 2000
    xs, ys, zs = axes(nx, ny, nz, 99)
    a = samples(M, 98)
    rng = np.random.default_rng(97)
    N = nx * ny * nz
    rho = (rng.standard_normal(N) + 1j * rng.standard_normal(N)).astype(np.complex64)
    k = [dev(a[n]) for n in ("kx", "ky", "kz")]
    ax = [dev(xs), dev(ys), dev(zs)]
    fr, fi = mri.forward_grid(*k, *ax, dev(rho.real), dev(rho.imag), trig="accurate")
    one = torch.ones(M, device="cuda")
    zero = torch.zeros(M, device="cuda")
    hr, hi = mri.fhd_grid(*k, *ax, one, zero, dev(a["rD"]), dev(a["iD"]), trig="accurate")
    d = a["rD"].astype(np.float64) + 1j * a["iD"]
    f_rho, fhd = cplx(fr, fi), cplx(hr, hi)
    lhs = np.vdot(d, f_rho)                         # <D, F rho>
    rhs = np.vdot(fhd, rho)                         # <F^H D, rho>
    scale = np.linalg.norm(d) * np.linalg.norm(f_rho) + np.linalg.norm(fhd) * np.linalg.norm(rho)
    assert abs(lhs - rhs) <= 1e-5 * scale
