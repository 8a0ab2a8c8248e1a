"""Edge shapes of the tensor-core grid paths against the oracle: one sample,
one row, sample counts just under / over a tile, row counts just over a
block, a padded coil group; at nx = 128 (one whole column block), nx = 9
(one mostly padded block, rows not 16-byte aligned: scalar stores) and
nx = 200 (a whole block and a partial one).  Every entry point that runs on
the tensor cores: F^H D, Q, batched F^H D, the forward model."""

import numpy as np
import pytest
import torch

import oracle
from non_cartesian_mri_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"accurate": 1e-5, "fast": 2e-4}
SHAPES = [(1, 1, 1), (1, 1, 31), (2, 3, 33), (5, 1, 64), (130, 1, 100), (1, 129, 257)]
WIDTHS = [128, 9, 200]


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


def case(nx, ny, nz, M, seed):
    rng = np.random.default_rng(seed)
    k = rng.uniform(-0.5, 0.5, (3, M)).astype(np.float32)
    if nx == 128:
        xs = (np.arange(128) - 64).astype(np.float32)
    else:
        xs = np.sort(rng.uniform(-64.0, 64.0, nx)).astype(np.float32)
    ys = (rng.permutation(256)[:ny] - 128).astype(np.float32) * 0.5
    zs = (rng.permutation(256)[:nz] - 128).astype(np.float32) * 0.5
    z, y, x = (a.reshape(-1) for a in np.meshgrid(zs, ys, xs, indexing="ij"))
    w = rng.standard_normal((4, M)).astype(np.float32)
    return k, xs, ys, zs, x, y, z, w, rng


def rel(got, ref):
    # a single sample can sum to an exact zero only by accident; guard anyway
    return oracle.rel_l2(got, ref) if np.linalg.norm(ref) > 0 else np.linalg.norm(got)


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("ny,nz,M", SHAPES)
@pytest.mark.parametrize("nx", WIDTHS)
def test_fhd_and_q_grid_shapes(mri, nx, ny, nz, M, trig):
    k, xs, ys, zs, x, y, z, w, _ = case(nx, ny, nz, M, nx + ny * 1000 + nz * 10 + M)
    kk = [dev(a) for a in k]
    axes = [dev(xs), dev(ys), dev(zs)]
    r, i = mri.fhd_grid(*kk, *axes, *[dev(a) for a in w], trig=trig)
    ref = oracle.fhd(k[0], k[1], k[2], x, y, z, w[0], w[1], w[2], w[3])
    assert rel(cplx(r, i), ref) <= TOL[trig]
    qr, qi = mri.q_grid(*kk, *axes, dev(w[0]), dev(w[1]), trig=trig)
    qref = oracle.q(k[0], k[1], k[2], x, y, z, w[0], w[1])
    assert rel(cplx(qr, qi), qref) <= TOL[trig]


@pytest.mark.parametrize("ny,nz,M", SHAPES)
@pytest.mark.parametrize("nx", WIDTHS)
def test_batched_grid_shapes(mri, nx, ny, nz, M):
    k, xs, ys, zs, x, y, z, w, rng = case(nx, ny, nz, M, 7 + nx + ny + nz + M)
    B = 5                                   # one padded group of 8
    rD = rng.standard_normal((B, M)).astype(np.float32)
    iD = rng.standard_normal((B, M)).astype(np.float32)
    r, i = mri.fhd_batched_grid(*[dev(a) for a in k], dev(xs), dev(ys), dev(zs), dev(w[0]),
                                dev(w[1]), dev(rD), dev(iD), trig="accurate")
    ref = oracle.fhd_batched(k[0], k[1], k[2], x, y, z, w[0], w[1], rD, iD)
    got = cplx(r, i)
    for b in range(B):
        assert rel(got[b], ref[b]) <= TOL["accurate"], b


@pytest.mark.parametrize("ny,nz,M", SHAPES)
@pytest.mark.parametrize("nx", WIDTHS)
def test_forward_grid_shapes(mri, nx, ny, nz, M):
    k, xs, ys, zs, x, y, z, _, rng = case(nx, ny, nz, M, 99 + nx + ny + nz + M)
    n = nx * ny * nz
    rho = (rng.standard_normal(n) + 1j * rng.standard_normal(n)).astype(np.complex64)
    r, i = mri.forward_grid(*[dev(a) for a in k], dev(xs), dev(ys), dev(zs), dev(rho.real),
                            dev(rho.imag), trig="accurate")
    ref = oracle.forward(k[0], k[1], k[2], x, y, z, rho)
    assert rel(cplx(r, i), ref) <= TOL["accurate"]
    assert mri.device_errors(clear=True) == 0
