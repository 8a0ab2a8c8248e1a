"""The gridding reconstruction (mri_gridding) on the GPU against the oracle
(oracle/gridding.py).

- random trajectories on non-cubic grids, one-voxel axes, ragged and tiny M,
  against the oracle element by element;
- samples on grid points: the result is F^H D (the oracle's and the GPU grid
  path's);
- the benchmarked size (128^3, 3D radial trajectory) in full against the
  oracle (which is cheap here: an interpolation and numpy's FFT);
- the longest FFT lines (1024), all samples at the origin (a constant
  image), accumulate, M = 0, argument errors.

Tolerance: the interpolation is exact arithmetic up to fp32 rounding of the
weights and of the atomic sums on the grid (whose order is not fixed), then
one fp32 inverse FFT (~1e-7 log2 N): 1e-5 relative L2.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import gridding as Gr

pytestmark = pytest.mark.gpu

TOL = 1e-5


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
    k = [rng.uniform(-kmax, kmax, M).astype(np.float32) for _ in range(3)]
    v = [rng.standard_normal(M).astype(np.float32) for _ in range(4)]
    return k, v


@pytest.mark.parametrize("shape,M", [((4, 8, 16), 1000), ((8, 8, 8), 4097), ((1, 4, 32), 333),
                                     ((2, 1, 1), 17), ((16, 32, 8), 1), ((32, 32, 32), 20000)])
def test_gridding_matches_oracle(mri, shape, M):
    k, v = samples(M, sum(shape) + M)
    r, i = mri.gridding(*(dev(a) for a in k), *(dev(a) for a in v), shape)
    ref = Gr.gridding_recon(*k, *v, shape).reshape(-1)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("shape", [(1, 1, 1024), (2, 1024, 1), (1024, 2, 2)])
def test_gridding_longest_lines(mri, shape):
    """An axis of 1024 voxels (the longest FFT line)."""
    k, v = samples(3000, sum(shape))
    r, i = mri.gridding(*(dev(a) for a in k), *(dev(a) for a in v), shape)
    ref = Gr.gridding_recon(*k, *v, shape).reshape(-1)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL


def test_samples_at_the_origin_give_a_constant_image(mri):
    """Every sample at k = 0: all weight on the grid point k_g = 0, and the
    image is the constant sum of Mu."""
    M = 777
    _, v = samples(M, 77)
    z = np.zeros(M, np.float32)
    r, i = mri.gridding(dev(z), dev(z), dev(z), *(dev(a) for a in v), (4, 8, 16))
    mu = Gr.mu(*v).sum()
    img = cplx(r, i)
    assert np.abs(img - mu).max() <= 1e-5 * abs(mu)


def test_on_grid_samples_give_fhd(mri):
    shape = (8, 16, 32)
    nz, ny, nx = shape
    rng = np.random.default_rng(9)
    M = 5000
    k = [((rng.integers(0, n, M) - n // 2) / n).astype(np.float32) for n in (nx, ny, nz)]
    v = [rng.standard_normal(M).astype(np.float32) for _ in range(4)]
    r, i = mri.gridding(*(dev(a) for a in k), *(dev(a) for a in v), shape)
    axes = [(np.arange(n) - n // 2).astype(np.float32) for n in (nx, ny, nz)]
    z, y, x = (a.reshape(-1) for a in np.meshgrid(axes[2], axes[1], axes[0], indexing="ij"))
    ref = oracle.fhd(*k, x, y, z, *v)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL
    gr, gi = mri.fhd_grid(*(dev(a) for a in k), *(dev(a) for a in axes), *(dev(a) for a in v),
                          trig="accurate")
    assert oracle.rel_l2(cplx(r, i), cplx(gr, gi)) <= 2 * TOL


def test_gridding_full_size_radial(mri):
    from non_cartesian_mri_gb300 import workloads as wl
    w = wl.make_workload("fhd_128_radial")
    shape = (w.L, w.L, w.L)
    args = [dev(a) for a in (w.kx, w.ky, w.kz, w.rPhi, w.iPhi, w.rD, w.iD)]
    r, i = mri.gridding(*args, shape)
    ref = Gr.gridding_recon(w.kx, w.ky, w.kz, w.rPhi, w.iPhi, w.rD, w.iD, shape).reshape(-1)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL
    # accumulate adds onto what is there
    out = (torch.full_like(r, 2.0), torch.full_like(i, -3.0))
    mri.gridding(*args, shape, accumulate=True, out=out)
    assert oracle.rel_l2(cplx(out[0] - 2.0, out[1] + 3.0), ref) <= TOL
    assert mri.device_errors(clear=True) == 0


def test_gridding_without_samples_is_zero(mri):
    e = torch.empty(0, device="cuda")
    r, i = mri.gridding(e, e, e, e, e, e, e, (4, 4, 8))
    assert torch.count_nonzero(r) == 0 and torch.count_nonzero(i) == 0


def test_gridding_argument_errors(mri):
    lib = mri.load()
    buf = torch.zeros(4096, device="cuda")
    P = ctypes.c_void_p
    p = P(buf.data_ptr())
    for nx, ny, nz in ((3, 4, 4), (4, 4, 2048), (0, 4, 4)):
        assert lib.mri_gridding(p, p, p, p, p, p, p, 16, nx, ny, nz, p, p, 0, None) == 2
    assert lib.mri_gridding(p, p, p, p, p, p, p, 16, 4, 4, 4, p, p, 2, None) == 5
    assert lib.mri_gridding(None, p, p, p, p, p, p, 16, 4, 4, 4, p, p, 0, None) == 1
