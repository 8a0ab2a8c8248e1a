"""Pins of the gridding oracle (oracle/gridding.py), no GPU.

- samples on grid points (k = (g - n/2)/n, exact in float32) are not
  interpolated, so the reconstruction is exactly the C oracle's F^H D at the
  voxel coordinates x = i - n/2 (catches the exponent's sign, the centring, a
  swapped axis on non-cubic grids);
- the eight weights of a sample sum to one, so the image at x = 0 is the sum
  of Mu, and they reproduce the sample's position (sum of w * k_g = k), which
  catches f and 1 - f swapped;
- a sample halfway between two grid points splits evenly;
- shifting k by a whole period gives the same grid (wrap-around);
- recon (numpy's inverse FFT with the centring) against recon_direct (three
  DFT matrices written out).
"""

import numpy as np
import pytest

import oracle
from oracle import gridding as Gr


def on_grid_samples(shape, M, seed):
    nz, ny, nx = shape
    rng = np.random.default_rng(seed)
    k = [((rng.integers(0, n, M) - n // 2) / n).astype(np.float32) for n in (nx, ny, nz)]
    vals = [rng.standard_normal(M).astype(np.float32) for _ in range(4)]
    return k, vals


@pytest.mark.parametrize("shape", [(4, 8, 16), (2, 4, 2), (8, 8, 8)])
def test_on_grid_samples_give_fhd(shape):
    nz, ny, nx = shape
    k, (rPhi, iPhi, rD, iD) = on_grid_samples(shape, 300, sum(shape))
    img = Gr.gridding_recon(*k, rPhi, iPhi, rD, iD, shape)
    z, y, x = np.meshgrid(np.arange(nz) - nz // 2, np.arange(ny) - ny // 2,
                          np.arange(nx) - nx // 2, indexing="ij")
    ref = oracle.fhd(*k, x.reshape(-1).astype(np.float32), y.reshape(-1).astype(np.float32),
                     z.reshape(-1).astype(np.float32), rPhi, iPhi, rD, iD)
    assert oracle.rel_l2(img.reshape(-1), ref) < 1e-12


def test_weights_partition_unity_and_reproduce_position():
    shape = (8, 16, 32)
    nz, ny, nx = shape
    rng = np.random.default_rng(3)
    M = 200
    # away from the wrap edge, so that the corners are not folded
    k = [rng.uniform(-0.45, 0.45, M) for _ in range(3)]
    mu = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    G = Gr.grid_samples(*k, mu, shape)
    assert abs(G.sum() - mu.sum()) < 1e-12 * np.abs(mu).sum()
    img = Gr.recon(G)
    assert abs(img[nz // 2, ny // 2, nx // 2] - mu.sum()) < 1e-10 * np.abs(mu).sum()
    for m in range(5):
        Gm = Gr.grid_samples(*(kk[m:m + 1] for kk in k), np.ones(1), shape)
        for axis, n, km in ((2, nx, k[0][m]), (1, ny, k[1][m]), (0, nz, k[2][m])):
            kg = (np.arange(n) - n // 2) / n
            shape_b = [1, 1, 1]
            shape_b[axis] = n
            assert abs((Gm.real * kg.reshape(shape_b)).sum() - km) < 1e-12


def test_halfway_sample_splits_evenly():
    shape = (4, 4, 8)
    # x halfway between g = 5 and 6; y and z on grid points 1 and 2
    kx = np.array([(5.5 - 4) / 8])
    ky = np.array([(1 - 2) / 4])
    kz = np.array([(2 - 2) / 4])
    G = Gr.grid_samples(kx, ky, kz, np.array([2.0 + 1.0j]), shape)
    nzr = np.argwhere(np.abs(G) > 0)
    assert sorted(map(tuple, nzr)) == [(2, 1, 5), (2, 1, 6)]
    assert G[2, 1, 5] == pytest.approx(1.0 + 0.5j) and G[2, 1, 6] == pytest.approx(1.0 + 0.5j)


def test_wrap_around_is_one_period():
    shape = (4, 8, 16)
    rng = np.random.default_rng(5)
    k = [rng.uniform(-0.5, 0.5, 64) for _ in range(3)]
    mu = rng.standard_normal(64) + 1j * rng.standard_normal(64)
    G = Gr.grid_samples(*k, mu, shape)
    G2 = Gr.grid_samples(k[0] - 1.0, k[1] + 1.0, k[2] - 1.0, mu, shape)
    assert np.abs(G - G2).max() < 1e-12
    # a sample just below +1/2 lands (almost) on the wrapped grid point 0
    Gw = Gr.grid_samples(np.array([0.5 - 2.0 ** -30]), np.zeros(1), np.zeros(1), np.ones(1),
                         shape)
    assert Gw[2, 4, 0] == pytest.approx(1.0, abs=1e-6)


@pytest.mark.parametrize("shape", [(2, 4, 8), (1, 2, 4), (4, 4, 4)])
def test_recon_equals_direct_sum(shape):
    rng = np.random.default_rng(sum(shape))
    G = rng.standard_normal(shape) + 1j * rng.standard_normal(shape)
    assert oracle.rel_l2(Gr.recon(G), Gr.recon_direct(G)) < 1e-12
