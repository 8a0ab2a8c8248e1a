"""fp64 oracle of the gridding reconstruction: the non-Cartesian samples
interpolated onto a Cartesian k-space grid, then an inverse DFT.

TEST INFRASTRUCTURE ONLY (as the rest of this package).

The chapter "Iterative MRI reconstruction" (section 17.1, Fig. 17.1B, and
the accuracy comparison of Fig. 17.19) names this as the usual alternative to
the iterative reconstruction: samples on a non-Cartesian trajectory are
interpolated ("gridded") onto a uniform grid, after which an inverse FFT gives
the image; its bilinear form reaches 16.8 dB against the iterative method's
27.6 dB on the pages' phantom.  Readings taken here, since the pages give no
more detail:

- the value gridded is the same Mu = conj(Phi) D that F^H D sums (Phi
  carries any density-compensation weight);
- the image is on the voxel grid x = i - n/2, i < n, per axis (unit spacing,
  the integer coordinates of the workloads), and the k-space grid is the one
  that grid's DFT uses: k_g = (g - n/2) / n, g < n;
- interpolation is the three-dimensional form of bilinear: each sample adds
  to the 2 x 2 x 2 grid points around it with weights (1 - f) or f per axis,
  f the fractional position; k is periodic with period 1 on the integer
  voxel grid (e^{i 2 pi (k + 1) x} = e^{i 2 pi k x}), so indices wrap modulo n;
- rho(x) = sum_g G[g] e^{+i 2 pi k_g . x}: no density or deapodisation
  correction beyond what Phi carries.

Functions: grid_samples (the interpolation, a plain loop over the eight
corners with numpy's unbuffered add), recon_direct (the sum above written out
as three small DFT matrices), recon (the same through numpy's inverse FFT,
with the centring written out).  Pinned in tests/test_oracle_gridding.py:
on-grid samples give exactly the oracle's F^H D, the weights of a sample sum
to one (the image at x = 0 is the sum of Mu), a sample halfway between grid
points splits evenly, wrap-around at k = +-1/2, and recon against
recon_direct.
"""

from __future__ import annotations

import numpy as np


def mu(rPhi, iPhi, rD, iD):
    """Mu = conj(Phi) D in complex128."""
    phi = np.asarray(rPhi, np.float64) + 1j * np.asarray(iPhi, np.float64)
    d = np.asarray(rD, np.float64) + 1j * np.asarray(iD, np.float64)
    return np.conj(phi) * d


def grid_samples(kx, ky, kz, values, shape):
    """G[gz, gy, gx] = sum_m values[m] * w_x w_y w_z over the 8 grid points
    around sample m: position u = (k + 1/2) n on each axis (grid point g sits
    at k_g = (g - n/2) / n), g0 = floor(u), f = u - g0, weight 1 - f for g0
    and f for g0 + 1, indices modulo n."""
    nz, ny, nx = shape
    values = np.asarray(values, np.complex128)
    pos = []
    for k, n in ((kx, nx), (ky, ny), (kz, nz)):
        u = (np.asarray(k, np.float64) + 0.5) * n
        g0 = np.floor(u)
        f = u - g0
        pos.append((g0.astype(np.int64), f, n))
    G = np.zeros(shape, np.complex128)
    for cz in (0, 1):
        for cy in (0, 1):
            for cx in (0, 1):
                (gx, fx, nx_), (gy, fy, ny_), (gz, fz, nz_) = pos
                w = ((fx if cx else 1 - fx) * (fy if cy else 1 - fy) * (fz if cz else 1 - fz))
                np.add.at(G, ((gz + cz) % nz_, (gy + cy) % ny_, (gx + cx) % nx_), values * w)
    return G


def _dft_matrix(n):
    """E[i, g] = e^{+i 2 pi k_g x_i}, x_i = i - n/2, k_g = (g - n/2) / n."""
    x = np.arange(n) - n // 2
    k = (np.arange(n) - n // 2) / n
    return np.exp(2j * np.pi * np.outer(x, k))


def recon_direct(G):
    """rho[iz, iy, ix] = sum_g G[g] e^{+i 2 pi k_g . x}, as three DFT matrices
    (small grids)."""
    nz, ny, nx = G.shape
    return np.einsum("zc,yb,xa,cba->zyx", _dft_matrix(nz), _dft_matrix(ny), _dft_matrix(nx), G)


def recon(G):
    """The same sum through numpy's inverse FFT: with g = j, x = i - n/2 and
    k_g = (j - n/2)/n per axis, e^{i 2 pi k_g x} = e^{i 2 pi j i / n}
    (-1)^j (-1)^i (-1)^{n/2}, so rho = c (-1)^i n^3 ifftn(G (-1)^j)."""
    nz, ny, nx = G.shape
    sz, sy, sx = (((-1.0) ** np.arange(n)) for n in (nz, ny, nx))
    sign = sz[:, None, None] * sy[None, :, None] * sx[None, None, :]
    c = (-1.0) ** (nz // 2 + ny // 2 + nx // 2)
    return c * sign * np.fft.ifftn(G * sign) * (nz * ny * nx)


def gridding_recon(kx, ky, kz, rPhi, iPhi, rD, iD, shape):
    """The whole reconstruction: Mu, interpolation, inverse DFT; complex128
    image [nz, ny, nx]."""
    return recon(grid_samples(kx, ky, kz, mu(rPhi, iPhi, rD, iD), shape))
