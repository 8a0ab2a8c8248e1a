"""Narrow grids on the tensor cores with folded rows, against the oracle.

For 8 <= nx <= 64 a block of 128 columns holds G = 128 / fw grid rows (fw =
nx rounded up to a power of two) when ny is a multiple of G.  Folding is
exact when every group of G rows has the same y offsets from its first row;
a check on the device decides, and otherwise the unfolded (padded) layout
runs.  Covered: every width class, y axes that fold (evenly spaced, and
groups with equal offsets but irregular gaps between groups) and axes that
must not (random, one irregular group), F^H D / Q / coil groups, accumulate,
sample splits, several and ragged row blocks.  All voxels are compared.
"""

import numpy as np
import pytest
import torch

import oracle
from non_cartesian_mri_gb300 import workloads as wl

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


def expand(xs, ys, zs):
    z, y, x = np.meshgrid(zs, ys, xs, indexing="ij")
    return x.reshape(-1), y.reshape(-1), z.reshape(-1)


def fold_of(nx, ny):
    if nx < 8 or nx > 64:
        return 1
    fw = 8
    while fw < nx:
        fw *= 2
    G = 128 // fw
    return G if ny % G == 0 else 1


def y_axis(kind, ny, G, rng):
    if kind == "even":
        return (np.arange(ny) * 0.75 - 7.0).astype(np.float32)
    if kind == "groups":
        # equal offsets inside every group of G rows, irregular gaps between groups
        base = np.cumsum(rng.integers(G + 1, 3 * G, ny // G)).astype(np.float32)
        return (np.repeat(base, G) + np.tile(np.arange(G), ny // G) - 20.0).astype(np.float32)
    if kind == "random":
        return np.sort(rng.uniform(-30, 30, ny)).astype(np.float32)
    # "one_off": evenly spaced but one row of the last group moved by a quarter
    y = (np.arange(ny) - ny // 2).astype(np.float32)
    y[-1] += 0.25
    return y


def inputs(M, seed):
    rng = np.random.default_rng(seed)
    k = rng.uniform(-0.5, 0.5, (3, M)).astype(np.float32)
    w = rng.standard_normal((4, M)).astype(np.float32)
    return k, w, rng


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("nx,ny,nz", [(64, 8, 3), (48, 4, 5), (32, 16, 3), (20, 8, 2),
                                      (16, 32, 2), (9, 8, 3), (8, 16, 2)])
@pytest.mark.parametrize("ykind", ["even", "groups", "random", "one_off"])
def test_fhd_grid_fold(mri, nx, ny, nz, ykind, trig):
    G = fold_of(nx, ny)
    assert G > 1
    M = 1000
    k, w, rng = inputs(M, nx * 100 + ny + nz)
    xs = (np.arange(nx) - nx // 2).astype(np.float32) * 1.25
    ys = y_axis(ykind, ny, G, rng)
    zs = (np.arange(nz) * 2.0 - 3.0).astype(np.float32)
    assert mri.plan_grid("fhd", M, nx, ny, nz)["grid_fold"] == G
    r, i = mri.fhd_grid(dev(k[0]), dev(k[1]), dev(k[2]), dev(xs), dev(ys), dev(zs),
                        *(dev(a) for a in w), trig=trig)
    x, y, z = expand(xs, ys, zs)
    ref = oracle.fhd(k[0], k[1], k[2], x, y, z, *w)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("trig", ["accurate", "fast"])
def test_q_grid_fold(mri, trig):
    nx, ny, nz, M = 32, 12, 4, 777           # G = 4
    k, w, _ = inputs(M, 5)
    xs = (np.arange(nx) - 16).astype(np.float32)
    ys = (np.arange(ny) - 6).astype(np.float32)
    zs = (np.arange(nz) - 2).astype(np.float32)
    r, i = mri.q_grid(dev(k[0]), dev(k[1]), dev(k[2]), dev(xs), dev(ys), dev(zs), dev(w[0]),
                      dev(w[1]), trig=trig)
    x, y, z = expand(xs, ys, zs)
    ref = oracle.q(k[0], k[1], k[2], x, y, z, w[0], w[1])
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]


@pytest.mark.parametrize("B", [8, 3])
def test_batched_grid_fold(mri, B):
    nx, ny, nz, M = 64, 6, 3, 900             # G = 2; B = 3 runs as a padded group of 4
    rng = np.random.default_rng(B)
    k = rng.uniform(-0.5, 0.5, (3, M)).astype(np.float32)
    phi = rng.standard_normal((2, M)).astype(np.float32)
    rD = rng.standard_normal((B, M)).astype(np.float32)
    iD = rng.standard_normal((B, M)).astype(np.float32)
    xs = (np.arange(nx) - 32).astype(np.float32)
    ys = (np.arange(ny) * 2.0).astype(np.float32)
    zs = np.array([-1.0, 0.0, 4.0], np.float32)
    r, i = mri.fhd_batched_grid(dev(k[0]), dev(k[1]), dev(k[2]), dev(xs), dev(ys), dev(zs),
                                dev(phi[0]), dev(phi[1]), dev(rD), dev(iD), trig="accurate")
    x, y, z = expand(xs, ys, zs)
    ref = oracle.fhd_batched(k[0], k[1], k[2], x, y, z, phi[0], phi[1], rD, iD)
    got = cplx(r, i)
    for b in range(B):
        assert oracle.rel_l2(got[b], ref[b]) <= TOL["accurate"], b


def test_fold_accumulate_splits_and_row_blocks(mri):
    """Many samples (split across CTAs), 9 planes x 16 = 144 row groups (two
    blocks of 128, the second ragged), added onto existing outputs."""
    nx, ny, nz, M = 32, 64, 9, 20000          # G = 4: 16 row groups per plane
    k, w, _ = inputs(M, 11)
    xs = (np.arange(nx) - 16).astype(np.float32)
    ys = (np.arange(ny) - 32).astype(np.float32)
    zs = (np.arange(nz) - 4).astype(np.float32)
    p = mri.plan_grid("fhd", M, nx, ny, nz)
    assert p["grid_fold"] == 4 and p["splits"] > 1 and p["voxel_ctas"] == 2
    N = nx * ny * nz
    out = (torch.full((N,), 0.5, device="cuda"), torch.full((N,), -1.5, device="cuda"))
    mri.fhd_grid(dev(k[0]), dev(k[1]), dev(k[2]), dev(xs), dev(ys), dev(zs),
                 *(dev(a) for a in w), trig="accurate", accumulate=True, out=out)
    x, y, z = expand(xs, ys, zs)
    idx = wl.voxel_subset(N, 3000, 7)
    ref = oracle.fhd(k[0], k[1], k[2], x, y, z, *w, idx=idx)
    got = cplx(out[0] - 0.5, out[1] + 1.5)[idx]
    assert oracle.rel_l2(got, ref) <= TOL["accurate"]
    assert mri.device_errors(clear=True) == 0
