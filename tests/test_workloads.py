"""Input generators: shapes, determinism and the stated trajectory geometry."""

import numpy as np
import pytest

from non_cartesian_mri_gb300 import workloads as wl

SIZES = {
    "fhd_tiny": (16 ** 3, 2048),
    "fhd_64": (64 ** 3, 32768),
    "fhd_128_radial": (128 ** 3, 262144),
    "q_128": (128 ** 3, 1048576),
    "fhd_batched_128": (128 ** 3, 524288),
}


@pytest.mark.parametrize("name", sorted(SIZES))
def test_sizes_and_dtypes(name):
    w = wl.make_workload(name, L=4)     # small grid keeps this fast; M unchanged
    N, M = SIZES[name]
    assert w.M == M
    assert w.N == 4 ** 3
    for a in (w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    kabs = np.sqrt(w.kx.astype(np.float64) ** 2 + w.ky ** 2 + w.kz ** 2)
    assert kabs.max() <= 0.5 * (1 + 1e-6) * (np.sqrt(3) if name == "fhd_tiny" else 1)
    if w.kind == "fhd_batched":
        assert w.rD.shape == (8, M) and w.B == 8
    elif w.kind == "fhd":
        assert w.rD.shape == (M,)


def test_full_grid_sizes():
    assert wl.voxel_grid(128)[0].size == 128 ** 3


def test_deterministic():
    a = wl.make_workload("fhd_tiny")
    b = wl.make_workload("fhd_tiny")
    for f in ("kx", "ky", "kz", "rPhi", "iPhi", "rD", "iD"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    c = wl.make_workload("fhd_tiny", seed=5)
    assert not np.array_equal(a.kx, c.kx)


def test_voxel_grid_order_x_fastest():
    x, y, z = wl.voxel_grid(4, 3, 2)
    assert x[:4].tolist() == [-2, -1, 0, 1]
    assert y[:5].tolist() == [-1, -1, -1, -1, 0]
    assert z[11] == -1 and z[12] == 0
    assert (x.min(), x.max(), y.min(), y.max(), z.min(), z.max()) == (-2, 1, -1, 1, -1, 0)


def test_radial_lines_pass_through_origin_without_a_zero_sample():
    kx, ky, kz = wl.traj_radial_fibonacci(16, 8)
    k = np.stack([kx, ky, kz]).astype(np.float64).reshape(3, 16, 8)
    assert np.all(np.abs(k).sum(axis=0) > 0)
    # the points of a line are symmetric about the origin
    np.testing.assert_allclose(k[:, :, ::-1], -k, atol=1e-7)
    np.testing.assert_allclose(np.linalg.norm(k[:, :, -1], axis=0), 0.5, rtol=1e-6)


def test_stack_of_spirals_is_point_symmetric():
    P, I, S = 8, 4, 32
    kx, ky, kz = wl.traj_stack_of_spirals(P, I, S, turns=2.0)
    k = np.stack([kx, ky, kz]).astype(np.float64).reshape(3, P, I, S)
    # plane p, interleave i  <->  plane P-1-p, interleave i+I/2
    mirror = k[:, ::-1][:, :, (np.arange(I) + I // 2) % I]
    np.testing.assert_allclose(mirror, -k, atol=1e-6)


def test_subset_sorted_distinct():
    idx = wl.voxel_subset(1000, 100, 3)
    assert idx.dtype == np.int64 and len(np.unique(idx)) == 100
    assert np.all(np.diff(idx) > 0)
