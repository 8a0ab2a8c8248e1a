"""Batched F^H D on a separable grid (mri_fhd_batched_grid) against the oracle.

nx >= 8 runs on the tensor cores in coil groups of 8 (a remainder of 2..4
coils as a padded group of 4, 5..7 as a padded group of 8, one coil alone);
other nx go through expanded coordinates and the general batched kernel.
The oracle gets the expanded voxel coordinates; tolerances as everywhere
(1e-5 accurate, 2e-4 fast), checked per coil so that a coil with small
weights next to large ones is held to the same relative bound.
"""

import numpy as np
import pytest
import torch

import oracle
from non_cartesian_mri_gb300 import workloads as wl
from tests.sampling import grid_blocks

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


def coil_data(w, B, M, seed, scales=None):
    """B coils of D on the first M samples of workload w (D_b = D * coil gain
    + noise); `scales` multiplies whole coils."""
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal(B) + 1j * rng.standard_normal(B)).astype(np.complex64)
    d = w.rD[:M] + 1j * w.iD[:M]
    dc = g[:, None] * d[None, :] + 0.1 * (rng.standard_normal((B, M)) + 1j * rng.standard_normal((B, M)))
    if scales is not None:
        dc = dc * np.asarray(scales, np.float64)[:, None]
    return dc.real.astype(np.float32), dc.imag.astype(np.float32)


def check_per_coil(got, ref, tol):
    for b in range(ref.shape[0]):
        assert oracle.rel_l2(got[b], ref[b]) <= tol, f"coil {b}"


@pytest.mark.parametrize("trig", ["accurate", "fast"])
@pytest.mark.parametrize("B", [1, 3, 8, 9, 13])
def test_tensor_core_coil_groups(mri, B, trig):
    """Groups of 1, a padded 4, a full 8 and 8 + padded 8; ragged rows
    (3 x 7 = 21) and a ragged sample count."""
    w = wl.make_workload("fhd_128_radial")
    M = 5001
    xs = (np.arange(128) - 64).astype(np.float32)
    # B = 9: a group of 8 and a single coil, on whole 128-row planes (each
    # CTA's rows one z plane)
    ys = (np.arange(128) - 64).astype(np.float32) if B == 9 else np.array([-40, 3, 57], np.float32)
    zs = np.array([-30.0, 6.0], np.float32) if B == 9 else (np.arange(7) * 9 - 30).astype(np.float32)
    rD, iD = coil_data(w, B, M, 10 + B)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    phi = [dev(w.rPhi[:M]), dev(w.iPhi[:M])]
    r, i = mri.fhd_batched_grid(*k, dev(xs), dev(ys), dev(zs), *phi, dev(rD), dev(iD), trig=trig)
    assert r.shape == (B, 128 * ys.size * zs.size)
    x, y, z = expand(xs, ys, zs)
    ref = oracle.fhd_batched(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, w.rPhi[:M], w.iPhi[:M],
                             rD, iD)
    check_per_coil(cplx(r, i), ref, TOL[trig])
    plan = mri.plan_grid_batched(B, M, 128, ys.size, zs.size)
    assert plan["tensor_cores"] == 1
    assert plan["coil_groups"] == {1: 1, 3: 1, 8: 1, 9: 2, 13: 2}[B]


def test_batched_grid_accumulates_and_matches_single_coil_calls(mri):
    w = wl.make_workload("fhd_128_radial")
    M, B = 3000, 5
    xs = (np.arange(128) - 64).astype(np.float32)
    ys = np.arange(4, dtype=np.float32) * 3 - 6
    zs = np.array([2.0, -9.0], np.float32)
    rD, iD = coil_data(w, B, M, 7)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    axes = [dev(xs), dev(ys), dev(zs)]
    phi = [dev(w.rPhi[:M]), dev(w.iPhi[:M])]
    r, i = mri.fhd_batched_grid(*k, *axes, *phi, dev(rD), dev(iD), trig="accurate")
    for b in range(B):
        rb, ib = mri.fhd_grid(*k, *axes, *phi, dev(rD[b]), dev(iD[b]), trig="accurate")
        assert oracle.rel_l2(cplx(r[b], i[b]), cplx(rb, ib)) <= 2e-6
    out = (torch.full_like(r, 1.5), torch.full_like(i, -2.0))
    mri.fhd_batched_grid(*k, *axes, *phi, dev(rD), dev(iD), trig="accurate", accumulate=True,
                         out=out)
    assert oracle.rel_l2(cplx(out[0] - 1.5, out[1] + 2.0), cplx(r, i)) <= 1e-6


def test_coils_of_very_different_scale(mri):
    """Each coil of a group has its own power-of-two operand scale: coils
    1e-6 and 1e4 times the others (a range no single f16 scale covers with
    full precision) still meet the relative bound each."""
    w = wl.make_workload("fhd_128_radial")
    M, B = 4000, 4
    xs = (np.arange(128) - 64).astype(np.float32)
    ys = np.array([0.0, 5.0], np.float32)
    zs = np.array([1.0], np.float32)
    rD, iD = coil_data(w, B, M, 3, scales=[1.0, 1e-6, 1e4, 1.0])
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    r, i = mri.fhd_batched_grid(*k, dev(xs), dev(ys), dev(zs), dev(w.rPhi[:M]),
                                dev(w.iPhi[:M]), dev(rD), dev(iD), trig="accurate")
    x, y, z = expand(xs, ys, zs)
    ref = oracle.fhd_batched(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, w.rPhi[:M], w.iPhi[:M],
                             rD, iD)
    check_per_coil(cplx(r, i), ref, TOL["accurate"])


_batched_ref = {}


def batched_ref(mri, w):
    """One voxel from every (row block, column block) of the 8-coil launch --
    16 grid rows per CTA, 1,024 blocks -- every coil; computed once."""
    if not _batched_ref:
        n = 128
        p = mri.plan_grid_batched(8, w.M, n, n, n)
        assert p["tensor_cores"] and p["voxel_ctas"] == n * n // 16
        idx = grid_blocks(n, n, n, 16, 301)
        _batched_ref["v"] = (idx, oracle.fhd_batched(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi,
                                                     w.iPhi, w.rD, w.iD, idx=idx))
    return _batched_ref["v"]


@pytest.mark.parametrize("trig", ["accurate", "fast"])
def test_batched_grid_128_workload(mri, trig):
    """The 8-coil 128^3 stack-of-spirals workload, sampled voxels."""
    w = wl.make_workload("fhd_batched_128")
    xs, ys, zs = w.axes()
    r, i = mri.fhd_batched_grid(dev(w.kx), dev(w.ky), dev(w.kz), dev(xs), dev(ys), dev(zs),
                                dev(w.rPhi), dev(w.iPhi), dev(w.rD), dev(w.iD), trig=trig)
    idx, ref = batched_ref(mri, w)
    check_per_coil(cplx(r, i)[:, idx], ref, TOL[trig])
    assert mri.device_errors(clear=True) == 0


def test_batched_grid_fallback_and_empty(mri):
    """nx = 6 goes through expanded coordinates and the general batched
    path (3 coils: the tensor-core coil kernel, not the grid kernel); M = 0
    gives zeros (or leaves accumulated outputs alone)."""
    w = wl.make_workload("fhd_64")
    M, B = 2500, 3
    xs = np.array([-30.0, -7.5, 0.0, 2.0, 19.0, 31.0], np.float32)
    ys = np.array([-3.0, 4.0, 11.0], np.float32)
    zs = np.array([0.0, 7.0], np.float32)
    rD, iD = coil_data(w, B, M, 5)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    r, i = mri.fhd_batched_grid(*k, dev(xs), dev(ys), dev(zs), dev(w.rPhi[:M]), dev(w.iPhi[:M]),
                                dev(rD), dev(iD), trig="accurate")
    x, y, z = expand(xs, ys, zs)
    ref = oracle.fhd_batched(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, w.rPhi[:M], w.iPhi[:M],
                             rD, iD)
    check_per_coil(cplx(r, i), ref, TOL["accurate"])
    p = mri.plan_grid_batched(B, M, 6, 3, 2)
    assert p["threads_per_cta"] == 320 and p["voxels_per_cta"] == 128 and p["grid_fold"] == 0
    e = torch.empty(0, device="cuda")
    eD = torch.empty((B, 0), device="cuda")
    rz, iz = mri.fhd_batched_grid(e, e, e, dev(xs), dev(ys), dev(zs), e, e, eD, eD)
    assert rz.shape == (B, 6 * 6) and torch.count_nonzero(rz) == 0
    assert torch.count_nonzero(iz) == 0
