"""Batched F^H D at arbitrary voxel coordinates on the tensor cores
(coils_tc_kernel) against the fp64 oracle.

Coil groups of 3 to 8 coils run there (a padded group of 8: absent coils
carry weight 0), one or two coils left over on the per-pair kernels.  Every
coil is held to the relative bound of its trig path (1e-5 accurate, 2e-4
fast), so a coil with small weights beside large ones is checked as strictly
as the rest.  Shapes are ragged in both axes: voxel counts that leave a
partial block of 128 (the MMA's rows) and sample counts that leave a partial
tile of 32.
"""

import numpy as np
import pytest
import torch

import oracle
from non_cartesian_mri_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"accurate": 1e-5, "fast": 2e-4, "fast_rr": 2e-4}
TRIGS = ["accurate", "fast", "fast_rr"]
KEYS = ("kx", "ky", "kz", "x", "y", "z", "rPhi", "iPhi", "rD", "iD")


@pytest.fixture(scope="module")
def mri():
    from non_cartesian_mri_gb300 import build
    build.build()
    import non_cartesian_mri_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def cplx(r, i):
    return r.cpu().numpy().astype(np.float64) + 1j * i.cpu().numpy().astype(np.float64)


def check_per_coil(got, ref, tol):
    assert got.shape == ref.shape
    for b in range(ref.shape[0]):
        assert oracle.rel_l2(got[b], ref[b]) <= tol, f"coil {b}"


def no_device_errors(mri):
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("trig", TRIGS)
@pytest.mark.parametrize("B", [3, 5, 8, 9, 10, 13])
def test_coil_groups(mri, B, trig):
    """3, 5: one padded group; 8: one full group; 9, 10: a group of 8 and the
    per-pair kernel for the rest; 13: groups of 8 and 5."""
    M, N = 1001, 1100
    a = wl.random_fhd_inputs(M, N, seed=40 + B, B=B)
    r, i = mri.fhd_batched(*[dev(a[k]) for k in KEYS], trig=trig)
    assert tuple(r.shape) == (B, N)
    check_per_coil(cplx(r, i), oracle.fhd_batched(**a), TOL[trig])
    p = mri.plan("fhd_batched", M, N, B=B)
    assert p["tensor_cores"] == 1 and p["voxels_per_cta"] == 128
    assert p["coil_groups"] == {3: 1, 5: 1, 8: 1, 9: 2, 10: 2, 13: 2}[B]
    no_device_errors(mri)


@pytest.mark.parametrize("M,N", [(1, 1), (31, 127), (32, 128), (33, 129), (64, 1)])
def test_tiny_shapes(mri, M, N):
    """One sample or voxel, a tile of 32 samples and a block of 128 voxels
    exactly, one past each.  With a handful of voxels a cancelling sum makes
    the relative error of the vector meaningless, so every output is held to
    the error bound of a sum instead: |error| <= tol * sum_m |Mu_b[m]| (the
    per-term error, mostly the fp32 rounding of the phase, times the terms'
    magnitudes)."""
    a = wl.random_fhd_inputs(M, N, seed=M * 131 + N, B=4)
    mu = np.abs((a["rPhi"] - 1j * a["iPhi"])[None, :] * (a["rD"] + 1j * a["iD"]))
    for trig in ("accurate", "fast"):
        r, i = mri.fhd_batched(*[dev(a[k]) for k in KEYS], trig=trig)
        err = np.abs(cplx(r, i) - oracle.fhd_batched(**a))
        assert np.all(err <= TOL[trig] * mu.sum(axis=1)[:, None]), trig
    no_device_errors(mri)


@pytest.mark.parametrize("B", [8, 13, 17])
def test_sample_splits_and_accumulate(mri, B):
    """Few voxels and many samples: the samples split across CTAs and the
    partial sums are reduced; accumulate adds onto the outputs.  13 and 17
    coils: a second group of 5 (its partials laid out for 5 coils in the
    buffer sized for 8), and a trailing single coil on the per-pair kernel."""
    M, N = 40000, 300
    p = mri.plan("fhd_batched", M, N, B=B)
    assert p["tensor_cores"] == 1 and p["splits"] > 1
    a = wl.random_fhd_inputs(M, N, seed=5 + B, B=B)
    args = [dev(a[k]) for k in KEYS]
    ref = oracle.fhd_batched(**a)
    r, i = mri.fhd_batched(*args, trig="accurate")
    check_per_coil(cplx(r, i), ref, TOL["accurate"])
    out = (torch.full((B, N), 1.5, device="cuda"), torch.full((B, N), -2.0, device="cuda"))
    mri.fhd_batched(*args, trig="accurate", accumulate=True, out=out)
    check_per_coil(cplx(out[0] - 1.5, out[1] + 2.0), ref, TOL["accurate"])
    no_device_errors(mri)


@pytest.mark.parametrize("k", [-100, 60])
def test_weight_scale_is_exact(mri, k):
    """The f16 weight operands are scaled by a power of two from the group's
    largest weight, so D * 2^k gives F^H D * 2^k bit for bit, far outside
    f16's range; all-zero weights give exact zeros."""
    M, N, B = 3000, 700, 6
    a = wl.random_fhd_inputs(M, N, seed=9, B=B)
    args = [dev(a[k]) for k in KEYS]
    s = float(2.0 ** k)
    for trig in ("accurate", "fast"):
        r0, i0 = mri.fhd_batched(*args, trig=trig)
        r1, i1 = mri.fhd_batched(*args[:8], args[8] * s, args[9] * s, trig=trig)
        assert torch.equal(r1, r0 * s) and torch.equal(i1, i0 * s), trig
        z = torch.zeros_like(args[8])
        rz, iz = mri.fhd_batched(*args[:8], z, z, trig=trig)
        assert torch.count_nonzero(rz) == 0 and torch.count_nonzero(iz) == 0
    no_device_errors(mri)


def test_coils_of_very_different_scale(mri):
    """Each coil has its own power-of-two operand scale: coils 1e-6 and 1e4
    times the others (a range no single f16 scale covers with full precision)
    still meet the relative bound each."""
    M, N, B = 4000, 500, 4
    a = wl.random_fhd_inputs(M, N, seed=12, B=B)
    g = np.array([1.0, 1e-6, 1e4, 1.0], np.float32)[:, None]
    a["rD"] = (a["rD"] * g).astype(np.float32)
    a["iD"] = (a["iD"] * g).astype(np.float32)
    r, i = mri.fhd_batched(*[dev(a[k]) for k in KEYS], trig="accurate")
    check_per_coil(cplx(r, i), oracle.fhd_batched(**a), TOL["accurate"])


def test_matches_single_coil_calls(mri):
    """Each coil of a group equals the single-weight call on that coil's D
    within the accurate path's error (the two paths round differently)."""
    M, N, B = 2500, 900, 5
    a = wl.random_fhd_inputs(M, N, seed=77, B=B)
    args = [dev(a[k]) for k in KEYS]
    r, i = mri.fhd_batched(*args, trig="accurate")
    for b in range(B):
        rb, ib = mri.fhd(*args[:8], args[8][b].contiguous(), args[9][b].contiguous(),
                         trig="accurate")
        assert oracle.rel_l2(cplx(r[b], i[b]), cplx(rb, ib)) <= 2e-6
