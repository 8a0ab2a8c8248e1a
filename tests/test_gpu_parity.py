"""CUDA path vs the fp64 oracle, element by element, on seeded inputs.

Tolerances: relative L2 error over real and imaginary parts of <= 1e-5 on the
accurate trig path and <= 2e-4 on the fast (SFU) paths, on every workload.
Full-size workloads run on the GPU in the launch configuration the benchmark
times; the oracle computes a seeded voxel subset (voxels are independent).
"""

import numpy as np
import pytest
import torch

import oracle
from non_cartesian_mri_gb300 import workloads as wl
from tests.sampling import gather_blocks

pytestmark = pytest.mark.gpu

TOL = {"accurate": 1e-5, "fast": 2e-4, "fast_rr": 2e-4}
TRIGS = ["accurate", "fast", "fast_rr"]


@pytest.fixture(scope="module")
def mri():
    from non_cartesian_mri_gb300 import build
    build.build()
    import non_cartesian_mri_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy().astype(np.float64)


def cplx(r, i):
    return host(r) + 1j * host(i)


def fhd_inputs(w):
    return [dev(a) for a in (w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD)]


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("trig", TRIGS)
def test_fhd_tiny_all_voxels(mri, trig):
    w = wl.make_workload("fhd_tiny")
    r, i = mri.fhd(*fhd_inputs(w), trig=trig)
    ref = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]


def plan_blocks(mri, kind, w, seed, per=1, B=1):
    """Voxels from every CTA block of the launch the call makes."""
    p = mri.plan(kind, w.M, w.N, B=B)
    vpc = p["voxels_per_cta"]
    assert p["voxel_ctas"] == -(-w.N // vpc)
    return gather_blocks(w.N, vpc, seed, per=per)


@pytest.mark.parametrize("trig", TRIGS)
def test_fhd_64_subset(mri, trig):
    w = wl.make_workload("fhd_64")
    r, i = mri.fhd(*fhd_inputs(w), trig=trig)
    idx = plan_blocks(mri, "fhd", w, 101, per=16)
    ref = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=idx)
    assert oracle.rel_l2(cplx(r, i)[idx], ref) <= TOL[trig]


@pytest.fixture(scope="module")
def radial():
    return wl.make_workload("fhd_128_radial")


@pytest.fixture(scope="module")
def radial_ref(mri, radial):
    w = radial
    idx = plan_blocks(mri, "fhd", w, 102)
    corners = np.array([0, w.N - 1, 127, w.N - 128], np.int64)   # largest |x|
    idx = np.unique(np.concatenate([idx, corners]))
    return idx, oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD, idx=idx)


@pytest.mark.parametrize("trig", TRIGS)
def test_fhd_128_radial_subset(mri, radial, radial_ref, trig):
    r, i = mri.fhd(*fhd_inputs(radial), trig=trig)
    idx, ref = radial_ref
    assert oracle.rel_l2(cplx(r, i)[idx], ref) <= TOL[trig]


@pytest.fixture(scope="module")
def q128():
    return wl.make_workload("q_128")


@pytest.fixture(scope="module")
def q128_ref(mri, q128):
    """One voxel from every CTA block of the full-size launch (1,024 blocks)."""
    w = q128
    idx = plan_blocks(mri, "q", w, 103)
    return idx, oracle.q(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, idx=idx)


@pytest.mark.parametrize("trig", TRIGS)
def test_q_128_subset(mri, q128, q128_ref, trig):
    w = q128
    args = [dev(a) for a in (w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi)]
    r, i = mri.q(*args, trig=trig)
    idx, ref = q128_ref
    assert oracle.rel_l2(cplx(r, i)[idx], ref) <= TOL[trig]


@pytest.fixture(scope="module")
def batched128():
    return wl.make_workload("fhd_batched_128")


@pytest.fixture(scope="module")
def batched128_ref(mri, batched128):
    """One voxel from every CTA block of the coil-group launch (2,048 blocks),
    all eight coils."""
    w = batched128
    idx = plan_blocks(mri, "fhd_batched", w, 104, B=8)
    return idx, oracle.fhd_batched(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD,
                                   w.iD, idx=idx)


@pytest.mark.parametrize("trig", ["accurate", "fast"])
def test_batched_128_subset(mri, batched128, batched128_ref, trig):
    w = batched128
    r, i = mri.fhd_batched(*fhd_inputs(w), trig=trig)
    assert tuple(r.shape) == (8, w.N)
    idx, ref = batched128_ref
    got = cplx(r, i)[:, idx]
    assert oracle.rel_l2(got, ref) <= TOL[trig]
    for b in range(8):                       # every coil, not just the total
        assert oracle.rel_l2(got[b], ref[b]) <= TOL[trig]


# ---------------------------------------------------------------------------
# ragged sizes, tails, degenerate cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N", [(1, 1), (1, 777), (3, 5), (255, 2049), (257, 4097),
                                 (1000, 2048 * 3 + 1), (4099, 300), (20000, 1500)])
@pytest.mark.parametrize("trig", ["accurate", "fast"])
def test_ragged_sizes(mri, M, N, trig):
    a = wl.random_fhd_inputs(M, N, seed=M * 7 + N)
    r, i = mri.fhd(*[dev(a[k]) for k in ("kx", "ky", "kz", "x", "y", "z", "rPhi", "iPhi",
                                          "rD", "iD")], trig=trig)
    ref = oracle.fhd(**a)
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig]


@pytest.mark.parametrize("B", [1, 2, 3, 5, 13])
def test_batched_coil_groups(mri, B):
    """Coil counts that need groups of 8, 4, 2 and 1."""
    a = wl.random_fhd_inputs(700, 1100, seed=B, B=B)
    r, i = mri.fhd_batched(*[dev(a[k]) for k in ("kx", "ky", "kz", "x", "y", "z", "rPhi",
                                                  "iPhi", "rD", "iD")], trig="accurate")
    ref = oracle.fhd_batched(**a)
    got = cplx(r, i)
    for b in range(B):
        assert oracle.rel_l2(got[b], ref[b]) <= TOL["accurate"]


def test_empty_samples_zero_or_keep(mri):
    x, y, z = (dev(v) for v in wl.voxel_grid(4))
    e = torch.empty(0, dtype=torch.float32, device="cuda")
    r, i = mri.fhd(e, e, e, x, y, z, e, e, e, e)
    assert torch.count_nonzero(r) == 0 and torch.count_nonzero(i) == 0
    old_r = torch.full_like(x, 3.0)
    old_i = torch.full_like(x, -2.0)
    mri.fhd(e, e, e, x, y, z, e, e, e, e, accumulate=True, out=(old_r, old_i))
    assert torch.all(old_r == 3.0) and torch.all(old_i == -2.0)


def test_empty_voxels_is_noop(mri):
    a = wl.random_fhd_inputs(10, 0, seed=1)
    r, i = mri.fhd(*[dev(a[k]) for k in ("kx", "ky", "kz", "x", "y", "z", "rPhi", "iPhi",
                                          "rD", "iD")])
    assert r.numel() == 0 and i.numel() == 0


@pytest.mark.parametrize("trig", TRIGS)
def test_single_sample_at_k0_is_mu_everywhere(mri, trig):
    """k = 0: the phase is exactly 0, so every voxel gets Mu[0] with no trig error."""
    rng = np.random.default_rng(3)
    x, y, z = wl.voxel_grid(16)
    zero = np.zeros(1, np.float32)
    rPhi, iPhi, rD, iD = (rng.standard_normal(1).astype(np.float32) for _ in range(4))
    r, i = mri.fhd(dev(zero), dev(zero), dev(zero), dev(x), dev(y), dev(z), dev(rPhi),
                   dev(iPhi), dev(rD), dev(iD), trig=trig)
    rmu, imu = mri.mu(dev(rPhi), dev(iPhi), dev(rD), dev(iD))
    assert torch.all(r == rmu[0]) and torch.all(i == imu[0])
    ref = oracle.mu(rPhi, iPhi, rD, iD)[0]
    assert abs(complex(float(rmu[0]), float(imu[0])) - ref) <= 4e-7 * abs(ref)


def test_mu_matches_oracle(mri):
    rng = np.random.default_rng(12)
    M = 100003
    a = [rng.standard_normal(M).astype(np.float32) for _ in range(4)]
    rmu, imu = mri.mu(*[dev(v) for v in a])
    ref = oracle.mu(*a)
    assert oracle.rel_l2(cplx(rmu, imu), ref) <= 1e-7


# ---------------------------------------------------------------------------
# properties at scale
# ---------------------------------------------------------------------------

def test_accumulate_adds_to_existing(mri):
    a = wl.random_fhd_inputs(3000, 5000, seed=77)
    args = [dev(a[k]) for k in ("kx", "ky", "kz", "x", "y", "z", "rPhi", "iPhi", "rD", "iD")]
    r0, i0 = mri.fhd(*args, trig="accurate")
    out = (torch.full_like(r0, 1.5), torch.full_like(i0, -0.25))
    mri.fhd(*args, trig="accurate", accumulate=True, out=out)
    torch.testing.assert_close(out[0], r0 + 1.5, rtol=1e-6, atol=1e-4)
    torch.testing.assert_close(out[1], i0 - 0.25, rtol=1e-6, atol=1e-4)


def test_chunked_accumulation_equals_one_call(mri, radial):
    """The pages' chunk-by-chunk host loop (Fig. 17.12) as accumulate calls."""
    w = radial
    args = fhd_inputs(w)
    r1, i1 = mri.fhd(*args, trig="accurate")
    M = w.M
    cuts = [0, 1000, 77777, 150001, M]
    out = (torch.zeros_like(r1), torch.zeros_like(i1))
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = [t[a:b] for t in args[:3]] + args[3:6] + [t[a:b] for t in args[6:]]
        mri.fhd(*part, trig="accurate", accumulate=True, out=out)
    num = torch.linalg.vector_norm(torch.complex(out[0] - r1, out[1] - i1))
    den = torch.linalg.vector_norm(torch.complex(r1, i1))
    assert float(num / den) <= 2e-6


def test_linear_in_D(mri):
    w = wl.make_workload("fhd_64")
    base = fhd_inputs(w)
    rng = np.random.default_rng(5)
    d2 = [dev(rng.standard_normal(w.M).astype(np.float32)) for _ in range(2)]
    r1, i1 = mri.fhd(*base, trig="accurate")
    r2, i2 = mri.fhd(*base[:8], *d2, trig="accurate")
    r3, i3 = mri.fhd(*base[:8], base[8] + 2 * d2[0], base[9] + 2 * d2[1], trig="accurate")
    a = torch.complex(r3, i3)
    b = torch.complex(r1 + 2 * r2, i1 + 2 * i2)
    assert float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b)) <= 3e-6


def test_q_at_origin_and_hermitian(mri):
    w = wl.make_workload("q_128")
    args = [dev(a) for a in (w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi)]
    r, i = mri.q(*args, trig="accurate")
    L = 128
    origin = (L // 2 * L + L // 2) * L + L // 2                 # voxel (0, 0, 0)
    wsum = float(np.sum(w.rPhi.astype(np.float64) ** 2 + w.iPhi.astype(np.float64) ** 2))
    assert abs(float(r[origin]) - wsum) <= 2e-6 * wsum
    assert abs(float(i[origin])) <= 2e-6 * wsum
    # Q(-x) = conj Q(x) for voxels whose mirror is on the grid
    xs, ys, zs = (np.array(v) for v in (w.x, w.y, w.z))
    sel = np.nonzero((xs > -64) & (ys > -64) & (zs > -64))[0][::997]
    mirror = (((-zs[sel] + 64) * L + (-ys[sel] + 64)) * L + (-xs[sel] + 64)).astype(np.int64)
    q = cplx(r, i)
    assert oracle.rel_l2(q[mirror], np.conj(q[sel])) <= 2e-5


def test_no_device_errors_recorded(mri):
    assert mri.device_errors(clear=True) == 0
