"""The separable-grid path (mri_fhd_grid / mri_q_grid) against the oracle.

The oracle gets the expanded voxel coordinates of the same grid; tolerances
as for the general path (1e-5 accurate, 2e-4 fast).  Covers the tensor-core
kernel (nx >= 8: whole and padded column blocks), the fallback through
expanded coordinates (nx < 8), ragged row counts, ragged sample counts,
non-uniform axes and accumulate.
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


def plan_grid_blocks(mri, kind, w, seed, per):
    """Voxels from every (row block, column block) the grid launch assigns to
    a CTA, `per` of them spread over each block's rows."""
    n = round(w.N ** (1 / 3))
    p = mri.plan_grid(kind, w.M, n, n, n)
    if not p["tensor_cores"]:
        return None
    # one weight: 128 MMA rows, each a group of grid_fold grid rows (64^3: 2)
    rows_per_cta = 128 * p["grid_fold"]
    assert p["voxel_ctas"] == -(-n * n // rows_per_cta) * -(-n // 128)
    return grid_blocks(n, n, n, rows_per_cta, seed, per=per)


_refs = {}


def grid_ref(mri, name, kind, per, seed):
    """Oracle values on the stratified subset, computed once per workload."""
    if name not in _refs:
        w = wl.make_workload(name)
        idx = plan_grid_blocks(mri, kind, w, seed, per)
        if kind == "q":
            origin = (64 * 128 + 64) * 128 + 64
            idx = np.unique(np.concatenate([idx, [origin]]))
            ref = oracle.q(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, idx=idx)
        else:
            ref = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD,
                             idx=idx)
        _refs[name] = (w, idx, ref)
    return _refs[name]


@pytest.mark.parametrize("trig", ["accurate", "fast", "fast_rr"])
@pytest.mark.parametrize("name,per", [("fhd_tiny", None), ("fhd_64", 64),
                                      ("fhd_128_radial", 8)])
def test_fhd_grid_workloads(mri, name, per, trig):
    if per is None:
        w = wl.make_workload(name)
        idx = None
        ref = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD)
    else:
        w, idx, ref = grid_ref(mri, name, "fhd", per, 201)
    xs, ys, zs = w.axes()
    r, i = mri.fhd_grid(dev(w.kx), dev(w.ky), dev(w.kz), dev(xs), dev(ys), dev(zs),
                        dev(w.rPhi), dev(w.iPhi), dev(w.rD), dev(w.iD), trig=trig)
    got = cplx(r, i) if idx is None else cplx(r, i)[idx]
    assert oracle.rel_l2(got, ref) <= TOL[trig]
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("trig", ["accurate", "fast"])
def test_q_grid_128(mri, trig):
    w, idx, ref = grid_ref(mri, "q_128", "q", 8, 202)
    xs, ys, zs = w.axes()
    r, i = mri.q_grid(dev(w.kx), dev(w.ky), dev(w.kz), dev(xs), dev(ys), dev(zs),
                      dev(w.rPhi), dev(w.iPhi), trig=trig)
    assert oracle.rel_l2(cplx(r, i)[idx], ref) <= TOL[trig]


@pytest.mark.parametrize("nx,ny,nz", [(16, 3, 5), (32, 7, 1), (256, 5, 3), (128, 17, 2),
                                      (64, 1, 1), (100, 4, 3), (8, 9, 9), (1, 40, 3),
                                      (7, 5, 4), (300, 2, 2)])
@pytest.mark.parametrize("M", [1, 33, 1000])
def test_grid_shapes(mri, nx, ny, nz, M):
    rng = np.random.default_rng(nx * 1000 + ny * 10 + nz + M)
    xs = np.sort(rng.uniform(-40, 40, nx)).astype(np.float32)       # non-uniform
    ys = (np.arange(ny) - ny // 2).astype(np.float32)
    zs = (np.arange(nz) * 1.5 - 2.0).astype(np.float32)
    a = wl.random_fhd_inputs(M, 1, seed=M + nx)
    x, y, z = expand(xs, ys, zs)
    for trig in ("accurate", "fast"):
        r, i = mri.fhd_grid(dev(a["kx"]), dev(a["ky"]), dev(a["kz"]), dev(xs), dev(ys), dev(zs),
                            dev(a["rPhi"]), dev(a["iPhi"]), dev(a["rD"]), dev(a["iD"]), trig=trig)
        ref = oracle.fhd(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"], a["rD"],
                         a["iD"])
        assert oracle.rel_l2(cplx(r, i), ref) <= TOL[trig], trig
    r, i = mri.q_grid(dev(a["kx"]), dev(a["ky"]), dev(a["kz"]), dev(xs), dev(ys), dev(zs),
                      dev(a["rPhi"]), dev(a["iPhi"]), trig="accurate")
    ref = oracle.q(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"])
    assert oracle.rel_l2(cplx(r, i), ref) <= TOL["accurate"]


def test_grid_matches_general_path_and_accumulates(mri):
    w = wl.make_workload("fhd_64")
    xs, ys, zs = w.axes()
    args = [dev(v) for v in (w.kx, w.ky, w.kz)]
    rest = [dev(v) for v in (w.rPhi, w.iPhi, w.rD, w.iD)]
    rg, ig = mri.fhd_grid(*args, dev(xs), dev(ys), dev(zs), *rest, trig="accurate")
    rf, i_f = mri.fhd(*args, dev(w.x), dev(w.y), dev(w.z), *rest, trig="accurate")
    assert oracle.rel_l2(cplx(rg, ig), cplx(rf, i_f)) <= 4e-6
    out = (torch.full_like(rg, 0.5), torch.full_like(ig, -0.5))
    mri.fhd_grid(*args, dev(xs), dev(ys), dev(zs), *rest, trig="accurate", accumulate=True,
                 out=out)
    assert oracle.rel_l2(cplx(out[0] - 0.5, out[1] + 0.5), cplx(rg, ig)) <= 1e-6


def test_grid_empty_and_no_errors(mri):
    e = torch.empty(0, device="cuda")
    xs = dev(np.arange(16, dtype=np.float32))
    r, i = mri.fhd_grid(e, e, e, xs, xs[:2], xs[:3], e, e, e, e)
    assert r.numel() == 96 and torch.count_nonzero(r) == 0
    assert mri.device_errors(clear=True) == 0


@pytest.mark.parametrize("trig", ["accurate", "fast"])
def test_tensor_core_width_against_general_path(mri, trig):
    """nx = 128 runs on the tensor cores: ragged rows (3 x 7 = 21 of 128 in
    a CTA), a sample count that splits unevenly, accumulate."""
    w = wl.make_workload("fhd_128_radial")
    M = 70001
    xs = (np.arange(128) - 64).astype(np.float32)
    ys = np.array([-40, 3, 57], np.float32)
    zs = (np.arange(7) * 9 - 30).astype(np.float32)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    wts = [dev(a[:M]) for a in (w.rPhi, w.iPhi, w.rD, w.iD)]
    rg, ig = mri.fhd_grid(*k, dev(xs), dev(ys), dev(zs), *wts, trig=trig)
    x, y, z = expand(xs, ys, zs)
    ref = oracle.fhd(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, w.rPhi[:M], w.iPhi[:M],
                     w.rD[:M], w.iD[:M])
    assert oracle.rel_l2(cplx(rg, ig), ref) <= TOL[trig]
    out = (torch.full_like(rg, 2.0), torch.full_like(ig, -1.0))
    mri.fhd_grid(*k, dev(xs), dev(ys), dev(zs), *wts, trig=trig, accumulate=True, out=out)
    assert oracle.rel_l2(cplx(out[0] - 2.0, out[1] + 1.0), ref) <= TOL[trig]
    qr, qi = mri.q_grid(*k, dev(xs), dev(ys), dev(zs), wts[0], wts[1], trig=trig)
    qref = oracle.q(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, w.rPhi[:M], w.iPhi[:M])
    assert oracle.rel_l2(cplx(qr, qi), qref) <= TOL[trig]
    assert mri.plan_grid("fhd", M, 128, 3, 7)["samples_per_tile"] == 32


@pytest.mark.parametrize("ny", [2, 128])
@pytest.mark.parametrize("k", [-100, 60])
def test_tensor_core_weight_scale_is_exact(mri, k, ny):
    """The tensor-core kernel scales its f16 operands by a power of two taken
    from the largest weight, so multiplying D by 2^k must multiply F^H D by
    exactly 2^k (the same bits up to the exponent), far outside f16's range;
    all-zero weights give exact zeros."""
    w = wl.make_workload("fhd_128_radial")
    M = 4099
    xs = (np.arange(128) - 64).astype(np.float32)
    ys = np.array([-7, 12], np.float32) if ny == 2 else (np.arange(128) - 64).astype(np.float32)
    zs = np.array([5], np.float32)
    k3 = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    axes = [dev(xs), dev(ys), dev(zs)]
    phi = [dev(w.rPhi[:M]), dev(w.iPhi[:M])]
    d = [dev(w.rD[:M]), dev(w.iD[:M])]
    for trig in ("accurate", "fast"):
        r0, i0 = mri.fhd_grid(*k3, *axes, *phi, *d, trig=trig)
        s = float(2.0 ** k)
        r1, i1 = mri.fhd_grid(*k3, *axes, *phi, d[0] * s, d[1] * s, trig=trig)
        assert torch.equal(r1, r0 * s) and torch.equal(i1, i0 * s), trig
        z = torch.zeros_like(d[0])
        rz, iz = mri.fhd_grid(*k3, *axes, *phi, z, z, trig=trig)
        assert torch.count_nonzero(rz) == 0 and torch.count_nonzero(iz) == 0


@pytest.mark.parametrize("trig", ["accurate", "fast"])
def test_tensor_core_two_row_blocks_per_plane(mri, trig):
    """ny = 256 (two blocks of 128 rows per plane) and three planes: the row
    coordinates of each CTA's block, across plane boundaries."""
    w = wl.make_workload("fhd_128_radial")
    M = 3001
    xs = (np.arange(128) - 64).astype(np.float32)
    ys = (np.arange(256) - 128).astype(np.float32) * 0.5
    zs = np.array([-21.0, 0.0, 13.0], np.float32)
    k = [dev(a[:M]) for a in (w.kx, w.ky, w.kz)]
    wts = [dev(a[:M]) for a in (w.rPhi, w.iPhi, w.rD, w.iD)]
    r, i = mri.fhd_grid(*k, dev(xs), dev(ys), dev(zs), *wts, trig=trig)
    x, y, z = expand(xs, ys, zs)
    idx = wl.voxel_subset(x.size, 4096, 17)
    ref = oracle.fhd(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, w.rPhi[:M], w.iPhi[:M],
                     w.rD[:M], w.iD[:M], idx=idx)
    assert oracle.rel_l2(cplx(r, i)[idx], ref) <= TOL[trig]
    qr, qi = mri.q_grid(*k, dev(xs), dev(ys), dev(zs), wts[0], wts[1], trig=trig)
    qref = oracle.q(w.kx[:M], w.ky[:M], w.kz[:M], x, y, z, w.rPhi[:M], w.iPhi[:M], idx=idx)
    assert oracle.rel_l2(cplx(qr, qi)[idx], qref) <= TOL[trig]
    assert mri.device_errors(clear=True) == 0
