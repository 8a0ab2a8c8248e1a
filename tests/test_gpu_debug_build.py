"""The MRI_DEBUG build: every TMA copy's tile index is checked against the
size of its table before it is issued (DEVERR_BOUNDS otherwise; the copy is
skipped, nothing traps).  Builds that variant in-tree and runs every kernel
family through it -- general gather (single, coil groups per pair and on the
tensor cores), tensor-core grid F^H D / Q (one coil, coil groups, several
column blocks), forward
model -- against the oracle, expecting no device error bit.  Runs in a child
process, since a process loads one library."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
import numpy as np
import torch
import oracle
import non_cartesian_mri_gb300 as mri
from non_cartesian_mri_gb300 import workloads as wl

TOL = {"accurate": 1e-5, "fast": 2e-4}
dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
cp = lambda r, i: r.cpu().numpy().astype(np.float64) + 1j * i.cpu().numpy()


def expand(xs, ys, zs):
    z, y, x = np.meshgrid(zs, ys, xs, indexing="ij")
    return x.reshape(-1), y.reshape(-1), z.reshape(-1)


rng = np.random.default_rng(5)
M = 1500
a = wl.random_fhd_inputs(M, 1, seed=9, B=3)
k = [dev(a[n]) for n in ("kx", "ky", "kz")]
for nx, ny, nz in ((16, 5, 3), (200, 3, 2), (16, 128, 1)):
    xs = np.sort(rng.uniform(-40, 40, nx)).astype(np.float32)
    ys = (np.arange(ny) - ny // 2).astype(np.float32)
    zs = (np.arange(nz) * 1.5 - 1.0).astype(np.float32)
    x, y, z = expand(xs, ys, zs)
    ax = [dev(xs), dev(ys), dev(zs)]
    w1 = [a["rPhi"], a["iPhi"], a["rD"][0], a["iD"][0]]
    for trig in ("fast", "accurate"):
        r, i = mri.fhd_grid(*k, *ax, *[dev(v) for v in w1], trig=trig)
        ref = oracle.fhd(a["kx"], a["ky"], a["kz"], x, y, z, *w1)
        assert oracle.rel_l2(cp(r, i), ref) <= TOL[trig], ("fhd_grid", nx, ny, trig)
        r, i = mri.q_grid(*k, *ax, dev(a["rPhi"]), dev(a["iPhi"]), trig=trig)
        ref = oracle.q(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"])
        assert oracle.rel_l2(cp(r, i), ref) <= TOL[trig], ("q_grid", nx, ny, trig)
        r, i = mri.fhd_batched_grid(*k, *ax, dev(a["rPhi"]), dev(a["iPhi"]), dev(a["rD"]),
                                    dev(a["iD"]), trig=trig)
        ref = oracle.fhd_batched(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"],
                                 a["rD"], a["iD"])
        g = cp(r, i)
        for b in range(3):
            assert oracle.rel_l2(g[b], ref[b]) <= TOL[trig], ("batched_grid", nx, b, trig)
        rho = (rng.standard_normal(x.size) + 1j * rng.standard_normal(x.size)).astype(np.complex64)
        r, i = mri.forward_grid(*k, *ax, dev(rho.real), dev(rho.imag), trig=trig)
        ref = oracle.forward(a["kx"], a["ky"], a["kz"], x, y, z, rho)
        assert oracle.rel_l2(cp(r, i), ref) <= TOL[trig], ("forward_grid", nx, ny, trig)
        if nx == 16 and ny == 5:
            X = [dev(v) for v in (x, y, z)]
            r, i = mri.fhd(*k, *X, *[dev(v) for v in w1], trig=trig)
            ref = oracle.fhd(a["kx"], a["ky"], a["kz"], x, y, z, *w1)
            assert oracle.rel_l2(cp(r, i), ref) <= TOL[trig], ("fhd", trig)
            r, i = mri.fhd_batched(*k, *X, dev(a["rPhi"]), dev(a["iPhi"]), dev(a["rD"]),
                                   dev(a["iD"]), trig=trig)
            ref = oracle.fhd_batched(a["kx"], a["ky"], a["kz"], x, y, z, a["rPhi"], a["iPhi"],
                                     a["rD"], a["iD"])
            g = cp(r, i)
            for b in range(3):
                assert oracle.rel_l2(g[b], ref[b]) <= TOL[trig], ("batched", b, trig)
            # two coils: the per-pair coil kernel (three run on the tensor cores)
            r, i = mri.fhd_batched(*k, *X, dev(a["rPhi"]), dev(a["iPhi"]), dev(a["rD"][:2]),
                                   dev(a["iD"][:2]), trig=trig)
            g = cp(r, i)
            for b in range(2):
                assert oracle.rel_l2(g[b], ref[b]) <= TOL[trig], ("batched2", b, trig)
        bits = mri.device_errors(clear=True)
        assert bits == 0, ("device error bits", bits, nx, ny, trig)
print("debug build: all kernels clean")
'''


def test_debug_build_checks_every_copy():
    from non_cartesian_mri_gb300 import build
    lib = build.build(defines=["MRI_DEBUG=1"],
                      out=os.path.join(build.BUILD, "debug", "libmri.so"))
    env = dict(os.environ, MRI_LIB=lib, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "all kernels clean" in r.stdout
