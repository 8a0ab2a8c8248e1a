"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes must give up, report through the device error word and leave the
context usable (the next F^H D call still matches the oracle)."""

import time

import numpy as np
import pytest
import torch

import oracle
from non_cartesian_mri_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mri():
    from non_cartesian_mri_gb300 import build
    build.build()
    import non_cartesian_mri_gb300 as m
    return m


def test_wait_that_completes_sets_no_error(mri):
    mri.device_errors(clear=True)
    mri.wait_selftest(True)
    assert mri.device_errors(clear=True) == 0


def test_wait_that_never_completes_times_out_and_reports(mri):
    mri.device_errors(clear=True)
    t0 = time.perf_counter()
    mri.wait_selftest(False)
    bits = mri.device_errors(clear=True)          # synchronises
    elapsed = time.perf_counter() - t0
    assert bits & 0x1, "tile-wait timeout bit"
    assert 0.9 < elapsed < 30.0
    assert mri.device_errors(clear=True) == 0     # cleared
    # the context still works
    w = wl.make_workload("fhd_tiny")
    args = [torch.from_numpy(a).cuda() for a in
            (w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD)]
    r, i = mri.fhd(*args, trig="accurate")
    got = r.cpu().numpy().astype(np.float64) + 1j * i.cpu().numpy()
    ref = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD)
    assert oracle.rel_l2(got, ref) <= 1e-5
    assert mri.device_errors(clear=True) == 0
