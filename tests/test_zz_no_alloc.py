"""mri_fhd_noalloc: F^H D for callers that may not allocate GPU memory.

Callers with a fixed, fully reserved device-memory budget, real-time loops
that must not wait on an allocator, or frameworks that own every allocation
cannot let a library allocate scratch.  mri_fhd_noalloc runs the same kernels
as mri_fhd with its scratch in a fixed array inside the library.  These tests
call it through the C ABI and check it against mri_fhd, twice in a row on
different problems (the array keeps the previous call's contents), with the
tolerances the parity tests use.
"""

import ctypes

import numpy as np
import pytest
import torch

from non_cartesian_mri_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"accurate": 1e-5, "fast": 2e-4}
TRIG = {"accurate": 0, "fast": 1}
P = ctypes.c_void_p
I64 = ctypes.c_int64
MRI_ERR_SIZE = 2


@pytest.fixture(scope="module")
def api():
    from non_cartesian_mri_gb300 import build
    build.build()
    import non_cartesian_mri_gb300 as mri
    lib = mri.load()
    f = lib.mri_fhd_noalloc
    f.argtypes = [P] * 10 + [I64, I64, P, P, ctypes.c_int, ctypes.c_int, P]
    f.restype = ctypes.c_int
    return mri, f


def ptr(t):
    return P(t.data_ptr())


def inputs(name):
    w = wl.make_workload(name)
    return w, [torch.from_numpy(np.ascontiguousarray(a)).cuda()
               for a in (w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD)]


def noalloc(f, t, M, N, out, trig, accumulate=0):
    stream = P(torch.cuda.current_stream().cuda_stream)
    return f(*[ptr(a) for a in t], M, N, ptr(out[0]), ptr(out[1]), TRIG[trig], accumulate,
             stream)


def rel(a, b):
    a = torch.complex(a[0].double(), a[1].double())
    b = torch.complex(b[0].double(), b[1].double())
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b))


def test_matches_mri_fhd_on_calls_in_a_row(api):
    mri, f = api
    # 128^3 (runs unsplit in the fixed array), then 64^3 (split), then 128^3 again
    for name, trig in (("fhd_128_radial", "accurate"), ("fhd_64", "fast"),
                       ("fhd_128_radial", "fast")):
        w, t = inputs(name)
        ref = mri.fhd(*t, trig=trig)
        out = (torch.full((w.N,), float("nan"), device="cuda"),
               torch.full((w.N,), float("nan"), device="cuda"))
        assert noalloc(f, t, w.M, w.N, out, trig) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out[0]).all() and torch.isfinite(out[1]).all()
        assert rel(out, ref) <= TOL[trig], name
    assert mri.device_errors(clear=True) == 0


def test_accumulate_and_ragged(api):
    mri, f = api
    a = wl.random_fhd_inputs(1001, 3333, seed=5)
    t = [torch.from_numpy(a[k]).cuda() for k in ("kx", "ky", "kz", "x", "y", "z", "rPhi",
                                                  "iPhi", "rD", "iD")]
    ref = mri.fhd(*t, trig="accurate")
    out = (torch.full((3333,), 2.0, device="cuda"), torch.full((3333,), -1.0, device="cuda"))
    assert noalloc(f, t, 1001, 3333, out, "accurate", accumulate=1) == 0
    torch.cuda.synchronize()
    assert rel((out[0] - 2.0, out[1] + 1.0), ref) <= TOL["accurate"]


def test_rejects_M_beyond_the_fixed_array(api):
    _, f = api
    limit = (32 * 1024 * 1024) // 5120 * 256           # samples whose records fit
    fake = [P(0x100000 + 256 * i) for i in range(12)]  # never dereferenced
    stream = P(torch.cuda.current_stream().cuda_stream)
    assert f(*fake[:10], limit + 1, 100, fake[10], fake[11], 0, 0, stream) == MRI_ERR_SIZE
