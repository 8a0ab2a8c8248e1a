"""The C ABI on a machine without a GPU: the library builds and loads, exports
every function the headers declare, and rejects bad arguments with the
documented status before any CUDA call.  The launch planner is host-only."""

import ctypes
import os
import re

import pytest

from non_cartesian_mri_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]

OK, NULL, SIZE, ALIGN, NOT_DEVICE, MODE, CUDA, UNSUPPORTED = range(8)


@pytest.fixture(scope="module")
def lib():
    path = lib_build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(mri_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_the_entry_points():
    names = declared_functions()
    for n in ("mri_mu", "mri_fhd", "mri_q", "mri_fhd_batched", "mri_status_string",
              "mri_plan_gather", "mri_device_errors", "mri_timing_begin", "mri_timing_end",
              "mri_microbench"):
        assert n in names


def test_every_declared_function_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_status_strings(lib):
    lib.mri_status_string.restype = ctypes.c_char_p
    seen = set()
    for s in range(8):
        txt = lib.mri_status_string(s).decode()
        assert txt and txt not in seen
        seen.add(txt)
    assert lib.mri_status_string(99).decode() == "unknown status"


P = ctypes.c_void_p
I64 = ctypes.c_int64


def _fhd(lib, ptrs, M, N, trig=1, acc=0):
    f = lib.mri_fhd
    f.argtypes = [P] * 10 + [I64, I64, P, P, ctypes.c_int, ctypes.c_int, P]
    f.restype = ctypes.c_int
    return f(*ptrs[:10], M, N, ptrs[10], ptrs[11], trig, acc, None)


def fake(n=12, addr=0x100000):
    """Distinct, aligned, never-dereferenced addresses."""
    return [P(addr + 256 * i) for i in range(n)]


def test_fhd_argument_checks_before_any_cuda_call(lib):
    good = fake()
    assert _fhd(lib, good, 10, 10, trig=7) == MODE
    assert _fhd(lib, good, 10, 10, acc=2) == MODE
    assert _fhd(lib, good, -1, 10) == SIZE
    assert _fhd(lib, good, 10, -5) == SIZE
    assert _fhd(lib, good, 1 << 40, 10) == SIZE
    assert _fhd(lib, good, 10, 0) == OK                 # N == 0 is a no-op
    for i in range(12):
        bad = list(good)
        bad[i] = P(None)
        assert _fhd(lib, bad, 10, 10) == NULL, f"NULL in slot {i}"
        bad[i] = P(0x100001 + 256 * i)
        assert _fhd(lib, bad, 10, 10) == ALIGN, f"misaligned slot {i}"


def test_sample_pointers_unused_when_M_is_zero(lib):
    ptrs = fake()
    for i in (0, 1, 2, 6, 7, 8, 9):          # kx ky kz rPhi iPhi rD iD
        ptrs[i] = P(None)
    # gets past the argument checks; stops at the device query without a GPU
    assert _fhd(lib, ptrs, 0, 10) in (OK, CUDA, UNSUPPORTED)
    ptrs[3] = P(None)                        # x is still required
    assert _fhd(lib, ptrs, 0, 10) == NULL


def test_batched_and_q_checks(lib):
    fb = lib.mri_fhd_batched
    fb.argtypes = [P] * 10 + [I64, I64, I64, P, P, ctypes.c_int, ctypes.c_int, P]
    fb.restype = ctypes.c_int
    g = fake()
    assert fb(*g[:10], 0, 10, 10, g[10], g[11], 0, 0, None) == SIZE     # B = 0
    assert fb(*g[:10], 2, 10, 10, g[10], g[11], 3, 0, None) == MODE
    q = lib.mri_q
    q.argtypes = [P] * 8 + [I64, I64, P, P, ctypes.c_int, ctypes.c_int, P]
    q.restype = ctypes.c_int
    assert q(*g[:8], 10, 10, P(None), g[9], 0, 0, None) == NULL
    mu = lib.mri_mu
    mu.argtypes = [P] * 6 + [I64, P]
    mu.restype = ctypes.c_int
    assert mu(*g[:6], -3, None) == SIZE
    assert mu(*g[:6], 0, None) == OK


class Plan(ctypes.Structure):
    _fields_ = [("threads_per_cta", ctypes.c_int), ("voxels_per_thread", ctypes.c_int),
                ("samples_per_tile", ctypes.c_int), ("splits", ctypes.c_int),
                ("voxel_ctas", ctypes.c_int64), ("tiles", ctypes.c_int64),
                ("coil_groups", ctypes.c_int), ("launches", ctypes.c_int),
                ("scratch_bytes", ctypes.c_int64), ("tensor_cores", ctypes.c_int),
                ("grid_fold", ctypes.c_int), ("fast_fp32_voxels", ctypes.c_int),
                ("voxels_per_cta", ctypes.c_int)]


def plan(lib, kind, B, M, N, sms=152):
    p = Plan()
    lib.mri_plan_gather.argtypes = [ctypes.c_int, I64, I64, I64, ctypes.c_int,
                                    ctypes.POINTER(Plan)]
    lib.mri_plan_gather.restype = ctypes.c_int
    assert lib.mri_plan_gather(kind, B, M, N, sms, ctypes.byref(p)) == OK
    return p


def test_plan_covers_every_voxel_and_sample(lib):
    for kind, B, M, N in [(0, 1, 262144, 128 ** 3), (1, 1, 1 << 20, 128 ** 3),
                          (2, 8, 524288, 128 ** 3), (0, 1, 32768, 64 ** 3),
                          (0, 1, 2048, 16 ** 3), (0, 1, 1, 1), (0, 1, 257, 2049)]:
        p = plan(lib, kind, B, M, N)
        vpc = p.voxels_per_cta
        if p.tensor_cores:
            assert vpc == 128                       # one voxel per tensor-memory lane
        else:
            assert vpc == p.threads_per_cta * p.voxels_per_thread
        assert p.voxel_ctas * vpc >= N > (p.voxel_ctas - 1) * vpc
        assert p.tiles * p.samples_per_tile >= M > (p.tiles - 1) * p.samples_per_tile
        assert 1 <= p.splits <= p.tiles
        # per group: prep and gather (tensor cores: also the weight tiles),
        # and the reduction of split partials
        per = 3 if p.tensor_cores else 2
        assert p.launches == p.coil_groups * (per + (1 if p.splits > 1 else 0))


def test_plan_invariants_over_shapes(lib):
    """Every plan over a sweep of shapes and SM counts: voxels and samples
    covered with no empty CTA column or tile, splits within the sample tiles
    (at most 1024, far inside the 65,535 a launch's y dimension allows), a
    voxel grid within 2^31 - 1 CTAs, the launch count of its groups, and
    scratch that holds the split partials."""
    for kind, Bs in ((0, (1,)), (1, (1,)), (2, (1, 2, 3, 5, 8, 9, 13, 17))):
        for B in Bs:
            for M in (1, 31, 32, 33, 1000, 32768, 262144, 1 << 20, 1 << 24):
                for N in (1, 127, 128, 129, 2049, 64 ** 3, 128 ** 3, 256 ** 3):
                    for sms in (1, 8, 152):
                        p = plan(lib, kind, B, M, N, sms)
                        vpc = p.voxels_per_cta
                        assert p.voxel_ctas * vpc >= N > (p.voxel_ctas - 1) * vpc
                        assert p.voxel_ctas <= 2 ** 31 - 1
                        spt = p.samples_per_tile
                        assert p.tiles * spt >= M > (p.tiles - 1) * spt
                        assert 1 <= p.splits <= min(p.tiles, 1024)
                        # groups of 8 (and one of 3-7) on the tensor cores, 3
                        # launches each; 1 or 2 coils left on the per-pair
                        # kernel, 2; one more per group whose samples split
                        if p.tensor_cores:
                            n_pair = int(B > 8 and B % 8 in (1, 2))
                        else:
                            n_pair = p.coil_groups
                        n_tc = p.coil_groups - n_pair
                        base = 3 * n_tc + 2 * n_pair
                        if n_pair == 0 or n_tc == 0:
                            assert p.launches == base + p.coil_groups * (p.splits > 1)
                        else:
                            assert base <= p.launches <= base + p.coil_groups
                        if p.splits > 1:
                            assert p.scratch_bytes >= p.splits * 2 * N * 4
                        assert p.scratch_bytes >= 0


def test_plan_splits_samples_when_voxels_underfill_the_gpu(lib):
    small = plan(lib, 0, 1, 32768, 64 ** 3)        # 128 voxel CTAs < 304 slots
    assert small.splits > 1
    # 1024 voxel CTAs on 304 slots is 3.37 waves: splitting must beat the tail
    big = plan(lib, 0, 1, 262144, 128 ** 3)
    waves = -(-big.voxel_ctas * big.splits // 304)
    eff = big.voxel_ctas * big.splits / (waves * 304)
    assert eff > 0.95


def test_plan_coil_groups(lib):
    # groups of 3..8 coils run on the tensor cores, 1 or 2 left over on the
    # per-pair kernels
    assert plan(lib, 2, 13, 1000, 5000).coil_groups == 2      # 8 + 5
    assert plan(lib, 2, 8, 1000, 5000).coil_groups == 1
    assert plan(lib, 2, 17, 1000, 5000).coil_groups == 3      # 8 + 8 + 1
    assert plan(lib, 2, 10, 1000, 5000).coil_groups == 2      # 8 + 2
    for B in (3, 5, 8):
        p = plan(lib, 2, B, 1000, 5000)
        assert p.tensor_cores == 1 and p.coil_groups == 1 and p.threads_per_cta == 320
    for B in (1, 2):
        p = plan(lib, 2, B, 1000, 5000)
        assert p.tensor_cores == 0 and p.coil_groups == 1
    assert plan(lib, 1, 1, 1000, 5000).tensor_cores == 0      # Q: the per-pair kernel
    p = plan(lib, 0, 1, 0, 100)
    assert p.launches == 2                                   # zero fill only


def test_batched_grid_plan_groups(lib):
    """Coil groups of the tensor-core grid path (host-only planning)."""
    f = lib.mri_plan_grid_batched
    f.argtypes = [I64, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.POINTER(Plan)]
    f.restype = ctypes.c_int
    for B, groups in [(1, 1), (2, 1), (4, 1), (5, 1), (8, 1), (9, 2), (13, 2), (16, 2), (17, 3)]:
        p = Plan()
        assert f(B, 524288, 128, 128, 128, 152, ctypes.byref(p)) == OK
        assert p.tensor_cores == 1 and p.coil_groups == groups, B
        assert p.samples_per_tile * p.tiles >= 524288
    p = Plan()
    assert f(0, 1000, 128, 4, 4, 152, ctypes.byref(p)) == SIZE
    # nx < 8: expanded coordinates and the general batched path (3 coils: the
    # tensor-core coil kernel, not the grid kernel; 1 coil: the per-pair kernel)
    assert f(3, 1000, 7, 4, 4, 152, ctypes.byref(p)) == OK and p.threads_per_cta == 320
    assert p.voxels_per_cta == 128 and p.voxel_ctas == 1
    assert f(1, 1000, 7, 4, 4, 152, ctypes.byref(p)) == OK and p.tensor_cores == 0
    # nx >= 8 runs on the tensor cores, one CTA column per block of 128
    # columns (the last one padded)
    assert f(3, 1000, 8, 4, 4, 152, ctypes.byref(p)) == OK and p.tensor_cores == 1
    c8 = p.voxel_ctas
    assert f(3, 1000, 64, 4, 4, 152, ctypes.byref(p)) == OK and p.voxel_ctas == c8
    assert f(3, 1000, 257, 4, 4, 152, ctypes.byref(p)) == OK and p.tensor_cores == 1
    assert p.voxel_ctas == 3 * c8
    assert lib.mri_plan_grid(2, 1000, 128, 4, 4, 152, ctypes.byref(p)) == MODE


def test_grid_fold_plan(lib):
    """Narrow grids (8 <= nx <= 64) fold 128 / fw grid rows into one block of
    128 columns, fw = nx rounded up to a power of two, when ny is a multiple
    of that; the plan counts the folded row blocks."""
    f = lib.mri_plan_grid
    f.argtypes = [ctypes.c_int, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.POINTER(Plan)]
    f.restype = ctypes.c_int
    for nx, ny, nz, fold in [(64, 64, 64, 2), (48, 64, 3, 2), (32, 64, 1, 4), (20, 8, 2, 4),
                             (16, 16, 4, 8), (9, 32, 1, 8), (8, 16, 2, 16), (8, 9, 9, 1),
                             (64, 1, 1, 1), (65, 64, 64, 1), (128, 128, 128, 1),
                             (32, 6, 5, 1), (7, 64, 64, 0)]:
        p = Plan()
        assert f(0, 32768, nx, ny, nz, 152, ctypes.byref(p)) == OK
        assert p.grid_fold == fold, (nx, ny, nz)
        if fold:
            assert p.voxel_ctas == -(-(ny // fold) * nz // 128) * -(-nx // 128)
            assert p.launches == 1 + (fold > 1) + 3 + (p.splits > 1)


def test_batched_grid_argument_checks(lib):
    f = lib.mri_fhd_batched_grid
    f.argtypes = ([P] * 3 + [P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int] + [P] * 4
                  + [I64, I64, P, P, ctypes.c_int, ctypes.c_int, P])
    f.restype = ctypes.c_int
    g = fake()
    args = lambda B=2, M=10, nx=128, trig=0, acc=0: (g[0], g[1], g[2], g[3], nx, g[4], 4, g[5], 4,
                                                     g[6], g[7], g[8], g[9], B, M, g[10], g[11],
                                                     trig, acc, None)
    assert f(*args(trig=5)) == MODE
    assert f(*args(acc=3)) == MODE
    assert f(*args(B=0)) == SIZE
    assert f(*args(M=-1)) == SIZE
    assert f(*args(nx=-2)) == SIZE


def test_forward_argument_checks(lib):
    f = lib.mri_forward
    f.argtypes = [P] * 8 + [I64, I64, P, P, ctypes.c_int, ctypes.c_int, P]
    f.restype = ctypes.c_int
    g = fake()
    assert f(*g[:8], 10, 10, g[8], g[9], 9, 0, None) == MODE
    assert f(*g[:8], -1, 10, g[8], g[9], 0, 0, None) == SIZE
    assert f(*g[:8], 10, -1, g[8], g[9], 0, 0, None) == SIZE
    assert f(*g[:8], 0, 10, g[8], g[9], 0, 0, None) == OK          # no samples: no-op
    bad = list(g[:8])
    bad[3] = P(None)                                                 # x
    assert f(*bad, 10, 10, g[8], g[9], 0, 0, None) == NULL
    bad = list(g[:8])
    bad[6] = P(0x100001)                                             # rRho misaligned
    assert f(*bad, 10, 10, g[8], g[9], 0, 0, None) == ALIGN


F32 = ctypes.c_float
INT = ctypes.c_int


def test_find_rho_argument_checks_before_any_cuda_call(lib):
    """mri_fft3, mri_toeplitz_kernel, mri_toeplitz_apply, mri_cg_solve: grid
    edges powers of two (FFT lines up to 1024, Toeplitz grids up to 512),
    modes, finite lambda and spacing, iteration bound, 8-byte alignment --
    all decided on the host."""
    g = fake()
    fft = lib.mri_fft3
    fft.argtypes = [P, INT, INT, INT, INT, P]
    fft.restype = INT
    assert fft(g[0], 6, 8, 8, 0, None) == SIZE
    assert fft(g[0], 8, 8, 2048, 0, None) == SIZE
    assert fft(g[0], 8, 8, 8, 2, None) == MODE
    assert fft(P(0x100004), 8, 8, 8, 0, None) == ALIGN
    ap = lib.mri_toeplitz_apply
    ap.argtypes = [P, INT, INT, INT, F32, P, P, P, P, INT, P]
    ap.restype = INT
    for n in ((3, 4, 4), (4, 4, 1024), (0, 4, 4), (4, -2, 4)):
        assert ap(g[0], *n, 0.0, *g[1:5], 0, None) == SIZE, n
    assert ap(g[0], 4, 4, 4, float("nan"), *g[1:5], 0, None) == SIZE
    assert ap(g[0], 4, 4, 4, 0.0, *g[1:5], 2, None) == MODE
    assert ap(P(0x100004), 4, 4, 4, 0.0, *g[1:5], 0, None) == ALIGN
    cg = lib.mri_cg_solve
    cg.argtypes = [P, INT, INT, INT, F32, P, P, P, P, INT, P, P]
    cg.restype = INT
    assert cg(g[0], 4, 4, 4, 0.0, *g[1:5], -1, g[5], None) == SIZE
    assert cg(g[0], 4, 4, 4, 0.0, *g[1:5], (1 << 20) + 1, g[5], None) == SIZE
    assert cg(g[0], 4, 4, 5, 0.0, *g[1:5], 3, g[5], None) == SIZE
    assert cg(g[0], 4, 4, 4, 0.0, *g[1:5], 3, P(0x100004), None) == ALIGN
    tk = lib.mri_toeplitz_kernel
    tk.argtypes = [P] * 5 + [I64, INT, INT, INT, F32, F32, F32, P, INT, P]
    tk.restype = INT
    assert tk(*g[:5], 10, 4, 4, 4, 1.0, float("inf"), 1.0, g[5], 0, None) == SIZE
    assert tk(*g[:5], 10, 4, 4, 4, 1.0, 1.0, 1.0, g[5], 9, None) == MODE
    assert tk(*g[:5], -1, 4, 4, 4, 1.0, 1.0, 1.0, g[5], 0, None) == SIZE
    assert tk(*g[:5], 10, 4, 6, 4, 1.0, 1.0, 1.0, g[5], 0, None) == SIZE


def test_gridding_argument_checks_before_any_cuda_call(lib):
    g = fake()
    f = lib.mri_gridding
    f.argtypes = [P] * 7 + [I64, INT, INT, INT, P, P, INT, P]
    f.restype = INT
    for n in ((3, 4, 4), (4, 4, 2048), (0, 4, 4)):
        assert f(*g[:7], 16, *n, g[7], g[8], 0, None) == SIZE, n
    assert f(*g[:7], -1, 4, 4, 4, g[7], g[8], 0, None) == SIZE
    assert f(*g[:7], 16, 4, 4, 4, g[7], g[8], 2, None) == MODE
    for i in range(9):
        bad = list(g[:9])
        bad[i] = P(None)
        assert f(*bad[:7], 16, 4, 4, 4, bad[7], bad[8], 0, None) == NULL, i
        bad[i] = P(0x100001 + 256 * i)
        assert f(*bad[:7], 16, 4, 4, 4, bad[7], bad[8], 0, None) == ALIGN, i
