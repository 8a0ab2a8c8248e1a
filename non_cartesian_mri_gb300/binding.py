"""Python binding of libmri.so: argument marshalling only.

Every computation runs in the library's CUDA kernels; this module checks
tensor types and shapes, allocates outputs with PyTorch, passes raw device
pointers and the current CUDA stream through ctypes, and raises on a non-OK
status.  There is no CPU fallback: if the library is not built or no sm_103a
device is present, calls raise.

Host (CPU) tensors or numpy arrays are accepted too: they are copied to the
current CUDA device, the call runs there, and the outputs are copied back to
host memory (this is the end-to-end path; the copies are the caller's cost).
"""

from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

TRIG = {"accurate": 0, "fast": 1, "fast_rr": 2}
KIND = {"fhd": 0, "q": 1, "fhd_batched": 2}

_lock = threading.Lock()
_lib = None


class MriError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class _Plan(ctypes.Structure):
    _fields_ = [("threads_per_cta", ctypes.c_int), ("voxels_per_thread", ctypes.c_int),
                ("samples_per_tile", ctypes.c_int), ("splits", ctypes.c_int),
                ("voxel_ctas", ctypes.c_int64), ("tiles", ctypes.c_int64),
                ("coil_groups", ctypes.c_int), ("launches", ctypes.c_int),
                ("scratch_bytes", ctypes.c_int64), ("tensor_cores", ctypes.c_int),
                ("grid_fold", ctypes.c_int), ("fast_fp32_voxels", ctypes.c_int),
                ("voxels_per_cta", ctypes.c_int)]


def lib_path() -> str:
    """The library to load: ``MRI_LIB`` if set (a variant build), else the default."""
    return os.environ.get("MRI_LIB") or _build.LIB


def load():
    """Load libmri.so (it must have been built: ``build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libmri.so is not built ({path}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.mri_mu.argtypes = [P] * 6 + [I64, P]
        lib.mri_fhd.argtypes = [P] * 10 + [I64, I64, P, P, I, I, P]
        lib.mri_q.argtypes = [P] * 8 + [I64, I64, P, P, I, I, P]
        lib.mri_fhd_batched.argtypes = [P] * 10 + [I64, I64, I64, P, P, I, I, P]
        lib.mri_forward.argtypes = [P] * 8 + [I64, I64, P, P, I, I, P]
        lib.mri_forward.restype = ctypes.c_int
        lib.mri_forward_grid.argtypes = ([P] * 3 + [P, I, P, I, P, I] + [P] * 2
                                         + [I64, P, P, I, I, P])
        lib.mri_forward_grid.restype = ctypes.c_int
        for f in (lib.mri_mu, lib.mri_fhd, lib.mri_q, lib.mri_fhd_batched):
            f.restype = ctypes.c_int
        lib.mri_status_string.argtypes = [ctypes.c_int]
        lib.mri_status_string.restype = ctypes.c_char_p
        lib.mri_plan_gather.argtypes = [I, I64, I64, I64, I, ctypes.POINTER(_Plan)]
        lib.mri_plan_gather.restype = ctypes.c_int
        lib.mri_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint), I]
        lib.mri_device_errors.restype = ctypes.c_int
        lib.mri_microbench.argtypes = [I, I, I, I64, P, P, P]
        lib.mri_wait_selftest.argtypes = [I, P]
        lib.mri_mma_probe.argtypes = [I, I, P, I64, P, P]
        F = ctypes.c_float
        lib.mri_fft3.argtypes = [P, I, I, I, I, P]
        lib.mri_toeplitz_kernel.argtypes = [P] * 5 + [I64, I, I, I, F, F, F, P, I, P]
        lib.mri_toeplitz_apply.argtypes = [P, I, I, I, F, P, P, P, P, I, P]
        lib.mri_cg_solve.argtypes = [P, I, I, I, F, P, P, P, P, I, P, P]
        lib.mri_gridding.argtypes = [P] * 7 + [I64, I, I, I, P, P, I, P]
        for f in (lib.mri_fft3, lib.mri_toeplitz_kernel, lib.mri_toeplitz_apply,
                  lib.mri_cg_solve, lib.mri_gridding):
            f.restype = ctypes.c_int
        lib.mri_mma_probe.restype = ctypes.c_int
        lib.mri_wait_selftest.restype = ctypes.c_int
        lib.mri_microbench.restype = ctypes.c_int
        lib.mri_fhd_grid.argtypes = ([P] * 3 + [P, I, P, I, P, I] + [P] * 4
                                     + [I64, P, P, I, I, P])
        lib.mri_fhd_grid.restype = ctypes.c_int
        lib.mri_q_grid.argtypes = ([P] * 3 + [P, I, P, I, P, I] + [P] * 2
                                   + [I64, P, P, I, I, P])
        lib.mri_q_grid.restype = ctypes.c_int
        lib.mri_plan_grid.argtypes = [I, I64, I, I, I, I, ctypes.POINTER(_Plan)]
        lib.mri_plan_grid.restype = ctypes.c_int
        lib.mri_fhd_batched_grid.argtypes = ([P] * 3 + [P, I, P, I, P, I] + [P] * 4
                                             + [I64, I64, P, P, I, I, P])
        lib.mri_fhd_batched_grid.restype = ctypes.c_int
        lib.mri_plan_grid_batched.argtypes = [I64, I64, I, I, I, I, ctypes.POINTER(_Plan)]
        lib.mri_plan_grid_batched.restype = ctypes.c_int
        lib.mri_timing_begin.argtypes = []
        lib.mri_timing_begin.restype = ctypes.c_int
        lib.mri_timing_end.argtypes = [ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(ctypes.c_int64)]
        lib.mri_timing_end.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().mri_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise MriError(status, where)


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(int(t.data_ptr()) if t is not None and t.numel() else None)


def _as_tensor(a):
    if isinstance(a, np.ndarray):
        return torch.from_numpy(np.ascontiguousarray(a))
    if not isinstance(a, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor or numpy array, got {type(a).__name__}")
    return a


class _Marshal:
    """Moves host inputs to the device (end-to-end path) and checks them."""

    def __init__(self, arrays):
        ts = [_as_tensor(a) for a in arrays]
        self.host = any(t.device.type != "cuda" for t in ts)
        if self.host:
            dev = torch.device("cuda", torch.cuda.current_device())
            ts = [t.to(dev, non_blocking=True) for t in ts]
        devs = {t.device for t in ts}
        if len(devs) != 1:
            raise ValueError(f"inputs on several devices: {sorted(map(str, devs))}")
        for t in ts:
            if t.dtype != torch.float32:
                raise TypeError(f"expected float32, got {t.dtype}")
            if not t.is_contiguous():
                raise ValueError("inputs must be contiguous")
        self.tensors = ts
        self.device = ts[0].device

    def result(self, outs):
        if self.host:
            return tuple(o.cpu() for o in outs)
        return tuple(outs)


def _outputs(out, shape, device):
    if out is None:
        return (torch.empty(shape, dtype=torch.float32, device=device),
                torch.empty(shape, dtype=torch.float32, device=device))
    r, i = out
    for t in (r, i):
        if (t.dtype != torch.float32 or t.device != device or tuple(t.shape) != tuple(shape)
                or not t.is_contiguous()):
            raise ValueError(f"out tensors must be contiguous float32 {tuple(shape)} on {device}")
    return r, i


def _same_len(name, ts, n):
    for t in ts:
        if t.dim() != 1 or t.shape[0] != n:
            raise ValueError(f"{name} arrays must be 1-D of length {n}")


def mu(rPhi, iPhi, rD, iD, *, stream=None):
    """cmpMu: (rMu, iMu) = conj(Phi) * D."""
    m = _Marshal([rPhi, iPhi, rD, iD])
    rPhi, iPhi, rD, iD = m.tensors
    M = rPhi.shape[0]
    _same_len("sample", m.tensors, M)
    rMu, iMu = _outputs(None, (M,), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_mu(_ptr(rPhi), _ptr(iPhi), _ptr(rD), _ptr(iD), _ptr(rMu), _ptr(iMu),
                             M, _stream_handle(stream)), "mri_mu")
    return m.result((rMu, iMu))


def fhd(kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD, *, trig="fast", accumulate=False,
        out=None, stream=None):
    """F^H D: (rFhD, iFhD)[n] = sum_m conj(Phi_m) D_m e^{+i 2 pi k_m . x_n}."""
    m = _Marshal([kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD])
    kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD = m.tensors
    M, N = kx.shape[0], x.shape[0]
    _same_len("sample", [kx, ky, kz, rPhi, iPhi, rD, iD], M)
    _same_len("voxel", [x, y, z], N)
    r, i = _outputs(out, (N,), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_fhd(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(x), _ptr(y), _ptr(z),
                              _ptr(rPhi), _ptr(iPhi), _ptr(rD), _ptr(iD), M, N, _ptr(r), _ptr(i),
                              TRIG[trig], int(bool(accumulate)), _stream_handle(stream)),
               "mri_fhd")
    return m.result((r, i))


def q(kx, ky, kz, x, y, z, rPhi, iPhi, *, trig="fast", accumulate=False, out=None,
      stream=None):
    """Q: (rQ, iQ)[n] = sum_m |Phi_m|^2 e^{+i 2 pi k_m . x_n}."""
    m = _Marshal([kx, ky, kz, x, y, z, rPhi, iPhi])
    kx, ky, kz, x, y, z, rPhi, iPhi = m.tensors
    M, N = kx.shape[0], x.shape[0]
    _same_len("sample", [kx, ky, kz, rPhi, iPhi], M)
    _same_len("voxel", [x, y, z], N)
    r, i = _outputs(out, (N,), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_q(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(x), _ptr(y), _ptr(z),
                            _ptr(rPhi), _ptr(iPhi), M, N, _ptr(r), _ptr(i), TRIG[trig],
                            int(bool(accumulate)), _stream_handle(stream)), "mri_q")
    return m.result((r, i))


def fhd_batched(kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD, *, trig="fast", accumulate=False,
                out=None, stream=None):
    """Batched F^H D over coil-major rD, iD [B, M]; returns (rFhD, iFhD) [B, N]."""
    m = _Marshal([kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD])
    kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD = m.tensors
    M, N = kx.shape[0], x.shape[0]
    _same_len("sample", [kx, ky, kz, rPhi, iPhi], M)
    _same_len("voxel", [x, y, z], N)
    if rD.dim() != 2 or rD.shape[1] != M or iD.shape != rD.shape:
        raise ValueError(f"rD, iD must be [B, {M}]")
    B = rD.shape[0]
    r, i = _outputs(out, (B, N), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_fhd_batched(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(x), _ptr(y), _ptr(z),
                                      _ptr(rPhi), _ptr(iPhi), _ptr(rD), _ptr(iD), B, M, N,
                                      _ptr(r), _ptr(i), TRIG[trig], int(bool(accumulate)),
                                      _stream_handle(stream)), "mri_fhd_batched")
    return m.result((r, i))


def forward(kx, ky, kz, x, y, z, rRho, iRho, *, trig="fast", accumulate=False, out=None,
            stream=None):
    """Forward model D[m] = sum_n rho[n] e^{-i2pi k_m.x_n}; returns (rD, iD) [M]."""
    m = _Marshal([kx, ky, kz, x, y, z, rRho, iRho])
    kx, ky, kz, x, y, z, rRho, iRho = m.tensors
    M, N = kx.shape[0], x.shape[0]
    _same_len("sample", [kx, ky, kz], M)
    _same_len("voxel", [x, y, z, rRho, iRho], N)
    r, i = _outputs(out, (M,), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_forward(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(x), _ptr(y), _ptr(z),
                                  _ptr(rRho), _ptr(iRho), M, N, _ptr(r), _ptr(i), TRIG[trig],
                                  int(bool(accumulate)), _stream_handle(stream)), "mri_forward")
    return m.result((r, i))


def forward_grid(kx, ky, kz, xs, ys, zs, rRho, iRho, *, trig="fast", accumulate=False,
                 out=None, stream=None):
    """Forward model of an image on the grid xs x ys x zs (rho [N], x fastest);
    returns (rD, iD) [M]."""
    m = _Marshal([kx, ky, kz, xs, ys, zs, rRho, iRho])
    kx, ky, kz, xs, ys, zs, rRho, iRho = m.tensors
    M = kx.shape[0]
    _same_len("sample", [kx, ky, kz], M)
    for t in (xs, ys, zs):
        if t.dim() != 1:
            raise ValueError("grid axes must be 1-D")
    nx, ny, nz = xs.shape[0], ys.shape[0], zs.shape[0]
    _same_len("voxel", [rRho, iRho], nx * ny * nz)
    r, i = _outputs(out, (M,), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_forward_grid(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(xs), nx, _ptr(ys), ny,
                                       _ptr(zs), nz, _ptr(rRho), _ptr(iRho), M, _ptr(r), _ptr(i),
                                       TRIG[trig], int(bool(accumulate)),
                                       _stream_handle(stream)), "mri_forward_grid")
    return m.result((r, i))


def fhd_grid(kx, ky, kz, xs, ys, zs, rPhi, iPhi, rD, iD, *, trig="fast", accumulate=False,
             out=None, stream=None):
    """F^H D on the separable grid xs x ys x zs; returns (rFhD, iFhD) [N], x fastest."""
    m = _Marshal([kx, ky, kz, xs, ys, zs, rPhi, iPhi, rD, iD])
    kx, ky, kz, xs, ys, zs, rPhi, iPhi, rD, iD = m.tensors
    M = kx.shape[0]
    _same_len("sample", [kx, ky, kz, rPhi, iPhi, rD, iD], M)
    for t in (xs, ys, zs):
        if t.dim() != 1:
            raise ValueError("grid axes must be 1-D")
    nx, ny, nz = xs.shape[0], ys.shape[0], zs.shape[0]
    r, i = _outputs(out, (nx * ny * nz,), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_fhd_grid(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(xs), nx, _ptr(ys), ny,
                                   _ptr(zs), nz, _ptr(rPhi), _ptr(iPhi), _ptr(rD), _ptr(iD), M,
                                   _ptr(r), _ptr(i), TRIG[trig], int(bool(accumulate)),
                                   _stream_handle(stream)), "mri_fhd_grid")
    return m.result((r, i))


def fhd_batched_grid(kx, ky, kz, xs, ys, zs, rPhi, iPhi, rD, iD, *, trig="fast",
                     accumulate=False, out=None, stream=None):
    """Batched F^H D on the separable grid xs x ys x zs over coil-major rD, iD
    [B, M]; returns (rFhD, iFhD) [B, N], x fastest."""
    m = _Marshal([kx, ky, kz, xs, ys, zs, rPhi, iPhi, rD, iD])
    kx, ky, kz, xs, ys, zs, rPhi, iPhi, rD, iD = m.tensors
    M = kx.shape[0]
    _same_len("sample", [kx, ky, kz, rPhi, iPhi], M)
    if rD.dim() != 2 or rD.shape[1] != M or iD.shape != rD.shape:
        raise ValueError(f"rD, iD must be [B, {M}]")
    for t in (xs, ys, zs):
        if t.dim() != 1:
            raise ValueError("grid axes must be 1-D")
    B = rD.shape[0]
    nx, ny, nz = xs.shape[0], ys.shape[0], zs.shape[0]
    r, i = _outputs(out, (B, nx * ny * nz), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_fhd_batched_grid(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(xs), nx, _ptr(ys),
                                           ny, _ptr(zs), nz, _ptr(rPhi), _ptr(iPhi), _ptr(rD),
                                           _ptr(iD), B, M, _ptr(r), _ptr(i), TRIG[trig],
                                           int(bool(accumulate)), _stream_handle(stream)),
               "mri_fhd_batched_grid")
    return m.result((r, i))


def q_grid(kx, ky, kz, xs, ys, zs, rPhi, iPhi, *, trig="fast", accumulate=False, out=None,
           stream=None):
    """Q on the separable grid xs x ys x zs; returns (rQ, iQ) [N], x fastest."""
    m = _Marshal([kx, ky, kz, xs, ys, zs, rPhi, iPhi])
    kx, ky, kz, xs, ys, zs, rPhi, iPhi = m.tensors
    M = kx.shape[0]
    _same_len("sample", [kx, ky, kz, rPhi, iPhi], M)
    nx, ny, nz = xs.shape[0], ys.shape[0], zs.shape[0]
    r, i = _outputs(out, (nx * ny * nz,), m.device)
    with torch.cuda.device(m.device):
        _check(load().mri_q_grid(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(xs), nx, _ptr(ys), ny,
                                 _ptr(zs), nz, _ptr(rPhi), _ptr(iPhi), M, _ptr(r), _ptr(i),
                                 TRIG[trig], int(bool(accumulate)), _stream_handle(stream)),
               "mri_q_grid")
    return m.result((r, i))


def plan_grid(kind: str, M: int, nx: int, ny: int, nz: int, num_sms: int = 0) -> dict:
    """The launch shape of mri_fhd_grid / mri_q_grid."""
    p = _Plan()
    _check(load().mri_plan_grid(KIND[kind], M, nx, ny, nz, num_sms, ctypes.byref(p)),
           "mri_plan_grid")
    return {name: getattr(p, name) for name, _ in _Plan._fields_}


def plan_grid_batched(B: int, M: int, nx: int, ny: int, nz: int, num_sms: int = 0) -> dict:
    """The launch shape of mri_fhd_batched_grid."""
    p = _Plan()
    _check(load().mri_plan_grid_batched(B, M, nx, ny, nz, num_sms, ctypes.byref(p)),
           "mri_plan_grid_batched")
    return {name: getattr(p, name) for name, _ in _Plan._fields_}


def plan(kind: str, M: int, N: int, B: int = 1, num_sms: int = 0) -> dict:
    """The launch shape libmri picks for a call (host-only when num_sms > 0)."""
    p = _Plan()
    _check(load().mri_plan_gather(KIND[kind], B, M, N, num_sms, ctypes.byref(p)),
           "mri_plan_gather")
    return {name: getattr(p, name) for name, _ in _Plan._fields_}


def wait_selftest(arrive: bool, stream=None) -> None:
    """Launch the bounded-wait self-test (see include/mri_microbench.h)."""
    _check(load().mri_wait_selftest(int(bool(arrive)), _stream_handle(stream)),
           "mri_wait_selftest")


def device_errors(clear: bool = True) -> int:
    """Device-side error bits (0: none).  Synchronises the current device."""
    bits = ctypes.c_uint(0)
    _check(load().mri_device_errors(ctypes.byref(bits), int(bool(clear))), "mri_device_errors")
    return int(bits.value)


class gather_timing:
    """Context manager: summed gather-kernel time (ms) of the calls inside it,
    measured with CUDA events on each launch's own stream.

        with gather_timing() as t:
            fhd(...)
        t.ms, t.launches
    """

    def __enter__(self):
        _check(load().mri_timing_begin(), "mri_timing_begin")
        self.ms = None
        self.launches = None
        return self

    def __exit__(self, *exc):
        ms = ctypes.c_double(0.0)
        n = ctypes.c_int64(0)
        _check(load().mri_timing_end(ctypes.byref(ms), ctypes.byref(n)), "mri_timing_end")
        self.ms = float(ms.value)
        self.launches = int(n.value)
        return False


PROBES = {"sin": 0, "cos": 1, "ffma": 2, "ex2": 3, "ffma2": 4}


def microbench(which: str, ctas_per_sm: int = 1, threads: int = 1024, iters: int = 1 << 14):
    """Results per SM per clock of one probed instruction (see mri_microbench.h).

    The rate is taken from each CTA's own elapsed cycles, which is the SM's
    busy time only when the SM holds one CTA: CTAs sharing an SM need not
    start and finish together, and their per-CTA counts then overstate the
    rate.  Keep ctas_per_sm = 1 (the default) for a roofline denominator."""
    dev = torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    grid = sms * ctas_per_sm
    cycles = torch.zeros(grid, dtype=torch.int64, device=dev)
    sink = torch.empty(grid * threads, dtype=torch.float32, device=dev)
    s = _stream_handle(None)
    _check(load().mri_microbench(PROBES[which], ctas_per_sm, threads, iters, _ptr(cycles),
                                 _ptr(sink), s), "mri_microbench")
    torch.cuda.synchronize(dev)
    cyc = cycles.double()
    ops_per_sm = ctas_per_sm * threads * iters * 8
    return {"probe": which, "per_sm_per_clk": float(ops_per_sm / cyc.median()),
            "per_sm_per_clk_min": float(ops_per_sm / cyc.max()),
            "cycles_median": float(cyc.median()), "sms": sms}


def mma_probe(mode: int = 1, tiles: int = 4096, b_tiles: int = 1024):
    """Pairs per SM per clock of the tensor-core grid kernel's MMA issue
    pattern alone (mode 0: A and B in shared memory; 1: A in tensor memory;
    2: A in tensor memory, B streamed by TMA from a table of b_tiles 48 KB
    tiles; see mri_mma_probe in mri_microbench.h)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device=dev)
    tab = torch.zeros(int(b_tiles) * 49152 if mode == 2 else 16, dtype=torch.uint8, device=dev)
    _check(load().mri_mma_probe(int(mode), int(tiles), _ptr(tab), int(b_tiles), _ptr(cycles),
                                _stream_handle(None)), "mri_mma_probe")
    torch.cuda.synchronize(dev)
    cyc = cycles.double()
    pairs = float(tiles) * 32 * 128 * 128
    return {"mode": int(mode), "tiles": int(tiles), "b_tiles": int(b_tiles),
            "pairs_per_sm_per_clk": float(pairs / cyc.median()),
            "pairs_per_sm_per_clk_min": float(pairs / cyc.max()),
            "cycles_median": float(cyc.median()), "sms": sms}


def fft3(data, inverse: bool = False, stream=None):
    """In-place 3-D FFT of a complex64 CUDA tensor of shape (Lz, Ly, Lx)
    (see mri_fft3); returns the tensor."""
    if data.dtype != torch.complex64 or not data.is_cuda or data.dim() != 3:
        raise ValueError("fft3 takes a 3-D complex64 CUDA tensor")
    data = data.contiguous()
    Lz, Ly, Lx = data.shape
    _check(load().mri_fft3(_ptr(data), Lx, Ly, Lz, int(bool(inverse)), _stream_handle(stream)),
           "mri_fft3")
    return data


def toeplitz_kernel(kx, ky, kz, rPhi, iPhi, shape, spacing=(1.0, 1.0, 1.0), *, trig="accurate",
                    stream=None):
    """Spectrum of F^H F on a grid of shape (nz, ny, nx) with voxel spacing
    (hx, hy, hz) (see mri_toeplitz_kernel): a real float32 tensor of shape
    (2nz, 2ny, 2nx)."""
    nz, ny, nx = (int(v) for v in shape)
    kx, ky, kz, rPhi, iPhi = (_as_tensor(t) for t in (kx, ky, kz, rPhi, iPhi))
    M = kx.numel()
    _same_len("samples", (kx, ky, kz, rPhi, iPhi), M)
    K = torch.empty((2 * nz, 2 * ny, 2 * nx), dtype=torch.float32, device=kx.device)
    hx, hy, hz = (float(v) for v in spacing)
    _check(load().mri_toeplitz_kernel(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(rPhi), _ptr(iPhi), M,
                                      nx, ny, nz, hx, hy, hz, _ptr(K), TRIG[trig],
                                      _stream_handle(stream)), "mri_toeplitz_kernel")
    return K


def _grid_shape(K):
    if K.dtype != torch.float32 or K.dim() != 3 or not K.is_cuda or not K.is_contiguous():
        raise ValueError("K must be the contiguous float32 CUDA tensor of toeplitz_kernel")
    return K.shape[0] // 2, K.shape[1] // 2, K.shape[2] // 2


def toeplitz_apply(K, rIn, iIn, *, lam: float = 0.0, accumulate=False, out=None, stream=None):
    """(F^H F + lam I) applied to a complex vector on the grid of K (see
    mri_toeplitz_apply); returns (rOut, iOut)."""
    nz, ny, nx = _grid_shape(K)
    rIn, iIn = _as_tensor(rIn), _as_tensor(iIn)
    N = nx * ny * nz
    _same_len("vector", (rIn, iIn), N)
    r, i = _outputs(out, (N,), rIn.device)
    _check(load().mri_toeplitz_apply(_ptr(K), nx, ny, nz, float(lam), _ptr(rIn), _ptr(iIn),
                                     _ptr(r), _ptr(i), int(bool(accumulate)),
                                     _stream_handle(stream)), "mri_toeplitz_apply")
    return r, i


def cg_solve(K, rB, iB, *, lam: float = 0.0, iters: int = 10, x0=None, stream=None):
    """Conjugate gradients on (F^H F + lam I) x = b (see mri_cg_solve).
    Returns (rX, iX, residual norms as a float64 CUDA tensor of iters + 1)."""
    nz, ny, nx = _grid_shape(K)
    rB, iB = _as_tensor(rB), _as_tensor(iB)
    N = nx * ny * nz
    _same_len("right-hand side", (rB, iB), N)
    if x0 is None:
        rX = torch.zeros(N, device=rB.device)
        iX = torch.zeros(N, device=rB.device)
    else:
        rX, iX = (_as_tensor(t).clone() for t in x0)
    norms = torch.empty(int(iters) + 1, dtype=torch.float64, device=rB.device)
    _check(load().mri_cg_solve(_ptr(K), nx, ny, nz, float(lam), _ptr(rB), _ptr(iB), _ptr(rX),
                               _ptr(iX), int(iters), _ptr(norms), _stream_handle(stream)),
           "mri_cg_solve")
    return rX, iX, norms


def gridding(kx, ky, kz, rPhi, iPhi, rD, iD, shape, *, accumulate=False, out=None, stream=None):
    """The gridding reconstruction on a grid of shape (nz, ny, nx) (see
    mri_gridding): trilinear interpolation of conj(Phi) D onto the Cartesian
    k-grid, then the inverse DFT onto the voxels x = i - n/2.  Returns
    (rOut, iOut) of nx*ny*nz floats."""
    nz, ny, nx = (int(v) for v in shape)
    kx, ky, kz, rPhi, iPhi, rD, iD = (_as_tensor(t) for t in (kx, ky, kz, rPhi, iPhi, rD, iD))
    M = kx.numel()
    _same_len("samples", (kx, ky, kz, rPhi, iPhi, rD, iD), M)
    r, i = _outputs(out, (nx * ny * nz,), kx.device)
    _check(load().mri_gridding(_ptr(kx), _ptr(ky), _ptr(kz), _ptr(rPhi), _ptr(iPhi), _ptr(rD),
                               _ptr(iD), M, nx, ny, nz, _ptr(r), _ptr(i), int(bool(accumulate)),
                               _stream_handle(stream)), "mri_gridding")
    return r, i
