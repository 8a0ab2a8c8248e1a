"""Mutation check of the numpy oracles (oracle/toeplitz.py, oracle/gridding.py),
no GPU: each plausible mistake (a wrong wrap or sign of the difference axis,
transposed axes, a conjugate, the wrong plane zeroed, a swapped CG ratio, the
interpolation weights swapped, the centring or the exponent's sign dropped,
Mu without the conjugate) is planted in a copy of the module's source, and at
least one of the pins below must then fail.  The unmutated modules pass all
of them.

The pins restate the ones of test_oracle_toeplitz.py and test_oracle_gridding.py
as functions of the module under test: F^H F against F^H (F rho) from the C
oracle's forward model and F^H D, the FFT route against the definition, the
real spectrum giving the same product, CG against a dense solve; on-grid
gridding against the C oracle's F^H D, partition of unity and position of the
weights, the halfway split, wrap-around, recon against the explicit DFT
matrices.
"""

import os
import types

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE = os.path.join(os.path.dirname(HERE), "oracle")


def caught(pins, mod):
    """A mutant is caught when a pin fails or the mutated code raises."""
    try:
        return not pins(mod)
    except Exception:
        return True


def load(name, old=None, new=None):
    src = open(os.path.join(ORACLE, name + ".py")).read()
    if old is not None:
        assert src.count(old) >= 1, f"mutation target not found: {old!r}"
        src = src.replace(old, new)
    mod = types.ModuleType("oracle_" + name + "_mut")
    mod.__package__ = "oracle"
    exec(compile(src, name + ".py", "exec"), mod.__dict__)
    return mod


# ---- Toeplitz pins ---------------------------------------------------------

def toeplitz_problem(shape, spacing, M, seed):
    rng = np.random.default_rng(seed)
    nz, ny, nx = shape
    hx, hy, hz = spacing
    k = rng.uniform(-0.5, 0.5, (3, M)).astype(np.float32)
    rPhi = rng.standard_normal(M).astype(np.float32)
    iPhi = rng.standard_normal(M).astype(np.float32)
    xs = (np.arange(nx) * hx - 3.0).astype(np.float32)
    ys = (np.arange(ny) * hy + 1.0).astype(np.float32)
    zs = (np.arange(nz) * hz - 0.5).astype(np.float32)
    z, y, x = np.meshgrid(zs, ys, xs, indexing="ij")
    rho = rng.standard_normal(shape) + 1j * rng.standard_normal(shape)
    return k, rPhi, iPhi, (x.reshape(-1), y.reshape(-1), z.reshape(-1)), rho


def toeplitz_pins_pass(T):
    shape, spacing = (2, 3, 4), (1.0, 0.75, 1.5)
    k, rPhi, iPhi, xyz, rho = toeplitz_problem(shape, spacing, 257, 9)
    Qc = T.q_difference_grid(k[0], k[1], k[2], rPhi, iPhi, shape, spacing)
    phi = rPhi.astype(np.float64) + 1j * iPhi
    v = phi * oracle.forward(k[0], k[1], k[2], *xyz, rho.reshape(-1))
    ref = oracle.fhd(k[0], k[1], k[2], *xyz, rPhi, iPhi, v.real, v.imag)
    direct = T.fhf_direct(Qc, rho)
    if not oracle.rel_l2(direct.reshape(-1), ref) < 1e-6:
        return False
    if not oracle.rel_l2(T.fhf_fft(Qc, rho), direct) < 1e-12:
        return False
    Kr, imag = T.toeplitz_spectrum(Qc)
    if not (imag < 1e-12 and oracle.rel_l2(T.fhf_spectrum(Kr, rho), direct) < 1e-12):
        return False
    N = int(np.prod(shape))
    A = np.zeros((N, N), np.complex128)
    for j in range(N):
        e = np.zeros(N, np.complex128)
        e[j] = 1.0
        A[:, j] = T.fhf_direct(Qc, e.reshape(shape)).reshape(-1)
    b = rho.reshape(-1)
    sol = np.linalg.solve(A + 0.3 * np.eye(N), b)
    apply = lambda vv: T.fhf_direct(Qc, vv.reshape(shape)).reshape(-1)   # noqa: E731
    x, norms = T.cg(apply, b, np.zeros(N), 0.3, 3 * N)
    return bool(np.abs(x - sol).max() < 1e-8 * np.abs(sol).max())


TOEPLITZ_MUTANTS = {
    "wrap off by one": ("np.where(i < n, i, i - 2 * n)", "np.where(i < n, i, i - 2 * n + 1)"),
    "difference sign": ("np.where(i < n, i, i - 2 * n)", "np.where(i < n, -i, i - 2 * n)"),
    "rolled axes transposed": ("np.roll(Qc, (jz, jy, jx), axis=(0, 1, 2))",
                               "np.roll(Qc, (jx, jy, jz), axis=(0, 1, 2))"),
    "conjugated Q": ("out += v * shifted[:nz, :ny, :nx]",
                     "out += v * np.conj(shifted[:nz, :ny, :nx])"),
    "wrong plane zeroed": ("Z[nz, :, :] = 0", "Z[nz - 1, :, :] = 0"),
    "FFT directions swapped": ("return np.fft.ifftn(Kr * np.fft.fftn(pad))[:nz, :ny, :nx]",
                               "return np.fft.fftn(Kr * np.fft.ifftn(pad))[:nz, :ny, :nx]"),
    "CG beta inverted": ("p = r + (rr_new / rr) * p", "p = r + (rr / rr_new) * p"),
    "CG step without lambda": ("return apply(v) + lam * v", "return apply(v)"),
}


def test_toeplitz_pins_pass_unmutated():
    assert toeplitz_pins_pass(load("toeplitz"))


@pytest.mark.parametrize("name", sorted(TOEPLITZ_MUTANTS))
def test_toeplitz_mutant_is_caught(name):
    old, new = TOEPLITZ_MUTANTS[name]
    assert caught(toeplitz_pins_pass, load("toeplitz", old, new)), name


# ---- gridding pins -----------------------------------------------------------

def gridding_pins_pass(Gr):
    shape = (4, 8, 16)
    nz, ny, nx = shape
    rng = np.random.default_rng(21)
    M = 300
    k = [((rng.integers(0, n, M) - n // 2) / n).astype(np.float32) for n in (nx, ny, nz)]
    vals = [rng.standard_normal(M).astype(np.float32) for _ in range(4)]
    img = Gr.gridding_recon(*k, *vals, shape)
    z, y, x = np.meshgrid(np.arange(nz) - nz // 2, np.arange(ny) - ny // 2,
                          np.arange(nx) - nx // 2, indexing="ij")
    ref = oracle.fhd(*k, x.reshape(-1).astype(np.float32), y.reshape(-1).astype(np.float32),
                     z.reshape(-1).astype(np.float32), *vals)
    if not oracle.rel_l2(img.reshape(-1), ref) < 1e-12:
        return False
    kk = [rng.uniform(-0.45, 0.45, 5) for _ in range(3)]
    for m in range(5):
        Gm = Gr.grid_samples(*(a[m:m + 1] for a in kk), np.ones(1), shape)
        if abs(Gm.sum() - 1.0) > 1e-12:
            return False
        for axis, n, km in ((2, nx, kk[0][m]), (1, ny, kk[1][m]), (0, nz, kk[2][m])):
            kg = (np.arange(n) - n // 2) / n
            bshape = [1, 1, 1]
            bshape[axis] = n
            if abs((Gm.real * kg.reshape(bshape)).sum() - km) > 1e-12:
                return False
    G = Gr.grid_samples(np.array([(5.5 - 8) / 16]), np.array([(1 - 4) / 8]),
                        np.array([(2 - 2) / 4]), np.array([2.0 + 1.0j]), shape)
    if sorted(map(tuple, np.argwhere(np.abs(G) > 0))) != [(2, 1, 5), (2, 1, 6)]:
        return False
    # wrap-around: a shift by one period gives the same grid, and a sample
    # just below +1/2 lands on the wrapped point 0
    kw = [rng.uniform(-0.5, 0.5, 64) for _ in range(3)]
    mw = rng.standard_normal(64) + 1j * rng.standard_normal(64)
    G1 = Gr.grid_samples(*kw, mw, shape)
    G2 = Gr.grid_samples(kw[0] - 1.0, kw[1] + 1.0, kw[2] - 1.0, mw, shape)
    if np.abs(G1 - G2).max() > 1e-12:
        return False
    Gw = Gr.grid_samples(np.array([0.5 - 2.0 ** -30]), np.zeros(1), np.zeros(1), np.ones(1),
                         shape)
    if abs(Gw[2, 4, 0] - 1.0) > 1e-6:
        return False
    R = rng.standard_normal((2, 4, 8)) + 1j * rng.standard_normal((2, 4, 8))
    return bool(oracle.rel_l2(Gr.recon(R), Gr.recon_direct(R)) < 1e-12)


GRIDDING_MUTANTS = {
    "weights swapped": ("(fx if cx else 1 - fx)", "(1 - fx if cx else fx)"),
    "no centring of k": ("u = (np.asarray(k, np.float64) + 0.5) * n",
                         "u = np.asarray(k, np.float64) * n"),
    "exponent sign": ("np.exp(2j * np.pi * np.outer(x, k))", "np.exp(-2j * np.pi * np.outer(x, k))"),
    "centring sign dropped": ("c = (-1.0) ** (nz // 2 + ny // 2 + nx // 2)", "c = 1.0"),
    "Mu without conjugate": ("return np.conj(phi) * d", "return phi * d"),
    "wrap index": ("((gz + cz) % nz_, (gy + cy) % ny_, (gx + cx) % nx_)",
                   "((gz + cz) % nz_, (gy + cy) % ny_, (gx + cx) % nx_ - (gx + cx) // nx_)"),
}


def test_gridding_pins_pass_unmutated():
    assert gridding_pins_pass(load("gridding"))


@pytest.mark.parametrize("name", sorted(GRIDDING_MUTANTS))
def test_gridding_mutant_is_caught(name):
    old, new = GRIDDING_MUTANTS[name]
    assert caught(gridding_pins_pass, load("gridding", old, new)), name
