"""Generate the minimax polynomials of the polynomial trig paths.

The gather needs sin(2*pi*t) and cos(2*pi*t).  Two reductions are used.

Quarter turns (the grid paths' per-factor trig): with u = 4t the kernel
reduces exactly, q = rint(u), f = u - q in [-1/2, 1/2], so the angle
phi = (pi/2) f lies in [-pi/4, pi/4], and evaluates

    sin(phi) ~ f * P(f^2)        (odd, degree 2*len(P) - 1)
    cos(phi) ~ Q(f^2)            (even, degree 2*len(Q) - 2)

then rotates by q quarter turns (a swap and sign flips from the two low bits
of q).

Half turns (the general gather, evaluated on pairs of floats): with u = 2t,
q = rint(u), f = u - q, phi = pi f in [-pi/2, pi/2], the same two series of
pi f, and e^{i 2 pi t} = (-1)^q e^{i phi}: only a sign flip from the low bit
of q, no swap, so every step but the flip is a floating-point operation that
the packed two-float instructions can do.

On these short intervals both series are well conditioned: the float32
evaluation stays within a few units in the last place and its mean error is
tiny, which matters because errors with a consistent sign add up coherently
in Q, whose weights |Phi|^2 are all positive.

P and Q are fitted with the Remez exchange algorithm (E. Ya. Remez, 1934):
minimise the maximum absolute error on s = f^2 in [0, 1/4], with the error
equioscillating on len(coeffs) + 1 points.  Work is in mpmath at 50 digits;
the coefficients are rounded to float32 and the float32 evaluation (Horner
with fused multiply-adds) is checked on a dense grid for its maximum and mean
error.  Writes ``sincospi_coeffs.h`` next to this file.

    python -m non_cartesian_mri_gb300.csrc.gen_sincospi
"""

from __future__ import annotations

import os

import mpmath as mp
import numpy as np

mp.mp.dps = 50
HERE = os.path.dirname(os.path.abspath(__file__))


def remez(f, basis_count, lo, hi, iters=40):
    """Minimax polynomial sum_j a_j s^j (j < basis_count) for f on [lo, hi]."""
    n = basis_count
    # initial reference: Chebyshev extrema
    xs = [lo + (hi - lo) * (1 - mp.cos(mp.pi * i / n)) / 2 for i in range(n + 1)]
    coeffs = None
    for _ in range(iters):
        # solve sum_j a_j x_i^j + (-1)^i E = f(x_i)
        A = mp.matrix(n + 1, n + 1)
        b = mp.matrix(n + 1, 1)
        for i, x in enumerate(xs):
            for j in range(n):
                A[i, j] = x ** j
            A[i, n] = (-1) ** i
            b[i] = f(x)
        sol = mp.lu_solve(A, b)
        coeffs = [sol[j] for j in range(n)]

        def err(x):
            return sum(c * x ** j for j, c in enumerate(coeffs)) - f(x)

        # new reference: extrema of the error on a fine grid, one per sign run
        grid = [lo + (hi - lo) * mp.mpf(k) / 4000 for k in range(4001)]
        ev = [err(x) for x in grid]
        runs = []
        cur = [0]
        for k in range(1, len(grid)):
            if mp.sign(ev[k]) == mp.sign(ev[cur[0]]) or ev[k] == 0:
                cur.append(k)
            else:
                runs.append(cur)
                cur = [k]
        runs.append(cur)
        ext = [max(r, key=lambda k: abs(ev[k])) for r in runs]
        if len(ext) < n + 1:
            break
        # keep n + 1 alternating extrema with the largest errors
        while len(ext) > n + 1:
            if abs(ev[ext[0]]) < abs(ev[ext[-1]]):
                ext.pop(0)
            else:
                ext.pop()
        new = [grid[k] for k in ext]
        if max(abs(a - b) for a, b in zip(new, xs)) < mp.mpf(10) ** -30:
            break
        xs = new
    return coeffs


def fit(p_terms=4, q_terms=5, turn=4):
    """P, Q for phi = (2 pi / turn) f, f in [-1/2, 1/2] (turn = 4: quarter
    turns, 2: half turns)."""
    quarter = mp.mpf(1) / 4                       # s = f^2 in [0, 1/4]
    half_pi = 2 * mp.pi / turn

    def sinc(s):                                  # sin(half_pi f) / f as a function of s
        if s == 0:
            return half_pi
        f = mp.sqrt(s)
        return mp.sin(half_pi * f) / f

    def cosq(s):
        return mp.cos(half_pi * mp.sqrt(s))

    def cosm1(s):                                 # (cos(half_pi f) - 1) / f^2
        if s == 0:
            return -half_pi ** 2 / 2
        return (mp.cos(half_pi * mp.sqrt(s)) - 1) / s

    P = remez(sinc, p_terms, mp.mpf(0), quarter)     # sin: degree 2p-1
    if turn == 4:
        Q = remez(cosq, q_terms, mp.mpf(0), quarter)     # cos: degree 2q-2
    else:
        # constant term fixed at 1, so that a whole number of half turns
        # (in particular a phase of exactly 0) gives cos = +-1 exactly
        Q = [mp.mpf(1)] + remez(cosm1, q_terms - 1, mp.mpf(0), quarter)
    return P, Q


def f32(x):
    return np.float32(float(x))


def fma32(a, b, c):
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def horner32(coeffs32, s):
    acc = coeffs32[-1]
    for c in reversed(coeffs32[:-1]):
        acc = fma32(acc, s, c)
    return acc


def quarter_turn_sincos32(P32, Q32, u):
    """The kernel's float32 sequence for sin and cos of (pi/2) u."""
    u = np.float32(u)
    magic = np.float32(12582912.0)
    v = np.float32(u + magic)
    q = int(np.float32(v - magic))
    f = np.float32(u - np.float32(q))
    s = np.float32(f * f)
    sf = np.float32(f * horner32(P32, s))
    cf = horner32(Q32, s)
    if q & 1:
        sf, cf = cf, sf
    sn = -sf if (q & 2) else sf
    cs = -cf if ((q + 1) & 2) else cf
    return np.float32(sn), np.float32(cs)


def half_turn_sincos32(P32, Q32, u):
    """The kernel's float32 sequence for sin and cos of pi u (u in half
    turns), vectorised over u."""
    u = np.asarray(u, np.float32)
    magic = np.float32(12582912.0)
    v = (u + magic).astype(np.float32)
    t = (v - magic).astype(np.float32)
    f = (u - t).astype(np.float32)
    s = (f * f).astype(np.float32)

    def horner(c):
        acc = np.full_like(s, c[-1])
        for ci in reversed(c[:-1]):
            acc = (acc.astype(np.float64) * s.astype(np.float64)
                   + np.float64(ci)).astype(np.float32)
        return acc

    sf = (f * horner(P32)).astype(np.float32)
    cf = horner(Q32)
    odd = (t.astype(np.int64) & 1) != 0
    return np.where(odd, -sf, sf), np.where(odd, -cf, cf)


def check(P32, Q32, n=20001):
    """Max and mean error of the float32 evaluation of sin/cos(2 pi t),
    t = u/4 over four turns."""
    u = np.linspace(-8.0, 8.0, n).astype(np.float32)
    es, ec = [], []
    for ui in u:
        sn, cs = quarter_turn_sincos32(P32, Q32, ui)
        x = np.pi / 2 * np.float64(ui)
        es.append(float(sn) - np.sin(x))
        ec.append(float(cs) - np.cos(x))
    es, ec = np.array(es), np.array(ec)
    return (float(np.abs(es).max()), float(np.abs(ec).max()),
            float(es.mean()), float(ec.mean()))


def check_half(P32, Q32, n=200001):
    """Max and mean error of the float32 evaluation of sin/cos(2 pi t),
    t = u/2 over four turns."""
    u = np.linspace(-8.0, 8.0, n).astype(np.float32)
    sn, cs = half_turn_sincos32(P32, Q32, u)
    x = np.pi * u.astype(np.float64)
    es = sn.astype(np.float64) - np.sin(x)
    ec = cs.astype(np.float64) - np.cos(x)
    return (float(np.abs(es).max()), float(np.abs(ec).max()),
            float(es.mean()), float(ec.mean()))


# (name, sin terms, cos terms, turn divisor)
SETS = (("Quarter", 4, 5, 4), ("Half", 5, 5, 2))


def main():
    lines = [
        "// sincospi_coeffs.h -- generated by gen_sincospi.py (Remez exchange, mpmath",
        "// 50 digits, coefficients rounded to float32).  Do not edit by hand.",
        "//   Quarter: u in quarter turns, f = u - rint(u) in [-1/2, 1/2], phi = (pi/2) f;",
        "//   Half:    u in half turns,    f = u - rint(u) in [-1/2, 1/2], phi = pi f;",
        "//   sin(phi) ~ f * P(f^2),  cos(phi) ~ Q(f^2).",
        "#pragma once",
        "#ifdef __CUDACC__",
        "#define MRI_HD __host__ __device__",
        "#else",
        "#define MRI_HD",
        "#endif",
        "namespace mri {",
    ]
    for name, pt, qt, turn in SETS:
        P, Q = fit(pt, qt, turn)
        P32 = [f32(c) for c in P]
        Q32 = [f32(c) for c in Q]
        es, ec, ms, mc = (check if turn == 4 else check_half)(P32, Q32)
        lines += [
            f"// {name}: degree {2 * pt - 1} / {2 * qt - 2}; float32 evaluation over four turns:",
            f"//   max |error| sin {es:.3e}, cos {ec:.3e}; mean error sin {ms:.2e}, cos {mc:.2e}",
            f"struct SinCos{name} {{",
            f"    static constexpr int P_TERMS = {pt};",
            f"    static constexpr int Q_TERMS = {qt};",
            "    MRI_HD static constexpr float P(int i)",
            "    {",
            "        return " + " : ".join(f"i == {j} ? {float(c):.9e}f" for j, c in
                                         enumerate(P32[:-1])) + f" : {float(P32[-1]):.9e}f;",
            "    }",
            "    MRI_HD static constexpr float Q(int i)",
            "    {",
            "        return " + " : ".join(f"i == {j} ? {float(c):.9e}f" for j, c in
                                         enumerate(Q32[:-1])) + f" : {float(Q32[-1]):.9e}f;",
            "    }",
            "};",
        ]
    lines += ["}  // namespace mri", ""]
    path = os.path.join(HERE, "sincospi_coeffs.h")
    with open(path, "w") as fh:
        fh.write("\n".join(lines))
    print("\n".join(lines))


if __name__ == "__main__":
    main()
