"""Generate the minimax polynomials of the polynomial trig paths.

The gather needs sin(2*pi*t) and cos(2*pi*t).  With u = 4t (quarter turns)
the kernel reduces exactly, q = rint(u), f = u - q in [-1/2, 1/2], so the
angle phi = (pi/2) f lies in [-pi/4, pi/4], and evaluates

    sin(phi) ~ f * P(f^2)        (odd, degree 2*len(P) - 1)
    cos(phi) ~ Q(f^2)            (even, degree 2*len(Q) - 2)

then rotates by q quarter turns (a swap and sign flips from the two low bits
of q).  On this short interval both series are well conditioned: the float32
evaluation stays within about one ulp and its mean error is tiny, which
matters because errors with a consistent sign add up coherently in Q, whose
weights |Phi|^2 are all positive.

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


def fit(p_terms=4, q_terms=5):
    quarter = mp.mpf(1) / 4                       # s = f^2 in [0, 1/4]
    half_pi = mp.pi / 2

    def sinc(s):                                  # sin((pi/2) f) / f as a function of s
        if s == 0:
            return half_pi
        f = mp.sqrt(s)
        return mp.sin(half_pi * f) / f

    def cosq(s):
        return mp.cos(half_pi * mp.sqrt(s))

    P = remez(sinc, p_terms, mp.mpf(0), quarter)     # sin: degree 2p-1
    Q = remez(cosq, q_terms, mp.mpf(0), quarter)     # cos: degree 2q-2
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


# (name, sin terms, cos terms)
SETS = (("Quarter", 4, 5),)


def main():
    lines = [
        "// sincospi_coeffs.h -- generated by gen_sincospi.py (Remez exchange, mpmath",
        "// 50 digits, coefficients rounded to float32).  Do not edit by hand.",
        "//   u in quarter turns, f = u - rint(u) in [-1/2, 1/2], phi = (pi/2) f:",
        "//   sin(phi) ~ f * P(f^2),  cos(phi) ~ Q(f^2).",
        "#pragma once",
        "#ifdef __CUDACC__",
        "#define MRI_HD __host__ __device__",
        "#else",
        "#define MRI_HD",
        "#endif",
        "namespace mri {",
    ]
    for name, pt, qt in SETS:
        P, Q = fit(pt, qt)
        P32 = [f32(c) for c in P]
        Q32 = [f32(c) for c in Q]
        es, ec, ms, mc = check(P32, Q32)
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
