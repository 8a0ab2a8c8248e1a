"""The minimax coefficients of the polynomial trig (sincospi_coeffs.h).

Checks on the CPU that the committed header is what gen_sincospi.py writes,
and that the float32 sequence the kernel performs (exact quarter-turn
reduction, Horner with fused multiply-adds, rotation by the quadrant) stays
within about one ulp of numpy's double-precision sin and cos, with a mean
error far below what a sum of a million positive weights could expose.
"""

import os
import re

import numpy as np
import pytest

from non_cartesian_mri_gb300.csrc import gen_sincospi as gen

HEADER = os.path.join(os.path.dirname(gen.__file__), "sincospi_coeffs.h")


def parse():
    text = open(HEADER).read()
    sets = {}
    for m in re.finditer(r"struct SinCos(\w+) \{(.*?)\n\};", text, re.S):
        name, body = m.group(1), m.group(2)
        co = {}
        for fname, expr in re.findall(
                r"static constexpr float (\w)\(int i\)\s*\{\s*return (.*?);\s*\}", body, re.S):
            co[fname] = [np.float32(float(v.rstrip("f")))
                         for v in re.findall(r"[-+]?\d\.\d+e[-+]\d+f", expr)]
        sets[name] = co
    return sets


@pytest.fixture(scope="module")
def coef():
    return parse()["Quarter"]


@pytest.fixture(scope="module")
def half():
    return parse()["Half"]


def test_header_matches_generator():
    sets = parse()
    assert sorted(sets) == sorted(name for name, *_ in gen.SETS)
    for name, pt, qt, turn in gen.SETS:
        P, Q = gen.fit(pt, qt, turn)
        assert [gen.f32(c) for c in P] == sets[name]["P"], name
        assert [gen.f32(c) for c in Q] == sets[name]["Q"], name


def test_half_turn_max_and_mean_error(half):
    """The general gather's sequence (half-turn reduction, Horner, sign flip
    by the parity of the half turn) over 32 turns either way."""
    u = np.linspace(-64.0, 64.0, 400001).astype(np.float32)
    sn, cs = gen.half_turn_sincos32(half["P"], half["Q"], u)
    x = np.pi * u.astype(np.float64)
    es = sn.astype(np.float64) - np.sin(x)
    ec = cs.astype(np.float64) - np.cos(x)
    assert np.abs(es).max() <= 1.5e-7 and np.abs(ec).max() <= 3e-7
    assert abs(es.mean()) <= 2e-9 and abs(ec.mean()) <= 2e-9


def test_whole_half_turns_are_exact(half):
    """A phase of a whole number of half turns (0 in particular) gives sin 0 and
    cos +-1 exactly: the cos series' constant term is 1 and f = 0."""
    u = np.array([0.0, 1.0, -1.0, 2.0, -3.0, 2e6, 2e6 + 1], np.float32)
    sn, cs = gen.half_turn_sincos32(half["P"], half["Q"], u)
    assert np.all(sn == 0.0)
    assert np.all(cs == np.where(u.astype(np.int64) % 2 == 0, 1.0, -1.0))


def test_max_and_mean_error(coef):
    u = np.linspace(-64.0, 64.0, 40001).astype(np.float32)     # 16 turns either way
    es, ec = [], []
    for ui in u:
        sn, cs = gen.quarter_turn_sincos32(coef["P"], coef["Q"], ui)
        x = np.pi / 2 * np.float64(ui)
        es.append(float(sn) - np.sin(x))
        ec.append(float(cs) - np.cos(x))
    es, ec = np.array(es), np.array(ec)
    assert np.abs(es).max() <= 1.2e-7 and np.abs(ec).max() <= 1.2e-7
    assert abs(es.mean()) <= 2e-9 and abs(ec.mean()) <= 2e-9


@pytest.mark.parametrize("u,ref", [(0.0, (0, 1)), (1.0, (1, 0)), (2.0, (0, -1)),
                                   (3.0, (-1, 0)), (-1.0, (-1, 0)), (-2.0, (0, -1)),
                                   (4e6, (0, 1)), (4e6 + 1, (1, 0))])
def test_whole_quarter_turns_are_exact(coef, u, ref):
    sn, cs = gen.quarter_turn_sincos32(coef["P"], coef["Q"], u)
    assert abs(float(sn) - ref[0]) <= 1e-7 and abs(float(cs) - ref[1]) <= 1e-7
