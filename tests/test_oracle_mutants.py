"""The oracle pins reject plausible mistakes.

Each case copies oracle.c, plants one mistake in the copy (CPU only), builds
it, routes the oracle to that build and runs every pin; at least one pin must
fail.  The unmodified source must pass all of them.
"""

import inspect
import os

import pytest

import oracle
import tests.test_oracle_pins as pins
from tests.conftest import read_golden

MUTANTS = {
    "exponent sign": [("double phase = TWO_PI *", "double phase = -TWO_PI *")],
    "no conjugate on Phi": [("rMu[m] = rp * rd + ip * id;", "rMu[m] = rp * rd - ip * id;"),
                            ("iMu[m] = rp * id - ip * rd;", "iMu[m] = rp * id + ip * rd;")],
    "y term uses x": [("(double)ky[m] * y\n", "(double)ky[m] * x\n"),
                      ("+ (double)ky[m] * y[n]\n", "+ (double)ky[m] * x[n]\n")],
    "z term dropped": [("\n                                 + (double)kz[m] * z);", ");"),
                       ("\n                                         + (double)kz[m] * z[n]);", ");")],
    "MAC sign": [("sr += wr[m] * c - wi[m] * s;", "sr += wr[m] * c + wi[m] * s;")],
    "Q weight |Phi| not |Phi|^2": [("w[m] = rp * rp + ip * ip;", "w[m] = sqrt(rp * rp + ip * ip);")],
    "Q sin/cos swapped": [("sr += wr[m] * cos(phase);", "sr += wr[m] * sin(phase);"),
                          ("si += wr[m] * sin(phase);", "si += wr[m] * cos(phase);")],
    "coil offset dropped": [("rD + b * M, iD + b * M", "rD, iD")],
    "forward sign": [("double phase = -TWO_PI * ((double)kx[m] * x[n]",
                      "double phase = TWO_PI * ((double)kx[m] * x[n]")],
    "2*pi missing": [("static const double TWO_PI = 6.283185307179586476925286766559;",
                      "static const double TWO_PI = 1.0;")],
}


def _pin_calls():
    """(name, zero-arg callable) for every pin, expanding parametrize marks."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        marks = getattr(fn, "pytestmark", [])
        cases = [{}]
        for mk in marks:
            if mk.name == "parametrize":
                argname, values = mk.args[0], mk.args[1]
                cases = [dict(c, **{argname: v}) for c in cases for v in values]
        for c in cases:
            kw = dict(c)
            if "golden" in params:
                kw["golden"] = read_golden
            calls.append((name, (lambda fn=fn, kw=kw: fn(**kw))))
    return calls


def _build_variant(tmp_path, edits):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    for old, new in edits:
        assert old in src, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "oracle_variant.c"
    path.write_text(src)
    return oracle.Oracle(oracle.build(force=True, src=str(path),
                                      out=str(tmp_path / "liboracle_variant.so")))


def _failing_pins(instance):
    prev = oracle.use(instance)
    failed = []
    try:
        for name, call in _pin_calls():
            try:
                call()
            except (AssertionError, IndexError, ValueError):
                failed.append(name)
    finally:
        oracle.use(prev)
    return failed


def test_unmodified_oracle_passes_every_pin(tmp_path):
    assert _failing_pins(_build_variant(tmp_path, [])) == []


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(mutant, tmp_path):
    failed = _failing_pins(_build_variant(tmp_path, MUTANTS[mutant]))
    assert failed, f"no pin caught the planted mistake: {mutant}"
