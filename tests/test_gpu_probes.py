"""Unit-rate probes (include/mri_microbench.h) on the GPU: they run, leave no
device error, and report rates inside what an sm_103 SM can deliver."""

import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mri():
    from non_cartesian_mri_gb300 import build
    build.build()
    import non_cartesian_mri_gb300 as m
    return m


def test_ffma_probe(mri):
    r = mri.microbench("ffma", ctas_per_sm=1, threads=1024, iters=1 << 10)
    assert 32.0 < r["per_sm_per_clk"] <= 130.0


def test_ffma2_and_sfu_probes(mri):
    """Packed pairs deliver (at most) the FMA pipe's 128 results per SM per
    clock, like scalar FMAs: the pair instruction saves issue slots, not pipe
    cycles.  The SFU gives 16 sin or cos per SM per clock."""
    r2 = mri.microbench("ffma2", iters=1 << 10)["per_sm_per_clk"]
    assert 32.0 < r2 <= 130.0
    for probe in ("sin", "cos"):
        r = mri.microbench(probe, iters=1 << 10)["per_sm_per_clk"]
        assert 8.0 < r <= 17.0, probe


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_mma_probe(mri, mode):
    """12 MMAs of 128 x 256 x 16 per 32 x 128 x 128 tile: at most 8192 f16
    flops per SM per clock, i.e. 8192 / 24 = 341 pairs."""
    r = mri.mma_probe(mode, tiles=512, b_tiles=64)
    assert 50.0 < r["pairs_per_sm_per_clk"] <= 342.0, r
    assert mri.device_errors(clear=True) == 0
