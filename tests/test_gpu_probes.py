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


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_mma_probe(mri, mode):
    """12 MMAs of 128 x 256 x 16 per 32 x 128 x 128 tile: at most 8192 f16
    flops per SM per clock, i.e. 8192 / 24 = 341 pairs."""
    r = mri.mma_probe(mode, tiles=512, b_tiles=64)
    assert 50.0 < r["pairs_per_sm_per_clk"] <= 342.0, r
    assert mri.device_errors(clear=True) == 0
