"""The GPU parity tests' own helpers, checked on the CPU: the row slices that
feed the oracle sampled rows of a full matrix, and the error measure."""
import numpy as np
import pytest

from gpu_helpers import max_rel, packed_rows, sample_rows, scale_rows
from oracle import oracle
from weight_only_quantized_qgemv_gb300 import synth

FMTS = [(synth.INT8_ROW, None), (synth.INT8_G, 64), (synth.INT4_ROW, None), (synth.INT4_G, 32),
        (synth.INT3_G64, None), (synth.MXFP4_G32, None), (synth.MXFP4_E8M0, None)]


@pytest.mark.parametrize("fmt,gs", FMTS)
def test_row_slices_equal_the_oracles_row_sample(fmt, gs):
    """oracle.qgemv on the sliced rows = the oracle's own row-sampled GEMV of the whole matrix, bit for bit."""
    O, I, s = 37, 256, 3
    g = synth.fixed_group(fmt, I, gs)
    rng = synth.generator(31, fmt)
    w = synth.draw_packed(fmt, O, I, rng)
    sc = synth.draw_scales(O, I, g, rng, "pow2" if fmt == synth.MXFP4_E8M0 else "lognormal", fmt=fmt)
    x = synth.draw_x(s, I, rng)
    rows = sample_rows(O, 10)
    got = oracle.qgemv(fmt, g, packed_rows(fmt, w, O, I, rows), scale_rows(sc, O, rows), x, len(rows), I)
    want = oracle.qgemv_rows(fmt, g, w, sc, x, O, I, rows)
    assert np.array_equal(got, want)
    full = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert np.array_equal(got, full[:, rows])


def test_sample_rows_holds_the_edges():
    rows = sample_rows(1000, 20)
    assert {0, 1, 998, 999, 500} <= set(rows.tolist())
    assert np.all(np.diff(rows) > 0) and rows.min() >= 0 and rows.max() < 1000
    assert np.array_equal(sample_rows(5, 20), np.arange(5))


def test_max_rel_is_per_output_vector():
    """max_o |y - y*| / max_o |y*|, the worst over the output vectors."""
    ystar = np.array([[1.0, -4.0, 2.0], [0.01, 0.0, 0.02]])
    y = ystar.copy()
    y[0, 0] += 0.004                 # 0.004 / 4 = 1e-3 in vector 0
    y[1, 1] += 0.00001               # 1e-5 / 0.02 = 5e-4 in vector 1
    assert max_rel(y, ystar) == pytest.approx(1e-3)
    y[1, 1] += 0.00003               # 4e-5 / 0.02 = 2e-3 in vector 1: the worst
    assert max_rel(y, ystar) == pytest.approx(2e-3)
