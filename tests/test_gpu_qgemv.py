"""Step a3 on the GPU: qgemv against the f64 oracle.

Small ragged sizes cover several tiles, partial warp steps (I not a multiple
of 32 chunks), row tails and token counts above one launch's 8.  The full
workload sizes run in the launch configuration the bench times and are
compared on sampled rows.  Integer-exact inputs must match bit for bit.
"""
import numpy as np
import pytest

from gpu_helpers import GATE, INT3_G64, INT4_G, INT8_ROW, MXFP4_G32, dev, empty_f32, host, max_rel, \
    packed_rows, sample_rows, scale_rows
from bounds import gemv_bound
from oracle import oracle
from weight_only_quantized_qgemv_gb300 import qgemv, synth

pytestmark = pytest.mark.gpu

# (fmt, gs argument, I): I spans one warp step, several, and a ragged last step.
SHAPES = [(INT8_ROW, 0, 16), (INT8_ROW, 0, 528), (INT8_ROW, 0, 1040),
          (INT4_G, 32, 32), (INT4_G, 32, 1184), (INT4_G, 32, 2080), (INT4_G, 64, 1152), (INT4_G, 128, 4096),
          (INT3_G64, 0, 64), (INT3_G64, 0, 2112), (INT3_G64, 0, 4160),
          (MXFP4_G32, 0, 32), (MXFP4_G32, 0, 1184), (MXFP4_G32, 0, 2080)]


def run_gemv(fmt, gs, w, sc, x, O, I):
    s = x.shape[0]
    y = empty_f32(s, O)
    qgemv(fmt, gs, dev(w), dev(sc), dev(x), O, I, s, y)
    return host(y)


def inputs(fmt, gs, O, I, s, seed):
    g = synth.fixed_group(fmt, I, gs or None)
    rng = synth.generator(seed, fmt, O, I, s)
    w = synth.draw_packed(fmt, O, I, rng)
    sc = synth.draw_scales(O, I, g, rng, "lognormal", -4.0)
    x = synth.draw_x(s, I, rng)
    return g, w, sc, x


@pytest.mark.parametrize("fmt,gs,I", SHAPES)
@pytest.mark.parametrize("O,s", [(1, 1), (37, 1), (130, 2), (77, 3), (200, 4), (45, 8), (29, 11)])
def test_qgemv_small(fmt, gs, I, O, s):
    g, w, sc, x = inputs(fmt, gs, O, I, s, 11)
    y = run_gemv(fmt, gs, w, sc, x, O, I)
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert max_rel(y, ystar) <= GATE
    # condition-aware bound of an f32 dot product of I terms in any order
    wd = oracle.dequant_f32(fmt, g, w, sc, O, I).astype(np.float64)
    cond = np.abs(x.astype(np.float64)) @ np.abs(wd).T
    assert np.all(np.abs(y - ystar) <= (I + 4) * 2.0 ** -24 * cond + 1e-30)


@pytest.mark.parametrize("fmt,gs,I", SHAPES)
def test_qgemv_integer_exact(fmt, gs, I):
    """Small-integer x and power-of-two scales: every partial sum is exact in f32."""
    O, s = 67, 3
    g = synth.fixed_group(fmt, I, gs or None)
    rng = synth.generator(13, fmt, I)
    w = synth.draw_packed(fmt, O, I, rng)
    sc = synth.draw_scales(O, I, g, rng, "pow2")
    x = rng.integers(-4, 5, size=(s, I)).astype(np.float32)
    y = run_gemv(fmt, gs, w, sc, x, O, I)
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert np.array_equal(y.astype(np.float64), ystar)


@pytest.mark.parametrize("fmt,gs,I", [(INT4_G, 32, 1184), (INT3_G64, 0, 2112), (MXFP4_G32, 0, 1184),
                                      (INT8_ROW, 0, 528)])
def test_qgemv_zero_scales_and_zero_x(fmt, gs, I):
    O, s = 50, 2
    g, w, sc, x = inputs(fmt, gs, O, I, s, 17)
    assert not run_gemv(fmt, gs, w, np.zeros_like(sc), x, O, I).any()
    assert not run_gemv(fmt, gs, w, sc, np.zeros_like(x), O, I).any()


def test_qgemv_linearity():
    fmt, gs, O, I = INT4_G, 32, 300, 2048
    g, w, sc, x = inputs(fmt, gs, O, I, 2, 19)
    y = run_gemv(fmt, gs, w, sc, x, O, I)
    y2 = run_gemv(fmt, gs, w, sc, np.float32(-0.5) * x, O, I)
    assert np.array_equal(y2, np.float32(-0.5) * y)       # power-of-two scaling is exact


@pytest.mark.parametrize("name", ["int8_row_1024x1024_s1", "int4_g32_16384x6144_s1", "int4_g32_16384x6144_s4",
                                  "int3_g64_6144x16384_s1"])
def test_qgemv_full_size_sampled(name):
    wl = synth.workload(name)
    w, sc = wl.weights()
    x = wl.x()
    y = run_gemv(wl.fmt, wl.gs if wl.fmt == INT4_G else 0, w, sc, x, wl.O, wl.I)
    assert np.isfinite(y).all()
    rows = sample_rows(wl.O, 96)
    pw, ps = packed_rows(wl.fmt, w, wl.O, wl.I, rows), scale_rows(sc, wl.O, rows)
    ystar = oracle.qgemv(wl.fmt, wl.gs, pw, ps, x, len(rows), wl.I)
    assert max_rel(y[:, rows], ystar) <= GATE
    # and every sampled element within the f32 dot-product bound of its own row
    assert np.all(np.abs(y[:, rows] - ystar) <= gemv_bound(wl.fmt, wl.gs, pw, ps, x, len(rows), wl.I))


def test_qgemv_full_size_repeatable():
    """Same inputs, same bits: the summation order is fixed per launch shape."""
    wl = synth.workload("int4_g32_16384x6144_s1")
    w, sc = wl.weights()
    x = wl.x()
    a = run_gemv(wl.fmt, wl.gs, w, sc, x, wl.O, wl.I)
    b = run_gemv(wl.fmt, wl.gs, w, sc, x, wl.O, wl.I)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fmt,gs,I", [(INT8_ROW, 0, 1040), (INT4_G, 32, 2080), (INT3_G64, 0, 2112),
                                      (MXFP4_G32, 0, 2080)])
def test_qgemv_row_bits_do_not_depend_on_batch(fmt, gs, I):
    """An activation row gets the same bits alone as in a batch of 5 (colibri's
    expert tier states the same of its per-row GEMV)."""
    O, s = 130, 5
    g, w, sc, x = inputs(fmt, gs, O, I, s, 29)
    ys = run_gemv(fmt, gs, w, sc, x, O, I)
    for t in range(s):
        y1 = run_gemv(fmt, gs, w, sc, x[t:t + 1], O, I)
        assert np.array_equal(y1[0], ys[t])


@pytest.mark.parametrize("fmt,gs,I", [(INT4_G, 32, 36864), (INT3_G64, 0, 43008), (INT8_ROW, 0, 36864),
                                      (MXFP4_G32, 0, 36864)])
def test_qgemv_longest_rows(fmt, gs, I):
    """Rows at the shared-memory staging limit (about 37,000 inputs; int3 43,000), ragged O, s = 1 and 3."""
    for O, s in [(100, 1), (33, 3)]:
        g, w, sc, x = inputs(fmt, gs, O, I, s, 211)
        y = run_gemv(fmt, gs, w, sc, x, O, I)
        assert max_rel(y, oracle.qgemv(fmt, g, w, sc, x, O, I)) <= GATE


def test_qgemv_rows_past_the_limit_are_rejected():
    from weight_only_quantized_qgemv_gb300 import QStatusError
    fmt, gs, O, I, s = INT4_G, 32, 8, 40960, 1
    g, w, sc, x = inputs(fmt, gs, O, I, s, 223)
    with pytest.raises(QStatusError) as e:
        run_gemv(fmt, gs, w, sc, x, O, I)
    assert e.value.status == -2
