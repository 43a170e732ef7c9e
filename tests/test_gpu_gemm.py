"""The prefill GEMM (qgemm, tensor cores) against the f64 oracle.

qgemm computes the same y as qgemv, for many activation rows at once, with f16
tensor-core products of exactly decoded codes and a two-part f16 split of x.
Its results are held to the f32 dot-product bound (not to qgemv's bits), to
the workloads' 1e-3 gate, and to exact equality where every partial sum is an
exactly representable integer.  Shapes cover ragged weight-row tiles (O not a
multiple of 128), ragged activation-row tiles of all three tile widths (32,
64, 128), odd multiples of 64 inputs, and every format.
"""
import numpy as np
import pytest

from gpu_helpers import (GATE, INT3_G64, INT4_G, INT4_ROW, INT8_G, INT8_ROW, MXFP4_E8M0, MXFP4_G32, cuda, dev,
                         empty_f32, host, max_rel, packed_rows, sample_rows, scale_rows, torch)
from oracle import oracle
from weight_only_quantized_qgemv_gb300 import qgemm, qgemm_workspace, qgemv, synth

pytestmark = pytest.mark.gpu

# (fmt, gs argument, I)
SHAPES = [(INT4_G, 32, 1024), (INT4_G, 64, 1152), (INT4_G, 256, 2048), (INT4_ROW, 0, 1088),
          (INT8_ROW, 0, 1088), (INT8_G, 32, 1088), (INT8_G, 256, 2048), (INT3_G64, 0, 1024),
          (MXFP4_G32, 0, 1088), (MXFP4_E8M0, 0, 1152)]


def run_gemm(fmt, gs, w, sc, x, O, I):
    s = x.shape[0]
    y = empty_f32(s, O)
    nb = qgemm_workspace(I, s)
    ws = torch.empty(nb, dtype=torch.uint8, device=cuda())
    qgemm(fmt, gs, dev(w), dev(sc), dev(x), O, I, s, y, ws, nb)
    return host(y)


def inputs(fmt, gs, O, I, s, seed, kind="lognormal"):
    g = synth.fixed_group(fmt, I, gs or None)
    rng = synth.generator(seed, fmt, O, I, s)
    w = synth.draw_packed(fmt, O, I, rng)
    sc = synth.draw_scales(O, I, g, rng, kind, -4.0, fmt=fmt)
    x = synth.draw_x(s, I, rng)
    return g, w, sc, x


def f32_bound(fmt, g, w, sc, x, O, I):
    """|y - y*| allowed per element: the f32 dot-product bound plus the x split's 2^-22."""
    wd = oracle.dequant_f32(fmt, g, w, sc, O, I).astype(np.float64)
    cond = np.abs(x.astype(np.float64)) @ np.abs(wd).T
    return ((I + 4) * 2.0 ** -24 + 2.0 ** -20) * cond + 1e-30


@pytest.mark.parametrize("fmt,gs,I", SHAPES)
@pytest.mark.parametrize("O,s", [(1, 1), (130, 16), (77, 33), (200, 70), (129, 130)])
def test_gemm_small(fmt, gs, I, O, s):
    g, w, sc, x = inputs(fmt, gs, O, I, s, 151)
    y = run_gemm(fmt, gs, w, sc, x, O, I)
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert max_rel(y, ystar) <= GATE
    assert np.all(np.abs(y - ystar) <= f32_bound(fmt, g, w, sc, x, O, I))


@pytest.mark.parametrize("fmt,gs,I", SHAPES)
def test_gemm_integer_exact(fmt, gs, I):
    """Small-integer x and power-of-two scales: the split is exact and every sum an exact f32."""
    O, s = 131, 40
    g = synth.fixed_group(fmt, I, gs or None)
    rng = synth.generator(157, fmt, I)
    w = synth.draw_packed(fmt, O, I, rng)
    sc = synth.draw_scales(O, I, g, rng, "pow2", fmt=fmt)
    x = rng.integers(-4, 5, size=(s, I)).astype(np.float32)
    y = run_gemm(fmt, gs, w, sc, x, O, I)
    assert np.array_equal(y.astype(np.float64), oracle.qgemv(fmt, g, w, sc, x, O, I))


def test_gemm_row_scaling():
    """Rows of very different magnitudes each keep their relative accuracy (per-row power of two)."""
    fmt, gs, O, I, s = INT4_G, 32, 96, 1024, 6
    g, w, sc, x = inputs(fmt, gs, O, I, s, 163)
    x = x * np.array([1e-30, 1e-8, 1.0, 1e8, 1e30, 0.0], dtype=np.float32)[:, None]
    y = run_gemm(fmt, gs, w, sc, x, O, I)
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert np.isfinite(y).all()
    assert not y[5].any()
    assert max_rel(y[:5], ystar[:5]) <= GATE
    assert np.all(np.abs(y - ystar) <= f32_bound(fmt, g, w, sc, x, O, I))


def test_gemm_rows_at_the_range_edges():
    """Rows near the ends of the split's range: largest magnitudes around 1e36
    and 1e37 (the split takes p near -105 and -109) and around 1e-33 (p near
    124) keep the f32 bound; a zero row gives zeros."""
    fmt, gs, O, I, s = INT4_G, 32, 130, 1024, 5
    g, w, sc, x = inputs(fmt, gs, O, I, s, 171)
    x = x * np.array([1e36, 1e37 / 4.0, 1e-33, 3e-33, 0.0], dtype=np.float32)[:, None]
    assert np.isfinite(x).all()
    y = run_gemm(fmt, gs, w, sc, x, O, I)
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert np.isfinite(y).all()
    assert not y[4].any()
    assert max_rel(y[:4], ystar[:4]) <= GATE
    assert np.all(np.abs(y - ystar) <= f32_bound(fmt, g, w, sc, x, O, I))


def test_gemm_agrees_with_gemv():
    """Same inputs through qgemv (groups of 8 rows) and qgemm: within the bound of each other."""
    fmt, gs, O, I, s = MXFP4_G32, 0, 300, 2048, 48
    g, w, sc, x = inputs(fmt, gs, O, I, s, 167)
    a = run_gemm(fmt, gs, w, sc, x, O, I)
    b = empty_f32(s, O)
    qgemv(fmt, gs, dev(w), dev(sc), dev(x), O, I, s, b)
    assert max_rel(a, host(b)) <= 1e-5


@pytest.mark.parametrize("name", ["int4_g32_16384x6144_s32_prefill", "int4_g32_16384x6144_s512_prefill"])
def test_gemm_full_size_sampled(name):
    """The prefill workloads the bench times (the int4-g32 16384 x 6144 matrix,
    32 and 512 activation rows, the same inputs), sampled rows against the oracle."""
    wl = synth.workload(name)
    w, sc = wl.weights()
    x = wl.x()
    assert wl.gemm and x.shape == (wl.s, wl.I)
    y = run_gemm(wl.fmt, wl.gs, w, sc, x, wl.O, wl.I)
    assert np.isfinite(y).all()
    rows = sample_rows(wl.O, 48)
    ystar = oracle.qgemv(wl.fmt, wl.gs, packed_rows(wl.fmt, w, wl.O, wl.I, rows), scale_rows(sc, wl.O, rows), x,
                         len(rows), wl.I)
    assert max_rel(y[:, rows], ystar) <= GATE


def test_gemm_repeatable():
    fmt, gs, O, I, s = INT4_G, 32, 260, 2048, 100
    g, w, sc, x = inputs(fmt, gs, O, I, s, 173)
    a = run_gemm(fmt, gs, w, sc, x, O, I)
    b = run_gemm(fmt, gs, w, sc, x, O, I)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("fmt,gs,O,I,s", [(INT3_G64, 0, 6144, 16384, 64), (MXFP4_E8M0, 0, 2048, 6144, 256),
                                          (INT8_ROW, 0, 1024, 1024, 300)])
def test_gemm_workload_shapes_sampled(fmt, gs, O, I, s):
    """Longer rows and the other workloads' shapes, sampled rows against the oracle."""
    g = synth.fixed_group(fmt, I, gs or None)
    rng = synth.generator(199, fmt, O, I, s)
    w = synth.draw_packed(fmt, O, I, rng)
    sc = synth.draw_scales(O, I, g, rng, "lognormal", -4.0, fmt=fmt)
    x = synth.draw_x(s, I, rng)
    y = run_gemm(fmt, gs, w, sc, x, O, I)
    rows = sample_rows(O, 40)
    ystar = oracle.qgemv(fmt, g, packed_rows(fmt, w, O, I, rows), scale_rows(sc, O, rows), x, len(rows), I)
    assert max_rel(y[:, rows], ystar) <= GATE


@pytest.mark.parametrize("fmt,gs", [(INT4_G, 32), (INT3_G64, 0)])
def test_gemm_longest_rows(fmt, gs):
    """The longest rows qgemm takes (2^20 inputs): 16384 steps along K in one CTA.

    At this length the worst-case f32 bound is looser than the gate itself,
    so the gate alone is checked."""
    O, I, s = 130, 1 << 20, 3
    g, w, sc, x = inputs(fmt, gs, O, I, s, 223)
    y = run_gemm(fmt, gs, w, sc, x, O, I)
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert np.isfinite(y).all()
    assert max_rel(y, ystar) <= GATE


def test_gemm_most_activation_rows():
    """The most activation rows qgemm takes (65536): 512 column tiles of 128 rows."""
    fmt, gs, O, I, s = INT4_G, 32, 96, 128, 1 << 16
    g, w, sc, x = inputs(fmt, gs, O, I, s, 227)
    y = run_gemm(fmt, gs, w, sc, x, O, I)
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert max_rel(y, ystar) <= GATE
    assert np.all(np.abs(y - ystar) <= f32_bound(fmt, g, w, sc, x, O, I))
