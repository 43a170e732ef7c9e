"""Both streaming kernels against each other and against the f64 oracle.

The library has two kernels for the same contraction: the per-lane copy ring
kernel and the tensor-copy tile kernel (qkernel_policy selects).  Every lane
accumulates its chunks in the same order in both, and the cross-lane sums take
the same butterfly, so the two must agree bit for bit; each must also pass the
oracle gate on its own.  Shapes cover ragged last slices (I not a multiple of
one warp step), tails of row tiles and several activation rows.
"""
import numpy as np
import pytest

from gpu_helpers import GATE, INT3_G64, INT4_G, INT8_ROW, MXFP4_G32, dev, empty_f32, host, max_rel
from oracle import oracle
from test_gpu_expert_group import oracle_group, run_group, small_store
from test_gpu_qgemv import inputs, run_gemv
from weight_only_quantized_qgemv_gb300 import _lib, qgate_up, synth

pytestmark = pytest.mark.gpu


def with_policy(policy, fn):
    prev = _lib.qkernel_policy(policy)
    try:
        return fn()
    finally:
        _lib.qkernel_policy(prev)


SHAPES = [(INT8_ROW, 0, 528), (INT8_ROW, 0, 1040), (INT4_G, 32, 1184), (INT4_G, 32, 6144), (INT4_G, 64, 1152),
          (INT4_G, 256, 4096), (INT3_G64, 0, 2112), (INT3_G64, 0, 4160), (MXFP4_G32, 0, 1184),
          (MXFP4_G32, 0, 2080)]


@pytest.mark.parametrize("fmt,gs,I", SHAPES)
@pytest.mark.parametrize("O,s", [(37, 1), (301, 1), (130, 2), (77, 4), (45, 8)])
def test_qgemv_ring_and_tile_agree(fmt, gs, I, O, s):
    g, w, sc, x = inputs(fmt, gs, O, I, s, 41)
    y_ring = with_policy(_lib.QKERNEL_RING, lambda: run_gemv(fmt, gs, w, sc, x, O, I))
    y_tile = with_policy(_lib.QKERNEL_TILE, lambda: run_gemv(fmt, gs, w, sc, x, O, I))
    assert np.array_equal(y_ring.view(np.uint32), y_tile.view(np.uint32))
    assert max_rel(y_tile, oracle.qgemv(fmt, g, w, sc, x, O, I)) <= GATE


@pytest.mark.parametrize("fmt,gs,D", [(INT4_G, 32, 1184), (INT3_G64, 0, 2112), (MXFP4_G32, 0, 2080),
                                      (INT8_ROW, 0, 528)])
@pytest.mark.parametrize("F,s", [(61, 1), (130, 3)])
def test_gate_up_ring_and_tile_agree(fmt, gs, D, F, s):
    g = synth.fixed_group(fmt, D, gs or None)
    rng = synth.generator(43, fmt, F, D, s)
    wg, wu = synth.draw_packed(fmt, F, D, rng), synth.draw_packed(fmt, F, D, rng)
    sg = synth.draw_scales(F, D, g, rng, "lognormal", -4.0)
    su = synth.draw_scales(F, D, g, rng, "lognormal", -4.0)
    x = synth.draw_x(s, D, rng)

    def run():
        h = empty_f32(s, F)
        qgate_up(fmt, gs, dev(wg), dev(sg), dev(wu), dev(su), dev(x), F, D, s, h)
        return host(h)

    h_ring = with_policy(_lib.QKERNEL_RING, run)
    h_tile = with_policy(_lib.QKERNEL_TILE, run)
    assert np.array_equal(h_ring.view(np.uint32), h_tile.view(np.uint32))
    assert max_rel(h_tile, oracle.qgate_up(fmt, g, wg, sg, wu, su, x, F, D)) <= GATE


@pytest.mark.parametrize("fmt,gs", [(INT8_ROW, 0), (INT4_G, 32), (INT3_G64, 0), (MXFP4_G32, 0)])
@pytest.mark.parametrize("E,s,k", [(6, 1, 4), (5, 8, 4), (64, 8, 8)])
def test_expert_group_ring_and_tile_agree(fmt, gs, E, s, k):
    D, F = 256, 128
    st = small_store(fmt, E, D, F, 47)
    rng = synth.generator(53, fmt, E, s, k)
    x = synth.draw_x(s, D, rng)
    ids = rng.integers(0, E, size=(s, k)).astype(np.int32)
    wts = rng.random((s, k)).astype(np.float32)
    out_ring, st_ring = with_policy(_lib.QKERNEL_RING, lambda: run_group(fmt, gs, st, E, D, F, x, ids, wts))
    out_tile, st_tile = with_policy(_lib.QKERNEL_TILE, lambda: run_group(fmt, gs, st, E, D, F, x, ids, wts))
    assert st_ring == 0 and st_tile == 0
    assert np.array_equal(out_ring.view(np.uint32), out_tile.view(np.uint32))
    want = oracle_group(fmt, synth.fixed_group(fmt, D, gs or None), st, E, D, F, x, ids, wts)
    assert max_rel(out_tile, want) <= GATE


ROW_SHAPES = [(INT8_ROW, 0, 1024), (INT8_ROW, 0, 2048), (INT4_G, 32, 1024), (INT4_G, 32, 6144), (INT4_G, 64, 2048),
              (INT4_G, 128, 4096), (INT3_G64, 0, 2048), (INT3_G64, 0, 16384), (MXFP4_G32, 0, 1024),
              (MXFP4_G32, 0, 6144)]


@pytest.mark.parametrize("fmt,gs,I", ROW_SHAPES)
@pytest.mark.parametrize("O", [1, 37, 301, 1000])
def test_qgemv_row_team_kernel(fmt, gs, I, O):
    """The row-team kernel (forced; one activation row, rows of whole warp
    steps) against the oracle: the gate, the per-element f32 bound, and the
    same bits on a second call."""
    from bounds import gemv_bound
    g, w, sc, x = inputs(fmt, gs, O, I, 1, 59)
    y = with_policy(_lib.QKERNEL_ROW, lambda: run_gemv(fmt, gs, w, sc, x, O, I))
    y2 = with_policy(_lib.QKERNEL_ROW, lambda: run_gemv(fmt, gs, w, sc, x, O, I))
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert max_rel(y, ystar) <= GATE
    assert np.all(np.abs(y - ystar) <= gemv_bound(fmt, g, w, sc, x, O, I))
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("fmt,gs,D", [(INT4_G, 32, 2048), (MXFP4_G32, 0, 6144), (INT3_G64, 0, 2048),
                                      (INT8_ROW, 0, 1024)])
@pytest.mark.parametrize("F", [7, 130])
def test_gate_up_row_team_kernel(fmt, gs, D, F):
    from bounds import glu_bound
    g = synth.fixed_group(fmt, D, gs or None)
    rng = synth.generator(61, fmt, F, D)
    wg, wu = synth.draw_packed(fmt, F, D, rng), synth.draw_packed(fmt, F, D, rng)
    sg = synth.draw_scales(F, D, g, rng, "lognormal", -4.0)
    su = synth.draw_scales(F, D, g, rng, "lognormal", -4.0)
    x = synth.draw_x(1, D, rng)

    def run():
        h = empty_f32(1, F)
        qgate_up(fmt, gs, dev(wg), dev(sg), dev(wu), dev(su), dev(x), F, D, 1, h)
        return host(h)

    h = with_policy(_lib.QKERNEL_ROW, run)
    hstar = oracle.qgate_up(fmt, g, wg, sg, wu, su, x, F, D)
    assert max_rel(h, hstar) <= GATE
    _, b = glu_bound(fmt, g, wg, sg, wu, su, x, F, D)
    assert np.all(np.abs(h - hstar) <= b)
