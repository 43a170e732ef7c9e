"""Step a4 on the GPU: qgate_up (silu(gate x) * (up x), x read once) against the oracle."""
import numpy as np
import pytest

from gpu_helpers import GATE, INT3_G64, INT4_G, INT8_ROW, MXFP4_G32, dev, empty_f32, host, max_rel, \
    packed_rows, sample_rows, scale_rows
from bounds import glu_bound
from oracle import oracle
from weight_only_quantized_qgemv_gb300 import qgate_up, synth

pytestmark = pytest.mark.gpu


def run(fmt, gs, wg, sg, wu, su, x, F, D):
    s = x.shape[0]
    h = empty_f32(s, F)
    qgate_up(fmt, gs, dev(wg), dev(sg), dev(wu), dev(su), dev(x), F, D, s, h)
    return host(h)


@pytest.mark.parametrize("fmt,gs,D", [(INT8_ROW, 0, 528), (INT4_G, 32, 1184), (INT4_G, 64, 2048),
                                      (INT3_G64, 0, 2112), (MXFP4_G32, 0, 1184)])
@pytest.mark.parametrize("F,s", [(1, 1), (37, 1), (130, 2), (61, 5), (33, 9)])
def test_gate_up_small(fmt, gs, D, F, s):
    g = synth.fixed_group(fmt, D, gs or None)
    rng = synth.generator(23, fmt, F, D, s)
    wg, wu = synth.draw_packed(fmt, F, D, rng), synth.draw_packed(fmt, F, D, rng)
    sg = synth.draw_scales(F, D, g, rng, "lognormal", -4.0)
    su = synth.draw_scales(F, D, g, rng, "lognormal", -4.0)
    x = synth.draw_x(s, D, rng)
    h = run(fmt, gs, wg, sg, wu, su, x, F, D)
    hstar = oracle.qgate_up(fmt, g, wg, sg, wu, su, x, F, D)
    assert max_rel(h, hstar) <= GATE


@pytest.mark.parametrize("fmt,scale_kind", [(INT4_G, "lognormal"), (MXFP4_G32, "pow2")])
def test_gate_up_expert_size(fmt, scale_kind):
    F, D, s = 2048, 6144, 1
    rng = synth.generator(29, fmt)
    wg, wu = synth.draw_packed(fmt, F, D, rng), synth.draw_packed(fmt, F, D, rng)
    sg = synth.draw_scales(F, D, 32, rng, scale_kind, -4.0)
    su = synth.draw_scales(F, D, 32, rng, scale_kind, -4.0)
    x = synth.draw_x(s, D, rng)
    h = run(fmt, 32 if fmt == INT4_G else 0, wg, sg, wu, su, x, F, D)
    rows = sample_rows(F, 64)
    pg, ps_g, pu, ps_u = (packed_rows(fmt, wg, F, D, rows), scale_rows(sg, F, rows), packed_rows(fmt, wu, F, D, rows),
                          scale_rows(su, F, rows))
    hstar = oracle.qgate_up(fmt, 32, pg, ps_g, pu, ps_u, x, len(rows), D)
    assert max_rel(h[:, rows], hstar) <= GATE
    # every sampled element within the bound the pre-activation f32 sums propagate through silu
    _, b = glu_bound(fmt, 32, pg, ps_g, pu, ps_u, x, len(rows), D)
    assert np.all(np.abs(h[:, rows] - hstar) <= b)
