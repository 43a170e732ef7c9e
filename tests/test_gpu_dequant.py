"""Steps a1 + a2 on the GPU: qdequant against the oracle, bit for bit."""
import numpy as np
import pytest

from gpu_helpers import INT3_G64, INT4_G, INT8_ROW, MXFP4_G32, dev, empty_f32, host, packed_rows, \
    sample_rows, scale_rows
from oracle import oracle
from weight_only_quantized_qgemv_gb300 import qdequant, synth

pytestmark = pytest.mark.gpu

CASES = [(INT8_ROW, 0, 16), (INT8_ROW, 0, 1040), (INT4_G, 32, 32), (INT4_G, 32, 1184), (INT4_G, 64, 1152),
         (INT4_G, 128, 2048), (INT3_G64, 0, 64), (INT3_G64, 0, 1216), (MXFP4_G32, 0, 32), (MXFP4_G32, 0, 1184)]


@pytest.mark.parametrize("fmt,gs,I", CASES)
def test_dequant_bit_exact(fmt, gs, I):
    O = 37
    g = synth.fixed_group(fmt, I, gs or None)
    rng = synth.generator(7, fmt, I)
    w = synth.draw_packed(fmt, O, I, rng)
    if fmt == INT8_ROW:
        w = rng.integers(0, 256, size=O * I, dtype=np.uint8)      # every byte value, -128 included
    sc = rng.lognormal(-4, 3.0, size=O * (I // g)).astype(np.float32)
    sc[0], sc[1], sc[-1] = np.float32(1e-41), np.float32(0.0), np.float32(-1e30)   # subnormal, zero, negative
    out = empty_f32(O, I)
    qdequant(fmt, gs, dev(w), dev(sc), O, I, out)
    got = host(out)
    want = oracle.dequant_f32(fmt, g, w, sc, O, I)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("name", ["int8_row_1024x1024_s1", "int4_g32_16384x6144_s1", "int3_g64_6144x16384_s1"])
def test_dequant_full_size_sampled_rows(name):
    wl = synth.workload(name)
    w, sc = wl.weights()
    out = empty_f32(wl.O, wl.I)
    qdequant(wl.fmt, wl.gs if wl.fmt == INT4_G else 0, dev(w), dev(sc), wl.O, wl.I, out)
    rows = sample_rows(wl.O, 24)
    got = host(out)[rows]
    want = oracle.dequant_f32(wl.fmt, wl.gs, packed_rows(wl.fmt, w, wl.O, wl.I, rows), scale_rows(sc, wl.O, rows),
                              len(rows), wl.I)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_dequant_mxfp4_every_code():
    # every byte value once: both nibble positions see all 16 e2m1 codes
    O, I = 1, 512
    w = np.arange(256, dtype=np.uint8)
    sc = np.ones(I // 32, dtype=np.float32)
    out = empty_f32(O, I)
    qdequant(MXFP4_G32, 0, dev(w), dev(sc), O, I, out)
    want = oracle.dequant_f32(MXFP4_G32, 32, w, sc, O, I)
    assert np.array_equal(host(out).view(np.uint32), want.view(np.uint32))
