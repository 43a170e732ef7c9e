"""The storage variants on the GPU: int4 per row, int8 grouped and MXFP4 with
ue8m0 scale bytes, against the oracle.

They reuse the int4, int8 and e2m1 decoders and change only where the scale
comes from, so besides the oracle comparisons the checks here tie them to the
base formats: ue8m0 bytes 127 + k must give the same bits as f32 scales 2^k,
and both streaming kernels the same bits.
"""
import numpy as np
import pytest

from gpu_helpers import (GATE, INT4_ROW, INT8_G, MXFP4_E8M0, MXFP4_G32, cuda, dev, empty_f32, host, max_rel,
                         packed_rows, sample_rows, scale_rows, torch)
from bounds import expert_bound, gemv_bound
from oracle import oracle
from test_gpu_expert_group import run_group, small_store
from weight_only_quantized_qgemv_gb300 import (QACT_SWIGLU_CLAMPED, _lib, qdequant, qgate_up, qgate_up_act, qgemv,
                                               synth)

pytestmark = pytest.mark.gpu

# (fmt, gs argument, I): one warp step, several, ragged last steps; I % 512 == 0
# lets the ue8m0 scale rows go through the tensor-copy kernel, other I use the
# per-lane copy kernel.
SHAPES = [(INT4_ROW, 0, 32), (INT4_ROW, 0, 1184), (INT4_ROW, 0, 2080),
          (INT8_G, 16, 528), (INT8_G, 64, 1152), (INT8_G, 32, 2080), (INT8_G, 512, 2048), (INT8_G, 128, 4096),
          (MXFP4_E8M0, 0, 128), (MXFP4_E8M0, 0, 1152), (MXFP4_E8M0, 0, 2048), (MXFP4_E8M0, 0, 4224)]


def inputs(fmt, gs, O, I, s, seed, kind="lognormal"):
    g = synth.fixed_group(fmt, I, gs or None)
    rng = synth.generator(seed, fmt, O, I, s)
    w = synth.draw_packed(fmt, O, I, rng)
    sc = synth.draw_scales(O, I, g, rng, kind, -4.0, fmt=fmt)
    x = synth.draw_x(s, I, rng)
    return g, w, sc, x


def run_gemv(fmt, gs, w, sc, x, O, I):
    s = x.shape[0]
    y = empty_f32(s, O)
    qgemv(fmt, gs, dev(w), dev(sc), dev(x), O, I, s, y)
    return host(y)


def with_policy(policy, fn):
    prev = _lib.qkernel_policy(policy)
    try:
        return fn()
    finally:
        _lib.qkernel_policy(prev)


@pytest.mark.parametrize("fmt,gs,I", SHAPES)
@pytest.mark.parametrize("O,s", [(1, 1), (37, 1), (130, 2), (77, 3), (45, 8), (29, 11)])
def test_variant_qgemv_small(fmt, gs, I, O, s):
    g, w, sc, x = inputs(fmt, gs, O, I, s, 101)
    y = run_gemv(fmt, gs, w, sc, x, O, I)
    ystar = oracle.qgemv(fmt, g, w, sc, x, O, I)
    assert max_rel(y, ystar) <= GATE
    wd = oracle.dequant_f32(fmt, g, w, sc, O, I).astype(np.float64)
    cond = np.abs(x.astype(np.float64)) @ np.abs(wd).T
    assert np.all(np.abs(y - ystar) <= (I + 4) * 2.0 ** -24 * cond + 1e-30)


@pytest.mark.parametrize("fmt,gs,I", SHAPES)
def test_variant_qgemv_integer_exact(fmt, gs, I):
    """Small-integer x and power-of-two scales: every partial sum is exact in f32."""
    O, s = 67, 3
    g = synth.fixed_group(fmt, I, gs or None)
    rng = synth.generator(103, fmt, I)
    w = synth.draw_packed(fmt, O, I, rng)
    sc = synth.draw_scales(O, I, g, rng, "pow2", fmt=fmt)
    x = rng.integers(-4, 5, size=(s, I)).astype(np.float32)
    y = run_gemv(fmt, gs, w, sc, x, O, I)
    assert np.array_equal(y.astype(np.float64), oracle.qgemv(fmt, g, w, sc, x, O, I))


@pytest.mark.parametrize("fmt,gs,I", SHAPES)
def test_variant_dequant_bitexact(fmt, gs, I):
    O = 19
    g, w, sc, _ = inputs(fmt, gs, O, I, 1, 107)
    out = empty_f32(O, I)
    qdequant(fmt, gs, dev(w), dev(sc), O, I, out)
    want = oracle.dequant_f32(fmt, g, w, sc, O, I)
    assert np.array_equal(host(out).view(np.uint32), want.view(np.uint32))


def e8m0_and_f32(O, I, rng):
    """ue8m0 bytes 127 + k and the f32 scales 2^k they stand for, k in [-8, 0]."""
    k = rng.integers(-8, 1, size=O * (I // 32))
    return (127 + k).astype(np.uint8), np.ldexp(np.ones(k.size, dtype=np.float32), k).astype(np.float32)


@pytest.mark.parametrize("I", [1152, 2048, 4224])
@pytest.mark.parametrize("O,s", [(37, 1), (130, 3), (29, 11)])
def test_e8m0_bytes_equal_expanded_f32_scales(I, O, s):
    """The host expansion of the pages' MXFP4 path and the raw bytes give the same bits."""
    rng = synth.generator(109, I, O, s)
    w = synth.draw_packed(MXFP4_G32, O, I, rng)
    b, f = e8m0_and_f32(O, I, rng)
    x = synth.draw_x(s, I, rng)
    y8 = run_gemv(MXFP4_E8M0, 0, w, b, x, O, I)
    y7 = run_gemv(MXFP4_G32, 0, w, f, x, O, I)
    assert np.array_equal(y8.view(np.uint32), y7.view(np.uint32))


def test_e8m0_extreme_bytes():
    """Bytes 0 (2^-127, an f32 subnormal), 1, 254 and 255 (NaN) decode as the
    oracle says; a NaN scale makes exactly the outputs of its row NaN."""
    O, I, s = 8, 256, 2
    rng = synth.generator(113)
    w = synth.draw_packed(MXFP4_E8M0, O, I, rng)
    b = np.full(O * I // 32, 127, dtype=np.uint8)
    b[0] = 0          # row 0, group 0
    b[9] = 1          # row 1
    b[17] = 254       # row 2
    b[3 * 8 + 5] = 255  # row 3, group 5
    b[4 * 8:5 * 8] = 0  # row 4: every scale subnormal
    out = empty_f32(O, I)
    qdequant(MXFP4_E8M0, 0, dev(w), dev(b), O, I, out)
    got, want = host(out), oracle.dequant_f32(MXFP4_E8M0, 32, w, b, O, I)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok].view(np.uint32), want[ok].view(np.uint32))
    x = synth.draw_x(s, I, rng)
    y = run_gemv(MXFP4_E8M0, 0, w, b, x, O, I)
    ystar = oracle.qgemv(MXFP4_E8M0, 32, w, b, x, O, I)
    assert np.isnan(y[:, 3]).all() and np.isnan(ystar[:, 3]).all()
    rows = np.array([0, 1, 4, 5, 6, 7])     # row 2's 2^127 scale overflows f32 products; row 3 is NaN
    assert np.isfinite(y[:, rows]).all()
    # f32 dot-product bound per element, plus one subnormal ulp (2^-149) per
    # operation for the rows whose terms are subnormal
    wd = np.abs(want[rows].astype(np.float64))
    cond = np.abs(x.astype(np.float64)) @ wd.T
    err = np.abs(y[:, rows] - ystar[:, rows])
    assert np.all(err <= (I + 4) * (2.0 ** -24 * cond + 2.0 ** -149))
    assert np.abs(y[:, 4]).max() > 0                                 # 2^-127 scales are not flushed to zero


@pytest.mark.parametrize("fmt,gs,I", [(INT4_ROW, 0, 2080), (INT8_G, 64, 2048), (INT8_G, 16, 1152),
                                      (MXFP4_E8M0, 0, 2048), (MXFP4_E8M0, 0, 2560)])
@pytest.mark.parametrize("s", [1, 3])
def test_variant_kernels_agree(fmt, gs, I, s):
    O = 130
    _, w, sc, x = inputs(fmt, gs, O, I, s, 127)
    a = with_policy(_lib.QKERNEL_RING, lambda: run_gemv(fmt, gs, w, sc, x, O, I))
    b = with_policy(_lib.QKERNEL_TILE, lambda: run_gemv(fmt, gs, w, sc, x, O, I))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def gate_up_inputs(fmt, gs, F, D, s, seed):
    g = synth.fixed_group(fmt, D, gs or None)
    rng = synth.generator(seed, fmt, F, D, s)
    wg, wu = synth.draw_packed(fmt, F, D, rng), synth.draw_packed(fmt, F, D, rng)
    sg = synth.draw_scales(F, D, g, rng, "lognormal", -4.0, fmt=fmt)
    su = synth.draw_scales(F, D, g, rng, "lognormal", -4.0, fmt=fmt)
    return g, wg, sg, wu, su, synth.draw_x(s, D, rng)


GATE_UP_SHAPES = [(INT4_ROW, 0, 1184), (INT8_G, 64, 1152), (INT8_G, 16, 2080), (MXFP4_E8M0, 0, 1152),
                  (MXFP4_E8M0, 0, 2048)]


@pytest.mark.parametrize("fmt,gs,D", GATE_UP_SHAPES)
@pytest.mark.parametrize("F,s", [(37, 1), (130, 3), (29, 9)])
def test_variant_gate_up(fmt, gs, D, F, s):
    g, wg, sg, wu, su, x = gate_up_inputs(fmt, gs, F, D, s, 131)
    h = empty_f32(s, F)
    qgate_up(fmt, gs, dev(wg), dev(sg), dev(wu), dev(su), dev(x), F, D, s, h)
    assert max_rel(host(h), oracle.qgate_up(fmt, g, wg, sg, wu, su, x, F, D)) <= GATE
    u = oracle.qgemv(fmt, g, wu, su, x, F, D)
    L = float(np.float32(np.median(np.abs(u))))
    qgate_up_act(fmt, gs, dev(wg), dev(sg), dev(wu), dev(su), dev(x), F, D, s, QACT_SWIGLU_CLAMPED, L, h)
    assert max_rel(host(h), oracle.qgate_up(fmt, g, wg, sg, wu, su, x, F, D, act=1, limit=L)) <= GATE


@pytest.mark.parametrize("fmt,gs", [(INT4_ROW, 0), (INT8_G, 32), (MXFP4_E8M0, 0)])
@pytest.mark.parametrize("E,s,k", [(6, 1, 1), (6, 1, 4), (6, 3, 2), (5, 8, 4), (64, 8, 8)])
def test_variant_expert_group(fmt, gs, E, s, k):
    D, F = 256, 128
    st = small_store(fmt, E, D, F, 137)
    rng = synth.generator(139, fmt, E, s, k)
    x = synth.draw_x(s, D, rng)
    ids = rng.integers(0, E, size=(s, k)).astype(np.int32)
    wts = rng.random((s, k)).astype(np.float32)
    out, status = run_group(fmt, gs, st, E, D, F, x, ids, wts)
    assert status == 0
    g = synth.fixed_group(fmt, D, gs or None)
    want = oracle.expert_group(fmt, g, st["gate"], st["gate_s"], st["up"], st["up_s"], st["down"], st["down_s"],
                               E, D, F, x, ids, wts)
    assert max_rel(out, want) <= GATE


@pytest.mark.parametrize("s,k", [(1, 8), (8, 8)])
def test_e8m0_expert_group_equals_expanded_f32(s, k):
    """The whole routed-expert MLP: ue8m0 bytes and their f32 expansion give the same bits."""
    E, D, F = 12, 2048, 512
    rng = synth.generator(149, s, k)
    b8, f32 = {}, {}
    for name, (O, I) in {"gate": (F, D), "up": (F, D), "down": (D, F)}.items():
        b8[name] = f32[name] = np.concatenate([synth.draw_packed(MXFP4_G32, O, I, rng) for _ in range(E)])
        pairs = [e8m0_and_f32(O, I, rng) for _ in range(E)]
        b8[name + "_s"] = np.concatenate([p[0] for p in pairs])
        f32[name + "_s"] = np.concatenate([p[1] for p in pairs])
    x = synth.draw_x(s, D, rng)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(s)]).astype(np.int32)
    wts = rng.random((s, k)).astype(np.float32)
    a, sa = run_group(MXFP4_E8M0, 0, b8, E, D, F, x, ids, wts)
    b, sb = run_group(MXFP4_G32, 0, f32, E, D, F, x, ids, wts)
    assert sa == 0 and sb == 0
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("name", ["int4_row_16384x6144_s1", "int8_g64_16384x6144_s1"])
def test_variant_full_size_sampled(name):
    """The storage-variant workloads in the launch configuration the bench times."""
    wl = synth.workload(name)
    w, sc = wl.weights()
    x = wl.x()
    y = run_gemv(wl.fmt, wl.gs if wl.fmt == INT8_G else 0, w, sc, x, wl.O, wl.I)
    assert np.isfinite(y).all()
    rows = sample_rows(wl.O, 96)
    pw, ps = packed_rows(wl.fmt, w, wl.O, wl.I, rows), scale_rows(sc, wl.O, rows)
    ystar = oracle.qgemv(wl.fmt, wl.gs, pw, ps, x, len(rows), wl.I)
    assert max_rel(y[:, rows], ystar) <= GATE
    assert np.all(np.abs(y[:, rows] - ystar) <= gemv_bound(wl.fmt, wl.gs, pw, ps, x, len(rows), wl.I))


def test_e8m0_expert_workload_full_size_sampled():
    from test_gpu_expert_group import full_store_on_device, compact_store
    wl = synth.workload("mxfp4_e8m0_experts_E256_D6144_F2048_s1_k8")
    d = full_store_on_device(wl)
    x = wl.x()
    ids, wts = wl.routing()
    out, status = run_group(wl.fmt, 0, None, wl.E, wl.D, wl.F, x, ids, wts, stores_on_device=d)
    assert status == 0 and np.isfinite(out).all()
    used = np.unique(ids)
    cids = np.vectorize({int(e): i for i, e in enumerate(used)}.get)(ids).astype(np.int32)
    cols = np.unique(np.concatenate([[0, 1, wl.D - 1], synth.generator(7).choice(wl.D, 61, replace=False)]))
    st = compact_store(wl, used)
    want = oracle.expert_group(wl.fmt, 32, st["gate"], st["gate_s"], st["up"], st["up_s"], st["down"], st["down_s"],
                               len(used), wl.D, wl.F, x, cids, wts, cols=cols)
    assert max_rel(out[:, cols], want) <= GATE
    b = expert_bound(wl.fmt, 32, 32, st, wl.D, wl.F, x, cids, wts, cols, [0])
    assert np.all(np.abs(out[:1, cols] - want) <= b)
    # the same store with its bytes expanded to f32 on the host: the same bits
    d7 = {n: (v if not n.endswith("_s") else torch.ldexp(torch.ones_like(v, dtype=torch.float32),
                                                             v.to(torch.int32) - 127)) for n, v in d.items()}
    out7, status7 = run_group(synth.MXFP4_G32, 0, None, wl.E, wl.D, wl.F, x, ids, wts, stores_on_device=d7)
    assert status7 == 0 and np.array_equal(out.view(np.uint32), out7.view(np.uint32))
