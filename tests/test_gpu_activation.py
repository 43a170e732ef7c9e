"""Clamped SwiGLU on the GPU: qgate_up_act and qexpert_group_act against the oracle.

The limit is chosen near the median |up| value so that about half of the
products are clamped; limit 0 must give zeros, an infinite limit the same
bits as plain SwiGLU, and both streaming kernels the same bits.
"""
import numpy as np
import pytest

from gpu_helpers import GATE, INT3_G64, INT4_G, INT8_ROW, MXFP4_G32, cuda, dev, empty_f32, host, max_rel, torch
from bounds import expert_bound
from oracle import oracle
from test_gpu_expert_group import small_store
from weight_only_quantized_qgemv_gb300 import (QACT_SWIGLU, QACT_SWIGLU_CLAMPED, _lib, qexpert_group_act,
                                               qexpert_group_workspace, qgate_up, qgate_up_act, synth)

pytestmark = pytest.mark.gpu

SHAPES = [(INT8_ROW, 0, 528), (INT4_G, 32, 1184), (INT4_G, 64, 2048), (INT3_G64, 0, 2112), (MXFP4_G32, 0, 1184)]


def gate_up_inputs(fmt, gs, F, D, s, seed):
    g = synth.fixed_group(fmt, D, gs or None)
    rng = synth.generator(seed, fmt, F, D, s)
    wg, wu = synth.draw_packed(fmt, F, D, rng), synth.draw_packed(fmt, F, D, rng)
    sg = synth.draw_scales(F, D, g, rng, "lognormal", -4.0)
    su = synth.draw_scales(F, D, g, rng, "lognormal", -4.0)
    x = synth.draw_x(s, D, rng)
    return g, wg, sg, wu, su, x


def run_act(fmt, gs, wg, sg, wu, su, x, F, D, act, limit):
    s = x.shape[0]
    h = empty_f32(s, F)
    qgate_up_act(fmt, gs, dev(wg), dev(sg), dev(wu), dev(su), dev(x), F, D, s, act, limit, h)
    return host(h)


@pytest.mark.parametrize("fmt,gs,D", SHAPES)
@pytest.mark.parametrize("F,s", [(37, 1), (130, 3)])
def test_gate_up_clamped(fmt, gs, D, F, s):
    g, wg, sg, wu, su, x = gate_up_inputs(fmt, gs, F, D, s, 61)
    u = oracle.qgemv(fmt, g, wu, su, x, F, D)
    L = float(np.float32(np.median(np.abs(u))))
    h = run_act(fmt, gs, wg, sg, wu, su, x, F, D, QACT_SWIGLU_CLAMPED, L)
    want = oracle.qgate_up(fmt, g, wg, sg, wu, su, x, F, D, act=1, limit=L)
    assert max_rel(h, want) <= GATE
    # the clamp bites: the plain product differs by far more than the gate
    assert max_rel(oracle.qgate_up(fmt, g, wg, sg, wu, su, x, F, D), want) > 10 * GATE
    assert not run_act(fmt, gs, wg, sg, wu, su, x, F, D, QACT_SWIGLU_CLAMPED, 0.0).any()


@pytest.mark.parametrize("fmt,gs,D", SHAPES)
def test_gate_up_infinite_limit_is_swiglu(fmt, gs, D):
    F, s = 77, 2
    g, wg, sg, wu, su, x = gate_up_inputs(fmt, gs, F, D, s, 67)
    plain = empty_f32(s, F)
    qgate_up(fmt, gs, dev(wg), dev(sg), dev(wu), dev(su), dev(x), F, D, s, plain)
    h = run_act(fmt, gs, wg, sg, wu, su, x, F, D, QACT_SWIGLU_CLAMPED, float("inf"))
    assert np.array_equal(h.view(np.uint32), host(plain).view(np.uint32))
    h0 = run_act(fmt, gs, wg, sg, wu, su, x, F, D, QACT_SWIGLU, 123.0)       # the limit is ignored
    assert np.array_equal(h0.view(np.uint32), host(plain).view(np.uint32))


@pytest.mark.parametrize("fmt,gs,D", [(INT4_G, 32, 1184), (MXFP4_G32, 0, 2080)])
def test_gate_up_clamped_kernels_agree(fmt, gs, D):
    F, s = 130, 2
    g, wg, sg, wu, su, x = gate_up_inputs(fmt, gs, F, D, s, 71)
    out = []
    for policy in (_lib.QKERNEL_RING, _lib.QKERNEL_TILE):
        prev = _lib.qkernel_policy(policy)
        try:
            out.append(run_act(fmt, gs, wg, sg, wu, su, x, F, D, QACT_SWIGLU_CLAMPED, 0.05))
        finally:
            _lib.qkernel_policy(prev)
    assert np.array_equal(out[0].view(np.uint32), out[1].view(np.uint32))


def run_group_act(fmt, gs, st, E, D, F, x, ids, wts, act, limit):
    s, k = ids.shape
    d = {n: dev(v) for n, v in st.items()}
    out = empty_f32(s, D)
    ws_bytes = qexpert_group_workspace(E, D, F, s, k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda())   # zeroed before first use
    status = torch.full((1,), 12345, dtype=torch.int32, device=cuda())
    qexpert_group_act(fmt, gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], E, D, F,
                      dev(x), s, k, dev(ids.astype(np.int32)), dev(wts.astype(np.float32)), act, limit, out, ws,
                      ws_bytes, status)
    return host(out), int(host(status)[0])


@pytest.mark.parametrize("fmt,gs", [(INT8_ROW, 0), (INT4_G, 32), (INT3_G64, 0), (MXFP4_G32, 0)])
@pytest.mark.parametrize("E,s,k", [(6, 1, 4), (5, 8, 4)])
def test_expert_group_clamped(fmt, gs, E, s, k):
    D, F = 256, 128
    st = small_store(fmt, E, D, F, 73)
    rng = synth.generator(79, fmt, E, s, k)
    x = synth.draw_x(s, D, rng)
    ids = rng.integers(0, E, size=(s, k)).astype(np.int32)
    wts = rng.random((s, k)).astype(np.float32)
    g = synth.fixed_group(fmt, D, gs or None)
    L = 0.5
    out, status = run_group_act(fmt, gs, st, E, D, F, x, ids, wts, QACT_SWIGLU_CLAMPED, L)
    assert status == 0
    want = oracle.expert_group(fmt, g, st["gate"], st["gate_s"], st["up"], st["up_s"], st["down"],
                               st["down_s"], E, D, F, x, ids, wts, act=1, limit=L)
    assert max_rel(out, want) <= GATE
    zero, status = run_group_act(fmt, gs, st, E, D, F, x, ids, wts, QACT_SWIGLU_CLAMPED, 0.0)
    assert status == 0 and not zero.any()
    inf, _ = run_group_act(fmt, gs, st, E, D, F, x, ids, wts, QACT_SWIGLU_CLAMPED, float("inf"))
    plain, _ = run_group_act(fmt, gs, st, E, D, F, x, ids, wts, QACT_SWIGLU, 0.0)
    assert np.array_equal(inf.view(np.uint32), plain.view(np.uint32))


def test_expert_group_clamped_full_size_sampled():
    """The clamped-SwiGLU configuration the bench times: the MXFP4 expert
    workload (256 experts, D = 6144, F = 2048, top 8) with limit 7, sampled
    output columns against the oracle."""
    from test_gpu_expert_group import compact_store, full_store_on_device
    wl = synth.workload("mxfp4_experts_E256_D6144_F2048_s1_k8")
    L = 7.0
    d = full_store_on_device(wl)
    x = wl.x()
    ids, wts = wl.routing()
    ws_bytes = qexpert_group_workspace(wl.E, wl.D, wl.F, wl.s, wl.k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda())   # zeroed before first use
    status = torch.full((1,), 12345, dtype=torch.int32, device=cuda())
    out = empty_f32(wl.s, wl.D)
    qexpert_group_act(wl.fmt, 0, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], wl.E, wl.D,
                      wl.F, dev(x), wl.s, wl.k, dev(ids.astype(np.int32)), dev(wts.astype(np.float32)),
                      QACT_SWIGLU_CLAMPED, L, out, ws, ws_bytes, status)
    assert int(host(status)[0]) == 0
    y = host(out)
    assert np.isfinite(y).all()
    used = np.unique(ids)
    remap = {int(e): i for i, e in enumerate(used)}
    cids = np.vectorize(remap.get)(ids).astype(np.int32)
    cols = np.unique(np.concatenate([[0, 1, wl.D - 1], synth.generator(11).choice(wl.D, 61, replace=False)]))
    st = compact_store(wl, used)
    want = oracle.expert_group(wl.fmt, wl.gs, st["gate"], st["gate_s"], st["up"], st["up_s"], st["down"],
                               st["down_s"], len(used), wl.D, wl.F, x, cids, wts.astype(np.float32), cols=cols,
                               act=1, limit=L)
    assert max_rel(y[:, cols], want) <= GATE
    b = expert_bound(wl.fmt, wl.gs, wl.gs, st, wl.D, wl.F, x, cids, wts.astype(np.float32), cols, [0], act=1,
                     limit=L)
    assert np.all(np.abs(y[:1, cols] - want) <= b)
