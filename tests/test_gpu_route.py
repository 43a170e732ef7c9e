"""The router on the GPU (qroute, qexpert_group_routed) against the oracle.

Softmax routing selects by the logits themselves, so its ids must equal the
oracle's exactly (ties: lower index first); sigmoid routing selects by f32
keys sigmoid(l) + bias, which equal the oracle's f64 keys up to rounding, so
its ids are held to the oracle's on random logits (gaps far above the
rounding) and to validity (every chosen key at least every unchosen one, up
to the rounding) on top.  Weights: within 1e-6 of the oracle's.
"""
import numpy as np
import pytest

from gpu_helpers import GATE, MXFP4_G32, INT4_G, cuda, dev, empty_f32, host, max_rel, torch
from bounds import expert_bound
from oracle import oracle
from test_gpu_expert_group import small_store
from weight_only_quantized_qgemv_gb300 import (QACT_SWIGLU, QROUTE_SIGMOID_BIAS, QROUTE_SOFTMAX, qexpert_group_act,
                                               qexpert_group_routed, qexpert_group_workspace, qroute, synth)

pytestmark = pytest.mark.gpu


def run_route(kind, logits, bias, k, renorm, scale):
    s, E = logits.shape
    ids = torch.empty((s, k), dtype=torch.int32, device=cuda())
    wts = torch.empty((s, k), dtype=torch.float32, device=cuda())
    qroute(kind, dev(logits), None if bias is None else dev(bias), s, E, k, renorm, scale, ids, wts)
    return host(ids), host(wts)


@pytest.mark.parametrize("E,k", [(8, 1), (8, 8), (64, 4), (256, 8), (256, 32), (1000, 6)])
@pytest.mark.parametrize("s", [1, 37])
@pytest.mark.parametrize("renorm,scale", [(0, 1.0), (1, 1.0), (1, 2.5)])
def test_route_softmax(E, k, s, renorm, scale):
    rng = synth.generator(181, E, k, s)
    logits = (2 * rng.standard_normal((s, E))).astype(np.float32)
    ids, w = run_route(QROUTE_SOFTMAX, logits, None, k, renorm, scale)
    want_ids, want_w = oracle.route(0, logits, k=k, renorm=bool(renorm), scale=scale)
    assert np.array_equal(ids, want_ids)
    assert np.abs(w - want_w).max() <= 1e-6 * np.abs(want_w).max()


@pytest.mark.parametrize("E,k", [(64, 4), (256, 8), (256, 32)])
@pytest.mark.parametrize("renorm,scale", [(0, 1.0), (1, 2.5)])
def test_route_sigmoid_bias(E, k, renorm, scale):
    s = 29
    rng = synth.generator(191, E, k)
    logits = (2 * rng.standard_normal((s, E))).astype(np.float32)
    bias = (0.2 * rng.standard_normal(E)).astype(np.float32)
    ids, w = run_route(QROUTE_SIGMOID_BIAS, logits, bias, k, renorm, scale)
    want_ids, want_w = oracle.route(1, logits, bias, k=k, renorm=bool(renorm), scale=scale)
    keys = 1 / (1 + np.exp(-logits.astype(np.float64))) + bias.astype(np.float64)
    for t in range(s):
        chosen = keys[t, ids[t]]
        rest = np.delete(keys[t], ids[t])
        assert len(set(ids[t].tolist())) == k
        assert chosen.min() >= rest.max() - 1e-6 and np.all(np.diff(chosen) <= 1e-6)
    assert np.array_equal(ids, want_ids)
    assert np.abs(w - want_w).max() <= 1e-6 * np.abs(want_w).max()


def test_route_ties_and_nan():
    """Equal keys: lower index first; NaN logits rank last."""
    E, k = 64, 8
    z = np.zeros((2, E), dtype=np.float32)
    z[1, 3] = np.nan
    z[1, 0] = np.nan
    ids, w = run_route(QROUTE_SOFTMAX, z, None, k, 1, 1.0)
    assert ids[0].tolist() == list(range(k))
    assert ids[1].tolist() == [1, 2, 4, 5, 6, 7, 8, 9]
    assert np.allclose(w, 1.0 / k)
    lg = np.full((1, E), -1.0, dtype=np.float32)
    lg[0, 10] = lg[0, 20] = 2.0
    ids, _ = run_route(QROUTE_SIGMOID_BIAS, lg, np.zeros(E, np.float32), 3, 1, 1.0)
    assert ids[0].tolist() == [10, 20, 0]


@pytest.mark.parametrize("kind", [QROUTE_SOFTMAX, QROUTE_SIGMOID_BIAS])
@pytest.mark.parametrize("s,k", [(1, 32), (65, 32)])
def test_route_largest_sizes(kind, s, k):
    """The most experts (1024) and the most choices per token (32) a call takes."""
    E = 1024
    rng = synth.generator(211, kind, s, k)
    logits = (2 * rng.standard_normal((s, E))).astype(np.float32)
    bias = (0.2 * rng.standard_normal(E)).astype(np.float32) if kind == QROUTE_SIGMOID_BIAS else None
    ids, w = run_route(kind, logits, bias, k, 1, 1.0)
    want_ids, want_w = oracle.route(kind, logits, bias, k=k, renorm=True)
    assert np.array_equal(ids, want_ids)
    assert np.abs(w - want_w).max() <= 1e-6 * np.abs(want_w).max()


@pytest.mark.parametrize("fmt,gs", [(MXFP4_G32, 0), (INT4_G, 32)])
@pytest.mark.parametrize("kind", [QROUTE_SOFTMAX, QROUTE_SIGMOID_BIAS])
@pytest.mark.parametrize("E", [16, 256, 300])
def test_expert_group_routed(fmt, gs, kind, E):
    """Routing and the expert group in one call: the two calls' bits, and the oracle's result.

    Up to 256 experts the routing runs inside the expert group's first kernel;
    past that it is a router launch of its own ahead of it (E = 300)."""
    D, F, s, k = 256, 128, 5, 4
    st = small_store(fmt, E, D, F, 193)
    rng = synth.generator(197, fmt, kind)
    x = synth.draw_x(s, D, rng)
    logits = rng.standard_normal((s, E)).astype(np.float32)
    bias = (0.3 * rng.standard_normal(E)).astype(np.float32)
    d = {n: dev(v) for n, v in st.items()}
    ws_bytes = qexpert_group_workspace(E, D, F, s, k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda())   # zeroed before first use
    status = torch.full((1,), 12345, dtype=torch.int32, device=cuda())
    out = empty_f32(s, D)
    ids = torch.empty((s, k), dtype=torch.int32, device=cuda())
    wts = torch.empty((s, k), dtype=torch.float32, device=cuda())
    qexpert_group_routed(fmt, gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], E, D, F,
                         dev(x), s, k, kind, dev(logits), dev(bias), 1, 1.0, QACT_SWIGLU, 0.0, out, ids, wts, ws,
                         ws_bytes, status)
    assert int(host(status)[0]) == 0
    want_ids, want_w = oracle.route(kind, logits, bias, k=k, renorm=True)
    assert np.array_equal(host(ids), want_ids)
    # the same expert group from the two separate calls
    out2 = empty_f32(s, D)
    qexpert_group_act(fmt, gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], E, D, F, dev(x),
                      s, k, ids, wts, QACT_SWIGLU, 0.0, out2, ws, ws_bytes, status)
    assert np.array_equal(host(out).view(np.uint32), host(out2).view(np.uint32))
    g = synth.fixed_group(fmt, D, gs or None)
    want = oracle.expert_group(fmt, g, st["gate"], st["gate_s"], st["up"], st["up_s"], st["down"], st["down_s"],
                               E, D, F, x, want_ids, want_w.astype(np.float32))
    assert max_rel(host(out), want) <= GATE


@pytest.mark.parametrize("name", ["mxfp4_experts_E256_D6144_F2048_s1_k8", "int4_g32_experts_E256_D6144_F2048_s8_k8"])
def test_expert_group_routed_full_size_sampled(name):
    """The device-routed configuration the bench times: the workload's 256-expert
    store, router logits [s][256], softmax top 8 renormalized (routing inside the
    prep kernel).  Ids exactly the oracle's, weights within 1e-6, sampled output
    columns against the oracle."""
    from test_gpu_expert_group import compact_store, full_store_on_device, oracle_group
    wl = synth.workload(name)
    d = full_store_on_device(wl)
    x = wl.x()
    logits = wl.router_logits()
    gs = wl.gs if wl.fmt == INT4_G else 0
    ws_bytes = qexpert_group_workspace(wl.E, wl.D, wl.F, wl.s, wl.k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda())   # zeroed before first use
    status = torch.full((1,), 12345, dtype=torch.int32, device=cuda())
    out = empty_f32(wl.s, wl.D)
    ids = torch.empty((wl.s, wl.k), dtype=torch.int32, device=cuda())
    wts = torch.empty((wl.s, wl.k), dtype=torch.float32, device=cuda())
    qexpert_group_routed(wl.fmt, gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], wl.E, wl.D,
                         wl.F, dev(x), wl.s, wl.k, QROUTE_SOFTMAX, dev(logits), None, 1, 1.0, QACT_SWIGLU, 0.0, out,
                         ids, wts, ws, ws_bytes, status)
    assert int(host(status)[0]) == 0
    want_ids, want_w = oracle.route(0, logits, k=wl.k, renorm=True)
    assert np.array_equal(host(ids), want_ids)
    assert np.abs(host(wts) - want_w).max() <= 1e-6 * np.abs(want_w).max()
    y = host(out)
    assert np.isfinite(y).all()
    used = np.unique(want_ids)
    remap = {int(e): i for i, e in enumerate(used)}
    cids = np.vectorize(remap.get)(want_ids).astype(np.int32)
    cols = np.unique(np.concatenate([[0, 1, wl.D - 1], synth.generator(7).choice(wl.D, 61, replace=False)]))
    st = compact_store(wl, used)
    want = oracle_group(wl.fmt, wl.gs, st, len(used), wl.D, wl.F, x, cids, want_w.astype(np.float32), cols=cols)
    assert max_rel(y[:, cols], want) <= GATE
    # element by element against the oracle on the device's own router weights
    w_dev = host(wts)
    want_d = oracle_group(wl.fmt, wl.gs, st, len(used), wl.D, wl.F, x, cids, w_dev, cols=cols)
    tokens = sorted({0, wl.s - 1})
    b = expert_bound(wl.fmt, wl.gs, wl.gs, st, wl.D, wl.F, x, cids, w_dev, cols, tokens)
    assert np.all(np.abs(y[tokens][:, cols] - want_d[tokens]) <= b)


def test_expert_group_routed_rejects_before_routing():
    """Past 256 experts the router is a launch of its own; a call the expert
    group would reject (here a gate not 16-byte aligned) is rejected before
    the router is enqueued: the routing outputs stay untouched."""
    from weight_only_quantized_qgemv_gb300 import QStatusError
    fmt, E, D, F, s, k = MXFP4_G32, 512, 256, 128, 3, 4
    st = small_store(fmt, E, D, F, 199)
    d = {n: dev(v) for n, v in st.items()}
    gate_off = torch.empty(d["gate"].numel() + 16, dtype=torch.uint8, device=cuda())[8:8 + d["gate"].numel()]
    logits = dev(synth.generator(211).standard_normal((s, E)).astype(np.float32))
    ws_bytes = qexpert_group_workspace(E, D, F, s, k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda())   # zeroed before first use
    out = empty_f32(s, D)
    ids = torch.full((s, k), -77, dtype=torch.int32, device=cuda())
    wts = torch.full((s, k), -7.0, dtype=torch.float32, device=cuda())
    with pytest.raises(QStatusError) as e:
        qexpert_group_routed(fmt, 0, gate_off, d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], E, D, F,
                             dev(synth.draw_x(s, D, synth.generator(213))), s, k, QROUTE_SOFTMAX, logits, None, 1,
                             1.0, QACT_SWIGLU, 0.0, out, ids, wts, ws, ws_bytes)
    assert e.value.status == -3
    assert (host(ids) == -77).all() and (host(wts) == -7.0).all()
