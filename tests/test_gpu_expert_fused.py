"""The routed-expert group as one persistent launch (up to 256 pairs) against
the f64 oracle: every format, ragged row lengths, repeated experts in a row,
bad ids, the workspace reused call after call (its barrier counters must come
back to zero), routing inside the launch, the four-launch path (the same
streaming passes, so the same bits), the launch count the library reports,
and a bounded device wait made to run out on purpose."""
import numpy as np
import pytest

from bounds import expert_bound
from gpu_helpers import (GATE, INT3_G64, INT4_G, INT4_ROW, INT8_G, INT8_ROW, MXFP4_E8M0, MXFP4_G32, cuda, dev,
                         empty_f32, host, max_rel, torch)
from oracle import oracle
from test_gpu_expert_group import oracle_group, small_store
from weight_only_quantized_qgemv_gb300 import (QACT_SWIGLU, QROUTE_SOFTMAX, _lib, qexpert_group,
                                               qexpert_group_launches, qexpert_group_routed, qexpert_group_workspace,
                                               synth)

pytestmark = pytest.mark.gpu


def call(fmt, gs, d, E, D, F, x, ids, wts, ws, ws_bytes):
    s, k = ids.shape
    out = empty_f32(s, D)
    status = torch.full((1,), 12345, dtype=torch.int32, device=cuda())
    qexpert_group(fmt, gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], E, D, F,
                  dev(x), s, k, dev(ids.astype(np.int32)), dev(wts.astype(np.float32)), out, ws, ws_bytes, status)
    return host(out), int(host(status)[0])


def workspace(E, D, F, s, k):
    n = qexpert_group_workspace(E, D, F, s, k)
    return torch.zeros(n, dtype=torch.uint8, device=cuda()), n


def routing(rng, s, k, E, repeats):
    if repeats:
        return rng.integers(0, E, size=(s, k)).astype(np.int32), rng.random((s, k)).astype(np.float32)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(s)]).astype(np.int32)
    return ids, rng.random((s, k)).astype(np.float32)


FMTS = [(INT4_G, 32), (MXFP4_G32, 0), (INT8_ROW, 0), (INT3_G64, 0), (INT4_ROW, 0), (INT8_G, 32), (MXFP4_E8M0, 0)]
# (E, D, F, s, k): several row tiles and slices, ragged rows (640 and 1152
# inputs end inside a slice), 256 pairs
SHAPES = [(5, 2048, 2048, 1, 1), (9, 2048, 2048, 1, 4), (12, 4096, 2048, 3, 4), (64, 2048, 2048, 8, 8),
          (7, 6144, 2048, 2, 3), (6, 640, 1152, 3, 2), (256, 1152, 640, 32, 8)]


@pytest.mark.parametrize("fmt,gs", FMTS)
@pytest.mark.parametrize("E,D,F,s,k", SHAPES)
@pytest.mark.parametrize("repeats", [False, True])
def test_fused_matches_oracle(fmt, gs, E, D, F, s, k, repeats):
    if repeats and (E, s, k) != (64, 8, 8) and (E, s, k) != (9, 1, 4):
        pytest.skip("repeated ids on two shapes")
    st = small_store(fmt, E, D, F, 301)
    d = {n: dev(v) for n, v in st.items()}
    rng = synth.generator(303, fmt, E, D, s, k)
    x = synth.draw_x(s, D, rng)
    ids, wts = routing(rng, s, k, E, repeats)
    ws, nb = workspace(E, D, F, s, k)
    assert qexpert_group_launches(fmt, gs, E, D, F, s, k) == 1
    out, status = call(fmt, gs, d, E, D, F, x, ids, wts, ws, nb)
    assert status == 0
    g_up, g_dn = synth.fixed_group(fmt, D, gs or None), synth.fixed_group(fmt, F, gs or None)   # row formats: I
    want = oracle_group(fmt, g_up, st, E, D, F, x, ids, wts)
    assert max_rel(out, want) <= GATE
    cols = np.arange(0, D, max(1, D // 61))
    tokens = sorted({0, s - 1})
    b = expert_bound(fmt, g_up, g_dn, st, D, F, x, ids, wts, cols, tokens)
    assert np.all(np.abs(out[tokens][:, cols] - want[tokens][:, cols]) <= b)


@pytest.mark.parametrize("fmt,gs", FMTS)
def test_fused_against_four_launch_path(fmt, gs):
    """The same call through the four-launch path (QKERNEL_TILE): the same
    streaming passes and the same rank-order sum, so the same bits."""
    E, D, F, s, k = 16, 2048, 1152, 4, 4
    st = small_store(fmt, E, D, F, 307)
    d = {n: dev(v) for n, v in st.items()}
    rng = synth.generator(309)
    x = synth.draw_x(s, D, rng)
    ids, wts = routing(rng, s, k, E, True)
    ws, nb = workspace(E, D, F, s, k)
    fused, st1 = call(fmt, gs, d, E, D, F, x, ids, wts, ws, nb)
    prev = _lib.qkernel_policy(_lib.QKERNEL_TILE)
    try:
        assert qexpert_group_launches(fmt, gs, E, D, F, s, k) == 4
        four, st2 = call(fmt, gs, d, E, D, F, x, ids, wts, ws, nb)
    finally:
        _lib.qkernel_policy(prev)
    assert st1 == 0 and st2 == 0
    assert np.array_equal(fused.view(np.uint32), four.view(np.uint32))
    # and the workspace still works for the fused launch after the other path used it
    again, st3 = call(fmt, gs, d, E, D, F, x, ids, wts, ws, nb)
    assert st3 == 0 and np.array_equal(again.view(np.uint32), fused.view(np.uint32))


def test_launch_counts():
    """One launch up to 256 pairs, four past that; a routed call over more than
    256 experts adds the router kernel."""
    assert qexpert_group_launches(INT4_G, 32, 256, 6144, 2048, 8, 8) == 1
    assert qexpert_group_launches(MXFP4_G32, 0, 256, 6144, 2048, 1, 8) == 1
    assert qexpert_group_launches(MXFP4_G32, 0, 256, 6144, 2048, 1, 8, routed=True) == 1
    assert qexpert_group_launches(INT4_G, 32, 256, 2048, 2048, 32, 8) == 1
    assert qexpert_group_launches(INT4_G, 32, 256, 2048, 2048, 33, 8) == 4
    assert qexpert_group_launches(INT4_G, 32, 512, 2048, 2048, 4, 8, routed=True) == 2
    with pytest.raises(_lib.QStatusError):
        qexpert_group_launches(INT4_G, 32, 256, 2048, 2048, 0, 8)


def test_fused_workspace_reused_call_after_call():
    """Ten calls on one workspace with different routings: each exact to the
    oracle's gate, so the grid-barrier counters came back to zero every time."""
    fmt, gs, E, D, F, s, k = INT4_G, 32, 24, 2048, 1024, 4, 4
    st = small_store(fmt, E, D, F, 311)
    d = {n: dev(v) for n, v in st.items()}
    ws, nb = workspace(E, D, F, s, k)
    for i in range(10):
        rng = synth.generator(313, i)
        x = synth.draw_x(s, D, rng)
        ids, wts = routing(rng, s, k, E, i % 2 == 1)
        out, status = call(fmt, gs, d, E, D, F, x, ids, wts, ws, nb)
        assert status == 0
        assert max_rel(out, oracle_group(fmt, gs, st, E, D, F, x, ids, wts)) <= GATE
    assert not host(ws[:1280].view(torch.int32)).any(), "the counters are back at zero"


def test_fused_bad_id_reports_on_device():
    fmt, gs, E, D, F, s, k = INT4_G, 32, 4, 2048, 1024, 2, 2
    st = small_store(fmt, E, D, F, 317)
    d = {n: dev(v) for n, v in st.items()}
    x = synth.draw_x(s, D, synth.generator(1))
    ws, nb = workspace(E, D, F, s, k)
    for bad in (4, -1):
        ids = np.array([[0, 1], [2, bad]], dtype=np.int32)
        out, status = call(fmt, gs, d, E, D, F, x, ids, np.ones((s, k), np.float32), ws, nb)
        assert status == -8
        assert not out.any()
    ids = np.array([[0, 1], [2, 3]], dtype=np.int32)
    out, status = call(fmt, gs, d, E, D, F, x, ids, np.ones((s, k), np.float32), ws, nb)
    assert status == 0


@pytest.mark.parametrize("E", [32, 256])
def test_fused_routed_in_the_launch(E):
    """qexpert_group_routed up to 256 experts: the routing runs in the launch's
    prologue; ids exactly the oracle's, weights within 1e-6, out against the
    oracle on the device's own weights."""
    fmt, gs, D, F, s, k = MXFP4_G32, 0, 2048, 2048, 5, 8
    st = small_store(fmt, E, D, F, 319)
    d = {n: dev(v) for n, v in st.items()}
    rng = synth.generator(321, E)
    x = synth.draw_x(s, D, rng)
    logits = rng.standard_normal((s, E)).astype(np.float32)
    ws, nb = workspace(E, D, F, s, k)
    out = empty_f32(s, D)
    ids = torch.empty((s, k), dtype=torch.int32, device=cuda())
    wts = torch.empty((s, k), dtype=torch.float32, device=cuda())
    status = torch.full((1,), 12345, dtype=torch.int32, device=cuda())
    qexpert_group_routed(fmt, gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], E, D, F,
                         dev(x), s, k, QROUTE_SOFTMAX, dev(logits), None, 1, 1.0, QACT_SWIGLU, 0.0, out, ids, wts, ws,
                         nb, status)
    assert int(host(status)[0]) == 0
    want_ids, want_w = oracle.route(0, logits, k=k, renorm=True)
    assert np.array_equal(host(ids), want_ids)
    w_dev = host(wts)
    assert np.abs(w_dev - want_w).max() <= 1e-6 * np.abs(want_w).max()
    want = oracle_group(fmt, 32, st, E, D, F, x, want_ids, w_dev)
    assert max_rel(host(out), want) <= GATE


def test_fused_timeout_path():
    """One CTA does not count its finished gate/up tiles (test hook): the
    waits of the CTAs that need them run out after 1 ms, the launch returns
    with QSTATUS_DEVICE_TIMEOUT in the status word and in qdevice_error,
    nothing faults, the counters are back at zero, and the next call on the
    same workspace is exact again."""
    fmt, gs, E, D, F, s, k = INT4_G, 32, 8, 2048, 1024, 2, 3
    st = small_store(fmt, E, D, F, 323)
    d = {n: dev(v) for n, v in st.items()}
    rng = synth.generator(325)
    x = synth.draw_x(s, D, rng)
    ids, wts = routing(rng, s, k, E, False)
    ws, nb = workspace(E, D, F, s, k)
    assert _lib.qdevice_error(clear=True) == 0
    _lib.qdebug_inject(_lib.QDEBUG_WITHHOLD_SIGNAL, 1_000_000)
    try:
        _, status = call(fmt, gs, d, E, D, F, x, ids, wts, ws, nb)
    finally:
        _lib.qdebug_inject(_lib.QDEBUG_NONE, 0)
    assert status == -7
    assert _lib.qdevice_error(clear=True) == -7
    assert not host(ws[:1280].view(torch.int32)).any(), "the counters are back at zero"
    out, status = call(fmt, gs, d, E, D, F, x, ids, wts, ws, nb)
    assert status == 0
    assert max_rel(out, oracle_group(fmt, gs, st, E, D, F, x, ids, wts)) <= GATE
    assert _lib.qdevice_error(clear=True) == 0
