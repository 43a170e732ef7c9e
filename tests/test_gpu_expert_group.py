"""Steps a4 + a5 + a6 on the GPU: qexpert_group against the f64 oracle.

Small stores cover every format, repeated experts in a row, experts with more
pairs than one batch holds, bad ids (reported on the device), one-hot and zero
router weights.  The two expert workloads run at full size (256 experts) and
are compared on sampled output columns.
"""
import numpy as np
import pytest

from gpu_helpers import GATE, INT3_G64, INT4_G, INT8_ROW, MXFP4_G32, cuda, dev, empty_f32, host, max_rel, torch
from bounds import expert_bound
from oracle import oracle
from weight_only_quantized_qgemv_gb300 import qexpert_group, qexpert_group_workspace, synth

pytestmark = pytest.mark.gpu


def small_store(fmt, E, D, F, seed):
    gs_up = synth.fixed_group(fmt, D)
    gs_dn = synth.fixed_group(fmt, F)
    rng = synth.generator(seed, fmt, E, D, F)
    m = {}
    for name, (O, I, g) in {"gate": (F, D, gs_up), "up": (F, D, gs_up), "down": (D, F, gs_dn)}.items():
        m[name] = np.concatenate([synth.draw_packed(fmt, O, I, rng) for _ in range(E)])
        m[name + "_s"] = np.concatenate([synth.draw_scales(O, I, g, rng, "lognormal", -4.0, fmt=fmt)
                                         for _ in range(E)])
    return m


def run_group(fmt, gs, st, E, D, F, x, ids, wts, stores_on_device=None):
    s, k = ids.shape
    d = stores_on_device or {n: dev(v) for n, v in st.items()}
    out = empty_f32(s, D)
    ws_bytes = qexpert_group_workspace(E, D, F, s, k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda())   # zeroed before first use
    status = torch.full((1,), 12345, dtype=torch.int32, device=cuda())
    qexpert_group(fmt, gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], E, D, F,
                  dev(x), s, k, dev(ids.astype(np.int32)), dev(wts.astype(np.float32)), out, ws, ws_bytes, status)
    return host(out), int(host(status)[0])


def oracle_group(fmt, gs, st, E, D, F, x, ids, wts, cols=None):
    return oracle.expert_group(fmt, gs, st["gate"], st["gate_s"], st["up"], st["up_s"], st["down"], st["down_s"],
                               E, D, F, x, ids, wts, cols=cols)


FMTS = [(INT8_ROW, 0), (INT4_G, 32), (INT3_G64, 0), (MXFP4_G32, 0)]


@pytest.mark.parametrize("fmt,gs", FMTS)
@pytest.mark.parametrize("E,s,k", [(6, 1, 1), (6, 1, 4), (6, 3, 2), (5, 8, 4), (2, 9, 4), (64, 8, 8)])
def test_expert_group_small(fmt, gs, E, s, k):
    D, F = 256, 128
    st = small_store(fmt, E, D, F, 31)
    rng = synth.generator(37, fmt, E, s, k)
    x = synth.draw_x(s, D, rng)
    ids = rng.integers(0, E, size=(s, k)).astype(np.int32)      # repeats allowed and summed
    wts = rng.random((s, k)).astype(np.float32)
    out, status = run_group(fmt, gs, st, E, D, F, x, ids, wts)
    assert status == 0
    want = oracle_group(fmt, synth.fixed_group(fmt, D, gs or None), st, E, D, F, x, ids, wts)
    assert max_rel(out, want) <= GATE


def test_expert_group_invariants():
    fmt, gs, E, D, F, s, k = INT4_G, 32, 7, 512, 256, 4, 3
    st = small_store(fmt, E, D, F, 41)
    rng = synth.generator(43)
    x = synth.draw_x(s, D, rng)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(s)]).astype(np.int32)
    wts = rng.random((s, k)).astype(np.float32)
    base, _ = run_group(fmt, gs, st, E, D, F, x, ids, wts)
    zero, _ = run_group(fmt, gs, st, E, D, F, x, ids, np.zeros_like(wts))
    assert not zero.any()
    onehot = np.zeros_like(wts)
    onehot[:, 2] = 1.0
    oh, _ = run_group(fmt, gs, st, E, D, F, x, ids, onehot)
    single, _ = run_group(fmt, gs, st, E, D, F, x, ids[:, 2:3].copy(), np.ones((s, 1), np.float32))
    assert np.array_equal(oh, single)
    perm, _ = run_group(fmt, gs, st, E, D, F, x, ids[:, ::-1].copy(), wts[:, ::-1].copy())
    assert max_rel(perm, base) <= 1e-5


def test_expert_group_bad_id_reports_on_device():
    fmt, gs, E, D, F, s, k = INT4_G, 32, 4, 256, 128, 2, 2
    st = small_store(fmt, E, D, F, 47)
    x = synth.draw_x(s, D, synth.generator(1))
    ids = np.array([[0, 1], [2, 4]], dtype=np.int32)     # 4 is outside [0, 4)
    out, status = run_group(fmt, gs, st, E, D, F, x, ids, np.ones((s, k), np.float32))
    assert status == -8
    assert not out.any()
    ids[1, 1] = -1
    out, status = run_group(fmt, gs, st, E, D, F, x, ids, np.ones((s, k), np.float32))
    assert status == -8


def full_store_on_device(wl):
    """The 256-expert store of a workload, drawn expert by expert into device memory."""
    d = {}
    for name, which in wl.MATRICES:
        nb, ns = wl.sizes(which)
        d[name] = torch.empty(wl.E * nb, dtype=torch.uint8, device=cuda())
        d[name + "_s"] = torch.empty(wl.E * ns, dtype=torch.uint8 if wl.fmt == synth.MXFP4_E8M0 else torch.float32,
                                     device=cuda())

    def sink(name, slot, w, sc):
        d[name][slot * w.size:(slot + 1) * w.size].copy_(torch.from_numpy(w))
        d[name + "_s"][slot * sc.size:(slot + 1) * sc.size].copy_(torch.from_numpy(sc))

    wl.generate(range(wl.E), sink)
    torch.cuda.synchronize()
    return d


def compact_store(wl, experts):
    return wl.store(experts)


@pytest.mark.parametrize("name", ["mxfp4_experts_E256_D6144_F2048_s1_k8", "int4_g32_experts_E256_D6144_F2048_s8_k8"])
def test_expert_group_full_size_sampled(name):
    wl = synth.workload(name)
    d = full_store_on_device(wl)
    x = wl.x()
    ids, wts = wl.routing()
    out, status = run_group(wl.fmt, wl.gs if wl.fmt == INT4_G else 0, None, wl.E, wl.D, wl.F, x, ids, wts,
                            stores_on_device=d)
    assert status == 0 and np.isfinite(out).all()
    used = np.unique(ids)
    remap = {int(e): i for i, e in enumerate(used)}
    cids = np.vectorize(remap.get)(ids).astype(np.int32)
    cols = np.unique(np.concatenate([[0, 1, wl.D - 1], synth.generator(5).choice(wl.D, 61, replace=False)]))
    st = compact_store(wl, used)
    want = oracle_group(wl.fmt, wl.gs, st, len(used), wl.D, wl.F, x, cids, wts, cols=cols)
    assert max_rel(out[:, cols], want) <= GATE
    # element by element, for the first and last token (all of them at s = 1)
    tokens = sorted({0, wl.s - 1})
    b = expert_bound(wl.fmt, wl.gs, wl.gs, st, wl.D, wl.F, x, cids, wts, cols, tokens)
    assert np.all(np.abs(out[tokens][:, cols] - want[tokens]) <= b)


def test_expert_group_most_pairs():
    """s * k = 4096 pairs (the limit), every expert routed many times, repeated ids in some rows."""
    fmt, gs, E, D, F, s, k = INT4_G, 32, 16, 256, 128, 512, 8
    st = small_store(fmt, E, D, F, 227)
    rng = synth.generator(229)
    x = synth.draw_x(s, D, rng)
    ids = rng.integers(0, E, size=(s, k)).astype(np.int32)
    wts = rng.random((s, k)).astype(np.float32)
    out, status = run_group(fmt, gs, st, E, D, F, x, ids, wts)
    assert status == 0
    assert max_rel(out, oracle_group(fmt, gs, st, E, D, F, x, ids, wts)) <= GATE
