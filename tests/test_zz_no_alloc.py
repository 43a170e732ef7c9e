"""The allocation-free routed-expert group, for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It must pass alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest

from gpu_helpers import GATE, INT4_G, MXFP4_G32, cuda, dev, empty_f32, host, max_rel, torch
from weight_only_quantized_qgemv_gb300 import _lib, qexpert_group, qexpert_group_workspace, synth

pytestmark = pytest.mark.gpu


def _store(fmt, E, D, F, seed):
    rng = synth.generator(seed, fmt, E)
    st = {}
    for name, (O, I) in (("gate", (F, D)), ("up", (F, D)), ("down", (D, F))):
        st[name] = np.concatenate([synth.draw_packed(fmt, O, I, rng) for _ in range(E)])
        st[name + "_s"] = np.concatenate([synth.draw_scales(O, I, 32, rng, "lognormal", -4.0) for _ in range(E)])
    return {n: dev(v) for n, v in st.items()}


def _noalloc_c_abi(fmt, gs, d, E, D, F, x, ids, wts, out, status):
    """Straight through the C ABI with ctypes."""
    L = _lib.lib()
    f = L.qexpert_group_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [I, I, P, P, P, P, P, P, I, I, I, P, I, I, P, P, P, P, P]
    f.restype = I
    s, k = ids.shape
    return f(fmt, gs, d["gate"].data_ptr(), d["gate_s"].data_ptr(), d["up"].data_ptr(), d["up_s"].data_ptr(),
             d["down"].data_ptr(), d["down_s"].data_ptr(), E, D, F, x.data_ptr(), s, k, ids.data_ptr(),
             wts.data_ptr(), out.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("fmt,gs", [(INT4_G, 32), (MXFP4_G32, 0)])
def test_noalloc_matches_workspace_entry_point_twice(fmt, gs):
    E, D, F, s, k = 9, 1024, 512, 4, 3
    d = _store(fmt, E, D, F, 51)
    for call in range(2):                      # two calls in a row share the built-in scratch
        rng = synth.generator(53, call)
        x = dev(synth.draw_x(s, D, rng))
        ids_np, wts_np = synth.draw_routing(s, k, E, rng)
        ids, wts = dev(ids_np), dev(wts_np)
        out_ref = empty_f32(s, D)
        ws_bytes = qexpert_group_workspace(E, D, F, s, k)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda())   # zeroed before first use
        qexpert_group(fmt, gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"], E, D, F,
                      x, s, k, ids, wts, out_ref, ws, ws_bytes)
        out = empty_f32(s, D)
        status = torch.full((1,), 99, dtype=torch.int32, device=cuda())
        assert _noalloc_c_abi(fmt, gs, d, E, D, F, x, ids, wts, out, status) == 0
        assert int(host(status)[0]) == 0
        assert max_rel(host(out), host(out_ref).astype(np.float64)) <= GATE


def test_noalloc_rejects_sizes_beyond_its_scratch():
    E, D, F, s, k = 4, 6144, 2048, 64, 8          # 512 pairs: ~16 MB of scratch, above the 4 MiB array
    assert qexpert_group_workspace(E, D, F, s, k) > (4 << 20)
    d = {n: torch.empty(16, dtype=torch.uint8, device=cuda()) for n in ("gate", "gate_s", "up", "up_s", "down",
                                                                       "down_s")}
    x = torch.empty(16, dtype=torch.float32, device=cuda())
    ids = torch.zeros((s, k), dtype=torch.int32, device=cuda())
    out = torch.empty(16, dtype=torch.float32, device=cuda())
    status = torch.zeros(1, dtype=torch.int32, device=cuda())
    assert _noalloc_c_abi(INT4_G, 32, d, E, D, F, x, ids, x, out, status) == -5    # QSTATUS_WORKSPACE
