"""Thin ctypes binding of the C ABI in include/qgemv.h.

Argument marshalling only: every computation runs in the CUDA library.  Array
arguments may be torch tensors (their data_ptr() is passed) or raw integer
device addresses; `stream` defaults to torch's current CUDA stream.  A negative
status raises QStatusError.  If the library has not been built, loading fails
loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

QFMT_INT8_ROW, QFMT_INT4_G, QFMT_INT3_G64, QFMT_MXFP4_G32 = 1, 4, 5, 7
QFMT_INT4_ROW, QFMT_MXFP4_E8M0, QFMT_INT8_G = 2, 8, 13

QSTATUS = {
    0: "QSTATUS_OK",
    -1: "QSTATUS_BAD_FMT",
    -2: "QSTATUS_BAD_DIM",
    -3: "QSTATUS_MISALIGNED",
    -4: "QSTATUS_NULL",
    -5: "QSTATUS_WORKSPACE",
    -6: "QSTATUS_LAUNCH",
    -7: "QSTATUS_DEVICE_TIMEOUT",
    -8: "QSTATUS_BAD_EXPERT_ID",
    -9: "QSTATUS_BAD_ACT",
    -10: "QSTATUS_BAD_ROUTE",
}

QACT_SWIGLU, QACT_SWIGLU_CLAMPED = 0, 1
QROUTE_SOFTMAX, QROUTE_SIGMOID_BIAS = 0, 1


class QStatusError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{QSTATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it was never built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"the CUDA library {path} is not built; run __graft_entry__.build() "
                               "(nvcc, sm_103a) first -- there is no CPU fallback")
        L = ctypes.CDLL(path)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.qgemv.argtypes = [I, I, P, P, P, I, I, I, P, P]
        L.qgemv.restype = I
        L.qgate_up.argtypes = [I, I, P, P, P, P, P, I, I, I, P, P]
        L.qgate_up.restype = I
        L.qexpert_group_workspace.argtypes = [I, I, I, I, I]
        L.qexpert_group_workspace.restype = Z
        L.qexpert_group_launches.argtypes = [I, I, I, I, I, I, I, I]
        L.qexpert_group_launches.restype = I
        L.qexpert_group.argtypes = [I, I, P, P, P, P, P, P, I, I, I, P, I, I, P, P, P, P, Z, P, P]
        L.qexpert_group.restype = I
        Fl = ctypes.c_float
        L.qgate_up_act.argtypes = [I, I, P, P, P, P, P, I, I, I, I, Fl, P, P]
        L.qgate_up_act.restype = I
        L.qexpert_group_act.argtypes = [I, I, P, P, P, P, P, P, I, I, I, P, I, I, P, P, I, Fl, P, P, Z, P, P]
        L.qexpert_group_act.restype = I
        L.qroute.argtypes = [I, P, P, I, I, I, I, Fl, P, P, P]
        L.qroute.restype = I
        L.qexpert_group_routed.argtypes = [I, I, P, P, P, P, P, P, I, I, I, P, I, I, I, P, P, I, Fl, I, Fl, P, P, P,
                                           P, Z, P, P]
        L.qexpert_group_routed.restype = I
        L.qgemm_workspace.argtypes = [I, I]
        L.qgemm_workspace.restype = Z
        L.qgemm.argtypes = [I, I, P, P, P, I, I, I, P, P, Z, P]
        L.qgemm.restype = I
        L.qdequant.argtypes = [I, I, P, P, I, I, P, P]
        L.qdequant.restype = I
        L.qstatus_string.argtypes = [I]
        L.qstatus_string.restype = ctypes.c_char_p
        L.qlast_cuda_error.argtypes = []
        L.qlast_cuda_error.restype = ctypes.c_char_p
        L.qdevice_error.argtypes = [I]
        L.qdevice_error.restype = I
        L.qkernel_policy.argtypes = [I]
        L.qkernel_policy.restype = I
        L.qdebug_inject.argtypes = [I, ctypes.c_longlong]
        L.qdebug_inject.restype = I
        _lib = L
    return _lib


def _ptr(a):
    """The device address of an array argument.  A tensor must live on a CUDA
    device and be contiguous (the library reads dense row-major arrays); a
    host tensor or a strided view is refused here, before any launch."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if not getattr(a, "is_cuda", False):
        raise ValueError(f"expected a CUDA tensor, got one on {getattr(a, 'device', type(a).__name__)}")
    if not a.is_contiguous():
        raise ValueError("expected a contiguous tensor (dense row-major layout)")
    return a.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != 0:
        L = lib()
        msg = L.qstatus_string(status).decode()
        if status == -6:
            msg += f" ({L.qlast_cuda_error().decode()})"
        raise QStatusError(status, msg)


def qstatus_string(status: int) -> str:
    return lib().qstatus_string(status).decode()


QKERNEL_AUTO, QKERNEL_RING, QKERNEL_TILE, QKERNEL_ROW = 0, 1, 2, 3


def qkernel_policy(policy: int) -> int:
    """Sets the process's kernel choice (QKERNEL_*); returns the previous one."""
    prev = lib().qkernel_policy(int(policy))
    if prev < 0:
        raise QStatusError(prev, qstatus_string(prev))
    return prev


QDEBUG_NONE, QDEBUG_WITHHOLD_SIGNAL = 0, 1


def qdebug_inject(kind: int, wait_ns: int = 1) -> None:
    """Arms a test fault for the next one-launch expert group (QDEBUG_*)."""
    _check(lib().qdebug_inject(int(kind), int(wait_ns)))


def qdevice_error(clear: bool = False) -> int:
    """QSTATUS_DEVICE_TIMEOUT if a bounded device-side wait ran out since the
    last clear, else QSTATUS_OK (synchronizes with the device)."""
    return lib().qdevice_error(1 if clear else 0)


def qgemv(fmt, gs, w, scales, x, O, I, s, y, stream=None):
    _check(lib().qgemv(fmt, gs, _ptr(w), _ptr(scales), _ptr(x), O, I, s, _ptr(y), _stream(stream)))


def qgate_up(fmt, gs, wg, sg, wu, su, x, F, D, s, h, stream=None):
    _check(lib().qgate_up(fmt, gs, _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(x), F, D, s, _ptr(h),
                          _stream(stream)))


def qgate_up_act(fmt, gs, wg, sg, wu, su, x, F, D, s, act, limit, h, stream=None):
    _check(lib().qgate_up_act(fmt, gs, _ptr(wg), _ptr(sg), _ptr(wu), _ptr(su), _ptr(x), F, D, s, int(act),
                              float(limit), _ptr(h), _stream(stream)))


def qexpert_group_workspace(E, D, F, s, k) -> int:
    return lib().qexpert_group_workspace(E, D, F, s, k)


def qexpert_group_launches(fmt, gs, E, D, F, s, k, routed=False) -> int:
    """Kernel launches of one expert-group call of these sizes (1: the fused launch)."""
    n = lib().qexpert_group_launches(fmt, gs, E, D, F, s, k, int(bool(routed)))
    _check(min(n, 0))
    return n


def qexpert_group(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids, wts, out,
                  workspace, ws_bytes, status_dev=None, stream=None):
    _check(lib().qexpert_group(fmt, gs, _ptr(gate), _ptr(gate_s), _ptr(up), _ptr(up_s), _ptr(down),
                               _ptr(down_s), E, D, F, _ptr(x), s, k, _ptr(ids), _ptr(wts), _ptr(out),
                               _ptr(workspace), ws_bytes, _ptr(status_dev), _stream(stream)))


def qexpert_group_act(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids, wts, act, limit,
                      out, workspace, ws_bytes, status_dev=None, stream=None):
    _check(lib().qexpert_group_act(fmt, gs, _ptr(gate), _ptr(gate_s), _ptr(up), _ptr(up_s), _ptr(down),
                                   _ptr(down_s), E, D, F, _ptr(x), s, k, _ptr(ids), _ptr(wts), int(act),
                                   float(limit), _ptr(out), _ptr(workspace), ws_bytes, _ptr(status_dev),
                                   _stream(stream)))


def qroute(kind, logits, bias, s, E, k, renorm, scale, ids, wts, stream=None):
    _check(lib().qroute(int(kind), _ptr(logits), _ptr(bias), s, E, k, int(renorm), float(scale), _ptr(ids), _ptr(wts),
                        _stream(stream)))


def qexpert_group_routed(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, route_kind, logits, bias,
                         renorm, route_scale, act, limit, out, ids_out, wts_out, workspace, ws_bytes,
                         status_dev=None, stream=None):
    _check(lib().qexpert_group_routed(fmt, gs, _ptr(gate), _ptr(gate_s), _ptr(up), _ptr(up_s), _ptr(down),
                                      _ptr(down_s), E, D, F, _ptr(x), s, k, int(route_kind), _ptr(logits), _ptr(bias),
                                      int(renorm), float(route_scale), int(act), float(limit), _ptr(out),
                                      _ptr(ids_out), _ptr(wts_out), _ptr(workspace), int(ws_bytes),
                                      _ptr(status_dev), _stream(stream)))


def qgemm_workspace(I, s) -> int:
    return int(lib().qgemm_workspace(I, s))


def qgemm(fmt, gs, w, scales, x, O, I, s, y, workspace, ws_bytes, stream=None):
    _check(lib().qgemm(fmt, gs, _ptr(w), _ptr(scales), _ptr(x), O, I, s, _ptr(y), _ptr(workspace), int(ws_bytes),
                       _stream(stream)))


def qdequant(fmt, gs, w, scales, O, I, out, stream=None):
    _check(lib().qdequant(fmt, gs, _ptr(w), _ptr(scales), O, I, _ptr(out), _stream(stream)))


def qexpert_group_noalloc(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids, wts, out,
                          status_dev=None, stream=None):
    """qexpert_group with its scratch in the library's own fixed device array
    (for callers that cannot allocate device memory)."""
    f = lib().qexpert_group_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [I, I, P, P, P, P, P, P, I, I, I, P, I, I, P, P, P, P, P]
    f.restype = I
    _check(f(fmt, gs, _ptr(gate), _ptr(gate_s), _ptr(up), _ptr(up_s), _ptr(down), _ptr(down_s), E, D, F, _ptr(x),
             s, k, _ptr(ids), _ptr(wts), _ptr(out), _ptr(status_dev), _stream(stream)))
