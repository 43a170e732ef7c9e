"""ctypes wrapper around the plain f64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE: imported only by the tests, by the package entry's smoke
check and by the bench's CPU-baseline leg.  The product path never loads it.

`build()` compiles oracle.c with gcc (OpenMP when the compiler has it).  The
`Oracle` class wraps one compiled copy; the module-level functions use the
default copy next to this file.  All results are numpy arrays in double.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

INT8_ROW, INT4_G, INT3_G64, MXFP4_G32 = 1, 4, 5, 7


def compile_oracle(src: str, out: str, openmp: bool = True) -> str:
    """gcc -O2 a copy of the oracle source into a shared library."""
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", out + ".tmp", src, "-lm"]
    if openmp:
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
            os.replace(out + ".tmp", out)
            return out
        except subprocess.CalledProcessError:
            pass
    subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (if stale); returns the path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_oracle(SRC, LIB)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _sc(fmt, a):
    """Scales as the format stores them: ue8m0 bytes for MXFP4_E8M0 (8), else f32."""
    return _u8(a) if fmt == 8 else _f32(a)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


class Oracle:
    """One compiled copy of the oracle."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        P, L, I = ctypes.c_void_p, ctypes.c_long, ctypes.c_int
        D = ctypes.c_double
        lib.oracle_packed_bytes.argtypes = [I, L, L]
        lib.oracle_packed_bytes.restype = L
        lib.oracle_code.argtypes = [I, P, L, L, L, L]
        lib.oracle_code.restype = I
        lib.oracle_e2m1.argtypes = [I]
        lib.oracle_e2m1.restype = D
        lib.oracle_code_value.argtypes = [I, I]
        lib.oracle_code_value.restype = D
        lib.oracle_weight.argtypes = [I, L, P, P, L, L, L, L]
        lib.oracle_weight.restype = D
        lib.oracle_dequant_f32.argtypes = [I, L, P, P, L, L, P]
        lib.oracle_qgemv.argtypes = [I, L, P, P, P, L, L, L, P]
        lib.oracle_qgemv_rows.argtypes = [I, L, P, P, P, L, L, L, P, L, P]
        lib.oracle_e8m0.argtypes = [I]
        lib.oracle_e8m0.restype = D
        lib.oracle_silu.argtypes = [D]
        lib.oracle_silu.restype = D
        lib.oracle_glu.argtypes = [I, D, D, D]
        lib.oracle_glu.restype = D
        lib.oracle_qgate_up_act.argtypes = [I, L, P, P, P, P, P, L, L, L, I, D, P]
        lib.oracle_qgate_up_rows_act.argtypes = [I, L, P, P, P, P, P, L, L, L, P, L, I, D, P]
        lib.oracle_expert_group_act_cols.argtypes = [I, L, P, P, P, P, P, P, L, L, L, P, L, L, P, P, I, D, P, L,
                                                     P, P]
        lib.oracle_qgate_up.argtypes = [I, L, P, P, P, P, P, L, L, L, P]
        lib.oracle_qgate_up_rows.argtypes = [I, L, P, P, P, P, P, L, L, L, P, L, P]
        lib.oracle_expert_group_cols.argtypes = [I, L, P, P, P, P, P, P, L, L, L, P, L, L, P, P, P, L, P, P]
        lib.oracle_sigmoid.argtypes = [D]
        lib.oracle_sigmoid.restype = D
        lib.oracle_route.argtypes = [I, P, P, L, L, L, I, D, P, P, P, P]
        lib.oracle_threads.restype = I
        lib.oracle_set_threads.argtypes = [I]
        lib.oracle_set_threads.restype = None
        self.lib = lib

    def threads(self) -> int:
        return self.lib.oracle_threads()

    def set_threads(self, n: int) -> None:
        """Threads of the OpenMP loops from here on (timing only: every output
        row is one thread's index-order sum whatever the count)."""
        self.lib.oracle_set_threads(int(n))

    def packed_bytes(self, fmt: int, O: int, I: int) -> int:
        return self.lib.oracle_packed_bytes(fmt, O, I)

    def codes(self, fmt: int, w, O: int, I: int) -> np.ndarray:
        """Raw codes [O][I] (step a1), element by element."""
        w = _u8(w)
        out = np.empty((O, I), dtype=np.int64)
        for o in range(O):
            for i in range(I):
                out[o, i] = self.lib.oracle_code(fmt, _p(w), O, I, o, i)
        return out

    def e2m1(self, code: int) -> float:
        return self.lib.oracle_e2m1(code)

    def code_value(self, fmt: int, code: int) -> float:
        return self.lib.oracle_code_value(fmt, code)

    def silu(self, z: float) -> float:
        return self.lib.oracle_silu(z)

    def dequant_f32(self, fmt: int, gs: int, w, scales, O: int, I: int) -> np.ndarray:
        """Dequantized weights rounded once to f32 [O][I] (step a2)."""
        w, scales = _u8(w), _sc(fmt, scales)
        out = np.empty((O, I), dtype=np.float32)
        self.lib.oracle_dequant_f32(fmt, gs, _p(w), _p(scales), O, I, _p(out))
        return out

    def qgemv(self, fmt: int, gs: int, w, scales, x, O: int, I: int) -> np.ndarray:
        """y [s][O] in double (step a3)."""
        w, scales, x = _u8(w), _sc(fmt, scales), _f32(x).reshape(-1, I)
        s = x.shape[0]
        y = np.empty((s, O), dtype=np.float64)
        self.lib.oracle_qgemv(fmt, gs, _p(w), _p(scales), _p(x), O, I, s, _p(y))
        return y

    def qgemv_rows(self, fmt: int, gs: int, w, scales, x, O: int, I: int, rows) -> np.ndarray:
        """y [s][len(rows)] for the sampled rows."""
        w, scales, x = _u8(w), _sc(fmt, scales), _f32(x).reshape(-1, I)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        s = x.shape[0]
        y = np.empty((s, len(rows)), dtype=np.float64)
        self.lib.oracle_qgemv_rows(fmt, gs, _p(w), _p(scales), _p(x), O, I, s, _p(rows), len(rows), _p(y))
        return y

    def e8m0(self, e: int) -> float:
        """Value of a ue8m0 scale byte."""
        return self.lib.oracle_e8m0(int(e))

    def glu(self, act: int, limit: float, g: float, u: float) -> float:
        """The gate/up activation of one (g, u) pair: act 0 SwiGLU, act 1 clamped SwiGLU."""
        return self.lib.oracle_glu(int(act), float(limit), float(g), float(u))

    def qgate_up(self, fmt: int, gs: int, wg, sg, wu, su, x, F: int, D: int, act: int = 0,
                 limit: float = 0.0) -> np.ndarray:
        """h [s][F] = act(gate x, up x) in double (step a4; act 0 = silu(g) * u)."""
        wg, sg, wu, su, x = _u8(wg), _sc(fmt, sg), _u8(wu), _sc(fmt, su), _f32(x).reshape(-1, D)
        s = x.shape[0]
        h = np.empty((s, F), dtype=np.float64)
        self.lib.oracle_qgate_up_act(fmt, gs, _p(wg), _p(sg), _p(wu), _p(su), _p(x), F, D, s, int(act),
                                     float(limit), _p(h))
        return h

    def qgate_up_rows(self, fmt: int, gs: int, wg, sg, wu, su, x, F: int, D: int, rows, act: int = 0,
                      limit: float = 0.0) -> np.ndarray:
        wg, sg, wu, su, x = _u8(wg), _sc(fmt, sg), _u8(wu), _sc(fmt, su), _f32(x).reshape(-1, D)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        s = x.shape[0]
        h = np.empty((s, len(rows)), dtype=np.float64)
        self.lib.oracle_qgate_up_rows_act(fmt, gs, _p(wg), _p(sg), _p(wu), _p(su), _p(x), F, D, s,
                                          _p(rows), len(rows), int(act), float(limit), _p(h))
        return h

    def expert_group(self, fmt: int, gs: int, gate, gate_s, up, up_s, down, down_s,
                     E: int, D: int, F: int, x, ids, wts, cols=None, act: int = 0,
                     limit: float = 0.0) -> np.ndarray:
        """out [s][D] (or [s][len(cols)]) in double (steps a4 + a5, rank order)."""
        gate, gate_s, up, up_s = _u8(gate), _sc(fmt, gate_s), _u8(up), _sc(fmt, up_s)
        down, down_s, x = _u8(down), _sc(fmt, down_s), _f32(x).reshape(-1, D)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        wts = _f32(wts)
        s = x.shape[0]
        k = ids.size // s
        if cols is None:
            ncols, cptr = D, None
        else:
            cols = np.ascontiguousarray(cols, dtype=np.int64)
            ncols, cptr = len(cols), _p(cols)
        out = np.empty((s, ncols), dtype=np.float64)
        h = np.empty(F, dtype=np.float64)
        self.lib.oracle_expert_group_act_cols(fmt, gs, _p(gate), _p(gate_s), _p(up), _p(up_s), _p(down),
                                              _p(down_s), E, D, F, _p(x), s, k, _p(ids), _p(wts), int(act),
                                              float(limit), cptr, ncols, _p(out), _p(h))
        return out


    def sigmoid(self, z: float) -> float:
        return self.lib.oracle_sigmoid(float(z))

    def route(self, kind: int, logits, bias=None, k: int = 8, renorm: bool = True, scale: float = 1.0):
        """(ids int32 [s][k], weights double [s][k]) of the router (kind 0 softmax, 1 sigmoid + bias)."""
        logits = _f32(logits)
        s, E = logits.shape
        b = _f32(np.zeros(E) if bias is None else bias)
        ids = np.empty((s, k), dtype=np.int32)
        w = np.empty((s, k), dtype=np.float64)
        keys = np.empty(E, dtype=np.float64)
        taken = np.empty(E, dtype=np.uint8)
        self.lib.oracle_route(int(kind), _p(logits), _p(b), s, E, k, int(bool(renorm)), float(scale), _p(ids),
                              _p(w), _p(keys), _p(taken))
        return ids, w


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from oracle.c next to this file."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def __getattr__(name):
    # Module-level access to the default copy's methods: oracle.qgemv(...), ...
    if name in {"threads", "set_threads", "packed_bytes", "codes", "e2m1", "code_value", "e8m0", "silu", "glu", "dequant_f32",
                "qgemv", "qgemv_rows", "qgate_up", "qgate_up_rows", "expert_group", "sigmoid", "route"}:
        return getattr(default(), name)
    raise AttributeError(name)
