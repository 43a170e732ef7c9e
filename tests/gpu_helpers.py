"""Helpers of the GPU parity tests: device upload, error measures, row slices."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

INT8_ROW, INT4_G, INT3_G64, MXFP4_G32 = 1, 4, 5, 7
INT4_ROW, MXFP4_E8M0, INT8_G = 2, 8, 13
GATE = 1e-3      # max_o |y - y*| / max_o |y*| per output vector, from the workloads' statement


def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def dev(a: np.ndarray):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a).to(cuda())


def host(t) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def empty_f32(*shape):
    return torch.empty(*shape, dtype=torch.float32, device=cuda())


def max_rel(y, ystar) -> float:
    """max |y - y*| / max |y*| over each output vector (last axis), worst vector."""
    y = np.asarray(y, dtype=np.float64).reshape(-1, np.shape(ystar)[-1])
    ystar = np.asarray(ystar, dtype=np.float64).reshape(y.shape)
    den = np.maximum(np.abs(ystar).max(axis=1), 1e-300)
    return float((np.abs(y - ystar).max(axis=1) / den).max())


def packed_rows(fmt: int, w: np.ndarray, O: int, I: int, rows) -> np.ndarray:
    """The packed bytes of the given rows, as a len(rows) x I matrix of format fmt."""
    rows = np.asarray(rows)
    if fmt in (INT8_ROW, INT8_G):
        return w.reshape(O, I)[rows].reshape(-1)
    if fmt in (INT4_G, INT4_ROW, MXFP4_G32, MXFP4_E8M0):
        return w.reshape(O, I // 2)[rows].reshape(-1)
    A = w[: O * I // 4].reshape(O, I // 4)[rows]
    B = w[O * I // 4:].reshape(O, I // 8)[rows]
    return np.concatenate([A.reshape(-1), B.reshape(-1)])


def scale_rows(scales: np.ndarray, O: int, rows) -> np.ndarray:
    return scales.reshape(O, -1)[np.asarray(rows)].reshape(-1)


def sample_rows(O: int, n: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set([0, 1, O - 1, O - 2, O // 2]) | set(rng.choice(O, size=min(n, O), replace=False).tolist())
    return np.array(sorted(r for r in pick if 0 <= r < O))
