"""Per-element error bounds for the parity tests.

The device computes every output as f32 sums of f32 products in some order.
Against the oracle's exact (f64) value y* of an output y = sum_i w_i x_i, such
a sum is off by at most (n + 4) 2^-24 sum_i |w_i x_i| (n terms: one rounding
per product and per addition along the longest chain, plus the scale
multiplication).  The gate/up activation and the expert group's down product
and weighted sum propagate those bounds:
  h = act(g, u): |dh| <= 1.1 Bg (|u| + Bu) + (|silu(g)| + 1.1 Bg) Bu + 8 2^-24 |h|
      (silu' <= 1.1 everywhere; the clamps of the clamped SwiGLU are
      1-Lipschitz; 8 ulps cover expf, the division and the two products),
  z = down h: |dz| <= |down| Bh + (F + 4) 2^-24 |down| (|h| + Bh),
  out = sum_r w_r z_r: |dout| <= sum_r |w_r| Bz_r + (k + 2) 2^-24 sum_r |w_r| (|z_r| + Bz_r).
The magnitudes |w| come from the oracle's dequantized weights; the exact
values g, u, h, z and out from the oracle itself.
"""
from __future__ import annotations

import numpy as np

from oracle import oracle

U = 2.0 ** -24
SILU_SLOPE = 1.1


def dot_bound(wd: np.ndarray, x: np.ndarray) -> np.ndarray:
    """(n + 4) 2^-24 |x| |W|^T for f32 rows wd [O][n] and activations x [s][n]."""
    n = wd.shape[1]
    return (n + 4) * U * (np.abs(np.asarray(x, dtype=np.float64)) @ np.abs(wd.astype(np.float64)).T) + 1e-30


def gemv_bound(fmt, gs, w, sc, x, O, I):
    """Bound on |y - y*| per element of y [s][O] = qgemv of (w, sc) and x."""
    return dot_bound(oracle.dequant_f32(fmt, gs, w, sc, O, I), np.asarray(x).reshape(-1, I))


def _act(g, u, act, limit):
    if act == 1:
        g = np.minimum(g, limit)
        u = np.clip(u, -limit, limit)
    with np.errstate(over="ignore"):          # exp(-g) -> inf for very negative g: silu -> -0
        silu = g / (1.0 + np.exp(-g))
    return silu, u


def glu_bound(fmt, gs, wg, sg, wu, su, x, F, D, act=0, limit=0.0):
    """(h*, bound) for h [s][F] = act(gate x, up x) computed on the device in f32."""
    x = np.asarray(x, dtype=np.float32).reshape(-1, D)
    gstar = oracle.qgemv(fmt, gs, wg, sg, x, F, D)
    ustar = oracle.qgemv(fmt, gs, wu, su, x, F, D)
    bg = dot_bound(oracle.dequant_f32(fmt, gs, wg, sg, F, D), x)
    bu = dot_bound(oracle.dequant_f32(fmt, gs, wu, su, F, D), x)
    silu, uc = _act(gstar, ustar, act, limit)
    hstar = silu * uc
    bound = SILU_SLOPE * bg * (np.abs(uc) + bu) + (np.abs(silu) + SILU_SLOPE * bg) * bu + 8 * U * np.abs(hstar)
    return hstar, bound + 1e-30


def expert_bound(fmt, gs_up, gs_dn, st, D, F, x, ids, wts, cols, tokens, act=0, limit=0.0):
    """Bound on |out - out*| for out[t][cols], t in tokens, of the expert group
    over the store st (gate, gate_s, up, up_s, down, down_s back to back per
    expert), routing ids / wts [s][k]."""
    from weight_only_quantized_qgemv_gb300 import synth
    cols = np.asarray(cols)
    k = ids.shape[1]
    nb_up, nb_dn = synth.packed_bytes(fmt, F, D), synth.packed_bytes(fmt, D, F)
    ns_up, ns_dn = F * (D // gs_up), D * (F // gs_dn)
    rows_dn = np.asarray(cols)
    out = np.zeros((len(tokens), len(cols)))
    for ti, t in enumerate(tokens):
        bsum = np.zeros(len(cols))
        mag = np.zeros(len(cols))
        for r in range(k):
            e = int(ids[t, r])
            g_w = st["gate"][e * nb_up:(e + 1) * nb_up]
            g_s = st["gate_s"][e * ns_up:(e + 1) * ns_up]
            u_w = st["up"][e * nb_up:(e + 1) * nb_up]
            u_s = st["up_s"][e * ns_up:(e + 1) * ns_up]
            hstar, bh = glu_bound(fmt, gs_up, g_w, g_s, u_w, u_s, x[t:t + 1], F, D, act, limit)
            hstar, bh = hstar[0], bh[0]
            d_w = st["down"][e * nb_dn:(e + 1) * nb_dn]
            d_s = st["down_s"][e * ns_dn:(e + 1) * ns_dn]
            wd = np.abs(oracle.dequant_f32(fmt, gs_dn, _rows(fmt, d_w, D, F, rows_dn),
                                           d_s.reshape(D, -1)[rows_dn].reshape(-1), len(rows_dn), F)
                        .astype(np.float64))
            bz = wd @ bh + (F + 4) * U * (wd @ (np.abs(hstar) + bh))
            zmag = wd @ np.abs(hstar)          # >= |z*|
            wr = abs(float(wts[t, r]))
            bsum += wr * bz
            mag += wr * (zmag + bz)
        out[ti] = bsum + (k + 2) * U * mag + 1e-30
    return out


def _rows(fmt, w, O, I, rows):
    from gpu_helpers import packed_rows
    return packed_rows(fmt, w, O, I, rows)
