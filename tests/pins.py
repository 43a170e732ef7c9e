"""Pins of the CPU oracle: checks against what the pages and the mathematics fix.

Each pin takes one compiled copy of the oracle (so the mutant tests can run the
same pins on copies with a planted mistake) and raises AssertionError when the
copy disagrees with:
  - the hand-built words under tests/golden/ (e2m1 table, int4 nibble - 8,
    int3 dual planes, int8 bytes), each fixture citing its passage;
  - IEEE f32 multiplication (numpy) for the f32 dequantized weight;
  - an independent dense evaluation (codes packed by the tests' own packer,
    numpy f64 matmul) for the GEMV, gate/up and the expert group;
  - closed forms: zero-scale groups give exact zeros, linearity in x, exact
    integer results for small-integer x and power-of-two scales, silu against
    scipy's logistic function, invariants of the routed sum (one-hot weights,
    zero weights, permuted ranks, repeated experts).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
from scipy.special import expit

from packing import (ALL_FMTS, INT3_G64, INT4_G, INT4_ROW, INT8_G, INT8_ROW, MXFP4_E8M0, MXFP4_G32, dense,
                     draw_scales, e2m1_table, group_of, load_table, pack, random_codes, scale_values,
                     to_stored_scales, values_of)


def _close(a, b, rtol=1e-12, atol=0.0):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(np.abs(b).max(), 1e-300)
    err = np.abs(a - b).max() / scale if a.size else 0.0
    assert err <= rtol or np.allclose(a, b, rtol=rtol, atol=atol), f"max rel err {err:.3e} > {rtol:.1e}"


# --- step a1/a2: codes and values on hand-built words -----------------------

def pin_e2m1(orc):
    tab = e2m1_table()
    for c in range(16):
        v = orc.e2m1(c)
        assert v == tab[c] and np.signbit(v) == np.signbit(tab[c]), f"e2m1 code {c:#x}: {v} != {tab[c]}"
        v = orc.code_value(MXFP4_G32, c)
        assert v == tab[c] and np.signbit(v) == np.signbit(tab[c])
    # every code through the packed path: byte b holds codes (b & 15, b >> 4)
    codes = np.array([[c for c in range(16)] * 2], dtype=np.int64)
    got = orc.codes(MXFP4_G32, pack(MXFP4_G32, codes), 1, 32)
    assert np.array_equal(got, codes)


def pin_int4_nibbles(orc):
    rows = load_table("int4_nibbles.txt")
    for byte_s, v_even, v_odd in rows:
        byte = int(byte_s, 16)
        for o, b in ((0, 0), (1, 5)):          # row 1, byte 5 -> inputs 10, 11
            w = np.full(2 * 16, 0x88, dtype=np.uint8)  # 2 rows x 32 inputs
            w[o * 16 + b] = byte
            c0 = orc.codes(INT4_G, w, 2, 32)[o, 2 * b]
            c1 = orc.codes(INT4_G, w, 2, 32)[o, 2 * b + 1]
            assert orc.code_value(INT4_G, int(c0)) == int(v_even), (byte_s, c0)
            assert orc.code_value(INT4_G, int(c1)) == int(v_odd), (byte_s, c1)


def pin_int3_planes(orc):
    O, I = 2, 64
    for r in load_table("int3_planes.txt"):
        A0, A1, B = (int(v, 16) for v in r[:3])
        want = [int(v) for v in r[3:]]
        w = np.zeros(O * I // 4 + O * I // 8, dtype=np.uint8)
        w[1 * 16 + 0] = A0                       # row 1, plane A bytes 0, 1
        w[1 * 16 + 1] = A1
        w[O * I // 4 + 1 * 8 + 0] = B           # plane B after the whole plane A
        got = orc.codes(INT3_G64, w, O, I)
        assert list(got[1, :8]) == want, (r, list(got[1, :8]))
        assert not got[0].any() and not got[1, 8:].any()
        for c, v in zip(want, got[1, :8]):
            assert orc.code_value(INT3_G64, int(v)) == c - 4
    # every code at every position of both rows
    for o in range(O):
        for p in range(I):
            for c in range(8):
                codes = np.zeros((O, I), dtype=np.int64)
                codes[o, p] = c
                w = np.zeros(O * I // 4 + O * I // 8, dtype=np.uint8)
                w[o * 16 + p // 4] |= (c & 3) << (2 * (p % 4))
                w[O * I // 4 + o * 8 + p // 8] |= ((c >> 2) & 1) << (p % 8)
                if p % 16 == 0 or c == 7:
                    assert np.array_equal(orc.codes(INT3_G64, w, O, I), codes), (o, p, c)


def pin_int8_bytes(orc):
    for byte_s, v in load_table("int8_bytes.txt"):
        w = np.zeros(2 * 16, dtype=np.uint8)
        w[16 + 3] = int(byte_s, 16)
        got = orc.codes(INT8_ROW, w, 2, 16)
        assert got[1, 3] == int(v) and orc.code_value(INT8_ROW, int(got[1, 3])) == int(v)


def pin_random_codes(orc):
    rng = np.random.default_rng(7)
    for fmt in ALL_FMTS:
        codes = random_codes(fmt, 3, 128, rng)
        got = orc.codes(fmt, pack(fmt, codes), 3, 128)
        assert np.array_equal(got, codes), f"fmt {fmt}"


def pin_e8m0(orc):
    for b, v in load_table("e8m0_scales.txt"):
        got = orc.e8m0(int(b))
        if v == "nan":
            assert np.isnan(got), b
        else:
            assert got == 2.0 ** int(v[2:]), (b, got, v)


def pin_format_variants(orc):
    """The three variant formats reduce to pinned ones: int4 with one scale per row is int4 with
    a group of the whole row, int8 grouped with a group of the whole row is int8 per row, and
    MXFP4 with ue8m0 byte 127 + k is MXFP4 with the f32 scale 2^k."""
    rng = np.random.default_rng(41)
    O, I, s = 3, 256, 2
    x = rng.standard_normal((s, I)).astype(np.float32)
    c4 = random_codes(INT4_ROW, O, I, rng)
    sr = rng.lognormal(-4, 0.5, size=O).astype(np.float32)
    assert np.array_equal(orc.qgemv(INT4_ROW, 0, pack(INT4_ROW, c4), sr, x, O, I),
                          orc.qgemv(INT4_G, I, pack(INT4_G, c4), sr, x, O, I))
    c8 = random_codes(INT8_G, O, I, rng)
    assert np.array_equal(orc.qgemv(INT8_G, I, pack(INT8_G, c8), sr, x, O, I),
                          orc.qgemv(INT8_ROW, 0, pack(INT8_ROW, c8), sr, x, O, I))
    cm = random_codes(MXFP4_E8M0, O, I, rng)
    k = rng.integers(-8, 3, size=O * (I // 32))
    assert np.array_equal(orc.qgemv(MXFP4_E8M0, 0, pack(MXFP4_E8M0, cm), (127 + k).astype(np.uint8), x, O, I),
                          orc.qgemv(MXFP4_G32, 0, pack(MXFP4_G32, cm), np.ldexp(1.0, k).astype(np.float32), x, O,
                                    I))
    # int8 grouped takes its groups along the row: groups of 32 with different scales
    sg = rng.lognormal(-4, 0.5, size=O * (I // 32)).astype(np.float32)
    want = x.astype(np.float64) @ (c8 * np.repeat(sg.reshape(O, -1).astype(np.float64), 32, axis=1)).T
    _close(orc.qgemv(INT8_G, 32, pack(INT8_G, c8), sg, x, O, I), want)


# --- step a2: f32 dequantized weights ----------------------------------------

def pin_dequant_f32(orc):
    rng = np.random.default_rng(11)
    for fmt in ALL_FMTS:
        for gs_req in (None, 64, 128):
            O, I = 3, 256
            gs = group_of(fmt, I, gs_req)
            if fmt not in (INT4_G, INT8_G) and gs_req is not None:
                continue
            codes = random_codes(fmt, O, I, rng)
            scales = draw_scales(fmt, O * (I // gs), rng, -4, 3.0)
            if fmt == MXFP4_E8M0:
                scales[0], scales[-1] = 0, 250           # 2^-127 (subnormal in f32) and 2^123
            else:
                scales[0] = np.float32(1e-41)      # subnormal scale
                scales[-1] = np.float32(1e36)       # large, no f32 overflow at |value| <= 128
            got = orc.dequant_f32(fmt, gs, pack(fmt, codes), scales, O, I)
            sv = scale_values(fmt, scales).astype(np.float32)    # exact: powers of two or f32 already
            want = values_of(fmt, codes).astype(np.float32) * np.repeat(sv.reshape(O, -1), gs, axis=1)
            assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32)), f"fmt {fmt} gs {gs}"


def pin_fixed_groups(orc):
    """int3-g64 groups 64 inputs and MXFP4 32 whatever gs says; int8 and int4 per row one per row."""
    rng = np.random.default_rng(12)
    for fmt, g in ((INT3_G64, 64), (MXFP4_G32, 32), (INT8_ROW, 256), (INT4_ROW, 256), (MXFP4_E8M0, 32)):
        O, I = 2, 256
        codes = random_codes(fmt, O, I, rng)
        scales = draw_scales(fmt, O * (I // g), rng, -4, 1.0)
        a = orc.dequant_f32(fmt, g, pack(fmt, codes), scales, O, I)
        for other in (32, 64, 128):
            b = orc.dequant_f32(fmt, other, pack(fmt, codes), scales, O, I)
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (fmt, other)


# --- step a3: the GEMV -------------------------------------------------------

def pin_gemv_bruteforce(orc):
    rng = np.random.default_rng(13)
    for fmt in ALL_FMTS:
        for gs_req in (None, 64):
            for s in (1, 4):
                O, I = 4, 64 if gs_req is None else 128
                gs = group_of(fmt, I, gs_req)
                if gs_req is not None and fmt not in (INT4_G, INT8_G):
                    continue
                codes = random_codes(fmt, O, I, rng)
                scales = draw_scales(fmt, O * (I // gs), rng)
                x = rng.standard_normal((s, I)).astype(np.float32)
                got = orc.qgemv(fmt, gs, pack(fmt, codes), scales, x, O, I)
                want = x.astype(np.float64) @ dense(fmt, codes, scales, gs).T
                _close(got, want)
                # scale 1: a plain dense matvec of the code values
                ones = to_stored_scales(fmt, np.ones(O * (I // gs)))
                got1 = orc.qgemv(fmt, gs, pack(fmt, codes), ones, x, O, I)
                _close(got1, x.astype(np.float64) @ values_of(fmt, codes).T)
                rows = np.array([3, 0, 2])
                _close(orc.qgemv_rows(fmt, gs, pack(fmt, codes), scales, x, O, I, rows), got[:, rows])


def pin_zero_scales(orc):
    rng = np.random.default_rng(17)
    for fmt in ALL_FMTS:
        if fmt == MXFP4_E8M0:
            continue                                 # ue8m0 has no zero
        O, I = 3, 128
        gs = group_of(fmt, I)
        codes = random_codes(fmt, O, I, rng)
        x = rng.standard_normal((2, I)).astype(np.float32)
        zero = np.zeros(O * (I // gs), dtype=np.float32)
        assert not orc.qgemv(fmt, gs, pack(fmt, codes), zero, x, O, I).any()
        if gs < I:
            scales = draw_scales(fmt, O * (I // gs), rng)
            scales.reshape(O, -1)[:, 1] = 0.0        # group 1 of every row is zero
            y1 = orc.qgemv(fmt, gs, pack(fmt, codes), scales, x, O, I)
            codes2 = codes.copy()
            codes2[:, gs:2 * gs] = random_codes(fmt, O, gs, rng)
            y2 = orc.qgemv(fmt, gs, pack(fmt, codes2), scales, x, O, I)
            assert np.array_equal(y1, y2), f"fmt {fmt}: a zero-scale group changed y"


def pin_linearity(orc):
    rng = np.random.default_rng(19)
    for fmt in ALL_FMTS:
        O, I = 4, 128
        gs = group_of(fmt, I)
        w = pack(fmt, random_codes(fmt, O, I, rng))
        scales = draw_scales(fmt, O * (I // gs), rng)
        x1 = rng.standard_normal(I).astype(np.float32)
        x2 = rng.standard_normal(I).astype(np.float32)
        x1[1::2] = 0.0                              # disjoint supports: a*x1 + b*x2 exact in f32
        x2[0::2] = 0.0
        a, b = np.float32(0.25), np.float32(-8.0)
        x3 = a * x1 + b * x2
        y1 = orc.qgemv(fmt, gs, w, scales, x1, O, I)
        y2 = orc.qgemv(fmt, gs, w, scales, x2, O, I)
        y3 = orc.qgemv(fmt, gs, w, scales, x3, O, I)
        _close(y3, float(a) * y1 + float(b) * y2, rtol=1e-12)


def pin_integer_exact(orc):
    rng = np.random.default_rng(23)
    for fmt in ALL_FMTS:
        O, I = 3, 256
        gs = group_of(fmt, I)
        codes = random_codes(fmt, O, I, rng)
        k = rng.integers(-8, 1, size=O * (I // gs))
        scales = to_stored_scales(fmt, np.ldexp(np.ones(k.size), k))
        x = rng.integers(-4, 5, size=(2, I)).astype(np.float32)
        got = orc.qgemv(fmt, gs, pack(fmt, codes), scales, x, O, I)
        vals = values_of(fmt, codes)
        for t in range(2):
            for o in range(O):
                exact = sum(Fraction(vals[o, i]) * Fraction(2) ** int(k[o * (I // gs) + i // gs]) * int(x[t, i])
                            for i in range(I))
                assert Fraction(got[t, o]) == exact, (fmt, t, o)


# --- step a4: silu and the fused gate/up --------------------------------------

def pin_silu(orc):
    assert orc.silu(0.0) == 0.0
    for z in np.linspace(-30, 30, 121):
        want = z * expit(z)
        got = orc.silu(float(z))
        assert abs(got - want) <= 1e-15 * max(1.0, abs(want)), (z, got, want)


def pin_gate_up(orc):
    rng = np.random.default_rng(29)
    for fmt in ALL_FMTS:
        F, D, s = 8, 128, 2
        gs = group_of(fmt, D)
        cg, cu = random_codes(fmt, F, D, rng), random_codes(fmt, F, D, rng)
        sg = draw_scales(fmt, F * (D // gs), rng)
        su = draw_scales(fmt, F * (D // gs), rng)
        x = rng.standard_normal((s, D)).astype(np.float32)
        got = orc.qgate_up(fmt, gs, pack(fmt, cg), sg, pack(fmt, cu), su, x, F, D)
        g = x.astype(np.float64) @ dense(fmt, cg, sg, gs).T
        u = x.astype(np.float64) @ dense(fmt, cu, su, gs).T
        _close(got, g * expit(g) * u)
        rows = np.array([7, 1])
        _close(orc.qgate_up_rows(fmt, gs, pack(fmt, cg), sg, pack(fmt, cu), su, x, F, D, rows), got[:, rows])


def pin_clamped_glu(orc):
    """Clamped SwiGLU (reading: silu(min(g, L)) * clamp(u, -L, L)): its closed
    cases and the structure a slip would break."""
    grid = np.linspace(-9, 9, 37)
    for g in grid:
        for u in grid:
            g, u = float(g), float(u)
            # a limit at or above both values changes nothing (the plain case is pinned above)
            assert orc.glu(1, 10.0, g, u) == orc.glu(0, 0.0, g, u)
            # limit 0 zeroes everything (the page: clamps "at any limit, including 0")
            assert orc.glu(1, 0.0, g, u) == 0.0
            # past the limit the value no longer depends on g (from above) or u (both sides)
            L = 2.0
            if g > L:
                assert orc.glu(1, L, g, u) == orc.glu(1, L, L, u)
            if u > L:
                assert orc.glu(1, L, g, u) == orc.glu(1, L, g, L)
            if u < -L:
                assert orc.glu(1, L, g, u) == orc.glu(1, L, g, -L)
    # the gate is capped from above only: a very negative gate keeps its own silu
    assert abs(orc.glu(1, 1.0, -5.0, 0.5) - (-5.0 * 0.0066928509242848554 * 0.5)) < 1e-15
    # sigmoid(1) = 0.7310585786300049 (tables): g = 5 and u = 7 both clamp to L = 1
    assert abs(orc.glu(1, 1.0, 5.0, 7.0) - 0.7310585786300049) < 1e-15
    # the clamp of u is symmetric: u = -7 clamps to -1
    assert abs(orc.glu(1, 1.0, 5.0, -7.0) + 0.7310585786300049) < 1e-15


def pin_gate_up_clamped(orc):
    rng = np.random.default_rng(37)
    for fmt in ALL_FMTS:
        F, D, s = 8, 128, 2
        gs = group_of(fmt, D)
        cg, cu = random_codes(fmt, F, D, rng), random_codes(fmt, F, D, rng)
        sg = draw_scales(fmt, F * (D // gs), rng, -3)
        su = draw_scales(fmt, F * (D // gs), rng, -3)
        x = rng.standard_normal((s, D)).astype(np.float32)
        g = x.astype(np.float64) @ dense(fmt, cg, sg, gs).T
        u = x.astype(np.float64) @ dense(fmt, cu, su, gs).T
        L = float(np.median(np.abs(u)))          # clamps about half of the values
        got = orc.qgate_up(fmt, gs, pack(fmt, cg), sg, pack(fmt, cu), su, x, F, D, act=1, limit=L)
        gc = np.minimum(g, L)
        _close(got, gc * expit(gc) * np.clip(u, -L, L))
        assert not orc.qgate_up(fmt, gs, pack(fmt, cg), sg, pack(fmt, cu), su, x, F, D, act=1, limit=0.0).any()


# --- step a5: the routed expert group ----------------------------------------

def _expert_store(fmt, E, D, F, rng):
    gs_gu, gs_dn = group_of(fmt, D), group_of(fmt, F)
    cg = [random_codes(fmt, F, D, rng) for _ in range(E)]
    cu = [random_codes(fmt, F, D, rng) for _ in range(E)]
    cd = [random_codes(fmt, D, F, rng) for _ in range(E)]
    sg = [draw_scales(fmt, F * (D // gs_gu), rng) for _ in range(E)]
    su = [draw_scales(fmt, F * (D // gs_gu), rng) for _ in range(E)]
    sd = [draw_scales(fmt, D * (F // gs_dn), rng) for _ in range(E)]
    packed = (np.concatenate([pack(fmt, c) for c in cg]), np.concatenate(sg),
              np.concatenate([pack(fmt, c) for c in cu]), np.concatenate(su),
              np.concatenate([pack(fmt, c) for c in cd]), np.concatenate(sd))
    dense_m = ([dense(fmt, cg[e], sg[e], gs_gu) for e in range(E)],
               [dense(fmt, cu[e], su[e], gs_gu) for e in range(E)],
               [dense(fmt, cd[e], sd[e], gs_dn) for e in range(E)])
    return packed, dense_m


def _dense_group(dense_m, x, ids, wts):
    G, U, Dn = dense_m
    s, k = ids.shape
    out = np.zeros((s, Dn[0].shape[0]))
    for t in range(s):
        for r in range(k):
            e = ids[t, r]
            g = G[e] @ x[t].astype(np.float64)
            u = U[e] @ x[t].astype(np.float64)
            out[t] += float(wts[t, r]) * (Dn[e] @ (g * expit(g) * u))
    return out


def pin_expert_group(orc):
    rng = np.random.default_rng(31)
    for fmt in ALL_FMTS:
        E, D, F, s, k = 5, 128, 64, 3, 2
        gs = group_of(fmt, D) if fmt != INT8_ROW else 0   # int8: one scale per row of each matrix
        packed, dense_m = _expert_store(fmt, E, D, F, rng)
        x = rng.standard_normal((s, D)).astype(np.float32)
        ids = np.array([[0, 3], [4, 4], [2, 1]], dtype=np.int32)   # token 1 routes expert 4 twice
        wts = rng.random((s, k)).astype(np.float32)
        got = orc.expert_group(fmt, gs, *packed, E, D, F, x, ids, wts)
        want = _dense_group(dense_m, x, ids, wts)
        _close(got, want, rtol=1e-11)
        # one-hot router weights reduce to one expert's MLP
        onehot = np.zeros_like(wts)
        onehot[:, 1] = 1.0
        _close(orc.expert_group(fmt, gs, *packed, E, D, F, x, ids, onehot),
               _dense_group(dense_m, x, ids[:, 1:], np.ones((s, 1), np.float32)), rtol=1e-11)
        # zero router weights give zeros
        assert not orc.expert_group(fmt, gs, *packed, E, D, F, x, ids, np.zeros_like(wts)).any()
        # the routed sum does not depend on the order of (id, weight) pairs
        perm = orc.expert_group(fmt, gs, *packed, E, D, F, x, ids[:, ::-1].copy(), wts[:, ::-1].copy())
        _close(perm, got, rtol=1e-12)
        # a sample of output columns equals those columns of the whole output
        cols = np.array([5, 127, 0])
        _close(orc.expert_group(fmt, gs, *packed, E, D, F, x, ids, wts, cols=cols), got[:, cols], rtol=1e-14)
        # clamped SwiGLU: a limit above every value is the plain group, limit 0 gives zeros
        _close(orc.expert_group(fmt, gs, *packed, E, D, F, x, ids, wts, act=1, limit=1e30), got, rtol=1e-15)
        assert not orc.expert_group(fmt, gs, *packed, E, D, F, x, ids, wts, act=1, limit=0.0).any()


# --- the router (softmax / sigmoid-with-bias top-k) -------------------------

def pin_route_selection(orc):
    """Hand-built keys: the k largest in decreasing order, equal keys lower index first."""
    l = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]], dtype=np.float32)
    assert orc.route(0, l, k=3)[0].tolist() == [[1, 2, 4]]
    assert orc.route(0, l, k=4)[0].tolist() == [[1, 2, 4, 3]]
    assert orc.route(0, l, k=5)[0].tolist() == [[1, 2, 4, 3, 0]]
    # the chosen set is the k largest on random rows (any k), ranks in decreasing logit
    rng = np.random.default_rng(53)
    L = rng.standard_normal((20, 64)).astype(np.float32)
    for k in (1, 4, 8, 64):
        ids, _ = orc.route(0, L, k=k)
        for t in range(20):
            want = np.argsort(-L[t].astype(np.float64), kind="stable")[:k]
            assert ids[t].tolist() == want.tolist()


def pin_route_softmax_weights(orc):
    """Softmax closed forms: ratios exp(l_i - l_j), a full set sums to 1, shift invariance, renorm."""
    rng = np.random.default_rng(59)
    L = (np.round(3 * rng.standard_normal((6, 32)) * 64) / 64).astype(np.float32)   # exact under + 4
    ids, w = orc.route(0, L, k=32, renorm=False)
    _close(w.sum(axis=1), np.ones(6), rtol=1e-14)
    for t in range(6):
        li = L[t, ids[t]].astype(np.float64)
        _close(w[t] / w[t, 0], np.exp(li - li[0]), rtol=1e-13)
    ids8, w8 = orc.route(0, L, k=8, renorm=False)
    _close(w8, w[:, :8], rtol=1e-14)                          # the same p, just fewer of them
    ids8r, w8r = orc.route(0, L, k=8, renorm=True, scale=2.5)
    _close(w8r, 2.5 * w8 / w8.sum(axis=1, keepdims=True), rtol=1e-14)
    assert (ids8r == ids8).all()
    _, ws = orc.route(0, L + np.float32(4.0), k=8, renorm=False)   # exact shift of every logit
    _close(ws, w8, rtol=1e-12)
    # equal logits: uniform
    _, wu = orc.route(0, np.zeros((1, 16), np.float32), k=16, renorm=False)
    _close(wu, np.full((1, 16), 1 / 16), rtol=1e-15)


def pin_route_sigmoid_bias(orc):
    """Sigmoid router: the bias picks, the unbiased scores weigh."""
    assert orc.sigmoid(0.0) == 0.5
    _close(orc.sigmoid(1.5) + orc.sigmoid(-1.5), 1.0, rtol=1e-15)
    _close(orc.sigmoid(2.0), 1 / (1 + np.exp(-2.0)), rtol=1e-15)
    l = np.zeros((1, 4), np.float32)
    b = np.array([0.0, 0.1, 0.0, 0.2], np.float32)
    ids, w = orc.route(1, l, b, k=2, renorm=False, scale=3.0)
    assert ids.tolist() == [[3, 1]]
    _close(w, [[1.5, 1.5]], rtol=1e-15)                         # 3 * sigmoid(0), bias not in the weight
    ids, w = orc.route(1, l, b, k=2, renorm=True)
    _close(w, [[0.5, 0.5]], rtol=1e-15)
    # a bias large enough overrides the logits; without bias the order follows the logits
    l2 = np.array([[2.0, -1.0, 0.5]], np.float32)
    assert orc.route(1, l2, np.zeros(3, np.float32), k=3)[0].tolist() == [[0, 2, 1]]
    assert orc.route(1, l2, np.array([0, 5, 0], np.float32), k=1)[0].tolist() == [[1]]
    ids, w = orc.route(1, l2, np.zeros(3, np.float32), k=2, renorm=True)
    s0, s2 = 1 / (1 + np.exp(-2.0)), 1 / (1 + np.exp(-0.5))
    _close(w, [[s0 / (s0 + s2), s2 / (s0 + s2)]], rtol=1e-14)


def pin_route_single_expert(orc):
    """One expert (E = k = 1): softmax weight 1, sigmoid weight sigmoid(l) or 1 renormalized, times scale."""
    l = np.array([[0.75], [-3.0]], np.float32)
    ids, w = orc.route(0, l, k=1, renorm=False, scale=2.0)
    assert ids.tolist() == [[0], [0]]
    _close(w, [[2.0], [2.0]], rtol=1e-15)
    ids, w = orc.route(1, l, np.array([0.3], np.float32), k=1, renorm=False, scale=2.0)
    assert ids.tolist() == [[0], [0]]
    _close(w, 2.0 / (1.0 + np.exp(-l.astype(np.float64))), rtol=1e-15)
    _, w = orc.route(1, l, np.array([0.3], np.float32), k=1, renorm=True, scale=2.0)
    _close(w, [[2.0], [2.0]], rtol=1e-15)


ALL_PINS = [pin_e2m1, pin_e8m0, pin_int4_nibbles, pin_int3_planes, pin_int8_bytes, pin_random_codes,
            pin_format_variants,
            pin_dequant_f32, pin_fixed_groups, pin_gemv_bruteforce, pin_zero_scales, pin_linearity,
            pin_integer_exact, pin_silu, pin_clamped_glu, pin_gate_up, pin_gate_up_clamped, pin_expert_group,
            pin_route_selection, pin_route_softmax_weights, pin_route_sigmoid_bias, pin_route_single_expert]
