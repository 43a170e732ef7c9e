"""The prefill GEMM's two-part split of x, restated from its definition and
checked on the CPU: the error bound the GEMM parity tests allow for it, and
the range the header states.

Definition (the cooperative-matrix reading): per activation row, p puts the
largest magnitude in [2^14, 2^15), clamped to [-126, 126]; a = x * 2^p (exact
in f32), hi = f16(a), lo = f16(a - hi) (the difference is exact in f32), and
the products run on hi + lo, scaled back by 2^-p.
"""
import numpy as np
import pytest

from weight_only_quantized_qgemv_gb300 import synth


def split(x):
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.abs(x).max())
    e = int((amax.view(np.uint32) >> 23) & 0xFF)
    p = 0 if (amax == 0 or e == 255) else (126 if e == 0 else 141 - e)
    p = max(-126, min(126, p))
    a = (x * np.float32(2.0 ** p)).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        hi = a.astype(np.float16)
        lo = (a - hi.astype(np.float32)).astype(np.float16)
    return p, a, hi, lo


@pytest.mark.parametrize("mag", [1e-33, 1e-25, 1e-12, 1e-3, 1.0, 7.5, 1e3, 1e12, 1e30, 1e34, 1e36, 3e37])
def test_split_error_is_22_bits(mag):
    """|a - hi - lo| <= 2^-22 |a| + 2^-25 per element, inside the stated range."""
    x = synth.draw_x(4, 4096, synth.generator(41)) * np.float32(mag)
    x[0, 7] = 0.0
    x[1, :100] *= np.float32(1e-6)              # small entries beside large ones
    for row in x:
        p, a, hi, lo = split(row)
        # [2^14, 2^15) unless p was clamped; always below the f16 overflow point here
        assert np.abs(a).max() < 65520.0 and np.isfinite(hi).all()
        if -126 < p < 126:
            assert 2.0 ** 14 <= np.abs(a).max() < 2.0 ** 15
        err = np.abs(a.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
        assert np.all(err <= 2.0 ** -22 * np.abs(a.astype(np.float64)) + 2.0 ** -25)
        # the dot product with any weights: within 2^-22 sum |x w| plus the absolute part
        w = synth.generator(43).standard_normal(row.size)
        got = (hi.astype(np.float64) + lo.astype(np.float64)) @ w * 2.0 ** -p
        want = row.astype(np.float64) @ w
        tol = 2.0 ** -22 * np.abs(row.astype(np.float64)) @ np.abs(w) + 2.0 ** -25 * 2.0 ** -p * np.abs(w).sum()
        assert abs(got - want) <= tol


def test_split_range_edges():
    """Every finite row fits (FLT_MAX takes p = -113).  Rows below 2^-112 take the
    clamp p = 126 and are scaled below 2^14; the split's error stays within
    2^-22 of each scaled element plus 2^-25 absolute, i.e. 2^-151 or less in
    x's units -- below f32's resolution -- down to rows of subnormals."""
    for mag in (1e35, 1e36, 3.0e38, np.finfo(np.float32).max):
        big = np.full(8, mag, dtype=np.float32)
        big[1] = -big[1]
        p, _, hi, _ = split(big)
        assert np.isfinite(hi).all() and p >= -126
    p, _, _, _ = split(np.full(4, np.finfo(np.float32).max, dtype=np.float32))
    assert p == -113
    for mag in (2.0 ** -108, 2.0 ** -113, 2.0 ** -120, 2.0 ** -137):
        row = (synth.draw_x(1, 512, synth.generator(47))[0] * np.float32(mag)).astype(np.float32)
        p, a, hi, lo = split(row)
        assert p == (126 if mag < 2.0 ** -112 else p) and p <= 126
        err = np.abs(a.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
        assert np.all(err <= 2.0 ** -22 * np.abs(a.astype(np.float64)) + 2.0 ** -25)
        err_x = err * 2.0 ** -p
        assert np.all(err_x <= 2.0 ** -22 * np.abs(row.astype(np.float64)) + 2.0 ** -151)
