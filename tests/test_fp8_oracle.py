"""The oracle's e4m3 quantiser and W8A8 base against the format's definition.

Every one of the 256 codes is decoded from its bit fields (sign, 4 exponent bits with bias
7, 3 mantissa bits; exponent 0 is subnormal, S.1111.111 is NaN): each finite value rounds
to itself, each midpoint between neighbours rounds to the one with an even mantissa,
values past 448 saturate.  The per-row and per-column scales put the largest magnitude at
448 exactly, the relative error of a normal value is at most 2^-4, and a base whose
inputs are already on the e4m3 grid (scale 1) equals the plain product.
"""
import numpy as np
import pytest

import oracle
from oracle import fp8


def decode(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


FINITE = sorted({decode(c) for c in range(256) if not np.isnan(decode(c))})


def test_decoder_facts():
    pos = [v for v in FINITE if v > 0]
    assert max(pos) == 448.0 and min(pos) == 2.0 ** -9
    assert len(pos) == 126 and len(FINITE) == 253  # 126 positive, 126 negative, zero


def rounding_pins(rnd):
    """Round trip, midpoints to even, nearest neighbours, saturation; AssertionError on a
    failure."""
    vals = np.array(FINITE, dtype=np.float32)
    assert np.array_equal(rnd(vals), vals.astype(np.float64))
    pos = [v for v in FINITE if v >= 0]
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = np.float32((lo + hi) / 2)  # exact in fp32
        lo_even = (int(round(lo / (hi - lo))) % 2) == 0 if lo > 0 else True
        want = lo if lo_even else hi
        assert rnd(mid) == want, (lo, hi)
        assert rnd(-mid) == -want
        # just off the midpoint goes to the nearer neighbour
        assert rnd(np.nextafter(mid, np.float32(0))) == lo
        assert rnd(np.nextafter(mid, np.float32(1e9))) == hi
    for big in (448.0, 449.0, 464.0, 479.9, 480.0, 1e6):
        assert rnd(big) == 448.0 and rnd(-big) == -448.0
    return True


def test_round_trip_midpoints_and_saturation():
    assert rounding_pins(fp8.e4m3_round)


def _truncating(v):  # mistake: rounds toward zero
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6)
    q = np.exp2(e - 3)
    return np.copysign(np.minimum(np.floor(a / q) * q, 448.0), v)


def _half_up(v):  # mistake: ties away from zero
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6)
    q = np.exp2(e - 3)
    return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, 448.0), v)


def _no_saturation(v):  # mistake: rounds past 448 instead of saturating
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6)
    q = np.exp2(e - 3)
    return np.copysign(np.rint(a / q) * q, v)


def _no_subnormals(v):  # mistake: the normal quantum below 2^-6 too
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = np.exp2(e - 3)
    return np.copysign(np.minimum(np.rint(a / q) * q, 448.0), v)


@pytest.mark.parametrize("mutant", [_truncating, _half_up, _no_saturation, _no_subnormals])
def test_rounding_pins_catch_planted_mistakes(mutant):
    with pytest.raises(AssertionError):
        rounding_pins(mutant)


def test_scales_and_error_bound():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((16, 300)) * rng.uniform(0.01, 50, size=(16, 1))).astype(np.float32)
    x[3] = 0.0
    xq, sx = fp8.quantize_rows(x)
    assert sx[3] == 1.0 and not xq[3].any()
    for i in range(16):
        if i != 3:
            assert np.abs(xq[i]).max() == 448.0
    deq = xq * sx[:, None]
    normal = np.abs(xq) >= 2.0 ** -6
    rel = np.abs(deq - x)[normal] / np.abs(x)[normal]
    assert rel.max() <= 2.0 ** -4 + 1e-7
    assert np.abs(deq - x)[~normal].max() <= 2.0 ** -10 * sx.max()
    W = x.T.copy()
    wq, sw = fp8.quantize_cols(W)
    assert np.array_equal(wq, xq.T) and np.array_equal(sw, sx)


def test_base_on_the_grid_equals_the_plain_product():
    rng = np.random.default_rng(1)
    grid = np.array(FINITE)
    x = rng.choice(grid, size=(9, 40))
    x[:, 0] = 448.0  # every row's largest magnitude is 448: scale 1
    W = rng.choice(grid, size=(40, 7))
    W[0, :] = -448.0
    base = fp8.base_w8a8(x.astype(np.float32), W.astype(np.float32))
    table = oracle.SlotTable([None], 40, 7)
    plain = oracle.forward_rows(x, W, table, np.full(9, -1, np.int32))
    assert np.array_equal(base, plain)
