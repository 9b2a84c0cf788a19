"""Pins for the oracle's division, min/max, abs and conversion E ops.

rocRoller, "Design Overview", section "Expression": the operations an
expression supports are a list (division, minimum, maximum, absolute value
and conversions among them); the pages fix none of their special cases, so
the oracle takes IEEE 754-2019 for floats (division rounded once to nearest
even; minimumNumber / maximumNumber; abs clears the sign bit; conversions
round to nearest even, float to int truncates and saturates, NaN gives 0)
and, for int32 division by 0 and INT_MIN / -1, the results the RISC-V ISA
manual fixes for DIV (-1 and INT_MIN). Each pin here checks the oracle
against something other than itself: numpy's binary32 / int32 routines,
exact rationals, Python integers and hand-worked values. CPU only."""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import specutil
from test_oracle_pins import _frac, _int_operands, _mixed_f32_bits, _rne_binary32, _run_binop

RNG_SEED = 20261203


def _rng(k=0):
    return np.random.default_rng(RNG_SEED + k)


def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def _run_unop(eop, x, dt_in, dt_out):
    n = x.size
    spec = dict(name="unop", seed=0, sizes=(n,),
                ops=[("load", "x", dt_in), ("exec", [(eop, "y", "x", None)]), ("store", "out", "y", dt_out)],
                views={k: dict(strides=(1,), alloc=n) for k in ("x", "out")}, inputs={})
    bufs = {"x": x, "out": specutil.sentinel_array(dt_out, n)}
    oracle.OracleCommand(spec, bufs).eval_range()
    return bufs["out"]


# ---- float division ------------------------------------------------------------

def test_fdiv_matches_numpy_binary32():
    """numpy's float32 true_divide is the IEEE binary32 division (one
    rounding to nearest even, denormals kept, IEEE zeros and infinities)."""
    rng = _rng(1)
    n = 1 << 18
    xb, yb = _mixed_f32_bits(rng, n), _mixed_f32_bits(rng, n)
    rng.shuffle(yb)
    # zero, infinite and NaN divisors and dividends in every combination
    sp = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0x3F800000, 0x00000001], dtype=np.uint32)
    xs, ys = np.meshgrid(sp, sp)
    xb = np.concatenate([xb, xs.ravel()])
    yb = np.concatenate([yb, ys.ravel()])
    x, y = _f32(xb), _f32(yb)
    got = _run_binop("div", x.copy(), y.copy(), "f32")
    with np.errstate(all="ignore"):
        want = np.divide(x, y)
    ok = specutil.same_bits_nan_as_class(got, want, "f32")
    assert ok.all(), f"{(~ok).sum()} mismatches, first at {np.argmin(ok)}"


def test_fdiv_exact_rational():
    """Finite quotients equal the exact rational x / y rounded once to binary32
    (the zero's sign is the xor of the operands' signs)."""
    rng = _rng(2)
    xb, yb = _mixed_f32_bits(rng, 3000), _mixed_f32_bits(rng, 3000)
    rng.shuffle(yb)
    # ties and near-ties: 1 / 3, 2^-149 / 2 (halfway to zero), 3 * 2^-150 / 1
    xb = np.concatenate([xb, np.array([0x3F800000, 0x00000001, 0x00000003, 0x7F7FFFFF], dtype=np.uint32)])
    yb = np.concatenate([yb, np.array([0x40400000, 0x40000000, 0x3F000000, 0x3F000000], dtype=np.uint32)])
    fin = (((xb & 0x7F800000) != 0x7F800000) & ((yb & 0x7F800000) != 0x7F800000)
           & ((yb & 0x7FFFFFFF) != 0))
    xb, yb = xb[fin], yb[fin]
    got = specutil.bits(_run_binop("div", _f32(xb).copy(), _f32(yb).copy(), "f32"))
    for i in range(xb.size):
        q = _frac(int(xb[i])) / _frac(int(yb[i]))
        want = _rne_binary32(q, (int(xb[i]) >> 31) ^ (int(yb[i]) >> 31))
        assert int(got[i]) == want, (hex(int(xb[i])), hex(int(yb[i])), hex(int(got[i])), hex(want))


# ---- int division --------------------------------------------------------------

def _trunc_div(a: int, b: int) -> int:
    """Truncating integer division from the definition: |a| // |b| with the
    sign of a * b; the special cases of the reading taken for this op."""
    if b == 0:
        return -1
    q = abs(a) // abs(b)
    q = q if (a < 0) == (b < 0) else -q
    return ((q + 2**31) % 2**32) - 2**31  # INT_MIN / -1 wraps to INT_MIN


def test_idiv_truncates_toward_zero():
    rng = _rng(3)
    n = 1 << 15
    x, y = _int_operands(rng, n), _int_operands(rng, n)
    rng.shuffle(y)
    # small divisors make non-trivial quotients; include every sign pair
    y[n // 2:] = rng.integers(-40, 41, size=n - n // 2).astype(np.int32)
    got = _run_binop("div", x, y, "i32")
    want = np.array([_trunc_div(int(a), int(b)) for a, b in zip(x, y)], dtype=np.int64).astype(np.int32)
    assert (got == want).all()


def test_idiv_hand_cases():
    L = oracle.lib()
    u = lambda v: v & 0xFFFFFFFF  # noqa: E731
    cases = [(7, 2, 3), (-7, 2, -3), (7, -2, -3), (-7, -2, 3), (1, 0, -1), (0, 0, -1), (-5, 0, -1),
             (-2**31, -1, -2**31), (-2**31, 1, -2**31), (2**31 - 1, -1, -(2**31 - 1)), (0, 5, 0), (4, 5, 0)]
    for a, b, q in cases:
        assert L.orc_idiv(u(a), u(b)) == u(q), (a, b)


# ---- min / max -----------------------------------------------------------------

def test_fmin_fmax_exact_order():
    """For two numbers, min/max is the operand whose exact value is smaller /
    larger; equal nonzero values are the same encoding."""
    rng = _rng(4)
    xb, yb = _mixed_f32_bits(rng, 1 << 12), _mixed_f32_bits(rng, 1 << 12)
    rng.shuffle(yb)
    yb[:512] = xb[:512] ^ np.uint32(0x80000000)  # opposite signs
    yb[512:768] = xb[512:768]                    # equal
    num = ((xb & 0x7FFFFFFF) <= 0x7F800000) & ((yb & 0x7FFFFFFF) <= 0x7F800000)
    xb, yb = xb[num], yb[num]
    gmin = specutil.bits(_run_binop("min", _f32(xb).copy(), _f32(yb).copy(), "f32"))
    gmax = specutil.bits(_run_binop("max", _f32(xb).copy(), _f32(yb).copy(), "f32"))
    for i in range(xb.size):
        a, b = int(xb[i]), int(yb[i])
        fa, fb = float(_f32([a])[0]), float(_f32([b])[0])
        if fa == fb and fa == 0.0:
            continue  # signed zeros: next test
        lo, hi = (a, b) if fa < fb else (b, a)
        if fa == fb:
            lo = hi = a
        assert int(gmin[i]) == lo and int(gmax[i]) == hi, (hex(a), hex(b))


def test_fmin_fmax_signed_zero_and_nan():
    """-0 counts as less than +0; a NaN operand loses to a number; two NaNs
    give a NaN (IEEE 754-2019, minimumNumber / maximumNumber)."""
    L = oracle.lib()
    P0, N0, QN, SN, ONE, NONE = 0, 0x80000000, 0x7FC00000, 0x7F800001, 0x3F800000, 0xBF800000
    for a, b in ((P0, N0), (N0, P0)):
        assert L.orc_fmin(a, b) == N0 and L.orc_fmax(a, b) == P0
    for nan in (QN, SN, QN | 0x80000000):
        for x in (ONE, NONE, P0, N0, 0x7F800000, 0xFF800000, 1):
            assert L.orc_fmin(nan, x) == x and L.orc_fmin(x, nan) == x
            assert L.orc_fmax(nan, x) == x and L.orc_fmax(x, nan) == x
        assert (L.orc_fmin(nan, QN) & 0x7FFFFFFF) > 0x7F800000
        assert (L.orc_fmax(QN, nan) & 0x7FFFFFFF) > 0x7F800000


def test_fmin_fmax_match_numpy_away_from_zero_ties():
    """numpy's fmin/fmax ignore a NaN operand like minimumNumber; they leave
    the sign of a zero tie open, so those pairs are left to the hand test."""
    rng = _rng(5)
    n = 1 << 16
    xb, yb = _mixed_f32_bits(rng, n), _mixed_f32_bits(rng, n)
    rng.shuffle(yb)
    keep = ~(((xb & 0x7FFFFFFF) == 0) & ((yb & 0x7FFFFFFF) == 0))
    x, y = _f32(xb[keep]), _f32(yb[keep])
    for eop, ref in (("min", np.fmin), ("max", np.fmax)):
        got = _run_binop(eop, x.copy(), y.copy(), "f32")
        ok = specutil.same_bits_nan_as_class(got, ref(x, y), "f32")
        assert ok.all(), (eop, (~ok).sum())


def test_imin_imax_match_numpy():
    rng = _rng(6)
    n = 1 << 16
    x, y = _int_operands(rng, n), _int_operands(rng, n)
    rng.shuffle(y)
    assert (_run_binop("min", x, y, "i32") == np.minimum(x, y)).all()
    assert (_run_binop("max", x, y, "i32") == np.maximum(x, y)).all()


# ---- abs -------------------------------------------------------------------------

def test_fabs_clears_sign_bit():
    rng = _rng(7)
    xb = _mixed_f32_bits(rng, 1 << 14)
    got = specutil.bits(_run_unop("abs", _f32(xb).copy(), "f32", "f32"))
    assert (got == (xb & np.uint32(0x7FFFFFFF))).all()
    # numpy agrees on every non-NaN value
    nn = (xb & 0x7FFFFFFF) <= 0x7F800000
    assert (got[nn] == specutil.bits(np.abs(_f32(xb)))[nn]).all()


def test_iabs_mod_2_32():
    rng = _rng(8)
    x = _int_operands(rng, 1 << 14)
    got = _run_unop("abs", x, "i32", "i32")
    want = np.array([((abs(int(v)) + 2**31) % 2**32) - 2**31 for v in x], dtype=np.int64).astype(np.int32)
    assert (got == want).all()
    assert oracle.lib().orc_iabs(0x80000000) == 0x80000000


# ---- conversions -----------------------------------------------------------------

def test_i2f_rounds_to_nearest_even():
    """int32 -> binary32: numpy's astype is the IEEE conversion; the exact
    rational rounding covers every tie region above 2^24."""
    rng = _rng(9)
    x = _int_operands(rng, 1 << 16)
    # values around each power of two from 2^24 up, where ties occur
    ties = np.array([s * ((1 << k) + d) for k in range(24, 31) for d in (-3, -2, -1, 0, 1, 2, 3, 5, 64, 127, 128, 129)
                     for s in (1, -1)], dtype=np.int64)
    x = np.concatenate([x, ties.astype(np.int32), np.array([2**31 - 1, -2**31, 16777217, 16777219], dtype=np.int32)])
    got = specutil.bits(_run_unop("to_f32", x, "i32", "f32"))
    assert (got == specutil.bits(x.astype(np.float32))).all()
    for i in range(0, x.size, 97):
        assert int(got[i]) == _rne_binary32(Fraction(int(x[i])), 0)


def _f2i_ref(bits: int) -> int:
    """binary32 -> int32 from the definition: truncate the exact value toward
    zero, saturate to [INT_MIN, INT_MAX]; NaN -> 0."""
    if (bits & 0x7FFFFFFF) > 0x7F800000:
        return 0
    if (bits & 0x7FFFFFFF) == 0x7F800000:
        return 2**31 - 1 if bits >> 31 == 0 else -2**31
    t = math.trunc(_frac(bits))
    return max(-2**31, min(2**31 - 1, t))


def test_f2i_truncates_and_saturates():
    rng = _rng(10)
    xb = _mixed_f32_bits(rng, 1 << 14)
    # around the int32 range ends and small halves
    edge = np.array([0x4F000000, 0x4EFFFFFF, 0xCF000000, 0xCF000001, 0x3F000000, 0xBF000000, 0x3FC00000,
                     0xBFC00000, 0x3F7FFFFF, 0x7FC00000, 0xFFC00000, 0x7F800000, 0xFF800000, 0x80000000],
                    dtype=np.uint32)
    xb = np.concatenate([xb, edge])
    got = _run_unop("to_i32", _f32(xb).copy(), "f32", "i32")
    want = np.array([_f2i_ref(int(b)) for b in xb], dtype=np.int64).astype(np.int32)
    assert (got == want).all()
    # numpy agrees where its cast is defined (inside the int32 range)
    with np.errstate(invalid="ignore"):
        inside = np.abs(_f32(xb).astype(np.float64)) < 2**31
    assert (got[inside] == np.trunc(_f32(xb)[inside]).astype(np.int32)).all()


def test_identity_conversions_and_round_trip():
    """to_f32 of a float and to_i32 of an int are the identity; |n| <= 2^24
    survives int -> float -> int."""
    rng = _rng(11)
    xb = _mixed_f32_bits(rng, 4096)
    assert (specutil.bits(_run_unop("to_f32", _f32(xb).copy(), "f32", "f32")) == xb).all()
    xi = _int_operands(rng, 4096)
    assert (_run_unop("to_i32", xi, "i32", "i32") == xi).all()
    small = rng.integers(-2**24, 2**24 + 1, size=4096).astype(np.int32)
    n = small.size
    spec = dict(name="rt", seed=0, sizes=(n,),
                ops=[("load", "x", "i32"), ("exec", [("to_f32", "f", "x", None), ("to_i32", "y", "f", None)]),
                     ("store", "out", "y", "i32")],
                views={k: dict(strides=(1,), alloc=n) for k in ("x", "out")}, inputs={})
    bufs = {"x": small, "out": specutil.sentinel_array("i32", n)}
    oracle.OracleCommand(spec, bufs).eval_range()
    assert (bufs["out"] == small).all()


def test_mixed_class_rules():
    """Binary ops need operands of one class; conversions change the class;
    a store's type must match its value's class."""
    n = 4
    base = {k: dict(strides=(1,), alloc=n) for k in ("x", "i", "out")}
    bad = dict(name="bad", seed=0, sizes=(n,),
               ops=[("load", "x", "f32"), ("load", "i", "i32"), ("exec", [("min", "y", "x", "i")]),
                    ("store", "out", "y", "f32")], views=base, inputs={})
    bufs = {"x": np.zeros(n, np.float32), "i": np.zeros(n, np.int32), "out": specutil.sentinel_array("f32", n)}
    with pytest.raises(ValueError):
        oracle.OracleCommand(bad, bufs).eval_range()
    good = dict(bad, ops=[("load", "x", "f32"), ("load", "i", "i32"),
                          ("exec", [("to_f32", "fi", "i", None), ("max", "y", "x", "fi")]),
                          ("store", "out", "y", "f32")])
    bufs["x"][:] = [-1.5, 2.0, -0.0, 7.25]
    bufs["i"][:] = [-2, 3, 0, 7]
    oracle.OracleCommand(good, bufs).eval_range()
    assert specutil.bits(bufs["out"]).tolist() == specutil.bits(np.array([-1.5, 3.0, 0.0, 7.25], np.float32)).tolist()
