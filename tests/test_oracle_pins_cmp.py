"""Pins for the oracle's comparisons, SELECT and packed-bit (b1) stores.

Readings (the Silk page, "AMDGPU Backend", section "Code Object Format",
names a threshold classification: a loaded u32, an unsigned threshold
comparison and a packed prediction store, and says no more): comparisons
give the int 1 or 0 (IEEE relations for floats, so a NaN makes all but !=
false; signed or unsigned 32-bit for ints); SELECT(c, a, b) is a where c is
nonzero; a b1 store puts (value != 0) at bit k % 32 of little-endian word
k / 32 for the element at bit offset k, and zeroes the last word's bits past
the last element. Each pin checks the oracle against numpy (comparison
ufuncs, where, packbits) or hand values. CPU only."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import specutil
from inputgen import workloads
from test_oracle_pins import _int_operands, _mixed_f32_bits

RNG_SEED = 20261204
REL = ["lt", "le", "gt", "ge", "eq", "ne"]
NP_REL = {"lt": np.less, "le": np.less_equal, "gt": np.greater, "ge": np.greater_equal,
          "eq": np.equal, "ne": np.not_equal}


def _rng(k=0):
    return np.random.default_rng(RNG_SEED + k)


def _run(ops, loads, stores, n):
    """Evaluate a one-block Command over n elements; loads: name -> (dtype,
    array); stores: name -> (src, dtype)."""
    spec_ops = [("load", k, dt) for k, (dt, _) in loads.items()]
    spec_ops += [("exec", ops)] + [("store", k, src, dt) for k, (src, dt) in stores.items()]
    views = {k: dict(strides=(1,), alloc=n) for k in loads}
    for k, (_, dt) in stores.items():
        views[k] = dict(strides=(1,), alloc=(n + 31) // 32 if dt == "b1" else n)
    spec = dict(name="t", seed=0, sizes=(n,), ops=spec_ops, views=views, inputs={})
    bufs = {k: a for k, (_, a) in loads.items()}
    for k, (_, dt) in stores.items():
        bufs[k] = specutil.sentinel_array(dt, views[k]["alloc"])
    oracle.OracleCommand(spec, bufs).eval_range()
    return bufs, spec


@pytest.mark.parametrize("rel", REL)
def test_float_comparisons_match_numpy(rel):
    """numpy's comparison ufuncs on float32 are the IEEE relations (NaN
    unordered, -0 == +0)."""
    rng = _rng(1)
    n = 1 << 16
    xb, yb = _mixed_f32_bits(rng, n), _mixed_f32_bits(rng, n)
    rng.shuffle(yb)
    yb[:4096] = xb[:4096]                              # equal pairs
    yb[4096:4608] = xb[4096:4608] ^ np.uint32(0x80000000)  # opposite signs, including +-0
    xb[5000:5010] = 0x7FC00000                         # NaNs
    yb[5010:5020] = 0xFFC00001
    x, y = xb.view(np.float32), yb.view(np.float32)
    bufs, _ = _run([(rel, "r", "x", "y")], {"x": ("f32", x), "y": ("f32", y)}, {"o": ("r", "i32")}, n)
    with np.errstate(invalid="ignore"):
        want = NP_REL[rel](x, y).astype(np.int32)
    assert (bufs["o"] == want).all()


@pytest.mark.parametrize("rel", REL)
def test_int_comparisons_match_numpy(rel):
    rng = _rng(2)
    n = 1 << 16
    x, y = _int_operands(rng, n), _int_operands(rng, n)
    rng.shuffle(y)
    y[:1000] = x[:1000]
    bufs, _ = _run([(rel, "r", "x", "y")], {"x": ("i32", x), "y": ("i32", y)}, {"o": ("r", "i32")}, n)
    assert (bufs["o"] == NP_REL[rel](x, y).astype(np.int32)).all()


@pytest.mark.parametrize("rel", ["ult", "ule", "ugt", "uge"])
def test_unsigned_comparisons_match_numpy(rel):
    rng = _rng(3)
    n = 1 << 16
    x, y = _int_operands(rng, n), _int_operands(rng, n)
    rng.shuffle(y)
    y[:1000] = x[:1000]
    bufs, _ = _run([(rel, "r", "x", "y")], {"x": ("i32", x), "y": ("i32", y)}, {"o": ("r", "i32")}, n)
    want = NP_REL[rel[1:]](x.view(np.uint32), y.view(np.uint32)).astype(np.int32)
    assert (bufs["o"] == want).all()
    # signed and unsigned orders differ exactly when the signs differ
    signed = NP_REL[rel[1:]](x, y)
    differ = (x < 0) != (y < 0)
    assert ((want.astype(bool) != signed) == (differ & (x != y))).all()


def test_comparison_hand_cases():
    L = oracle.lib()
    K = oracle.KINDS
    nan, p0, n0, one, inf = 0x7FC00000, 0, 0x80000000, 0x3F800000, 0x7F800000
    for rel in ("lt", "le", "gt", "ge", "eq"):
        assert L.orc_compare(K[rel], 0, nan, one) == 0 and L.orc_compare(K[rel], 0, one, nan) == 0
        assert L.orc_compare(K[rel], 0, nan, nan) == 0
    assert L.orc_compare(K["ne"], 0, nan, nan) == 1 and L.orc_compare(K["ne"], 0, nan, one) == 1
    assert L.orc_compare(K["eq"], 0, p0, n0) == 1 and L.orc_compare(K["lt"], 0, n0, p0) == 0
    assert L.orc_compare(K["le"], 0, inf, inf) == 1 and L.orc_compare(K["lt"], 0, one, inf) == 1
    # int: -1 < 0 signed, 0xFFFFFFFF > 0 unsigned; INT_MIN is the smallest signed, 2^31 unsigned
    assert L.orc_compare(K["lt"], 1, 0xFFFFFFFF, 0) == 1
    assert L.orc_compare(K["ugt"], 1, 0xFFFFFFFF, 0) == 1
    assert L.orc_compare(K["lt"], 1, 0x80000000, 0x7FFFFFFF) == 1
    assert L.orc_compare(K["ult"], 1, 0x7FFFFFFF, 0x80000000) == 1
    assert L.orc_compare(K["uge"], 1, 0xA0000000, 0xA0000000) == 1
    assert L.orc_compare(K["uge"], 1, 0x9FFFFFFF, 0xA0000000) == 0


def test_select_matches_numpy_where():
    """SELECT picks bit patterns: NaN payloads, -0 and int values pass
    unchanged; any nonzero condition counts as true."""
    rng = _rng(4)
    n = 1 << 15
    ab, bb = _mixed_f32_bits(rng, n), _mixed_f32_bits(rng, n)
    c = rng.integers(-3, 4, size=n).astype(np.int32)
    c[:8] = [0, 1, -1, 2**31 - 1, -2**31, 0, 7, 0]
    xi, yi = _int_operands(rng, n), _int_operands(rng, n)
    bufs, _ = _run([("select", "f", "a", "b", "c"), ("select", "i", "xi", "yi", "c")],
                   {"a": ("f32", ab.view(np.float32)), "b": ("f32", bb.view(np.float32)), "c": ("i32", c),
                    "xi": ("i32", xi), "yi": ("i32", yi)},
                   {"of": ("f", "f32"), "oi": ("i", "i32")}, n)
    assert (specutil.bits(bufs["of"]) == np.where(c != 0, ab, bb)).all()
    assert (bufs["oi"] == np.where(c != 0, xi, yi)).all()


@pytest.mark.parametrize("n", [1, 31, 32, 33, 1000, 4096, 4099])
def test_b1_store_matches_packbits(n):
    """Bits in element order, least significant first within each byte and
    little-endian words: numpy's packbits with bitorder 'little', read as
    u32. The last word's bits past n are 0, the words after it untouched."""
    rng = _rng(5 + n)
    x = rng.integers(-5, 5, size=n).astype(np.int32)
    bufs, _ = _run([("ne", "nz", "x", "zero")], {"x": ("i32", x), "zero": ("i32", np.zeros(n, np.int32))},
                   {"bits": ("nz", "b1")}, n)
    nb = (n + 31) // 32
    packed = np.packbits((x != 0).astype(np.uint8), bitorder="little")
    packed = np.concatenate([packed, np.zeros(nb * 4 - packed.size, np.uint8)]).view("<u4")
    assert (bufs["bits"].view(np.uint32) == packed).all()
    # the bit of an int value is value != 0, not its low bit
    bufs2, _ = _run([("add", "v", "x", "zero")], {"x": ("i32", np.full(n, 2, np.int32)),
                                                   "zero": ("i32", np.zeros(n, np.int32))},
                    {"bits": ("v", "b1")}, n)
    assert (bufs2["bits"].view(np.uint32)[: n // 32] == 0xFFFFFFFF).all()


def test_b1_points_and_class_rule():
    n = 100
    x = np.arange(n, dtype=np.int32) - 50
    spec = dict(name="p", seed=0, sizes=(n,),
                ops=[("load", "x", "i32"), ("scalar", "t", "i32", 10), ("exec", [("ge", "p", "x", "t")]),
                     ("store", "bits", "p", "b1")],
                views={"x": dict(strides=(1,), alloc=n), "bits": dict(strides=(1,), alloc=4)}, inputs={})
    bufs = {"x": x, "bits": specutil.sentinel_array("b1", 4)}
    oc = oracle.OracleCommand(spec, bufs)
    pts = oc.eval_points(np.array([0, 59, 60, 99]))
    assert pts["bits"].tolist() == [0, 0, 1, 1]
    # a float value cannot be stored as b1
    bad = dict(spec, ops=[("load", "f", "f32"), ("store", "bits", "f", "b1")],
               views={"f": dict(strides=(1,), alloc=n), "bits": dict(strides=(1,), alloc=4)})
    with pytest.raises(ValueError):
        oracle.OracleCommand(bad, {"f": np.zeros(n, np.float32), "bits": bufs["bits"]}).eval_range()


def test_threshold_workloads_match_numpy():
    for f in (workloads.threshold_u32, workloads.threshold_bits):
        spec = f(50_000)
        bufs = specutil.host_buffers(spec)
        oracle.OracleCommand(spec, bufs).eval_range()
        pred = bufs["x"].view(np.uint32) >= np.uint32(workloads.THRESHOLD)
        assert 0.3 < pred.mean() < 0.45
        if spec["name"] == "threshold_u32":
            assert (bufs["out"] == pred.astype(np.int32)).all()
        else:
            packed = np.packbits(pred.astype(np.uint8), bitorder="little")
            nb = (pred.size + 31) // 32
            packed = np.concatenate([packed, np.zeros(nb * 4 - packed.size, np.uint8)]).view("<u4")
            assert (bufs["bits"].view(np.uint32) == packed).all()


def test_planted_op_mistakes_are_caught():
    """Plausible mistakes in the new ops (each written here as the mistaken
    formula) disagree with the oracle on inputs the pins above use, so a pin
    would fail if the oracle made that mistake."""
    L = oracle.lib()
    u = lambda v: v & 0xFFFFFFFF  # noqa: E731
    s32 = lambda v: ((v + 2**31) % 2**32) - 2**31  # noqa: E731
    # int division flooring instead of truncating (-7 / 2 = -4)
    assert s32(L.orc_idiv(u(-7), 2)) != -7 // 2
    # x / 0 as 0 (a common convention) instead of -1
    assert L.orc_idiv(5, 0) != 0
    # an ordered != (false on NaN)
    assert L.orc_compare(oracle.KINDS["ne"], 0, 0x7FC00000, 0x3F800000) == 1
    # comparing signed where unsigned is asked
    assert L.orc_compare(oracle.KINDS["ult"], 1, 1, u(-1)) == 1 and L.orc_compare(oracle.KINDS["lt"], 1, 1, u(-1)) == 0
    # float -> int rounding to nearest instead of truncating (1.5 -> 2)
    assert L.orc_f2i(0x3FC00000) == 1
    # int -> float truncating instead of rounding (2^24 + 3 -> 2^24 + 4 under RNE)
    assert L.orc_i2f(16777219) == 0x4B800002
    # min as (a < b ? a : b): min(+0, -0) would be -0 only by accident of order
    assert L.orc_fmin(0, 0x80000000) == 0x80000000 and L.orc_fmax(0x80000000, 0) == 0
    # select testing only the low bit of the condition
    n = 4
    bufs, _ = _run([("select", "s", "a", "b", "c")],
                   {"a": ("i32", np.full(n, 1, np.int32)), "b": ("i32", np.full(n, 2, np.int32)),
                    "c": ("i32", np.array([2, -2, 0, 1], np.int32))}, {"o": ("s", "i32")}, n)
    assert bufs["o"].tolist() == [1, 1, 2, 1]  # c = 2 and -2 are true (low bit 0)
    # bits most significant first
    bufs, _ = _run([("ne", "nz", "x", "zero")], {"x": ("i32", np.array([1] + [0] * 31, np.int32)),
                                                   "zero": ("i32", np.zeros(32, np.int32))},
                   {"bits": ("nz", "b1")}, 32)
    assert bufs["bits"].view(np.uint32)[0] == 1  # element 0 is bit 0, not bit 31
