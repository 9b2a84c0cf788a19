"""Pins for the CPU oracle, against things other than the oracle itself:
hand-worked cases (tests/golden), exact rational arithmetic, numpy/torch
library routines for the special cases they cover, algebraic invariants and
brute force over small strided views. CPU only."""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from inputgen import workloads
import specutil

RNG_SEED = 20261202


def _rng(k=0):
    return np.random.default_rng(RNG_SEED + k)


def _mixed_f32_bits(rng, n):
    """Random binary32 patterns: raw bits, nearby exponents, subnormals, edges."""
    raw = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    k = n // 4
    # operands of similar magnitude (cancellation and ties in sums)
    near = (rng.integers(0x3E000000, 0x41000000, size=k, dtype=np.uint64).astype(np.uint32)
            | (rng.integers(0, 2, size=k, dtype=np.uint64).astype(np.uint32) << 31))
    raw[:k] = near
    # subnormals and tiny normals
    sub = rng.integers(0, 0x01000000, size=k, dtype=np.uint64).astype(np.uint32)
    raw[k:2 * k] = sub | (rng.integers(0, 2, size=k, dtype=np.uint64).astype(np.uint32) << 31)
    edges = np.array([0, 0x80000000, 1, 0x80000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0xFF7FFFFF,
                      0x7F800000, 0xFF800000, 0x3F800000, 0xBF800000, 0x33800000, 0x34000000],
                     dtype=np.uint32)
    raw[2 * k:2 * k + edges.size] = edges
    return raw


def _binop_spec(n, eop, dt="f32"):
    st = (1,)
    return dict(name="binop", seed=0, sizes=(n,),
                ops=[("load", "x", dt), ("load", "y", dt), ("exec", [(eop, "z", "x", "y")]),
                     ("store", "out", "z", dt)],
                views={k: dict(strides=st, alloc=n) for k in ("x", "y", "out")}, inputs={})


def _run_binop(eop, x, y, dt):
    spec = _binop_spec(x.size, eop, dt)
    bufs = {"x": x, "y": y, "out": specutil.sentinel_array(dt, x.size)}
    oracle.OracleCommand(spec, bufs).eval_range()
    return bufs["out"]


# ---- float E ops ---------------------------------------------------------

@pytest.mark.parametrize("eop", ["add", "sub", "mul"])
def test_f32_ops_match_numpy_binary32(eop):
    """numpy's binary32 ufuncs are IEEE operations in single precision (no
    contraction, no flush to zero): an independent implementation of one
    rounding per op."""
    rng = _rng(1)
    n = 1 << 18
    xb = _mixed_f32_bits(rng, n)
    yb = _mixed_f32_bits(rng, n)
    rng.shuffle(yb)
    x, y = xb.view(np.float32), yb.view(np.float32)
    got = _run_binop(eop, x.copy(), y.copy(), "f32")
    with np.errstate(all="ignore"):
        want = {"add": np.add, "sub": np.subtract, "mul": np.multiply}[eop](x, y)
    ok = specutil.same_bits_nan_as_class(got, want, "f32")
    assert ok.all(), f"{(~ok).sum()} mismatches, first at {np.argmin(ok)}"


def _rne_binary32(q: Fraction, zero_sign: int) -> int:
    """Exact rational -> binary32 bits, round to nearest even (IEEE 754 4.3.1),
    written from the definition with integer arithmetic only."""
    if q == 0:
        return zero_sign << 31
    sign = 1 if q < 0 else 0
    a = -q if sign else q
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    qe = max(e, -126) - 23
    m = a / (Fraction(2) ** qe)
    M = m.numerator // m.denominator
    rem = m - M
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and M % 2 == 1):
        M += 1
    if M == 0:
        return sign << 31
    if M == 1 << 24:
        M >>= 1
        qe += 1
    if M < (1 << 23):  # subnormal
        return (sign << 31) | M
    E = qe + 23
    if E > 127:
        return (sign << 31) | 0x7F800000
    return (sign << 31) | ((E + 127) << 23) | (M - (1 << 23))


def _frac(bits_u32: int) -> Fraction:
    f = float(np.array([bits_u32], dtype=np.uint32).view(np.float32)[0])
    return Fraction(f)


@pytest.mark.parametrize("eop", ["add", "sub", "mul"])
def test_f32_ops_exact_rational(eop):
    """Per-op results equal the exact rational result rounded once to binary32."""
    rng = _rng(2)
    xb = _mixed_f32_bits(rng, 3000)
    yb = _mixed_f32_bits(rng, 3000)
    rng.shuffle(yb)
    # finite operands only; ties: 1 + 2^-24 and 1 + 3*2^-24
    extra_x = np.array([0x3F800000, 0x3F800000, 0x00000001, 0x80000000, 0x7F7FFFFF, 0x00800000],
                       dtype=np.uint32)
    extra_y = np.array([0x33800000, 0x34400000, 0x00000001, 0x80000000, 0x7F7FFFFF, 0x80000001],
                       dtype=np.uint32)
    xb = np.concatenate([xb, extra_x])
    yb = np.concatenate([yb, extra_y])
    fin = ((xb & 0x7F800000) != 0x7F800000) & ((yb & 0x7F800000) != 0x7F800000)
    xb, yb = xb[fin], yb[fin]
    got = specutil.bits(_run_binop(eop, xb.view(np.float32).copy(), yb.view(np.float32).copy(), "f32"))
    for i in range(xb.size):
        xv, yv = _frac(int(xb[i])), _frac(int(yb[i]))
        sx, sy = int(xb[i]) >> 31, int(yb[i]) >> 31
        if eop == "add":
            q, zs = xv + yv, (1 if (sx and sy) else 0)
        elif eop == "sub":
            q, zs = xv - yv, (1 if (sx and not sy) else 0)
        else:
            q, zs = xv * yv, sx ^ sy
        want = _rne_binary32(q, zs)
        assert int(got[i]) == want, (eop, hex(int(xb[i])), hex(int(yb[i])), hex(int(got[i])), hex(want))


def test_f32_invariants():
    rng = _rng(3)
    n = 1 << 16
    xb = _mixed_f32_bits(rng, n)
    yb = _mixed_f32_bits(rng, n)
    fin = ((xb & 0x7F800000) != 0x7F800000) & ((yb & 0x7F800000) != 0x7F800000)
    x, y = xb[fin].view(np.float32).copy(), yb[fin].view(np.float32).copy()
    b = specutil.bits
    # commutativity, bitwise
    assert (b(_run_binop("add", x, y, "f32")) == b(_run_binop("add", y, x, "f32"))).all()
    assert (b(_run_binop("mul", x, y, "f32")) == b(_run_binop("mul", y, x, "f32"))).all()
    one = np.ones_like(x)
    zero = np.zeros_like(x)
    assert (b(_run_binop("mul", x, one, "f32")) == b(x)).all()
    # x - x == +0 for finite x
    assert (b(_run_binop("sub", x, x.copy(), "f32")) == 0).all()
    # x + 0 == x except x = -0, which gives +0
    got = b(_run_binop("add", x, zero, "f32"))
    want = np.where(b(x) == 0x80000000, 0, b(x))
    assert (got == want).all()


def test_neg_is_sign_flip_and_involution():
    rng = _rng(4)
    xb = _mixed_f32_bits(rng, 1 << 14)
    n = xb.size
    spec = dict(name="neg", seed=0, sizes=(n,),
                ops=[("load", "x", "f32"), ("exec", [("neg", "y", "x", None), ("neg", "z", "y", None)]),
                     ("store", "oy", "y", "f32"), ("store", "oz", "z", "f32")],
                views={k: dict(strides=(1,), alloc=n) for k in ("x", "oy", "oz")}, inputs={})
    bufs = {"x": xb.view(np.float32), "oy": specutil.sentinel_array("f32", n),
            "oz": specutil.sentinel_array("f32", n)}
    oracle.OracleCommand(spec, bufs).eval_range()
    assert (specutil.bits(bufs["oy"]) == (xb ^ np.uint32(0x80000000))).all()
    assert (specutil.bits(bufs["oz"]) == xb).all()


# ---- int32 E ops -----------------------------------------------------------

INT_EDGES = np.array([0, 1, -1, 2**31 - 1, -2**31, 0x10000, -0x10000, 3, 7], dtype=np.int64)


def _int_operands(rng, n):
    x = rng.integers(-2**31, 2**31, size=n, dtype=np.int64)
    x[:INT_EDGES.size] = INT_EDGES
    return x.astype(np.int32)


@pytest.mark.parametrize("eop", ["add", "sub", "mul"])
def test_i32_ops_are_mod_2_32(eop):
    """Results equal the exact integer result reduced modulo 2^32."""
    rng = _rng(5)
    n = 1 << 16
    x, y = _int_operands(rng, n), _int_operands(rng, n)
    rng.shuffle(y)
    got = _run_binop(eop, x, y, "i32").view(np.uint32).astype(np.uint64)
    xi, yi = x.astype(object), y.astype(object)
    exact = {"add": xi + yi, "sub": xi - yi, "mul": xi * yi}[eop]
    want = np.array([int(v) % (1 << 32) for v in exact], dtype=np.uint64)
    assert (got == want).all()


def test_i32_invariants():
    rng = _rng(6)
    n = 1 << 14
    x, y = _int_operands(rng, n), _int_operands(rng, n)
    spec = dict(name="inv", seed=0, sizes=(n,),
                ops=[("load", "x", "i32"), ("load", "y", "i32"),
                     ("exec", [("add", "s", "x", "y"), ("sub", "r", "s", "y"),
                               ("neg", "nx", "x", None), ("neg", "nnx", "nx", None),
                               ("mul", "xy", "x", "y"), ("mul", "yx", "y", "x")]),
                     ("store", "o_r", "r", "i32"), ("store", "o_nnx", "nnx", "i32"),
                     ("store", "o_xy", "xy", "i32"), ("store", "o_yx", "yx", "i32"),
                     ("store", "o_nx", "nx", "i32")],
                views={k: dict(strides=(1,), alloc=n)
                       for k in ("x", "y", "o_r", "o_nnx", "o_xy", "o_yx", "o_nx")}, inputs={})
    bufs = {"x": x, "y": y}
    for k in ("o_r", "o_nnx", "o_xy", "o_yx", "o_nx"):
        bufs[k] = specutil.sentinel_array("i32", n)
    oracle.OracleCommand(spec, bufs).eval_range()
    assert (bufs["o_r"] == x).all()            # x + y - y == x
    assert (bufs["o_nnx"] == x).all()          # -(-x) == x
    assert (bufs["o_xy"] == bufs["o_yx"]).all()
    # Neg(INT_MIN) == INT_MIN; INT_MAX + 1 == INT_MIN; 0x10000 * 0x10000 == 0
    i = int(np.where(x == -2**31)[0][0])
    assert bufs["o_nx"][i] == -2**31
    L = oracle.lib()
    assert L.orc_iadd(0x7FFFFFFF, 1) == 0x80000000
    assert L.orc_imul(0x10000, 0x10000) == 0
    assert L.orc_ineg(0x80000000) == 0x80000000


# ---- conversions -----------------------------------------------------------

def _dense_f32_patterns():
    """Every upper half (sign, exponent, top mantissa bits) with low halves
    around both rounding positions (ties at 0x1000 for binary16 normals and at
    0x8000 for bfloat16), plus random low halves."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x3000,
                     0x5000, 0x7FFF, 0x8000, 0x8001, 0x9000, 0xC000, 0xF000, 0xFFFF],
                    dtype=np.uint32)
    rnd = _rng(7).integers(0, 1 << 16, size=16, dtype=np.uint64).astype(np.uint32)
    lows = np.concatenate([lows, rnd])
    return (hi[:, None] | lows[None, :]).ravel()


def test_f32_to_f16_matches_numpy():
    x = _dense_f32_patterns()
    got = oracle.f32_to_f16_bits(x)
    with np.errstate(all="ignore"):
        want = x.view(np.float32).astype(np.float16).view(np.uint16)
    ok = specutil.same_bits_nan_as_class(got, want, "f16")
    assert ok.all(), hex(int(x[np.argmin(ok)]))


def test_f32_to_bf16_matches_torch():
    x = _dense_f32_patterns()
    got = oracle.f32_to_bf16_bits(x)
    want = (torch.from_numpy(x.view(np.float32).copy()).to(torch.bfloat16)
            .view(torch.int16).numpy().view(np.uint16))
    ok = specutil.same_bits_nan_as_class(got, want, "bf16")
    assert ok.all(), hex(int(x[np.argmin(ok)]))


def _widen(dt, raw16):
    n = raw16.size
    spec = dict(name="widen", seed=0, sizes=(n,),
                ops=[("load", "x", dt), ("store", "out", "x", "f32")],
                views={k: dict(strides=(1,), alloc=n) for k in ("x", "out")}, inputs={})
    bufs = {"x": raw16.view(specutil.NP[dt]), "out": specutil.sentinel_array("f32", n)}
    oracle.OracleCommand(spec, bufs).eval_range()
    return bufs["out"]


def test_f16_widening_exhaustive():
    raw = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = _widen("f16", raw)
    want = raw.view(np.float16).astype(np.float32)
    assert specutil.same_bits_nan_as_class(got, want, "f32").all()


def test_bf16_widening_exhaustive():
    raw = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = _widen("bf16", raw)
    want = torch.from_numpy(raw.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert specutil.same_bits_nan_as_class(got, want, "f32").all()


# ---- hand-worked cases -------------------------------------------------------

@pytest.mark.parametrize("case", sorted(specutil.golden_cases()))
def test_golden_hand_case(case):
    spec, bufs, expect = specutil.golden_spec(specutil.golden_cases()[case])
    oracle.OracleCommand(spec, bufs).eval_range()
    dts = workloads.tensor_dtypes(spec)
    for name, want in expect.items():
        got = bufs[name]
        assert (specutil.bits(got) == specutil.bits(want)).all(), (name, got, want)
    # the points API gives the same values
    pts = oracle.OracleCommand(spec, {k: v.copy() for k, v in bufs.items()}).eval_points(
        np.arange(int(np.prod(spec["sizes"]))))
    for name, want in expect.items():
        if spec["views"][name]["strides"] == workloads._dense(spec["sizes"])[0]:
            assert (specutil.bits(pts[name]) == specutil.bits(want)).all()
    del dts


# ---- brute force over small strided views -----------------------------------

def _view(buf, sizes, strides):
    return np.lib.stride_tricks.as_strided(
        buf, shape=sizes, strides=[s * buf.itemsize for s in strides], writeable=False)


def _modes(rows, cols):
    """(strides, alloc) pairs: row-major with padded leading dims, and
    transposed views of a cols x rows buffer with padded leading dims."""
    out = []
    for ld in (cols, cols + 1, cols + 3):
        out.append(((ld, 1), (rows - 1) * ld + cols))
    for ld in (rows, rows + 2):
        out.append(((1, ld), (cols - 1) * ld + rows))
    return out


@pytest.mark.parametrize("rows", [1, 2, 3, 5, 7])
@pytest.mark.parametrize("cols", [1, 2, 4, 6, 9])
def test_strided_views_brute_force(rows, cols):
    """Every combination of view modes for A, B and out on a rows x cols
    Command out = A*B - A: values match numpy over strided views, every
    element of the output view is written and nothing outside it (guard bands
    before and after each buffer) changes."""
    rng = _rng(100 + rows * 10 + cols)
    modes = _modes(rows, cols)
    G = 4  # guard elements each side
    for ma in modes:
        for mb in modes:
            for mo in modes[:4]:
                spec = dict(name="bf", seed=0, sizes=(rows, cols),
                            ops=[("load", "A", "f32"), ("load", "B", "f32"),
                                 ("exec", [("mul", "AB", "A", "B"), ("sub", "r", "AB", "A")]),
                                 ("store", "out", "r", "f32")],
                            views={"A": dict(strides=ma[0], alloc=ma[1]),
                                   "B": dict(strides=mb[0], alloc=mb[1]),
                                   "out": dict(strides=mo[0], alloc=mo[1])}, inputs={})
                fullA = rng.standard_normal(ma[1] + 2 * G).astype(np.float32)
                fullB = rng.standard_normal(mb[1] + 2 * G).astype(np.float32)
                fullO = specutil.sentinel_array("f32", mo[1] + 2 * G)
                A, B, O = fullA[G:G + ma[1]], fullB[G:G + mb[1]], fullO[G:G + mo[1]]
                A0, B0 = fullA.copy(), fullB.copy()
                oracle.OracleCommand(spec, {"A": A, "B": B, "out": O}).eval_range()
                vA, vB = _view(A, (rows, cols), ma[0]), _view(B, (rows, cols), mb[0])
                want = vA * vB - vA
                vO = _view(O, (rows, cols), mo[0])
                assert (specutil.bits(np.ascontiguousarray(vO)) == specutil.bits(want)).all()
                written = np.zeros(fullO.size, dtype=bool)
                idx = (np.arange(rows)[:, None] * mo[0][0] + np.arange(cols)[None, :] * mo[0][1]).ravel()
                written[G + idx] = True
                assert (specutil.bits(fullO[~written]) == specutil.SENTINEL_BITS["f32"]).all()
                assert (specutil.bits(fullA) == specutil.bits(A0)).all()
                assert (specutil.bits(fullB) == specutil.bits(B0)).all()


@pytest.mark.parametrize("perm", [(0, 1, 2), (2, 1, 0), (1, 0, 2), (0, 2, 1), (2, 0, 1)])
def test_rank3_permuted_views(perm):
    """A rank-3 view that permutes a contiguous buffer, and a stride-0
    broadcast load, against numpy transposes and broadcasting."""
    rng = _rng(200)
    phys = (3, 4, 5)
    buf = rng.standard_normal(60).astype(np.float32)
    pst = (20, 5, 1)
    sizes = tuple(phys[p] for p in perm)
    strides = tuple(pst[p] for p in perm)
    bvec = rng.standard_normal(sizes[2]).astype(np.float32)
    dense = workloads._dense(sizes)[0]
    n = int(np.prod(sizes))
    spec = dict(name="r3", seed=0, sizes=sizes,
                ops=[("load", "X", "f32"), ("load", "b", "f32"),
                     ("exec", [("add", "r", "X", "b")]), ("store", "out", "r", "f32")],
                views={"X": dict(strides=strides, alloc=60), "b": dict(strides=(0, 0, 1), alloc=sizes[2]),
                       "out": dict(strides=dense, alloc=n)}, inputs={})
    out = specutil.sentinel_array("f32", n)
    oracle.OracleCommand(spec, {"X": buf, "b": bvec, "out": out}).eval_range()
    want = np.transpose(buf.reshape(phys), perm) + bvec[None, None, :]
    assert (specutil.bits(out) == specutil.bits(np.ascontiguousarray(want).ravel())).all()


# ---- the workloads at small sizes against library expressions -----------------

def test_workload_add_matches_numpy():
    spec = workloads.add_f32(1000)
    bufs = specutil.host_buffers(spec)
    oracle.OracleCommand(spec, bufs).eval_range()
    assert (specutil.bits(bufs["out"]) == specutil.bits(bufs["x"] + bufs["y"])).all()


def test_workload_chain_matches_numpy():
    spec = workloads.chain_f32(4099)
    bufs = specutil.host_buffers(spec)
    oracle.OracleCommand(spec, bufs).eval_range()
    a, b, c = bufs["a"], bufs["b"], bufs["c"]
    want = (a * b) - ((c + a) * np.float32(0.75))
    assert (specutil.bits(bufs["out"]) == specutil.bits(want)).all()


def test_workload_wrap_matches_numpy():
    spec = workloads.wrap_i32(4099)
    bufs = specutil.host_buffers(spec)
    oracle.OracleCommand(spec, bufs).eval_range()
    x, y, z, w = (bufs[k] for k in "xyzw")
    with np.errstate(over="ignore"):
        want = x * y + z - w
    assert (bufs["out"] == want).all()
    # modular arithmetic is associative: a second grouping gives the same bits
    with np.errstate(over="ignore"):
        assert (bufs["out"] == (z - w) + (y * x)).all()


def test_workload_strided_matches_torch():
    m, n, ld = 40, 48, 52
    spec = workloads.strided_bf16(m, n, ld)
    bufs = specutil.host_buffers(spec)
    oracle.OracleCommand(spec, bufs).eval_range()
    A = torch.from_numpy(bufs["A"].view(np.int16).copy()).view(torch.bfloat16)
    A = torch.as_strided(A, (m, n), (ld, 1)).float()
    B = torch.from_numpy(bufs["B"].view(np.int16).copy()).view(torch.bfloat16).reshape(n, m).float().t()
    want = (A * B - A + 0.5).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).ravel()
    assert (bufs["out"] == want).all()


def test_workload_wide_dag_matches_numpy():
    spec = workloads.wide_dag(3001)
    bufs = specutil.host_buffers(spec)
    oracle.OracleCommand(spec, bufs).eval_range()
    v = {k: bufs[k] for k in "abcdef"}
    v["s"], v["r"] = np.float32(1.5), np.float32(-0.25)
    for eop, name, a, b in workloads.WIDE_DAG:
        if eop == "neg":
            v[name] = -v[a]
        else:
            v[name] = {"add": np.add, "sub": np.subtract, "mul": np.multiply}[eop](v[a], v[b])
    assert (specutil.bits(bufs["out0"]) == specutil.bits(v["t16"].astype(np.float32))).all()
    with np.errstate(all="ignore"):
        want16 = v["t13"].astype(np.float16)
    assert specutil.same_bits_nan_as_class(bufs["out1"], want16, "f16").all()


def test_points_match_range():
    spec = workloads.wide_dag(5000)
    bufs = specutil.host_buffers(spec)
    oc = oracle.OracleCommand(spec, bufs)
    oc.eval_range()
    idx = _rng(9).integers(0, 5000, size=300)
    pts = oc.eval_points(idx)
    assert (specutil.bits(pts["out0"]) == specutil.bits(bufs["out0"][idx])).all()
    assert (specutil.bits(pts["out1"]) == specutil.bits(bufs["out1"][idx])).all()


def test_planted_mistakes_are_caught():
    """A wrong sign, a dropped term or swapped operands in the Command change
    the oracle's answer on these inputs, so the cross-checks above would see
    such a mistake in the oracle's walk."""
    spec = workloads.chain_f32(2048)
    bufs = specutil.host_buffers(spec)
    oracle.OracleCommand(spec, bufs).eval_range()
    ref = bufs["out"].copy()
    variants = []
    bad = dict(spec)
    bad["ops"] = [o if o[0] != "exec" else ("exec", [("mul", "ab", "a", "b"), ("add", "ca", "c", "a"),
                                                     ("mul", "cas", "ca", "s"), ("sub", "r", "cas", "ab")])
                  for o in spec["ops"]]
    variants.append(bad)
    bad2 = dict(spec)
    bad2["ops"] = [o if o[0] != "exec" else ("exec", [("mul", "ab", "a", "b"), ("add", "ca", "c", "b"),
                                                      ("mul", "cas", "ca", "s"), ("sub", "r", "ab", "cas")])
                   for o in spec["ops"]]
    variants.append(bad2)
    for v in variants:
        b2 = {k: x.copy() for k, x in bufs.items()}
        b2["out"] = specutil.sentinel_array("f32", 2048)
        oracle.OracleCommand(v, b2).eval_range()
        assert not (specutil.bits(b2["out"]) == specutil.bits(ref)).all()


def test_workload_batched_transpose_matches_numpy():
    spec = workloads.batched_transpose(3, 40, 24)
    bufs = specutil.host_buffers(spec)
    oracle.OracleCommand(spec, bufs).eval_range()
    A = bufs["A"].reshape(3, 24, 40).transpose(0, 2, 1)
    B = bufs["B"].reshape(3, 40, 24)
    want = np.ascontiguousarray(A * B - A).ravel()
    assert (specutil.bits(bufs["out"]) == specutil.bits(want)).all()


def test_workload_div_clamp_i32_matches_numpy():
    """numpy binary32 division, fmax/fmin, truncation to int32 (values are
    clamped into range first) and truncating int division from |q| // 3."""
    spec = workloads.div_clamp_i32(20000)
    bufs = specutil.host_buffers(spec)
    oracle.OracleCommand(spec, bufs).eval_range()
    x = bufs["x"]
    y = np.divide(x, np.float32(0.0074))
    c = np.fmin(np.fmax(y, np.float32(-128.0)), np.float32(127.0))
    q = np.trunc(c).astype(np.int32)
    r = (np.sign(q) * (np.abs(q) // 3)).astype(np.int32)
    assert (bufs["oq"] == q).all()
    assert (bufs["or"] == r).all()
    clamped = (np.abs(q) >= 127).mean()
    assert 0.2 < clamped < 0.5, clamped  # the clamp is exercised
