"""The workloads: Commands, views and input recipes, as plain data.

A workload ("spec") is a dict:

``name``      short identifier
``seed``      generator seed; tensor ``k`` of ``inputs`` draws stream ``k``
``sizes``     logical sizes shared by every tensor of the Command (row-major)
``ops``       the Command, in tag order:
              ``("load", name, dtype)``            Load_Tensor
              ``("scalar", name, dtype, value)``   Load_Scalar
              ``("exec", [(eop, name, a, b), ...])`` one T_Execute block;
                                                   eop in add/sub/mul/div/
                                                   min/max and the compares
                                                   lt/le/gt/ge/eq/ne/ult/ule/
                                                   ugt/uge (binary), neg/abs/
                                                   to_f32/to_i32 (b None), or
                                                   ("select", name, a, b, c)
                                                   for c ? a : b
              ``("store", name, src, dtype)``      Store_Tensor
``views``     per load/store name: ``strides`` (elements) and ``alloc``
              (elements in the physical buffer; 32-bit words for a b1 store)
``inputs``    per load name: (distribution kind, lo, hi) for inputgen
``offsets``   (optional) per tensor name: elements between its allocation's
              start and the view's base (a view placed off the vector
              alignment); absent names start at their allocation

Nothing here computes the Command; the oracle side and the CUDA side each
build their own Command from the same spec.
"""
from __future__ import annotations

DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "i32": 4}  # b1 stores: 32 elements per 4-byte word


def _dense(sizes):
    strides, acc = [], 1
    for s in reversed(sizes):
        strides.append(acc)
        acc *= s
    return tuple(reversed(strides)), acc


def add_f32(n: int = 1 << 20) -> dict:
    """z = x + y, fp32, contiguous 1-D, x and y uniform[-1, 1], seed 0."""
    st, al = _dense((n,))
    return dict(
        name="add_f32", seed=0, sizes=(n,),
        ops=[("load", "x", "f32"), ("load", "y", "f32"),
             ("exec", [("add", "z", "x", "y")]),
             ("store", "out", "z", "f32")],
        views={k: dict(strides=st, alloc=al) for k in ("x", "y", "out")},
        inputs={"x": ("uniform_f32", -1.0, 1.0), "y": ("uniform_f32", -1.0, 1.0)},
    )


def chain_f32(n: int = 1 << 26) -> dict:
    """out = (a*b) - (c + a)*s, s = 0.75, fp32 contiguous, a, b, c normal(0,1).

    Tag ``a`` is referenced twice; it is still read from memory once."""
    st, al = _dense((n,))
    return dict(
        name="chain_f32", seed=1, sizes=(n,),
        ops=[("load", "a", "f32"), ("load", "b", "f32"), ("load", "c", "f32"),
             ("scalar", "s", "f32", 0.75),
             ("exec", [("mul", "ab", "a", "b"),
                       ("add", "ca", "c", "a"),
                       ("mul", "cas", "ca", "s"),
                       ("sub", "r", "ab", "cas")]),
             ("store", "out", "r", "f32")],
        views={k: dict(strides=st, alloc=al) for k in ("a", "b", "c", "out")},
        inputs={k: ("normal_f32", 0.0, 0.0) for k in ("a", "b", "c")},
    )


def chain_bf16(n: int = 1 << 27) -> dict:
    """The chain Command, out = (a*b) - (c + a)*s with s = 0.75, on bf16
    tensors (computed in fp32, rounded once on the store), a, b, c uniform
    [-4, 4] truncated to bf16, seed 9: the contiguous path's 2-byte loads."""
    st, al = _dense((n,))
    return dict(
        name="chain_bf16", seed=9, sizes=(n,),
        ops=[("load", "a", "bf16"), ("load", "b", "bf16"), ("load", "c", "bf16"),
             ("scalar", "s", "f32", 0.75),
             ("exec", [("mul", "ab", "a", "b"),
                       ("add", "ca", "c", "a"),
                       ("mul", "cas", "ca", "s"),
                       ("sub", "r", "ab", "cas")]),
             ("store", "out", "r", "bf16")],
        views={k: dict(strides=st, alloc=al) for k in ("a", "b", "c", "out")},
        inputs={k: ("uniform_bf16_trunc", -4.0, 4.0) for k in ("a", "b", "c")},
    )


def wrap_i32(n: int = 1 << 28) -> dict:
    """out = x*y + z - w in int32 with two's-complement wraparound, seed 2."""
    st, al = _dense((n,))
    return dict(
        name="wrap_i32", seed=2, sizes=(n,),
        ops=[("load", "x", "i32"), ("load", "y", "i32"), ("load", "z", "i32"),
             ("load", "w", "i32"),
             ("exec", [("mul", "xy", "x", "y"),
                       ("add", "xyz", "xy", "z"),
                       ("sub", "r", "xyz", "w")]),
             ("store", "out", "r", "i32")],
        views={k: dict(strides=st, alloc=al) for k in ("x", "y", "z", "w", "out")},
        inputs={k: ("u32", 0.0, 0.0) for k in ("x", "y", "z", "w")},
    )


def strided_bf16(m: int = 8192, n: int = 8192, ld_a: int = 8320) -> dict:
    """out = A*B^T - A + 0.5 in fp32, bf16 in and out, values uniform[-4, 4].

    A is m x n row-major with leading dimension ld_a; B is an n x m row-major
    tensor read through its transpose view (strides {1, m}); out is dense."""
    return dict(
        name="strided_bf16", seed=3, sizes=(m, n),
        ops=[("load", "A", "bf16"), ("load", "B", "bf16"),
             ("scalar", "h", "f32", 0.5),
             ("exec", [("mul", "AB", "A", "B"),
                       ("sub", "ABA", "AB", "A"),
                       ("add", "r", "ABA", "h")]),
             ("store", "out", "r", "bf16")],
        views={"A": dict(strides=(ld_a, 1), alloc=(m - 1) * ld_a + n if m else 0),
               "B": dict(strides=(1, m), alloc=m * n),
               "out": dict(strides=(n, 1), alloc=m * n)},
        inputs={"A": ("uniform_bf16_trunc", -4.0, 4.0),
                "B": ("uniform_bf16_trunc", -4.0, 4.0)},
    )


# The 16 E ops of the wide DAG, in tag order; ``t10`` repeats ``t1`` with its
# operands swapped, so common-subexpression reuse maps it onto ``t1``.
WIDE_DAG = [
    ("add", "t1", "a", "b"),
    ("mul", "t2", "c", "d"),
    ("sub", "t3", "t1", "t2"),
    ("mul", "t4", "e", "s"),
    ("neg", "t5", "f", None),
    ("add", "t6", "t3", "t4"),
    ("mul", "t7", "t1", "t5"),
    ("sub", "t8", "t6", "t7"),
    ("add", "t9", "t2", "r"),
    ("add", "t10", "b", "a"),
    ("mul", "t11", "t10", "t9"),
    ("neg", "t12", "t3", None),
    ("add", "t13", "t11", "t12"),
    ("mul", "t14", "t8", "t13"),
    ("sub", "t15", "t4", "t5"),
    ("add", "t16", "t14", "t15"),
]


def wide_dag(n: int = 1 << 27) -> dict:
    """Six fp32 inputs normal(0,1), scalars 1.5 and -0.25, 16 E ops with
    shared subexpressions, stores out0 (fp32) <- t16 and out1 (fp16) <- t13."""
    st, al = _dense((n,))
    names = ("a", "b", "c", "d", "e", "f")
    return dict(
        name="wide_dag", seed=4, sizes=(n,),
        ops=[("load", k, "f32") for k in names]
        + [("scalar", "s", "f32", 1.5), ("scalar", "r", "f32", -0.25),
           ("exec", list(WIDE_DAG)),
           ("store", "out0", "t16", "f32"), ("store", "out1", "t13", "f16")],
        views={k: dict(strides=st, alloc=al) for k in names + ("out0", "out1")},
        inputs={k: ("normal_f32", 0.0, 0.0) for k in names},
    )


def batched_transpose(b: int = 64, m: int = 1024, n: int = 1024) -> dict:
    """out = A^T*B - A^T per batch (A^T: each m x n slice of A read through its
    transpose, strides {m*n, 1, m}), fp32, normal(0,1), seed 5: the batched
    coordinate transform of the generalised tile path."""
    dense = (m * n, n, 1)
    return dict(
        name="batched_transpose", seed=5, sizes=(b, m, n),
        ops=[("load", "A", "f32"), ("load", "B", "f32"),
             ("exec", [("mul", "AB", "A", "B"), ("sub", "r", "AB", "A")]),
             ("store", "out", "r", "f32")],
        views={"A": dict(strides=(m * n, 1, m), alloc=b * m * n),
               "B": dict(strides=dense, alloc=b * m * n),
               "out": dict(strides=dense, alloc=b * m * n)},
        inputs={"A": ("normal_f32", 0.0, 0.0), "B": ("normal_f32", 0.0, 0.0)},
    )


def div_clamp_i32(n: int = 1 << 27) -> dict:
    """q = to_i32(min(max(x / s, lo), hi)) and r = q / 3 (int32, truncating):
    x normal(0, 1), s = 0.0074 (so the clamp at lo = -128 / hi = 127 is
    active for about a third of the elements), seed 6. Float division, max,
    min, the float-to-int conversion and int division in one pass; stores q
    and r as int32."""
    st, al = _dense((n,))
    return dict(
        name="div_clamp_i32", seed=6, sizes=(n,),
        ops=[("load", "x", "f32"), ("scalar", "s", "f32", 0.0074), ("scalar", "lo", "f32", -128.0),
             ("scalar", "hi", "f32", 127.0), ("scalar", "k", "i32", 3),
             ("exec", [("div", "y", "x", "s"), ("max", "c0", "y", "lo"), ("min", "c", "c0", "hi"),
                       ("to_i32", "q", "c", None), ("div", "r", "q", "k")]),
             ("store", "oq", "q", "i32"), ("store", "or", "r", "i32")],
        views={k: dict(strides=st, alloc=al) for k in ("x", "oq", "or")},
        inputs={"x": ("normal_f32", 0.0, 0.0)},
    )


THRESHOLD = 0xA0000000  # 3/8 of uniform u32 values are at or above it


def threshold_u32(n: int = 1 << 28) -> dict:
    """Threshold classification, one prediction word per element: pred =
    UGE(x, t) stored as int32 0/1, x uniform over all u32 values (int32 bits),
    t = 0xA0000000 (so about 3/8 of the predictions are 1), seed 7."""
    st, al = _dense((n,))
    return dict(
        name="threshold_u32", seed=7, sizes=(n,),
        ops=[("load", "x", "i32"), ("scalar", "t", "i32", THRESHOLD - (1 << 32)),
             ("exec", [("uge", "pred", "x", "t")]),
             ("store", "out", "pred", "i32")],
        views={k: dict(strides=st, alloc=al) for k in ("x", "out")},
        inputs={"x": ("u32", 0.0, 0.0)},
    )


def threshold_bits(n: int = 1 << 28) -> dict:
    """Threshold classification with packed predictions: the same comparison
    as threshold_u32, stored one bit per element (b1: 32 predictions per
    word, bit i of the buffer for element i), seed 8."""
    st, _ = _dense((n,))
    return dict(
        name="threshold_bits", seed=8, sizes=(n,),
        ops=[("load", "x", "i32"), ("scalar", "t", "i32", THRESHOLD - (1 << 32)),
             ("exec", [("uge", "pred", "x", "t")]),
             ("store", "bits", "pred", "b1")],
        views={"x": dict(strides=st, alloc=n), "bits": dict(strides=st, alloc=(n + 31) // 32)},
        inputs={"x": ("u32", 0.0, 0.0)},
    )


def tile4_f32(m: int = 4096, n: int = 4096) -> dict:
    """out = A*B^T + C^T*s - A, fp32, with A row-direct (leading dimension
    n + 32) and B, C read through their transposes: three staged loads and
    a value kept live beside them put the program in the 4-slot tier of the
    tile executor, normal(0,1), seed 10 (a profiling case, not a headline)."""
    ld = n + 32
    return dict(
        name="tile4_f32", seed=10, sizes=(m, n),
        ops=[("load", "A", "f32"), ("load", "B", "f32"), ("load", "C", "f32"),
             ("scalar", "s", "f32", 0.5),
             ("exec", [("mul", "AB", "A", "B"), ("mul", "Cs", "C", "s"), ("add", "t", "AB", "Cs"),
                       ("sub", "r", "t", "A")]),
             ("store", "out", "r", "f32")],
        views={"A": dict(strides=(ld, 1), alloc=(m - 1) * ld + n),
               "B": dict(strides=(1, m), alloc=n * m),
               "C": dict(strides=(1, m), alloc=n * m),
               "out": dict(strides=(n, 1), alloc=m * n)},
        inputs={k: ("normal_f32", 0.0, 0.0) for k in ("A", "B", "C")},
    )


def wide32_f32(n: int = 1 << 24) -> dict:
    """A sum of products over nine fp32 inputs, x0*x1 + x2*x3 + ... + x8:
    nine loads live at once put the program past eight slots, in the 32-slot
    tier of the contiguous executor, normal(0,1), seed 11 (a profiling case,
    not a headline)."""
    st, al = _dense((n,))
    names = tuple(f"x{k}" for k in range(9))
    body = [("mul", "p0", "x0", "x1"), ("mul", "p1", "x2", "x3"), ("mul", "p2", "x4", "x5"),
            ("mul", "p3", "x6", "x7"), ("add", "q0", "p0", "p1"), ("add", "q1", "p2", "p3"),
            ("add", "q2", "q0", "q1"), ("add", "r", "q2", "x8")]
    return dict(
        name="wide32_f32", seed=11, sizes=(n,),
        ops=[("load", k, "f32") for k in names] + [("exec", body), ("store", "out", "r", "f32")],
        views={k: dict(strides=st, alloc=al) for k in names + ("out",)},
        inputs={k: ("normal_f32", 0.0, 0.0) for k in names},
    )


def rows_chain_f32(m: int = 8192, n: int = 8192) -> dict:
    """The chain Command over padded rows: a, b and c are m x n views of
    wider row-major tensors (leading dimensions 8320, 8256 and 8200), out is
    dense; normal(0,1), seed 12 (the contiguous executor's row walk)."""
    lds = {"a": n + 128, "b": n + 64, "c": n + 8, "out": n}
    spec = chain_f32(0)
    spec.update(name="rows_chain_f32", seed=12, sizes=(m, n),
                views={k: dict(strides=(ld, 1), alloc=(m - 1) * ld + n) for k, ld in lds.items()})
    return spec


def stencil_f32(n: int = 1 << 26) -> dict:
    """out = (x1 - x0) * s + x2, s = 0.5, fp32, with x1 and x2 one and two
    elements past the vector alignment and x0 and out on it (the layout of
    a difference of neighbouring slices; normal(0,1), seed 13): the
    contiguous executor with shifted loads. ``offsets`` gives each tensor's
    element offset into its allocation."""
    st, al = _dense((n,))
    return dict(
        name="stencil_f32", seed=13, sizes=(n,),
        ops=[("load", "x0", "f32"), ("load", "x1", "f32"), ("load", "x2", "f32"),
             ("scalar", "s", "f32", 0.5),
             ("exec", [("sub", "d", "x1", "x0"), ("mul", "e", "d", "s"), ("add", "r", "e", "x2")]),
             ("store", "out", "r", "f32")],
        views={k: dict(strides=st, alloc=al) for k in ("x0", "x1", "x2", "out")},
        inputs={k: ("normal_f32", 0.0, 0.0) for k in ("x0", "x1", "x2")},
        offsets={"x1": 1, "x2": 2},
    )


# Full-size workloads, in the order they are listed for this path.
FULL = {
    "add_f32": add_f32,
    "chain_f32": chain_f32,
    "wrap_i32": wrap_i32,
    "strided_bf16": strided_bf16,
    "wide_dag": wide_dag,
    "batched_transpose": batched_transpose,
    "div_clamp_i32": div_clamp_i32,
    "threshold_u32": threshold_u32,
    "threshold_bits": threshold_bits,
    "chain_bf16": chain_bf16,
}

# Layouts the contiguous executor takes beyond dense ranges (padded rows,
# loads off the stores' alignment): the benchmark's per-workload table
# lists them after the ones above.
LAYOUT = {
    "rows_chain_f32": rows_chain_f32,
    "stencil_f32": stencil_f32,
}

# Cases that run the executor objects the workloads above do not reach (the
# 4-slot tile tier, the 32-slot tier), for profiling; bench.py accepts them
# by name but they are not part of its per-workload table.
PROFILE = {
    "tile4_f32": tile4_f32,
    "wide32_f32": wide32_f32,
}


def load_names(spec: dict) -> list:
    return [op[1] for op in spec["ops"] if op[0] == "load"]


def store_names(spec: dict) -> list:
    return [op[1] for op in spec["ops"] if op[0] == "store"]


def tensor_dtypes(spec: dict) -> dict:
    out = {}
    for op in spec["ops"]:
        if op[0] in ("load", "store"):
            out[op[1]] = op[2] if op[0] == "load" else op[3]
    return out


def numel(spec: dict) -> int:
    n = 1
    for s in spec["sizes"]:
        n *= s
    return n


def store_bytes(dtype: str, n: int) -> int:
    """Bytes a store of n elements writes (packed bits: whole 4-byte words)."""
    return (n + 31) // 32 * 4 if dtype == "b1" else n * DTYPE_BYTES[dtype]


def algorithmic_bytes(spec: dict, live_loads=None) -> int:
    """Bytes one pass moves: every live loaded tensor read once and every
    store written once, over the logical elements (padding not counted)."""
    dt = tensor_dtypes(spec)
    n = numel(spec)
    loads = live_loads if live_loads is not None else load_names(spec)
    return (n * sum(DTYPE_BYTES[dt[k]] for k in loads)
            + sum(store_bytes(dt[k], n) for k in store_names(spec)))
