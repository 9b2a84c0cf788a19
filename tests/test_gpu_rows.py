"""Row-contiguous launches on the GPU: two merged dims, every view unit-stride
along the columns, each row starting on a 4-element boundary and a whole
number of the contiguous executor's warp chunks long (padded or sliced
row-major tensors, a load read as one row for every row). The contiguous
kernel walks (row, chunk) pairs; every element of every store buffer, the
padding between rows included (it keeps its sentinel), against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import gpuutil
import oracle
import layouts
import specutil

pytestmark = pytest.mark.gpu

# elements per slot per thread of the contiguous executor by tier (the base
# 4-slot tier runs 16 when every load is 2-byte)
VEC = {0: 16, 1: 8, 2: 8, 3: 2, 4: 4}


def _chunk(spec):
    c, _ = T.command_from_spec(spec)
    info = c.lower()[0]
    half2 = all(dt in ("f16", "bf16") for dt in (W.tensor_dtypes(spec)[n] for n in W.load_names(spec)))
    v = 16 if (info["tier"] == 1 and not info["extended"] and half2) else VEC[info["tier"]]
    return 32 * v, info


CHAIN = [("mul", "ab", "a", "b"), ("add", "ca", "c", "a"), ("mul", "cas", "ca", "s"), ("sub", "r", "ab", "cas")]


def _cases():
    out = []
    # 2-slot tier, f32 and bf16: x + y
    for dt in ("f32", "bf16"):
        out.append(("add_" + dt, 37, 1024, {"x": (dt, 1032), "y": (dt, 1024 + 64)},
                    {"out": ("z", dt, 1028)}, [("add", "z", "x", "y")], ()))
    # 4-slot tier: the chain Command in f32 (256-element chunks) and bf16
    # (the 16-element build, 512-element chunks)
    out.append(("chain_f32", 45, 768, {"a": ("f32", 800), "b": ("f32", 772), "c": ("f32", 768 + 256)},
                {"out": ("r", "f32", 776)}, CHAIN, (("s", "f32", 0.75),)))
    out.append(("chain_bf16", 45, 1536, {"a": ("bf16", 1544), "b": ("bf16", 1600), "c": ("bf16", 1540)},
                {"out": ("r", "bf16", 1536 + 8)}, CHAIN, (("s", "f32", 0.75),)))
    # int32, a load read as one row for every row, two stores
    out.append(("wrap_bcast_i32", 29, 512, {"x": ("i32", 516), "y": ("i32", 0), "z": ("i32", 640)},
                {"o1": ("t2", "i32", 512 + 4), "o2": ("t1", "i32", 520)},
                [("mul", "t0", "x", "y"), ("add", "t1", "t0", "z"), ("sub", "t2", "t1", "x")], ()))
    # 8-slot tier: the wide DAG's ops with fp32 and fp16 stores
    wide_loads = {k: ("f32", 256 * 3 + 4 * i) for i, k in enumerate("abcdef")}
    out.append(("wide_dag", 23, 768, wide_loads, {"out0": ("t16", "f32", 772), "out1": ("t13", "f16", 768)},
                W.WIDE_DAG, (("s", "f32", 1.5), ("r", "f32", -0.25))))
    # extended ops (division, comparison, select) in the 2- and 4-slot tiers
    out.append(("div_sel", 31, 1024, {"x": ("f32", 1036), "y": ("f32", 1024)}, {"out": ("r", "f32", 1040)},
                [("div", "q", "x", "y"), ("gt", "g", "q", "x"), ("select", "r", "q", "y", "g")], ()))
    out.append(("div_f32", 33, 1024, {"x": ("f32", 1036), "y": ("f32", 1024 + 32)}, {"out": ("q", "f32", 1024)},
                [("div", "q", "x", "y")], ()))
    out.append(("div_sel4", 31, 512, {"x": ("f32", 516), "y": ("f32", 520), "w": ("f32", 512)},
                {"out": ("r", "f32", 524), "o2": ("m", "f32", 512)},
                [("div", "q", "x", "y"), ("mul", "m", "w", "y"), ("lt", "g", "q", "m"),
                 ("select", "r", "q", "w", "g")], ()))
    # 16- and 32-slot tiers: 10 and 17 loads live to the end
    for nl in (10, 17 - 1):
        names = [f"x{i}" for i in range(nl)]
        block = [("add", "c0", "x0", names[-1])] + [("mul" if i % 2 else "sub", f"c{i}", f"c{i - 1}", names[i])
                                                     for i in range(1, nl)]
        block += [("mul", "m", names[0], names[1]), ("add", "r", f"c{nl - 1}", "m")]
        if nl > 10:
            # keep 17 values live: every product computed before any is summed
            block += [("mul", f"p{i}", names[i], names[(i + 1) % nl]) for i in range(nl)]
            acc = "r"
            for i in range(nl):
                block.append(("add", f"s{i}", acc, f"p{i}"))
                acc = f"s{i}"
            block.append(("neg", "q", acc, None))
        else:
            block.append(("neg", "q", "r", None))
        out.append((f"wide{nl}", 13, 512, {k: ("f32", 512 + 4 * i) for i, k in enumerate(names)},
                    {"out": ("r", "f32", 516), "out2": ("q", "bf16", 512 + 8)}, block, ()))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_padded_rows_on_the_contiguous_executor(case):
    name, rows, cols, loads, stores, block, scalars = case
    spec, bufs = layouts.padded_spec(name, rows, cols, loads, stores, block, scalars, seed=len(name) * 7 + rows)
    w, info = _chunk(spec)
    assert cols % w == 0, (cols, w, info)
    plan = gpuutil.parity(spec, bufs)
    assert plan["path"] == "contig" and plan["merged_rank"] == 2, plan


@pytest.mark.parametrize("rows,chunks", [(2, 100), (3000, 3), (4864, 1), (4865, 1), (9733, 2), (1, 7)])
def test_row_walk_with_carries(rows, chunks):
    """Row counts and chunks per row around the grid's warp count (the
    (row, chunk) pair is stepped by it with a carry): every row written
    once, the padding untouched. One row merges to a dense range."""
    cols = 512 * chunks
    spec, bufs = layouts.padded_spec(f"walk{rows}x{chunks}", rows, cols, {"x": ("f32", cols + 16), "y": ("f32", cols + 4)},
                             {"out": ("z", "f32", cols + 8)}, [("sub", "z", "x", "y")], seed=rows + chunks)
    plan = gpuutil.parity(spec, bufs)
    assert plan["path"] == "contig" and plan["merged_rank"] == (2 if rows > 1 else 1), plan


def test_padded_rows_in_place():
    """The store's view is the load's padded view (x = x * y + x, in place)."""
    rows, cols, ld = 40, 1024, 1040
    spec, bufs = layouts.padded_spec("inplace", rows, cols, {"x": ("f32", ld), "y": ("f32", cols)},
                             {"xo": ("r", "f32", ld)}, [("mul", "p", "x", "y"), ("add", "r", "p", "x")], seed=3)
    ref = {k: v.copy() for k, v in bufs.items()}
    ref["xo"] = bufs["x"].copy()
    oracle.OracleCommand(spec, ref).eval_range()
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    x = gpuutil.to_device(bufs["x"], "f32")
    y = gpuutil.to_device(bufs["y"], "f32")
    views = {tags["x"]: T.TensorView(x.data_ptr(), (rows, cols), (ld, 1)),
             tags["y"]: T.TensorView(y.data_ptr(), (rows, cols), (cols, 1)),
             tags["xo"]: T.TensorView(x.data_ptr(), (rows, cols), (ld, 1))}
    assert k.plan(views)["path"] == "contig"
    k.launch(views)
    k.sync()
    torch.cuda.synchronize()
    gpuutil.compare(x.cpu().numpy(), ref["xo"], "f32", "in place over padded rows")


def test_sliced_torch_tensor():
    """x[:, :n] of a wider torch tensor, the plain way a padded view arises."""
    rows, cols, wide = 300, 2048, 2048 + 96
    g = torch.Generator().manual_seed(5)
    xw = torch.randn(rows, wide, generator=g)
    yw = torch.randn(rows, wide, generator=g)
    spec = dict(name="sliced", seed=0, sizes=(rows, cols),
                ops=[("load", "x", "f32"), ("load", "y", "f32"), ("exec", [("mul", "z", "x", "y")]),
                     ("store", "out", "z", "f32")],
                views={"x": dict(strides=(wide, 1), alloc=(rows - 1) * wide + cols),
                       "y": dict(strides=(wide, 1), alloc=(rows - 1) * wide + cols),
                       "out": dict(strides=(cols, 1), alloc=rows * cols)}, inputs={})
    bufs = {"x": xw.numpy().reshape(-1)[:spec["views"]["x"]["alloc"]].copy(),
            "y": yw.numpy().reshape(-1)[:spec["views"]["y"]["alloc"]].copy(),
            "out": specutil.sentinel_array("f32", rows * cols)}
    want = gpuutil.oracle_every_element(spec, bufs)
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    xd, yd = xw.cuda(), yw.cuda()
    out = torch.empty(rows, cols, device="cuda")
    k.launch({tags["x"]: xd[:, :cols], tags["y"]: yd[:, :cols], tags["out"]: out})
    k.sync()
    torch.cuda.synchronize()
    gpuutil.compare(out.cpu().numpy().reshape(-1), want["out"], "f32", "x[:, :n] * y[:, :n]")


def _shifted_rows_cases():
    out = []
    # x one element in, y and out aligned: 2-slot tier (512-element chunks), the
    # row's first 4 and last 7 columns per element
    out.append(("add_x1", 37, 2059, {"x": ("f32", 2064), "y": ("f32", 2060)}, {"out": ("z", "f32", 2060)},
                [("add", "z", "x", "y")], (), {"x": 1}))
    # bf16 chain (4-slot tier, 256-element chunks) with the store two elements in
    out.append(("chain_bf16", 19, 2059, {"a": ("bf16", 2064), "b": ("bf16", 2080), "c": ("bf16", 2060)},
                {"out": ("r", "bf16", 2064)}, CHAIN, (("s", "f32", 0.75),), {"a": 3, "b": 1, "out": 2}))
    # a load read as one row for every row, at an offset
    out.append(("bcast_i32", 29, 1037, {"x": ("i32", 1040), "y": ("i32", 0)}, {"o": ("t", "i32", 1044)},
                [("mul", "t", "x", "y")], (), {"y": 2, "x": 1}))
    # the wide DAG (8-slot tier)
    wide_loads = {k: ("f32", 1040 + 4 * i) for i, k in enumerate("abcdef")}
    out.append(("wide_dag", 11, 1037, wide_loads, {"out0": ("t16", "f32", 1040), "out1": ("t13", "f16", 1044)},
                W.WIDE_DAG, (("s", "f32", 1.5), ("r", "f32", -0.25)), {"a": 1, "d": 2, "f": 3}))
    return out


@pytest.mark.parametrize("case", _shifted_rows_cases(), ids=lambda c: c[0])
def test_rows_at_offsets_take_the_row_walk_with_shifted_loads(case):
    """2-D views whose rows start at different offsets from the vector
    alignment (x[:, 1:] of a wider x and the like; row strides whole vectors):
    each row's first columns up to where the stores align plus 4 and its last
    4 or more run per element, the rest on the row walk with shifted loads."""
    name, rows, cols, loads, stores, block, scalars, offsets = case
    spec, bufs = layouts.padded_spec(name, rows, cols, loads, stores, block, scalars, seed=rows + cols)
    plan = gpuutil.parity(spec, bufs, offsets)
    assert plan["path"] == "contig" and plan["merged_rank"] == 2, plan


def test_rows_at_offsets_with_short_rows_run_per_element():
    """More than an eighth of each row would run per element: the whole
    launch does."""
    spec, bufs = layouts.padded_spec("short_rows", 40, 700, {"x": ("f32", 704), "y": ("f32", 708)},
                             {"out": ("z", "f32", 700)}, [("sub", "z", "x", "y")], seed=2)
    plan = gpuutil.parity(spec, bufs, {"x": 1})
    assert plan["path"] == "generic", plan


def test_sliced_columns_of_torch_tensors():
    """out[:, :n] = x[:, 1:n + 1] * y[:, :n] over (300, 4112) tensors: x's rows
    start one element past a vector boundary."""
    rows, wide, cols = 300, 4112, 4109
    g = torch.Generator().manual_seed(8)
    xw = torch.randn(rows, wide, generator=g)
    yw = torch.randn(rows, wide, generator=g)
    spec = dict(name="sliced_cols", seed=0, sizes=(rows, cols),
                ops=[("load", "x", "f32"), ("load", "y", "f32"), ("exec", [("mul", "z", "x", "y")]),
                     ("store", "out", "z", "f32")],
                views={k: dict(strides=(wide, 1), alloc=(rows - 1) * wide + cols) for k in ("x", "y", "out")},
                inputs={})
    alloc = spec["views"]["x"]["alloc"]
    bufs = {"x": xw.numpy().reshape(-1)[1:1 + alloc].copy(), "y": yw.numpy().reshape(-1)[:alloc].copy(),
            "out": specutil.sentinel_array("f32", alloc)}
    want = gpuutil.oracle_every_element(spec, bufs)["out"]
    want = np.concatenate([want, np.zeros(wide - cols, np.float32)]).reshape(rows, wide)[:, :cols]
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    xd, yd = xw.cuda(), yw.cuda()
    outw = torch.empty(rows, wide, device="cuda")
    views = {tags["x"]: xd[:, 1:1 + cols], tags["y"]: yd[:, :cols], tags["out"]: outw[:, :cols]}
    plan = k.plan(views)
    assert plan["path"] == "contig" and plan["merged_rank"] == 2, plan
    k.launch(views)
    k.sync()
    torch.cuda.synchronize()
    gpuutil.compare(outw[:, :cols].cpu().numpy().reshape(-1), want.reshape(-1), "f32", "x[:, 1:n + 1] * y[:, :n]")
