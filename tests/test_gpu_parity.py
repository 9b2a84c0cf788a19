"""GPU parity: the CUDA path (through the C ABI) against the oracle, element
by element on the same seeded inputs. Bit-exact for int32 and fp32; within
1 ulp (and in fact exact) for fp16/bf16 stores."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import gpuutil
import specutil

pytestmark = pytest.mark.gpu


# ---- the workloads at sizes the oracle finishes in seconds ------------------------

@pytest.mark.parametrize("spec,path", [
    (W.add_f32((1 << 20) + 37), "contig"),
    (W.add_f32(1 << 20), "contig"),
    (W.chain_f32((1 << 18) + 5), "contig"),
    (W.wrap_i32((1 << 18) + 3), "contig"),
    (W.strided_bf16(320, 264, 272), "tile2d"),
    (W.strided_bf16(200, 136, 144), "tile2d"),
    (W.strided_bf16(192, 128, 136), "tile2d"),
    (W.strided_bf16(100, 70, 75), "generic"),
    (W.wide_dag((1 << 18) + 11), "contig"),
    (W.wide_dag(37), "contig"),
    (W.div_clamp_i32((1 << 18) + 9), "contig"),
    (W.div_clamp_i32(100), "contig"),
    (W.threshold_u32((1 << 18) + 13), "contig"),
    (W.threshold_bits((1 << 18) + 13), "contig"),
    (W.threshold_bits(77), "contig"),
    (W.chain_bf16((1 << 18) + 7), "contig"),
    (W.chain_bf16(511), "contig"),
    (W.tile4_f32(132, 72), "tile2d"),
    (W.wide32_f32((1 << 16) + 7), "contig"),
], ids=lambda x: x["name"] + str(x["sizes"]) if isinstance(x, dict) else x)
def test_workload_small(spec, path):
    plan = gpuutil.parity(spec)
    assert plan["path"] == path


# ---- the workloads at full size, every element --------------------------------------

@pytest.mark.parametrize("name", list(W.FULL))
def test_workload_full_size_every_element(name):
    """Each workload at its full size (the five headline configurations
    among them: add 2^20, chain 2^26, int32 wraparound 2^28, the strided
    bf16 product 8192 x 8192 with A's leading dimension 8320 and B read
    through strides {1, 8192}, the 16-op DAG 2^27) in the launch
    configuration the benchmark times, every element of every store
    compared with the oracle (rocRoller, Design Overview, "Operations": a
    T_Execute applies to every element; "Kernel Graph": every index of the
    view)."""
    spec = W.FULL[name]()
    plan, checked, max_ulp = gpuutil.full_parity(spec)
    assert plan["path"] == ("tile2d" if name in ("strided_bf16", "batched_transpose") else "contig")
    # whole store buffers (a packed-bit store: its 32-bit words) were compared
    assert checked == sum(spec["views"][n]["alloc"] for n in W.store_names(spec))
    assert max_ulp == 0


@pytest.mark.parametrize("name", list(W.LAYOUT))
def test_layout_workload_full_size_every_element(name):
    """The benchmark's layout workloads at full size (the chain Command over
    8192 x 8192 padded rows; the 2^26-element stencil with two loads off the
    alignment), their offsets applied, every element against the oracle."""
    spec = W.LAYOUT[name]()
    plan, checked, max_ulp = gpuutil.full_parity(spec)
    assert plan["path"] == "contig" and plan["merged_rank"] == (2 if name == "rows_chain_f32" else 1), plan
    if name == "stencil_f32":
        assert plan["shifted_loads"] == 2, plan
    assert checked == sum(spec["views"][n]["alloc"] for n in W.store_names(spec))


# ---- tile executor over dtypes, ragged tiles and several transposed loads -------------

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("rows,cols", [(64, 64), (130, 72), (8, 200), (257, 40)])
def test_tile_paths(dt, rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    es = 2 if dt in ("f16", "bf16") else 4
    al = 16 // es  # strides must keep 16-byte rows
    ldA = (cols + al + al - 1) // al * al
    ldB = (rows + al - 1) // al * al
    ldC = (rows + 2 * al - 1) // al * al
    cls_int = dt == "i32"
    st = "i32" if cls_int else "f32"
    spec = dict(name=f"tile_{dt}", seed=0, sizes=(rows, cols),
                ops=[("load", "A", dt), ("load", "B", dt), ("load", "C", dt),
                     ("scalar", "s", st, 3 if cls_int else 0.5),
                     ("exec", [("mul", "AB", "A", "B"), ("sub", "t", "AB", "C"), ("add", "r", "t", "s"),
                               ("neg", "q", "B", None)]),
                     ("store", "out", "r", "i32" if cls_int else dt),
                     ("store", "out2", "q", "i32" if cls_int else "f32")],
                views={"A": dict(strides=(ldA, 1), alloc=(rows - 1) * ldA + cols),
                       "B": dict(strides=(1, ldB), alloc=(cols - 1) * ldB + rows),
                       "C": dict(strides=(1, ldC), alloc=(cols - 1) * ldC + rows),
                       "out": dict(strides=(cols, 1), alloc=rows * cols),
                       "out2": dict(strides=(ldA, 1), alloc=(rows - 1) * ldA + cols)},
                inputs={})
    bufs = {}
    for name in ("A", "B", "C"):
        n = spec["views"][name]["alloc"]
        if cls_int:
            bufs[name] = rng.integers(-2**31, 2**31, size=n).astype(np.int32)
        else:
            f = rng.standard_normal(n).astype(np.float32) * 4
            if dt == "f32":
                bufs[name] = f
            elif dt == "f16":
                bufs[name] = f.astype(np.float16)
            else:
                bufs[name] = (f.view(np.uint32) >> 16).astype(np.uint16)
    for name in ("out", "out2"):
        odt = W.tensor_dtypes(spec)[name]
        bufs[name] = specutil.sentinel_array(odt, spec["views"][name]["alloc"])
    plan = gpuutil.parity(spec, bufs)
    assert plan["path"] == "tile2d" and plan["n_transposed"] == 2


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("n_trans,n_live,tier", [(1, 0, 0), (2, 0, 1), (2, 4, 2)])
def test_tile_transposed_reads_in_every_tier(dt, n_trans, n_live, tier):
    """One row-direct and n_trans transposed loads, plus n_live values kept
    live together, put the program in the 2-, 4- or 8-slot tier of the tile
    executor: the two-row readers (2- and 4-slot) and the one-row reader
    (8-slot) over a ragged 130 x 72 index space, every element against the
    oracle. (At most three loads: a stage of the tile executor holds 48 KB.)"""
    rows, cols = 130, 72
    es = 2 if dt in ("f16", "bf16") else 4
    al = 16 // es
    ldA = (cols + al - 1) // al * al + al
    ldB = (rows + al - 1) // al * al + al
    rng = np.random.default_rng(n_trans * 10 + n_live + len(dt))
    bs = [f"B{i}" for i in range(n_trans)]
    ops3 = ("add", "mul", "sub")
    block, acc = [], "A"
    for i, b in enumerate(bs):
        block.append((ops3[i % 3], f"t{i}", acc, b))
        acc = f"t{i}"
    qs = [f"q{k}" for k in range(n_live)]
    for k, q in enumerate(qs):   # all computed before any is consumed
        block.append((ops3[(k + 1) % 3], q, "A", bs[k % n_trans]))
    for k, q in enumerate(qs):
        block.append((ops3[k % 3], f"u{k}", acc, q))
        acc = f"u{k}"
    spec = dict(name=f"tile_t{tier}_{dt}", seed=0, sizes=(rows, cols),
                ops=[("load", "A", dt)] + [("load", b, dt) for b in bs] + [("exec", block), ("store", "out", acc, dt)],
                views=dict({"A": dict(strides=(ldA, 1), alloc=(rows - 1) * ldA + cols),
                            "out": dict(strides=(cols, 1), alloc=rows * cols)},
                           **{b: dict(strides=(1, ldB), alloc=(cols - 1) * ldB + rows) for b in bs}),
                inputs={})
    bufs = {}
    for name in ["A"] + bs:
        n = spec["views"][name]["alloc"]
        if dt == "i32":
            bufs[name] = rng.integers(-2**31, 2**31, size=n).astype(np.int32)
        else:
            f = (rng.standard_normal(n) * 2).astype(np.float32)
            bufs[name] = f if dt == "f32" else f.astype(np.float16) if dt == "f16" else \
                (f.view(np.uint32) >> 16).astype(np.uint16)
    bufs["out"] = specutil.sentinel_array(dt, rows * cols)
    c, _ = T.command_from_spec(spec)
    assert c.lower()[0]["tier"] == tier
    plan = gpuutil.parity(spec, bufs)
    assert plan["path"] == "tile2d" and plan["n_transposed"] == n_trans


# ---- randomized Commands ---------------------------------------------------------------

def _dense_strides(shape):
    st, acc = [], 1
    for s in reversed(shape):
        st.append(acc)
        acc *= s
    return tuple(reversed(st)), acc


def _random_view(rng, sizes, allow_broadcast):
    rank = len(sizes)
    mode = rng.choice(["dense", "padded", "permuted", "broadcast"] if allow_broadcast
                      else ["dense", "padded", "permuted"])
    if mode == "dense":
        st, n = _dense_strides(sizes)
        return st, n
    if mode == "padded":
        pad = int(rng.integers(1, 9))
        st = [0] * rank
        acc = 1
        for k in range(rank - 1, -1, -1):
            st[k] = acc
            acc = acc * sizes[k] + (pad if k == rank - 1 else 0)
        n = sum((s - 1) * t for s, t in zip(sizes, st)) + 1
        return tuple(st), n
    if mode == "permuted":
        perm = rng.permutation(rank)
        phys = [sizes[p] for p in perm]
        pst, n = _dense_strides(phys)
        st = [0] * rank
        for q, p in enumerate(perm):
            st[p] = pst[q]
        return tuple(st), n
    st, n = _dense_strides(sizes)
    st = list(st)
    for k in range(rank):
        if rng.random() < 0.5:
            st[k] = 0
    n = sum((s - 1) * t for s, t in zip(sizes, st)) + 1
    return tuple(st), n


def _random_values(rng, dt, n):
    if dt == "i32":
        return rng.integers(-2**31, 2**31, size=n).astype(np.int32)
    f = (rng.standard_normal(n) * rng.choice([1.0, 100.0, 1e-3])).astype(np.float32)
    if dt == "f32":
        return f
    if dt == "f16":
        return f.astype(np.float16)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def random_case(seed):
    rng = np.random.default_rng(seed)
    rank = int(rng.integers(0, 4))
    sizes = tuple(int(x) for x in rng.integers(1, 24, size=rank))
    if rank and rng.random() < 0.3:
        sizes = sizes[:-1] + (int(rng.integers(100, 700)),)
    is_int = rng.random() < 0.3
    ops, views, bufs, vals = [], {}, {}, []
    n_loads = int(rng.integers(1, 7))
    for i in range(n_loads):
        dt = "i32" if is_int else str(rng.choice(["f32", "f16", "bf16"]))
        name = f"L{i}"
        ops.append(("load", name, dt))
        st, n = _random_view(rng, sizes, allow_broadcast=True)
        views[name] = dict(strides=st, alloc=n)
        bufs[name] = _random_values(rng, dt, n)
        vals.append(name)
    for i in range(int(rng.integers(0, 3))):
        name = f"S{i}"
        if is_int:
            ops.append(("scalar", name, "i32", int(rng.integers(-2**31, 2**31))))
        else:
            ops.append(("scalar", name, "f32", float(np.float32(rng.standard_normal()))))
        vals.append(name)
    block = []
    for i in range(int(rng.integers(1, 22))):
        eop = str(rng.choice(["add", "sub", "mul", "neg"]))
        a = str(rng.choice(vals))
        b = None if eop == "neg" else str(rng.choice(vals))
        name = f"E{i}"
        block.append((eop, name, a, b))
        vals.append(name)
    ops.append(("exec", block))
    for i in range(int(rng.integers(1, 4))):
        src = vals[-1 - int(rng.integers(0, min(4, len(vals))))]
        dt = "i32" if is_int else str(rng.choice(["f32", "f16", "bf16"]))
        name = f"O{i}"
        ops.append(("store", name, src, dt))
        st, n = _random_view(rng, sizes, allow_broadcast=False)
        views[name] = dict(strides=st, alloc=n)
        bufs[name] = specutil.sentinel_array(dt, n)
    return dict(name=f"random{seed}", seed=seed, sizes=sizes, ops=ops, views=views, inputs={}), bufs


@pytest.mark.parametrize("seed", range(60))
def test_random_commands(seed):
    spec, bufs = random_case(seed)
    gpuutil.parity(spec, bufs)


# ---- edge cases -------------------------------------------------------------------------

def test_empty_launch_is_a_no_op():
    spec = W.add_f32(0)
    bufs = {k: np.zeros(0, np.float32) for k in ("x", "y", "out")}
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    views = {tags[n]: T.TensorView(0, (0,), (1,)) for n in ("x", "y", "out")}
    assert k.plan(views)["path"] == "none"
    k.launch(views)
    k.sync()
    del bufs


@pytest.mark.parametrize("n", [1, 2, 3, 255, 256, 257, 1023, 1025, 4097])
def test_ragged_lengths(n):
    gpuutil.parity(W.wide_dag(n))
    gpuutil.parity(W.chain_f32(n))


def test_rank0_single_element():
    spec = W.chain_f32(1)
    spec["sizes"] = ()
    for k in spec["views"]:
        spec["views"][k] = dict(strides=(), alloc=1)
    gpuutil.parity(spec)


def test_fill_copy_and_in_place():
    n = 5000
    spec = dict(name="fill", seed=0, sizes=(n,),
                ops=[("load", "x", "f32"), ("scalar", "s", "f32", -2.5),
                     ("store", "fill", "s", "bf16"), ("store", "copy", "x", "f16"),
                     ("exec", [("mul", "y", "x", "s")]), ("store", "x_out", "y", "f32")],
                views={k: dict(strides=(1,), alloc=n) for k in ("x", "fill", "copy", "x_out")},
                inputs={"x": ("normal_f32", 0, 0)})
    bufs = specutil.host_buffers(spec)
    gpuutil.parity(spec, bufs)
    # in place: the store's view is the load's view
    dts = W.tensor_dtypes(spec)
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    dev = {name: gpuutil.to_device(bufs[name], dts[name]) for name in ("x", "fill", "copy")}
    views = {tags[nm]: T.TensorView(dev[nm].data_ptr(), (n,), (1,)) for nm in dev}
    views[tags["x_out"]] = views[tags["x"]]
    k.launch(views, {tags["s"]: -2.5})
    k.sync()
    torch.cuda.synchronize()
    ref = {kk: v.copy() for kk, v in bufs.items()}
    oracle.OracleCommand(spec, ref).eval_range()
    gpuutil.compare(dev["x"].cpu().numpy(), ref["x_out"], "f32", "in place")


@pytest.mark.parametrize("off", [1, 2, 3])
def test_misaligned_bases_use_the_generic_path(off):
    spec = W.wide_dag(10000)
    plan = gpuutil.parity(spec, offsets={"a": off, "out1": off})
    assert plan["path"] == "generic"


@pytest.mark.parametrize("off", [1, 2, 3])
@pytest.mark.parametrize("n", [2, 3, 517, 10000, 70001])
@pytest.mark.parametrize("wl", ["wide_dag", "chain_bf16"])
def test_bases_off_by_one_count_peel_a_head(wl, off, n):
    """Every view off its vector alignment by the same number of elements
    (f32 inputs and outputs with an f16 output, or bf16 throughout, all
    sliced off elements into their allocations): the first 4 - off elements
    run per element and the rest on the contiguous executor, once there are
    more than 4 - off; every element and the bytes around the views against
    the oracle."""
    spec = W.FULL[wl](n)
    names = W.load_names(spec) + W.store_names(spec)
    plan = gpuutil.parity(spec, offsets={k: off for k in names})
    assert plan["path"] == ("contig" if n > 4 - off else "generic")


def test_wide_tier_program():
    rng = np.random.default_rng(5)
    n = 3000
    names = [f"x{i}" for i in range(16)]
    block = [("add", "c0", "x0", "x15")] + [("mul", f"c{i}", f"c{i-1}", names[i]) for i in range(1, 16)]
    block += [("sub", f"d{i}", names[i], f"c{i}") for i in range(16)]
    block += [("add", "e0", "d0", "d1")] + [("add", f"e{i}", f"e{i-1}", f"d{i+1}") for i in range(1, 15)]
    spec = dict(name="wide", seed=0, sizes=(n,),
                ops=[("load", k, "f32") for k in names] + [("exec", block), ("store", "out", "e14", "f32"),
                                                            ("store", "out2", "c15", "bf16")],
                views={k: dict(strides=(1,), alloc=n) for k in names + ["out", "out2"]}, inputs={})
    bufs = {k: (rng.standard_normal(n) * 1.5).astype(np.float32) for k in names}
    bufs["out"] = specutil.sentinel_array("f32", n)
    bufs["out2"] = specutil.sentinel_array("bf16", n)
    c, _ = T.command_from_spec(spec)
    info = c.lower()[0]
    assert info["tier"] == 3 and info["n_slots"] > 16
    assert gpuutil.parity(spec, bufs)["path"] == "contig"


@pytest.mark.parametrize("strided", [False, True])
@pytest.mark.parametrize("n_loads", [9, 12, 15])
def test_sixteen_slot_tier_program(n_loads, strided):
    """Programs with 9 to 16 live values run the 16-slot tier (two-level
    dispatch, 4 elements per slot): every load live until the end, sums and
    products chained over them, an f32 and a bf16 store; dense views on the
    contiguous executor, stride-2 views on the generic one."""
    rng = np.random.default_rng(n_loads)
    n = 4099
    st = 2 if strided else 1
    names = [f"x{i}" for i in range(n_loads)]
    block = [("add", "c0", "x0", names[-1])] + [("mul" if i % 2 else "sub", f"c{i}", f"c{i-1}", names[i])
                                                 for i in range(1, n_loads)]
    block += [("mul", "m", names[0], names[1]), ("add", "r", f"c{n_loads - 1}", "m"), ("neg", "q", "r", None)]
    spec = dict(name=f"tier16_{n_loads}", seed=0, sizes=(n,),
                ops=[("load", k, "f32") for k in names] + [("exec", block), ("store", "out", "r", "f32"),
                                                            ("store", "out2", "q", "bf16")],
                views={k: dict(strides=(st,), alloc=st * (n - 1) + 1) for k in names + ["out", "out2"]},
                inputs={})
    bufs = {k: (rng.standard_normal(spec["views"][k]["alloc"]) * 1.5).astype(np.float32) for k in names}
    bufs["out"] = specutil.sentinel_array("f32", spec["views"]["out"]["alloc"])
    bufs["out2"] = specutil.sentinel_array("bf16", spec["views"]["out2"]["alloc"])
    c, _ = T.command_from_spec(spec)
    info = c.lower()[0]
    assert info["tier"] == 4 and 8 < info["n_slots"] <= 16, info
    assert gpuutil.parity(spec, bufs)["path"] == ("generic" if strided else "contig")


def test_special_values():
    """Denormals, signed zeros, infinities and NaNs flow through every op
    like the oracle's IEEE arithmetic (NaN payloads are not compared)."""
    specials = np.array([0, 0x80000000, 1, 0x80000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0xFF7FFFFF,
                         0x7F800000, 0xFF800000, 0x7FC00000, 0x3F800000, 0x33800000, 0x477FF000,
                         0x477FEFFF, 0x387FC000, 0x33000000, 0x00400000], dtype=np.uint32)
    x = np.repeat(specials, specials.size)
    y = np.tile(specials, specials.size)
    n = x.size
    spec = dict(name="specials", seed=0, sizes=(n,),
                ops=[("load", "x", "f32"), ("load", "y", "f32"),
                     ("exec", [("add", "s", "x", "y"), ("sub", "d", "x", "y"), ("mul", "p", "x", "y"),
                               ("neg", "m", "p", None)]),
                     ("store", "o1", "s", "f32"), ("store", "o2", "d", "f16"), ("store", "o3", "p", "bf16"),
                     ("store", "o4", "m", "f32")],
                views={k: dict(strides=(1,), alloc=n) for k in ("x", "y", "o1", "o2", "o3", "o4")}, inputs={})
    bufs = {"x": x.view(np.float32), "y": y.view(np.float32)}
    for k, dt in (("o1", "f32"), ("o2", "f16"), ("o3", "bf16"), ("o4", "f32")):
        bufs[k] = specutil.sentinel_array(dt, n)
    gpuutil.parity(spec, bufs)


def test_int_edge_values():
    e = np.array([0, 1, -1, 2**31 - 1, -2**31, 0x10000, -0x10000, 46341, -46341], dtype=np.int64)
    x = np.repeat(e, e.size).astype(np.int32)
    y = np.tile(e, e.size).astype(np.int32)
    n = x.size
    spec = dict(name="ints", seed=0, sizes=(n,),
                ops=[("load", "x", "i32"), ("load", "y", "i32"), ("scalar", "k", "i32", -2**31),
                     ("exec", [("mul", "p", "x", "y"), ("sub", "d", "p", "k"), ("neg", "m", "x", None),
                               ("add", "a", "m", "d")]),
                     ("store", "o", "a", "i32"), ("store", "o2", "m", "i32")],
                views={k: dict(strides=(1,), alloc=n) for k in ("x", "y", "o", "o2")}, inputs={})
    bufs = {"x": x, "y": y, "o": specutil.sentinel_array("i32", n), "o2": specutil.sentinel_array("i32", n)}
    gpuutil.parity(spec, bufs)


def test_sixteen_loads_and_eight_stores():
    rng = np.random.default_rng(11)
    n = 2049
    names = [f"x{i}" for i in range(16)]
    block = [("add", "s0", "x0", "x1")] + [("add", f"s{i}", f"s{i-1}", names[i + 1]) for i in range(1, 15)]
    stores = [(f"o{j}", f"s{14 - j}", ["f32", "f16", "bf16"][j % 3]) for j in range(8)]
    spec = dict(name="many", seed=0, sizes=(n,),
                ops=[("load", k, "f32") for k in names] + [("exec", block)]
                + [("store", o, s, dt) for o, s, dt in stores],
                views={k: dict(strides=(1,), alloc=n) for k in names + [o for o, _, _ in stores]}, inputs={})
    bufs = {k: rng.standard_normal(n).astype(np.float32) for k in names}
    for o, _, dt in stores:
        bufs[o] = specutil.sentinel_array(dt, n)
    gpuutil.parity(spec, bufs)


def test_launch_on_a_side_stream_and_relaunch():
    spec = W.chain_f32(70000)
    bufs = specutil.host_buffers(spec)
    s = torch.cuda.Stream()
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    for _ in range(3):
        got, _ = gpuutil.run_cuda(spec, bufs, stream=s, kernel=k)
    ref = {kk: v.copy() for kk, v in bufs.items()}
    oracle.OracleCommand(spec, ref).eval_range()
    gpuutil.compare(got["out"], ref["out"], "f32", "side stream")


def test_many_kernels_and_slot_reuse():
    """Compile more kernels than the constant table holds over time: destroyed
    kernels free their program slots for later compiles."""
    spec = W.add_f32(4096)
    bufs = specutil.host_buffers(spec)
    for i in range(120):
        c, _ = T.command_from_spec(spec)
        k = c.compile()
        if i % 40 == 0:
            got, _ = gpuutil.run_cuda(spec, bufs, kernel=k)
            gpuutil.compare(got["out"], bufs["x"] + bufs["y"], "f32", f"kernel {i}")
        del k, c


def test_exhaustive_store_conversion():
    """Every binary32 bit pattern stored as f16 and as bf16 through the GPU
    path equals the oracle's converter (NaNs compared as a class)."""
    from concurrent.futures import ThreadPoolExecutor
    chunk = 1 << 27
    spec = dict(name="conv", seed=0, sizes=(chunk,),
                ops=[("load", "x", "f32"), ("store", "h", "x", "f16"), ("store", "b", "x", "bf16")],
                views={k: dict(strides=(1,), alloc=chunk) for k in ("x", "h", "b")}, inputs={})
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    x = torch.empty(chunk, dtype=torch.int32, device="cuda")
    h = torch.empty(chunk, dtype=torch.int16, device="cuda")
    b = torch.empty(chunk, dtype=torch.int16, device="cuda")
    views = {tags["x"]: T.TensorView(x.data_ptr(), (chunk,), (1,)),
             tags["h"]: T.TensorView(h.data_ptr(), (chunk,), (1,)),
             tags["b"]: T.TensorView(b.data_ptr(), (chunk,), (1,))}
    ramp = torch.arange(chunk, dtype=torch.int64, device="cuda")
    pool = ThreadPoolExecutor(max_workers=16)
    for start in range(0, 1 << 32, chunk):
        x.copy_((ramp + start - (1 << 31)).to(torch.int32) ^ (-(1 << 31)))  # bit pattern start + i
        k.launch(views)
        k.sync()
        got_h = h.cpu().numpy().view(np.uint16)
        got_b = b.cpu().numpy().view(np.uint16)
        bits = (np.arange(chunk, dtype=np.uint64) + start).astype(np.uint32)
        parts = np.array_split(bits, 16)
        want_h = np.concatenate(list(pool.map(oracle.f32_to_f16_bits, parts)))
        want_b = np.concatenate(list(pool.map(oracle.f32_to_bf16_bits, parts)))
        gpuutil.compare(got_h, want_h, "f16", f"f16 from {start:#x}")
        gpuutil.compare(got_b, want_b, "bf16", f"bf16 from {start:#x}")


def test_device_wait_timeout_is_reported_and_the_context_recovers():
    """Force the tile executor's consumer warps to wait on a barrier nothing
    completes, with a 1 ms limit: the kernel must give up, the error must be
    reported by cmd_sync_status, and the next launch must work normally."""
    spec = W.strided_bf16(256, 192, 200)
    bufs = specutil.host_buffers(spec)
    dts = W.tensor_dtypes(spec)
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    dev = {n: gpuutil.to_device(bufs[n], dts[n]) for n in W.load_names(spec) + W.store_names(spec)}
    views = {tags[n]: T.TensorView(t.data_ptr(), spec["sizes"], spec["views"][n]["strides"]) for n, t in dev.items()}
    scal = T.spec_scalars(spec, tags)
    assert k.plan(views, scal)["path"] == "tile2d"
    T.cmd_configure_waits(1_000_000, True)
    try:
        k.launch(views, scal)
        with pytest.raises(T.CmdError) as e:
            k.sync()
        assert e.value.name == "CMD_ERR_DEVICE_TIMEOUT"
    finally:
        T.cmd_configure_waits(2_000_000_000, False)
    k.sync()  # the error word was cleared when reported
    gpuutil.parity(spec, bufs)


# ---- batched, permuted and broadcast views on the tile executor --------------------

def _nd_case(name, sizes, views, dts, seed=0):
    """out = A*B - A over rank-3 views; views/dts map A, B, out."""
    rng = np.random.default_rng(seed)
    spec = dict(name=name, seed=0, sizes=sizes,
                ops=[("load", "A", dts["A"]), ("load", "B", dts["B"]),
                     ("exec", [("mul", "AB", "A", "B"), ("sub", "r", "AB", "A")]),
                     ("store", "out", "r", dts["out"])],
                views={}, inputs={})
    bufs = {}
    for k in ("A", "B", "out"):
        st = views[k]
        alloc = sum((s - 1) * t for s, t in zip(sizes, st)) + 1
        spec["views"][k] = dict(strides=st, alloc=alloc)
        if k == "out":
            bufs[k] = specutil.sentinel_array(dts[k], alloc)
        else:
            bufs[k] = _random_values(rng, dts[k], alloc)
    return spec, bufs


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("case", ["batched_transpose", "perm_210", "batch_broadcast", "row_broadcast",
                                  "col_broadcast", "padded_batched"])
@pytest.mark.parametrize("sizes", [(3, 96, 136), (2, 64, 64), (5, 40, 72), (4, 40, 60), (2, 33, 100)])
def test_nd_views_on_the_tile_executor(dt, case, sizes):
    B, R, C = sizes
    dense = (R * C, C, 1)
    views = {
        "batched_transpose": {"A": (R * C, 1, R), "B": dense},
        "perm_210": {"A": (1, B, B * R), "B": dense},
        "batch_broadcast": {"A": (0, C, 1), "B": dense},
        "row_broadcast": {"A": (C, 0, 1), "B": dense},
        "col_broadcast": {"A": (R, 1, 0), "B": dense},
        "padded_batched": {"A": (R * (C + 8), C + 8, 1), "B": (R * C + 64, 1, R)},
    }[case]
    views = dict(views, out=dense)
    spec, bufs = _nd_case(f"{case}_{dt}", sizes, views, {"A": dt, "B": dt, "out": dt}, seed=B * 1000 + R)
    plan = gpuutil.parity(spec, bufs)
    es = 2 if dt == "bf16" else 4
    aligned = all((s * es) % 16 == 0 for s in (B, R, C, R * C))
    if case == "batch_broadcast" and aligned and (R * C) % 512 == 0:
        # (row, column) merge into rows of R * C elements, whole warp chunks
        # of the 2-slot tier: A's rows are one row read for every batch
        assert plan["path"] == "contig" and plan["merged_rank"] == 2, plan
    elif case in ("batched_transpose", "padded_batched", "batch_broadcast", "row_broadcast", "col_broadcast") \
            and aligned:
        assert plan["path"] == "tile2d", plan
    if case == "perm_210" and aligned and (B * es) % 16 == 0:
        assert plan["path"] == "tile2d", plan


def test_rank4_batched_transpose_with_two_batch_dims():
    sizes = (2, 3, 64, 80)
    A, R, C = sizes[1], sizes[2], sizes[3]
    dense = (A * R * C, R * C, C, 1)
    bt = (A * R * C, R * C, 1, R)
    spec, bufs = _nd_case("rank4", sizes, {"A": bt, "B": dense, "out": dense},
                          {"A": "f32", "B": "f32", "out": "f32"}, seed=4)
    plan = gpuutil.parity(spec, bufs)
    assert plan["path"] == "tile2d" and plan["merged_rank"] == 3  # the two batch dims merge


def test_rank4_with_two_batch_dims_that_do_not_merge():
    sizes = (2, 3, 64, 80)
    _, A, R, C = sizes
    dense = (A * R * C, R * C, C, 1)
    # A is a (3, 2, 80, 64) buffer: its two batch dims are swapped and its
    # tile is transposed, so nothing merges
    swapped = (R * C, 2 * R * C, 1, R)
    spec, bufs = _nd_case("rank4b", sizes, {"A": swapped, "B": dense, "out": dense},
                          {"A": "f32", "B": "f32", "out": "f32"}, seed=5)
    plan = gpuutil.parity(spec, bufs)
    assert plan["path"] == "tile2d" and plan["merged_rank"] == 4


# ---- division, min/max, abs and conversions ----------------------------------------------

BIN_OPS = ["add", "sub", "mul", "div", "min", "max"]
UN_OPS = ["neg", "abs", "to_f32", "to_i32"]


def random_mixed_case(seed):
    """A random Command over every E op, with float and int values mixed:
    binary ops take two values of one class, to_f32 / to_i32 cross over,
    and each store's type matches its value's class."""
    rng = np.random.default_rng(10_000 + seed)
    rank = int(rng.integers(0, 4))
    sizes = tuple(int(x) for x in rng.integers(1, 24, size=rank))
    if rank and rng.random() < 0.3:
        sizes = sizes[:-1] + (int(rng.integers(100, 700)),)
    ops, views, bufs = [], {}, {}
    vals = {"f": [], "i": []}
    for i in range(int(rng.integers(1, 7))):
        dt = str(rng.choice(["f32", "f16", "bf16", "i32"]))
        name = f"L{i}"
        ops.append(("load", name, dt))
        st, n = _random_view(rng, sizes, allow_broadcast=True)
        views[name] = dict(strides=st, alloc=n)
        bufs[name] = _random_values(rng, dt, n)
        if dt == "i32" and rng.random() < 0.5:
            bufs[name] = rng.integers(-9, 10, size=n).astype(np.int32)  # small: zeros and -1 as divisors
        vals["i" if dt == "i32" else "f"].append(name)
    for i in range(int(rng.integers(0, 3))):
        name = f"S{i}"
        if rng.random() < 0.5:
            ops.append(("scalar", name, "i32", int(rng.choice([0, -1, 3, -7, int(rng.integers(-2**31, 2**31))]))))
            vals["i"].append(name)
        else:
            ops.append(("scalar", name, "f32", float(np.float32(rng.choice([0.0, -0.0, 2.5, rng.standard_normal()])))))
            vals["f"].append(name)
    block, last = [], []
    for i in range(int(rng.integers(1, 22))):
        name = f"E{i}"
        eop = str(rng.choice(BIN_OPS + UN_OPS))
        cls = str(rng.choice([c for c in ("f", "i") if vals[c]]))
        a = str(rng.choice(vals[cls]))
        if eop in BIN_OPS:
            b = str(rng.choice(vals[cls]))
            out_cls = cls
        else:
            b = None
            out_cls = {"to_f32": "f", "to_i32": "i"}.get(eop, cls)
        block.append((eop, name, a, b))
        vals[out_cls].append(name)
        last.append((name, out_cls))
    ops.append(("exec", block))
    for i in range(int(rng.integers(1, 4))):
        src, cls = last[-1 - int(rng.integers(0, min(4, len(last))))]
        dt = "i32" if cls == "i" else str(rng.choice(["f32", "f16", "bf16"]))
        name = f"O{i}"
        ops.append(("store", name, src, dt))
        st, n = _random_view(rng, sizes, allow_broadcast=False)
        views[name] = dict(strides=st, alloc=n)
        bufs[name] = specutil.sentinel_array(dt, n)
    return dict(name=f"mixed{seed}", seed=seed, sizes=sizes, ops=ops, views=views, inputs={}), bufs


@pytest.mark.parametrize("seed", range(80))
def test_random_mixed_commands(seed):
    spec, bufs = random_mixed_case(seed)
    gpuutil.parity(spec, bufs)


F_SPECIALS = np.array([0, 0x80000000, 1, 0x80000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0xFF7FFFFF,
                       0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000, 0x3F800000, 0xBF800000, 0x40400000,
                       0x4F000000, 0xCF000000, 0x4EFFFFFF, 0x3F000000, 0xBFC00000, 0x33800000], dtype=np.uint32)
I_SPECIALS = np.array([0, 1, -1, 2, -2, 7, -7, 2**31 - 1, -2**31, 0x10000, -0x10000, 16777217, -16777219],
                      dtype=np.int64)


def _pairs(vals):
    return np.repeat(vals, vals.size), np.tile(vals, vals.size)


@pytest.mark.parametrize("tier_pad", [0, 9, 14])
def test_new_float_ops_on_special_values(tier_pad):
    """Every pair of special floats through div / min / max (both operand
    orders reach the reversed forms), abs and to_i32; tier_pad extra live
    values push the program to a wider tier."""
    xb, yb = _pairs(F_SPECIALS)
    n = xb.size
    pad = [f"p{i}" for i in range(tier_pad)]
    block = [("div", "q", "x", "y"), ("div", "r", "y", "q"), ("min", "lo", "x", "y"), ("max", "hi", "y", "x"),
             ("abs", "ax", "x", None), ("to_i32", "ti", "x", None), ("div", "qs", "x", "k"),
             ("min", "ms", "k", "y")]
    block += [("add", f"s{i}", p, "x") for i, p in enumerate(pad)]
    acc = "r"
    for i in range(tier_pad):
        block.append(("add", f"a{i}", acc, f"s{i}"))
        acc = f"a{i}"
    ops = ([("load", "x", "f32"), ("load", "y", "f32")] + [("load", p, "f32") for p in pad]
           + [("scalar", "k", "f32", -0.0), ("exec", block)]
           + [("store", o, s, dt) for o, s, dt in (("o_q", "q", "f32"), ("o_r", acc, "f32"), ("o_lo", "lo", "f32"),
                                                   ("o_hi", "hi", "bf16"), ("o_ax", "ax", "f16"),
                                                   ("o_ti", "ti", "i32"), ("o_qs", "qs", "f32"),
                                                   ("o_ms", "ms", "f32"))])
    names = ["x", "y"] + pad + ["o_q", "o_r", "o_lo", "o_hi", "o_ax", "o_ti", "o_qs", "o_ms"]
    spec = dict(name="fspecials", seed=0, sizes=(n,), ops=ops,
                views={k: dict(strides=(1,), alloc=n) for k in names}, inputs={})
    bufs = {"x": xb.view(np.float32), "y": yb.view(np.float32)}
    rng = np.random.default_rng(3)
    for p in pad:
        bufs[p] = rng.standard_normal(n).astype(np.float32)
    for o, _, dt in [(op[1], None, op[3]) for op in ops if op[0] == "store"]:
        bufs[o] = specutil.sentinel_array(dt, n)
    if tier_pad:
        c, _ = T.command_from_spec(spec)
        # (9 pads: 13-14 slots, the 16-slot tier; 14 pads: 18-19, the 32-slot tier)
        assert c.lower()[0]["tier"] == (4 if tier_pad < 14 else 3)
    gpuutil.parity(spec, bufs)


@pytest.mark.parametrize("tier_pad", [0, 9, 14])
def test_new_int_ops_on_edge_values(tier_pad):
    """Every pair of int32 edge values through division (zero and -1
    divisors, INT_MIN / -1, both operand orders), min / max, abs and
    to_f32 (rounding above 2^24)."""
    x, y = (v.astype(np.int32) for v in _pairs(I_SPECIALS))
    n = x.size
    pad = [f"p{i}" for i in range(tier_pad)]
    block = [("div", "q", "x", "y"), ("div", "r", "y", "x"), ("min", "lo", "x", "y"), ("max", "hi", "x", "y"),
             ("abs", "ax", "x", None), ("to_f32", "f", "x", None), ("div", "qs", "x", "k"),
             ("div", "sq", "k", "y")]
    block += [("add", f"s{i}", p, "q") for i, p in enumerate(pad)]
    acc = "r"
    for i in range(tier_pad):
        block.append(("mul", f"a{i}", acc, f"s{i}"))
        acc = f"a{i}"
    ops = ([("load", "x", "i32"), ("load", "y", "i32")] + [("load", p, "i32") for p in pad]
           + [("scalar", "k", "i32", -1), ("exec", block)]
           + [("store", o, s, dt) for o, s, dt in (("o_q", "q", "i32"), ("o_r", acc, "i32"), ("o_lo", "lo", "i32"),
                                                   ("o_hi", "hi", "i32"), ("o_ax", "ax", "i32"),
                                                   ("o_f", "f", "f32"), ("o_qs", "qs", "i32"),
                                                   ("o_sq", "sq", "i32"))])
    names = ["x", "y"] + pad + ["o_q", "o_r", "o_lo", "o_hi", "o_ax", "o_f", "o_qs", "o_sq"]
    spec = dict(name="ispecials", seed=0, sizes=(n,), ops=ops,
                views={k: dict(strides=(1,), alloc=n) for k in names}, inputs={})
    bufs = {"x": x, "y": y}
    rng = np.random.default_rng(4)
    for p in pad:
        bufs[p] = rng.integers(-2**31, 2**31, size=n).astype(np.int32)
    for o, dt in [(op[1], op[3]) for op in ops if op[0] == "store"]:
        bufs[o] = specutil.sentinel_array(dt, n)
    if tier_pad:
        c, _ = T.command_from_spec(spec)
        # (9 pads: 13-14 slots, the 16-slot tier; 14 pads: 18-19, the 32-slot tier)
        assert c.lower()[0]["tier"] == (4 if tier_pad < 14 else 3)
    gpuutil.parity(spec, bufs)


@pytest.mark.parametrize("path", ["contig", "tile2d", "generic"])
def test_new_ops_on_each_executor(path):
    """One Command with every new op, on a dense view (contig), a transposed
    2-D view (tile2d) and a padded odd-offset view (generic)."""
    rng = np.random.default_rng(21)
    m, nn = 96, 136
    spec = dict(name=f"newops_{path}", seed=0, sizes=(m, nn),
                ops=[("load", "A", "f32"), ("load", "B", "f32"), ("load", "I", "i32"),
                     ("exec", [("div", "q", "A", "B"), ("min", "lo", "q", "A"), ("max", "hi", "lo", "B"),
                               ("abs", "ab", "hi", None), ("to_i32", "ti", "ab", None),
                               ("div", "id", "I", "ti"), ("max", "im", "id", "I"), ("to_f32", "fi", "im", None),
                               ("sub", "r", "fi", "q")]),
                     ("store", "o1", "r", "f32"), ("store", "o2", "im", "i32")],
                views={}, inputs={})
    dense = ((nn, 1), m * nn)
    if path == "contig":
        a_view = dense
    elif path == "tile2d":
        a_view = ((1, m), m * nn)
    else:
        a_view = ((nn + 3, 1), (m - 1) * (nn + 3) + nn)
    spec["views"] = {"A": dict(strides=a_view[0], alloc=a_view[1]), "B": dict(strides=dense[0], alloc=dense[1]),
                     "I": dict(strides=dense[0], alloc=dense[1]), "o1": dict(strides=dense[0], alloc=dense[1]),
                     "o2": dict(strides=dense[0], alloc=dense[1])}
    bufs = {"A": (rng.standard_normal(a_view[1]) * 40).astype(np.float32),
            "B": (rng.standard_normal(dense[1]) * 3).astype(np.float32),
            "I": rng.integers(-1000, 1000, size=dense[1]).astype(np.int32),
            "o1": specutil.sentinel_array("f32", dense[1]), "o2": specutil.sentinel_array("i32", dense[1])}
    offsets = {"A": 1} if path == "generic" else None
    plan = gpuutil.parity(spec, bufs, offsets)
    assert plan["path"] == path


# ---- comparisons, select and packed-bit stores --------------------------------------------

CMP_OPS = ["lt", "le", "gt", "ge", "eq", "ne"]
UCMP_OPS = ["ult", "ule", "ugt", "uge"]


def random_cmp_case(seed):
    """A random Command over every E op including comparisons and select,
    float and int values mixed; some int results are stored as packed bits
    (dense views only, as b1 requires)."""
    rng = np.random.default_rng(20_000 + seed)
    rank = int(rng.integers(0, 4))
    sizes = tuple(int(x) for x in rng.integers(1, 24, size=rank))
    if rank and rng.random() < 0.4:
        sizes = sizes[:-1] + (int(rng.integers(100, 700)),)
    ops, views, bufs = [], {}, {}
    vals = {"f": [], "i": []}
    for i in range(int(rng.integers(1, 7))):
        dt = str(rng.choice(["f32", "f16", "bf16", "i32"]))
        name = f"L{i}"
        ops.append(("load", name, dt))
        st, n = _random_view(rng, sizes, allow_broadcast=True)
        views[name] = dict(strides=st, alloc=n)
        bufs[name] = _random_values(rng, dt, n)
        if dt == "i32" and rng.random() < 0.5:
            bufs[name] = rng.integers(-3, 4, size=n).astype(np.int32)  # ties in comparisons
        if dt == "f32" and rng.random() < 0.3:
            bufs[name][::7] = np.float32(np.nan)
            bufs[name][1::11] = np.float32(-0.0)
        vals["i" if dt == "i32" else "f"].append(name)
    for i in range(int(rng.integers(0, 3))):
        name = f"S{i}"
        if rng.random() < 0.5:
            ops.append(("scalar", name, "i32", int(rng.choice([0, 1, -1, int(rng.integers(-2**31, 2**31))]))))
            vals["i"].append(name)
        else:
            ops.append(("scalar", name, "f32", float(np.float32(rng.choice([0.0, -0.0, 0.5, rng.standard_normal()])))))
            vals["f"].append(name)
    block, last = [], []
    for i in range(int(rng.integers(1, 22))):
        name = f"E{i}"
        kind = rng.choice(["bin", "un", "cmp", "ucmp", "sel"], p=[0.3, 0.1, 0.3, 0.1, 0.2])
        cls = str(rng.choice([c for c in ("f", "i") if vals[c]]))
        a = str(rng.choice(vals[cls]))
        if kind == "bin":
            eop, b, out = str(rng.choice(BIN_OPS)), str(rng.choice(vals[cls])), cls
            block.append((eop, name, a, b))
        elif kind == "un":
            eop = str(rng.choice(UN_OPS))
            out = {"to_f32": "f", "to_i32": "i"}.get(eop, cls)
            block.append((eop, name, a, None))
        elif kind == "cmp" or (kind == "ucmp" and cls == "f"):
            block.append((str(rng.choice(CMP_OPS)), name, a, str(rng.choice(vals[cls]))))
            out = "i"
        elif kind == "ucmp":
            block.append((str(rng.choice(UCMP_OPS)), name, a, str(rng.choice(vals["i"]))))
            out = "i"
        else:
            if not vals["i"]:
                continue
            block.append(("select", name, a, str(rng.choice(vals[cls])), str(rng.choice(vals["i"]))))
            out = cls
        vals[out].append(name)
        last.append((name, out))
    if not block:
        block.append(("ne", "E0", vals["i"][0] if vals["i"] else vals["f"][0],
                      vals["i"][0] if vals["i"] else vals["f"][0]))
        last.append(("E0", "i"))
    ops.append(("exec", block))
    n_el = int(np.prod(sizes)) if sizes else 1
    for i in range(int(rng.integers(1, 4))):
        src, cls = last[-1 - int(rng.integers(0, min(4, len(last))))]
        if cls == "i":
            dt = "b1" if rng.random() < 0.5 else "i32"
        else:
            dt = str(rng.choice(["f32", "f16", "bf16"]))
        name = f"O{i}"
        ops.append(("store", name, src, dt))
        if dt == "b1":
            st, _ = _dense_strides(sizes)
            views[name] = dict(strides=st, alloc=(n_el + 31) // 32)
        else:
            st, n = _random_view(rng, sizes, allow_broadcast=False)
            views[name] = dict(strides=st, alloc=n)
        bufs[name] = specutil.sentinel_array(dt, views[name]["alloc"])
    return dict(name=f"cmp{seed}", seed=seed, sizes=sizes, ops=ops, views=views, inputs={}), bufs


@pytest.mark.parametrize("seed", range(100))
def test_random_compare_select_commands(seed):
    spec, bufs = random_cmp_case(seed)
    gpuutil.parity(spec, bufs)


def random_wide_case(seed):
    """A random Command whose lowered program needs more than 8 slots (the
    16- and 32-slot tiers): 9 to 16 loads of mixed types, operands drawn
    from the whole history so that early values stay live, 2 to 6 stores
    (int results sometimes as packed bits). By seed % 3: every E op including
    division, comparisons and select (the extended variant); only the base
    ops (add, sub, mul, min, max, neg, abs, conversions); or the base ops
    with a closing sum over 20 independent products, which keeps more than
    16 values live (the 32-slot tier). Drawn again (from the same seed's
    stream) until the program is past 8 slots (past 16 for the third kind)."""
    rng = np.random.default_rng(40_000 + seed)
    mode = seed % 3
    bin_ops = BIN_OPS if mode == 0 else [o for o in BIN_OPS if o != "div"]
    kinds, kp = (["bin", "un", "cmp", "sel"], [0.55, 0.15, 0.2, 0.1]) if mode == 0 else (["bin", "un"], [0.8, 0.2])
    while True:
        rank = int(rng.integers(1, 3))
        sizes = tuple(int(x) for x in rng.integers(2, 40, size=rank))
        if rng.random() < 0.5:
            sizes = sizes[:-1] + (int(rng.integers(300, 3000)),)
        ops, views, bufs = [], {}, {}
        vals = {"f": [], "i": []}
        for i in range(int(rng.integers(9, 17))):
            dt = str(rng.choice(["f32", "f16", "bf16", "i32"], p=[0.4, 0.15, 0.15, 0.3]))
            name = f"L{i}"
            ops.append(("load", name, dt))
            st, n = _random_view(rng, sizes, allow_broadcast=True) if rng.random() < 0.4 else _dense_strides(sizes)
            views[name] = dict(strides=st, alloc=n)
            bufs[name] = _random_values(rng, dt, n)
            if dt == "i32" and rng.random() < 0.5:
                bufs[name] = rng.integers(-5, 6, size=n).astype(np.int32)
            vals["i" if dt == "i32" else "f"].append(name)
        for i in range(int(rng.integers(0, 4))):
            name = f"S{i}"
            if rng.random() < 0.5:
                ops.append(("scalar", name, "i32", int(rng.choice([0, -1, 3, int(rng.integers(-2**31, 2**31))]))))
                vals["i"].append(name)
            else:
                ops.append(("scalar", name, "f32", float(np.float32(rng.choice([0.0, -0.0, 1.5, rng.standard_normal()])))))
                vals["f"].append(name)
        block, last = [], []
        for i in range(int(rng.integers(10, 40))):
            name = f"E{i}"
            kind = rng.choice(kinds, p=kp)
            cls = str(rng.choice([c for c in ("f", "i") if vals[c]]))
            a = str(rng.choice(vals[cls]))
            if kind == "bin":
                block.append((str(rng.choice(bin_ops)), name, a, str(rng.choice(vals[cls]))))
                out = cls
            elif kind == "un":
                eop = str(rng.choice(UN_OPS))
                out = {"to_f32": "f", "to_i32": "i"}.get(eop, cls)
                block.append((eop, name, a, None))
            elif kind == "cmp":
                block.append((str(rng.choice(CMP_OPS)), name, a, str(rng.choice(vals[cls]))))
                out = "i"
            else:
                if not vals["i"]:
                    continue
                block.append(("select", name, a, str(rng.choice(vals[cls])), str(rng.choice(vals["i"]))))
                out = cls
            vals[out].append(name)
            last.append((name, out))
        if mode == 2:
            # 20 products of loads, all live until the closing sum
            cls = "f" if len(vals["f"]) >= 2 else "i"
            pool = [v for v in vals[cls] if v.startswith("L")] or vals[cls]
            prods = []
            for k in range(20):
                name = f"P{k}"
                block.append(("mul", name, str(rng.choice(pool)), str(rng.choice(pool))))
                prods.append(name)
            acc = prods[0]
            for k in range(1, 20):
                block.append(("add", f"Q{k}", acc, prods[k]))
                acc = f"Q{k}"
            last.append((acc, cls))
        ops.append(("exec", block))
        n_el = int(np.prod(sizes))
        for i in range(int(rng.integers(2, 7))):
            src, cls = last[-1 - int(rng.integers(0, min(12, len(last))))]
            dt = ("b1" if rng.random() < 0.3 else "i32") if cls == "i" else str(rng.choice(["f32", "f16", "bf16"]))
            name = f"O{i}"
            ops.append(("store", name, src, dt))
            if dt == "b1":
                st, _ = _dense_strides(sizes)
                views[name] = dict(strides=st, alloc=(n_el + 31) // 32)
            else:
                st, n = _random_view(rng, sizes, allow_broadcast=False) if rng.random() < 0.3 else _dense_strides(sizes)
                views[name] = dict(strides=st, alloc=n)
            bufs[name] = specutil.sentinel_array(dt, views[name]["alloc"])
        spec = dict(name=f"wide{seed}", seed=seed, sizes=sizes, ops=ops, views=views, inputs={})
        c, _ = T.command_from_spec(spec)
        if c.lower()[0]["n_slots"] > (16 if mode == 2 else 8):
            return spec, bufs


@pytest.mark.parametrize("seed", range(60))
def test_random_wide_commands(seed):
    spec, bufs = random_wide_case(seed)
    c, _ = T.command_from_spec(spec)
    assert c.lower()[0]["tier"] in (3, 4)
    gpuutil.parity(spec, bufs)


@pytest.mark.parametrize("pad", [0, 4, 9])
def test_comparisons_and_select_on_special_values(pad):
    """Every pair of special floats and of int edge values through every
    comparison (slot and scalar forms, both operand orders) and select;
    pad extra live values move the program to the 8- and 32-slot tiers."""
    xb, yb = _pairs(F_SPECIALS)
    n = xb.size
    xi = np.resize(np.repeat(I_SPECIALS, I_SPECIALS.size), n).astype(np.int32)
    yi = np.resize(np.tile(I_SPECIALS, I_SPECIALS.size), n).astype(np.int32)
    pads = [f"p{i}" for i in range(pad)]
    block, outs = [], []
    for rel in CMP_OPS:
        block += [(rel, f"f{rel}", "x", "y"), (rel, f"fs{rel}", "x", "k"), (rel, f"fr{rel}", "k", "y"),
                  (rel, f"i{rel}", "xi", "yi")]
        outs += [f"f{rel}", f"fs{rel}", f"fr{rel}", f"i{rel}"]
    for rel in UCMP_OPS:
        block += [(rel, f"u{rel}", "xi", "yi"), (rel, f"us{rel}", "ki", "yi")]
        outs += [f"u{rel}", f"us{rel}"]
    block += [("select", "sf", "x", "y", "flt"), ("select", "si", "xi", "yi", "xi"),
              ("select", "ss", "x", "k", "ige"), ("select", "sk", "k", "y", "ine")]
    block += [("add", f"q{i}", p, "x") for i, p in enumerate(pads)]
    acc = "sf"
    for i in range(pad):
        block.append(("add", f"a{i}", acc, f"q{i}"))
        acc = f"a{i}"
    # every result stored, comparisons alternately as i32 words and packed
    # bits; at most 8 stores per Command, so the results are split over several
    all_stores = [(f"o_{o}", o, "b1" if j % 2 else "i32") for j, o in enumerate(outs)]
    all_stores += [("o_sf", acc, "f32"), ("o_si", "si", "i32"), ("o_ss", "ss", "f32"), ("o_sk", "sk", "bf16")]
    names = ["x", "y", "xi", "yi"] + pads
    loads = [("load", "x", "f32"), ("load", "y", "f32"), ("load", "xi", "i32"), ("load", "yi", "i32")]
    loads += [("load", p, "f32") for p in pads]
    scal = [("scalar", "k", "f32", -0.0), ("scalar", "ki", "i32", -2**31)]
    rng = np.random.default_rng(7)
    base = {"x": xb.view(np.float32), "y": yb.view(np.float32), "xi": xi, "yi": yi}
    for p in pads:
        base[p] = rng.standard_normal(n).astype(np.float32)
    for gi in range(0, len(all_stores), 8):
        group = all_stores[gi:gi + 8]
        ops = loads + scal + [("exec", block)] + [("store", o, src, dt) for o, src, dt in group]
        views = {k: dict(strides=(1,), alloc=n) for k in names}
        bufs = dict(base)
        for o, _, dt in group:
            views[o] = dict(strides=(1,), alloc=(n + 31) // 32 if dt == "b1" else n)
            bufs[o] = specutil.sentinel_array(dt, views[o]["alloc"])
        spec = dict(name=f"cmpspecials{gi}", seed=0, sizes=(n,), ops=ops, views=views, inputs={})
        if pad >= 4 and any(src == acc for _, src, _ in group):
            # (4 pads: 13 slots, the 16-slot tier; 9 pads: 18 slots, the 32-slot tier)
            c, _ = T.command_from_spec(spec)
            assert c.lower()[0]["tier"] == (4 if pad < 9 else 3)
        gpuutil.parity(spec, bufs)


@pytest.mark.parametrize("n", [1, 31, 32, 33, 255, 256, 257, 1000, 4097, (1 << 20) + 5])
def test_packed_bits_ragged_lengths(n):
    """b1 stores over the contiguous executor (with its generic tail) at
    ragged lengths: whole words, last word's extra bits zero, and the words
    after the buffer untouched (sentinel guard)."""
    rng = np.random.default_rng(n)
    x = rng.integers(-2**31, 2**31, size=n).astype(np.int32)
    nb = (n + 31) // 32
    spec = dict(name=f"bits{n}", seed=0, sizes=(n,),
                ops=[("load", "x", "i32"), ("scalar", "t", "i32", 0),
                     ("exec", [("lt", "neg", "x", "t"), ("ugt", "big", "x", "t")]),
                     ("store", "b_neg", "neg", "b1"), ("store", "b_big", "big", "b1")],
                views={"x": dict(strides=(1,), alloc=n), "b_neg": dict(strides=(1,), alloc=nb + 2),
                       "b_big": dict(strides=(1,), alloc=nb)}, inputs={})
    bufs = {"x": x, "b_neg": specutil.sentinel_array("b1", nb + 2), "b_big": specutil.sentinel_array("b1", nb)}
    plan = gpuutil.parity(spec, bufs)
    assert plan["path"] == "contig"


@pytest.mark.parametrize("case", ["strided_input", "transposed_input", "misaligned"])
def test_packed_bits_on_the_generic_executor(case):
    """A b1 store next to views the contiguous executor cannot take: the plan
    falls to the generic executor (never to the tile one)."""
    rng = np.random.default_rng(3)
    m, nn = 70, 133
    n = m * nn
    nb = (n + 31) // 32
    a_view = {"strided_input": ((nn + 5, 1), (m - 1) * (nn + 5) + nn),
              "transposed_input": ((1, m), n),
              "misaligned": ((nn, 1), n)}[case]
    spec = dict(name=f"bits_{case}", seed=0, sizes=(m, nn),
                ops=[("load", "A", "f32"), ("load", "B", "f32"),
                     ("exec", [("gt", "g", "A", "B"), ("select", "r", "A", "B", "g")]),
                     ("store", "bits", "g", "b1"), ("store", "mx", "r", "f32")],
                views={"A": dict(strides=a_view[0], alloc=a_view[1]), "B": dict(strides=(nn, 1), alloc=n),
                       "bits": dict(strides=(nn, 1), alloc=nb), "mx": dict(strides=(nn, 1), alloc=n)},
                inputs={})
    bufs = {"A": rng.standard_normal(a_view[1]).astype(np.float32), "B": rng.standard_normal(n).astype(np.float32),
            "bits": specutil.sentinel_array("b1", nb), "mx": specutil.sentinel_array("f32", n)}
    plan = gpuutil.parity(spec, bufs, {"A": 1} if case == "misaligned" else None)
    assert plan["path"] == "generic"


def test_packed_bits_view_must_be_dense():
    n = 64
    spec = dict(name="bad", seed=0, sizes=(2, n // 2),
                ops=[("load", "x", "i32"), ("exec", [("ne", "p", "x", "x")]), ("store", "bits", "p", "b1")],
                views={"x": dict(strides=(n // 2, 1), alloc=n), "bits": dict(strides=(1, 2), alloc=2)}, inputs={})
    bufs = {"x": np.zeros(n, np.int32), "bits": specutil.sentinel_array("b1", 2)}
    with pytest.raises(T.CmdError) as e:
        gpuutil.run_cuda(spec, bufs)
    assert e.value.name == "CMD_ERR_SHAPE"


@pytest.mark.parametrize("pad", [0, 2, 6])
def test_scalar_compare_into_the_tiers_last_slot(pad):
    """A comparison with a scalar reads no staging slot, so its result may sit
    in the tier's last slot (a fault of this kind once ended the program
    there without storing anything)."""
    n = 1000
    rng = np.random.default_rng(pad)
    names = ["x"] + [f"p{i}" for i in range(pad)]
    block = [("ne", "k", "s", "s"), ("add", "kx", "k", "x")]
    acc = "kx"
    for i in range(pad):
        block.append(("add", f"a{i}", acc, f"p{i}"))
        acc = f"a{i}"
    spec = dict(name=f"lastslot{pad}", seed=0, sizes=(n,),
                ops=[("load", k, "i32") for k in names] + [("scalar", "s", "i32", 3), ("exec", block),
                                                          ("store", "o", acc, "i32"), ("store", "ob", "k", "b1")],
                views={**{k: dict(strides=(1,), alloc=n) for k in names + ["o"]},
                       "ob": dict(strides=(1,), alloc=(n + 31) // 32)}, inputs={})
    bufs = {k: rng.integers(-100, 100, size=n).astype(np.int32) for k in names}
    bufs["o"] = specutil.sentinel_array("i32", n)
    bufs["ob"] = specutil.sentinel_array("b1", (n + 31) // 32)
    gpuutil.parity(spec, bufs)


@pytest.mark.parametrize("spec", [W.chain_f32(5000), W.wide_dag(4099), W.strided_bf16(130, 72, 80),
                                  W.threshold_bits(3000), W.div_clamp_i32(777), W.batched_transpose(2, 64, 96)],
                         ids=lambda s: s["name"])
def test_kernel_from_text_form(spec):
    """A Command written with cmd_to_yaml and read back with cmd_from_yaml
    compiles to a kernel whose results match the oracle element by element
    (rocRoller, "Design Overview", section "Serialization")."""
    c, _ = T.command_from_spec(spec)
    k = T.Command.from_yaml(c.to_yaml()).compile()
    bufs = specutil.host_buffers(spec)
    got, _ = gpuutil.run_cuda(spec, bufs, kernel=k)
    ref = {n: v.copy() for n, v in bufs.items()}
    oracle.OracleCommand(spec, ref).eval_range()
    dts = W.tensor_dtypes(spec)
    for name in W.store_names(spec):
        gpuutil.compare(got[name], ref[name], dts[name], f"{spec['name']}:{name} (from text)")


@pytest.mark.parametrize("n,path", [(1 << 20, "contig"), (5000, "contig"), (3 * 64 * 96, "tile2d"),
                                    (500, "generic"), (64 * 1024, "rows"), (70_001, "shifted")])
def test_back_to_back_dependent_launches(n, path):
    """Launches may begin while the previous kernel on the stream runs
    (programmatic dependent launch), but each waits for it before touching
    memory: a chain of launches where each reads what the last one wrote
    and overwrites what the last one read, with no synchronisation between
    them, gives the same result as running them one at a time."""
    rng = np.random.default_rng(n)
    if path == "tile2d":
        sizes, st_x = (3, 64, 96), (64 * 96, 1, 64)  # x read through a transposed view
    elif path == "rows":
        sizes, st_x = (64, 1024), (1040, 1)  # x's rows padded: the contiguous executor walks rows
    else:
        sizes, st_x = (n,), (1,)
    dense = W._dense(sizes)[0]
    x = torch.from_numpy(rng.integers(-2**31, 2**31, size=n).astype(np.int32)).cuda()
    if path in ("generic", "shifted"):  # x one element off the vector alignment, y on it: too short
        # for one warp chunk, per element; longer, the loads are shifted
        big = torch.empty(n + 1, dtype=torch.int32, device="cuda")
        big[1:].copy_(x)
        x = big[1:]
    pad = None
    if path == "rows":
        pad = torch.full((64, 1040), -5, dtype=torch.int32, device="cuda")
        pad[:, :1024].copy_(x.view(64, 1024))
        x = pad.view(-1)
    y = torch.empty(n, dtype=torch.int32, device="cuda")
    # A: y = x * x + k (reads x, writes y);  B: x = -y (reads y, overwrites x)
    ca = T.Command()
    xa = ca.load_tensor("i32", len(sizes))
    ka = ca.load_scalar("i32")
    ta = ca.execute([("mul", xa, xa), ("add", T.CMD_LOCAL(0), ka)])
    ya = ca.store(ta[1], "i32", len(sizes))
    cb = T.Command()
    yb = cb.load_tensor("i32", len(sizes))
    tb = cb.execute([("neg", yb, None)])
    xb = cb.store(tb[0], "i32", len(sizes))
    ka_k, kb_k = ca.compile(), cb.compile()
    vx = T.TensorView(x.data_ptr(), sizes, st_x)
    vy = T.TensorView(y.data_ptr(), sizes, dense)
    args_a = ka_k.args({xa: vx, ya: vy}, {ka: 7})
    args_b = kb_k.args({yb: vy, xb: vx}, {})
    assert ka_k.plan({xa: vx, ya: vy}, {ka: 7})["path"] == ("contig" if path in ("rows", "shifted") else path)
    host = (pad[:, :1024].reshape(-1) if pad is not None else x).cpu().numpy().astype(np.int64)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(12):
        ka_k.launch_args(args_a, stream)
        kb_k.launch_args(args_b, stream)
        yv = (host * host + 7) % 2**32                 # A, modulo 2^32
        host = ((-yv) % 2**32 + 2**31) % 2**32 - 2**31  # B, back to int32
    torch.cuda.synchronize()
    if pad is not None:
        # the view's elements follow the recurrence; the row padding is untouched
        assert (pad[:, :1024].cpu().numpy().reshape(-1) == host.astype(np.int32)).all()
        assert (pad[:, 1024:].cpu().numpy() == -5).all()
        return
    # every physical element of x follows the same recurrence (a view is a
    # permutation of its buffer), so the buffers compare directly
    assert (x.cpu().numpy() == host.astype(np.int32)).all()


def test_concurrent_compile_launch_destroy_from_threads():
    """Eight host threads, each on its own stream, repeatedly compile a
    distinct Command, launch it, check it against the oracle and destroy it
    (slots are reused), with no locking on the caller's side."""
    import threading
    errors = []
    specs = [W.chain_f32(3000 + 17 * t) if t % 3 == 0 else
             W.wrap_i32(2000 + 5 * t) if t % 3 == 1 else
             W.threshold_bits(4000 + 33 * t) for t in range(8)]
    refs = []
    for spec in specs:
        bufs = specutil.host_buffers(spec)
        ref = {k: v.copy() for k, v in bufs.items()}
        oracle.OracleCommand(spec, ref).eval_range()
        refs.append((bufs, ref))

    def worker(t):
        try:
            spec = specs[t]
            bufs, ref = refs[t]
            s = torch.cuda.Stream()
            dts = W.tensor_dtypes(spec)
            for _ in range(6):
                with torch.cuda.stream(s):
                    c, _ = T.command_from_spec(spec)
                    k = c.compile()
                    got, _ = gpuutil.run_cuda(spec, bufs, stream=s.cuda_stream, kernel=k)
                for name in W.store_names(spec):
                    gpuutil.compare(got[name], ref[name], dts[name], f"thread {t}: {name}")
                del k, c
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(8)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(300)
    assert not errors, errors[:3]
