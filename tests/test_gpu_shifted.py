"""1-D launches whose loads sit off the stores' vector alignment by other
numbers of elements (x[1:] - x[:-1] and the like), on the GPU: the head runs
per element up to where the stores align plus 4 elements, the contiguous
kernel reads each such load as aligned vectors and takes the end of every
lane's elements from its right neighbour (the last lane from the next group,
or one more vector after the chunk), and a tail of at least 4 elements runs
per element. Every element of every store buffer, and the bytes around the
views (sentinels), against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import gpuutil
import layouts
import specutil

pytestmark = pytest.mark.gpu


def case(name, n, loads, stores, block, scalars=(), seed=0):
    """loads: {name: dtype}; stores: {name: (source, dtype)}."""
    ops = [("load", k, dt) for k, dt in loads.items()] + [("scalar", k, dt, v) for k, dt, v in scalars]
    ops += [("exec", block)] + [("store", k, src, dt) for k, (src, dt) in stores.items()]
    views = {k: dict(strides=(1,), alloc=n) for k in list(loads) + list(stores)}
    spec = dict(name=name, seed=seed, sizes=(n,), ops=ops, views=views, inputs={})
    rng = np.random.default_rng(seed)
    bufs = {k: layouts.values(rng, dt, n) for k, dt in loads.items()}
    for k, (_, dt) in stores.items():
        bufs[k] = specutil.sentinel_array(dt, n)
    return spec, bufs


def _check(spec, bufs, offsets, want_path="contig"):
    plan = gpuutil.parity(spec, bufs, offsets)
    assert plan["path"] == want_path, (plan, offsets)
    return plan


ADD = [("add", "z", "x", "y")]
STENCIL = [("sub", "d", "x", "y"), ("mul", "e", "d", "s"), ("add", "z", "e", "w")]


@pytest.mark.parametrize("dt", ["f32", "i32", "bf16", "f16"])
@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 3, 0), (2, 1, 0), (3, 3, 1), (1, 2, 3), (0, 0, 2)])
def test_two_input_add_every_phase(dt, offs):
    """Load and store offsets in elements (x, y, out): every load shift 1..3
    against every store phase, ragged length."""
    n = (1 << 15) + 37
    odt = dt
    spec, bufs = case(f"add_{dt}", n, {"x": dt, "y": dt}, {"out": ("z", odt)}, ADD, seed=sum(offs) + len(dt))
    _check(spec, bufs, dict(zip(("x", "y", "out"), offs)))


@pytest.mark.parametrize("n", [7 + 512 + 4, 7 + 512 + 5, 7 + 1024 + 4, 4 * 512 + 9, (1 << 20) + 3])
def test_lengths_around_one_chunk(n):
    """Launch lengths at the threshold (head + one chunk + 4) and above."""
    spec, bufs = case("add_len", n, {"x": "f32", "y": "f32"}, {"out": ("z", "f32")}, ADD, seed=n % 97)
    _check(spec, bufs, {"x": 2, "y": 0, "out": 1})


def test_shorter_than_the_threshold_runs_per_element():
    n = 7 + 512 + 3
    spec, bufs = case("add_short", n, {"x": "f32", "y": "f32"}, {"out": ("z", "f32")}, ADD, seed=1)
    _check(spec, bufs, {"x": 2, "y": 0, "out": 1}, want_path="generic")


@pytest.mark.parametrize("offs", [(1, 0, 0, 0), (1, 2, 3, 0), (0, 1, 2, 3), (3, 0, 1, 2)])
def test_stencil_in_the_4_slot_tier(offs):
    """(x - y) * s + w with w live across: the 4-slot tier (256-element
    chunks), three loads at mixed offsets."""
    n = 100_003
    spec, bufs = case("stencil", n, {"x": "f32", "y": "f32", "w": "f32"}, {"out": ("z", "f32")}, STENCIL,
                      (("s", "f32", 0.5),), seed=7)
    c, _ = T.command_from_spec(spec)
    assert c.lower()[0]["tier"] == 1
    _check(spec, bufs, dict(zip(("x", "y", "w", "out"), offs)))


def test_mixed_widths_and_two_stores():
    """A bf16 and an f32 load at different offsets, an f16 and an f32 store
    at the same offset."""
    n = 70_001
    spec, bufs = case("mixed", n, {"x": "bf16", "y": "f32"}, {"o1": ("z", "f16"), "o2": ("d", "f32")},
                      [("mul", "d", "x", "y"), ("add", "z", "d", "x")], seed=3)
    _check(spec, bufs, {"x": 3, "y": 1, "o1": 2, "o2": 2})


@pytest.mark.parametrize("offs", [(1, 0, 0), (2, 3, 1)])
def test_extended_ops_shifted(offs):
    """Division, a comparison and a select (the extended variant), shifted."""
    n = 50_017
    spec, bufs = case("divsel", n, {"x": "f32", "y": "f32"}, {"out": ("r", "f32")},
                      [("div", "q", "x", "y"), ("gt", "g", "q", "x"), ("select", "r", "q", "y", "g")], seed=5)
    c, _ = T.command_from_spec(spec)
    assert c.lower()[0]["extended"] == 1
    _check(spec, bufs, dict(zip(("x", "y", "out"), offs)))


def test_finite_difference_of_one_tensor():
    """out = x[1:] - x[:-1] on one torch buffer: the two loads are views of
    the same memory one element apart."""
    n = (1 << 18) + 1
    g = torch.Generator().manual_seed(11)
    xh = torch.randn(n, generator=g)
    spec = dict(name="diff", seed=0, sizes=(n - 1,),
                ops=[("load", "a", "f32"), ("load", "b", "f32"), ("exec", [("sub", "d", "a", "b")]),
                     ("store", "out", "d", "f32")],
                views={"a": dict(strides=(1,), alloc=n - 1), "b": dict(strides=(1,), alloc=n - 1),
                       "out": dict(strides=(1,), alloc=n - 1)}, inputs={})
    bufs = {"a": xh.numpy()[1:].copy(), "b": xh.numpy()[:-1].copy(), "out": specutil.sentinel_array("f32", n - 1)}
    want = gpuutil.oracle_every_element(spec, bufs)
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    x = xh.cuda()
    out = torch.empty(n - 1, device="cuda")
    views = {tags["a"]: x[1:], tags["b"]: x[:-1], tags["out"]: out}
    assert k.plan(views)["path"] == "contig"
    k.launch(views)
    k.sync()
    torch.cuda.synchronize()
    gpuutil.compare(out.cpu().numpy(), want["out"], "f32", "x[1:] - x[:-1]")


@pytest.mark.parametrize("offs", [{"a": 1, "c": 2}, {"b": 3, "out0": 2, "out1": 2}, {"f": 1, "e": 2, "d": 3}])
def test_wide_dag_in_the_8_slot_tier(offs):
    """The 16-op DAG (8-slot tier, its shifted kernel at two CTAs per SM),
    fp32 and fp16 stores at one offset, loads at others."""
    spec = W.wide_dag(60_013)
    bufs = specutil.host_buffers(spec)
    c, _ = T.command_from_spec(spec)
    assert c.lower()[0]["tier"] == 2
    _check(spec, bufs, offs)


def test_extended_ops_in_the_8_slot_tier():
    """The DAG with a division appended: the extended 8-slot tier is built
    with the dense-range kernel only, so such views run per element."""
    spec = W.wide_dag(40_009)
    ops = list(spec["ops"])
    i = next(k for k, o in enumerate(ops) if o[0] == "exec")
    ops[i] = ("exec", list(ops[i][1]) + [("div", "t17", "t16", "t4")])
    ops = [("store", "out0", "t17", "f32") if (o[0] == "store" and o[1] == "out0") else o for o in ops]
    spec = dict(spec, ops=ops, name="wide_dag_div")
    bufs = specutil.host_buffers(spec)
    c, _ = T.command_from_spec(spec)
    info = c.lower()[0]
    assert info["tier"] == 2 and info["extended"] == 1, info
    _check(spec, bufs, {"a": 2, "e": 1}, want_path="generic")


@pytest.mark.parametrize("offs", [{"x0": 1}, {"x0": 1, "x5": 2, "x8": 3, "out": 1}])
def test_sixteen_slot_tier_shifted(offs):
    """Nine loads live at once (the 16-slot tier), shifted loads."""
    spec = W.wide32_f32((1 << 16) + 7)
    bufs = specutil.host_buffers(spec)
    c, _ = T.command_from_spec(spec)
    assert c.lower()[0]["tier"] == 4
    _check(spec, bufs, offs)


@pytest.mark.parametrize("seed", range(80))
def test_random_layouts(seed):
    spec, bufs, offsets = layouts.random_layout_case(seed)
    gpuutil.parity(spec, bufs, offsets)
