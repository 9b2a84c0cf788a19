"""Launches captured into CUDA graphs and replayed, every element against the
oracle.

cmd_launch only enqueues kernels on the caller's stream and makes no call that
waits on the device, so a launch can be captured (global capture mode, the
strictest): each executor (contiguous with its generic head and tail, TMA
tile, generic) in a graph; one graph of two dependent Commands, the second
reading what the first wrote; a graph replayed after new values were written
into its captured input buffers; and, in a fresh process, capture of each
executor's very first launch, whose one-time setup (kernel attributes, grid
size, the tensor-map entry point) then runs inside the capture."""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import gpuutil
import specutil

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _setup(spec, bufs, offsets=None):
    """Device copies of bufs, the compiled kernel, its views and scalars."""
    dts = W.tensor_dtypes(spec)
    dev = {n: gpuutil.to_device(bufs[n], dts[n], offset_elems=(offsets or {}).get(n, 0))
           for n in W.load_names(spec) + W.store_names(spec)}
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    views = {tags[n]: T.TensorView(t.data_ptr(), spec["sizes"], spec["views"][n]["strides"]) for n, t in dev.items()}
    return dev, k, views, T.spec_scalars(spec, tags)


def _check(spec, dev, want, what):
    dts = W.tensor_dtypes(spec)
    for n in W.store_names(spec):
        got = dev[n].cpu().numpy().view(specutil.NP[dts[n]])
        gpuutil.compare(got, want[n], dts[n], f"{spec['name']} {what}: {n}")


CASES = [
    (W.chain_f32((1 << 16) + 5), None, "contig"),               # contiguous + ragged tail
    (W.chain_f32((1 << 16) + 5), {"a": 1, "b": 1, "c": 1, "out": 1}, "contig"),  # + head
    (W.threshold_bits(5000), None, "contig"),
    (W.strided_bf16(128, 72, 80), None, "tile2d"),
    (W.batched_transpose(3, 64, 96), None, "tile2d"),
    (W.strided_bf16(100, 70, 75), None, "generic"),
]


@pytest.mark.parametrize("spec,offsets,planned", CASES,
                         ids=["chain_f32-tail", "chain_f32-head-tail", "threshold_bits", "strided_bf16-tile",
                              "batched_transpose", "strided_bf16-generic"])
def test_executor_launch_in_a_graph(spec, offsets, planned):
    bufs = specutil.host_buffers(spec)
    want = gpuutil.oracle_every_element(spec, bufs)
    dev, k, views, scal = _setup(spec, bufs, offsets)
    assert k.plan(views, scal)["path"] == planned
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="global"):
        k.launch(views, scal, stream=s)
    torch.cuda.synchronize()
    # capture records the launch without running it: the outputs still hold
    # their sentinels
    dts = W.tensor_dtypes(spec)
    for n in W.store_names(spec):
        got = dev[n].cpu().numpy().view(specutil.NP[dts[n]])
        assert np.array_equal(specutil.bits(got), specutil.bits(bufs[n])), f"{n} written during capture"
    for replay in range(2):
        g.replay()
        torch.cuda.synchronize()
        k.sync()
        _check(spec, dev, want, f"replay {replay}")


def test_dependent_commands_in_one_graph():
    """First = the chain Command into `out`; second = out + a (the two-input
    add reading the first's output). Both in one graph, in that order."""
    n = (1 << 17) + 3
    s1 = W.chain_f32(n)
    s2 = W.add_f32(n)
    b1 = specutil.host_buffers(s1)
    w1 = gpuutil.oracle_every_element(s1, b1)
    b2 = specutil.host_buffers(s2)
    b2 = {"x": w1["out"], "y": b1["a"], "out": b2["out"]}
    w2 = gpuutil.oracle_every_element(s2, b2)
    dev1, k1, v1, sc1 = _setup(s1, b1)
    out2 = gpuutil.to_device(b2["out"], "f32")
    c2, tags2 = T.command_from_spec(s2)
    k2 = c2.compile()
    v2 = {tags2["x"]: T.TensorView(dev1["out"].data_ptr(), (n,), (1,)),
          tags2["y"]: T.TensorView(dev1["a"].data_ptr(), (n,), (1,)),
          tags2["out"]: T.TensorView(out2.data_ptr(), (n,), (1,))}
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="global"):
        k1.launch(v1, sc1, stream=s)
        k2.launch(v2, {}, stream=s)
    g.replay()
    torch.cuda.synchronize()
    k1.sync()
    k2.sync()
    _check(s1, dev1, w1, "first in graph")
    gpuutil.compare(out2.cpu().numpy(), w2["out"], "f32", "second in graph (reads the first's output)")


def test_replay_after_new_input_values():
    """The graph holds pointers, not values: new inputs written into the
    captured buffers between replays give the new results."""
    spec = W.wrap_i32((1 << 16) + 9)
    bufs = specutil.host_buffers(spec)
    dev, k, views, scal = _setup(spec, bufs)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="global"):
        k.launch(views, scal, stream=s)
    for seed in (spec["seed"], 1234, 77):
        new = specutil.host_buffers(dict(spec, seed=seed))
        for n in W.load_names(spec):
            dev[n].copy_(torch.from_numpy(new[n].view(np.int32)))
        want = gpuutil.oracle_every_element(spec, new)
        g.replay()
        torch.cuda.synchronize()
        k.sync()
        _check(spec, dev, want, f"inputs of seed {seed}")


def first_launches_in_capture():
    """Run in a fresh process: the first launch of each executor object this
    process makes is captured (global mode) and replayed."""
    for spec, planned in ((W.chain_f32((1 << 15) + 7), "contig"),
                          (W.strided_bf16(128, 72, 80), "tile2d"),
                          (W.strided_bf16(100, 70, 75), "generic")):
        bufs = specutil.host_buffers(spec)
        want = gpuutil.oracle_every_element(spec, bufs)
        dev, k, views, scal = _setup(spec, bufs)
        assert k.plan(views, scal)["path"] == planned
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s, capture_error_mode="global"):
            k.launch(views, scal, stream=s)
        g.replay()
        torch.cuda.synchronize()
        k.sync()
        _check(spec, dev, want, "first launch, captured")
    print("first-launch capture ok")


def test_first_launch_of_each_executor_captured_in_a_fresh_process():
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([ROOT, HERE, os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, "-c", "import test_gpu_graph as t; t.first_launches_in_capture()"],
                       cwd=HERE, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "first-launch capture ok" in r.stdout
