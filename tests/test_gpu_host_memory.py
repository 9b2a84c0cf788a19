"""Launches whose tensors lie in pinned host memory: the kernel reads and
writes them across the host link (their addresses are valid on the device
under unified addressing), every element against the oracle. Views that
would take the tile executor run on the generic one (its TMA copies are
issued on device memory only). Only page-locked buffers are used: pageable
host memory is outside the library's contract."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import gpuutil
import specutil

pytestmark = pytest.mark.gpu


def _pinned(arr: np.ndarray, dt: str) -> torch.Tensor:
    """A page-locked copy of arr whose first element is 64-byte aligned (as
    device allocations are, so that the planner sees the same alignment)."""
    src = torch.from_numpy(np.ascontiguousarray(arr).view(gpuutil.NP_OF[dt]))
    nbytes = src.numel() * src.element_size()
    raw = torch.empty(nbytes + 64, dtype=torch.uint8, pin_memory=True)
    off = (-raw.data_ptr()) % 64
    out = raw[off:off + nbytes].view(src.dtype)
    out.copy_(src)
    return out


@pytest.mark.parametrize("spec,planned", [
    (W.wrap_i32((1 << 16) + 5), "contig"),
    (W.chain_bf16((1 << 14) + 3), "contig"),
    (W.wide_dag(4099), "contig"),
    (W.threshold_bits(5000), "contig"),
    (W.strided_bf16(128, 72, 80), "tile2d"),
    (W.strided_bf16(100, 70, 75), "generic"),
], ids=lambda x: x["name"] + str(x["sizes"]) if isinstance(x, dict) else x)
def test_launch_on_pinned_host_buffers(spec, planned):
    bufs = specutil.host_buffers(spec)
    dts = W.tensor_dtypes(spec)
    want = gpuutil.oracle_every_element(spec, bufs)
    host = {n: _pinned(bufs[n], dts[n]) for n in W.load_names(spec) + W.store_names(spec)}
    assert all(t.is_pinned() for t in host.values())
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    views = {tags[n]: T.TensorView(t.data_ptr(), spec["sizes"], spec["views"][n]["strides"]) for n, t in host.items()}
    scal = T.spec_scalars(spec, tags)
    assert k.plan(views, scal)["path"] == planned
    for call in range(2):
        k.launch(views, scal)
        k.sync()
        torch.cuda.synchronize()
        for n in W.store_names(spec):
            got = host[n].numpy().view(specutil.NP[dts[n]])
            gpuutil.compare(got, want[n], dts[n], f"pinned host, call {call}: {n}")


def test_padded_rows_on_pinned_host_buffers():
    """Padded rows (the contiguous executor's row walk) over pinned host
    memory."""
    import layouts
    spec, bufs = layouts.padded_spec("rows_host", 37, 1024, {"x": ("f32", 1032), "y": ("bf16", 1088)},
                               {"out": ("z", "f32", 1028)}, [("add", "z", "x", "y")], seed=4)
    want = gpuutil.oracle_every_element(spec, bufs)
    dts = W.tensor_dtypes(spec)
    host = {n: _pinned(bufs[n], dts[n]) for n in bufs}
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    views = {tags[n]: T.TensorView(t.data_ptr(), spec["sizes"], spec["views"][n]["strides"]) for n, t in host.items()}
    plan = k.plan(views)
    assert plan["path"] == "contig" and plan["merged_rank"] == 2
    k.launch(views)
    k.sync()
    torch.cuda.synchronize()
    gpuutil.compare(host["out"].numpy().view(specutil.NP["f32"]), want["out"], "f32", "padded rows, pinned host")


def test_shifted_loads_on_pinned_host_buffers():
    """x one element and y three elements past a 16-byte boundary, out on
    it (shifted loads) over pinned host memory."""
    n = 50_021
    rng = np.random.default_rng(9)
    x = rng.standard_normal(n).astype(np.float32)
    y = rng.standard_normal(n).astype(np.float32)
    spec = dict(name="shift_host", seed=0, sizes=(n,),
                ops=[("load", "x", "f32"), ("load", "y", "f32"), ("exec", [("mul", "z", "x", "y")]),
                     ("store", "out", "z", "f32")],
                views={k: dict(strides=(1,), alloc=n) for k in ("x", "y", "out")}, inputs={})
    bufs = {"x": x, "y": y, "out": specutil.sentinel_array("f32", n)}
    want = gpuutil.oracle_every_element(spec, bufs)
    hx = _pinned(np.concatenate([np.zeros(1, np.float32), x]), "f32")[1:]
    hy = _pinned(np.concatenate([np.zeros(3, np.float32), y]), "f32")[3:]
    ho = _pinned(bufs["out"], "f32")
    c, tags = T.command_from_spec(spec)
    k = c.compile()
    views = {tags["x"]: hx, tags["y"]: hy, tags["out"]: ho}
    assert k.plan(views)["path"] == "contig"
    for call in range(2):
        k.launch(views)
        k.sync()
        torch.cuda.synchronize()
        gpuutil.compare(ho.numpy(), want["out"], "f32", f"shifted loads, pinned host, call {call}")
