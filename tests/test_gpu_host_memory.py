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
