"""The allocation-free compile entry point, cmd_compile_static_scratch.

It serves callers that cannot call cudaMalloc: programs whose device memory
all belongs to their own pool or to a framework's allocator. Its kernels keep
their one device error word in a static array of the library instead of an
allocation. Like cmd_compile it is called outside any stream capture.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import pytest
import torch

import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import gpuutil
import specutil

pytestmark = pytest.mark.gpu


def _views(spec, tags, dev):
    return {tags[n]: T.TensorView(t.data_ptr(), spec["sizes"], spec["views"][n]["strides"]) for n, t in dev.items()}


def _run(kernel, spec, tags, bufs):
    """One launch of kernel on fresh device copies of bufs; the store buffers
    come back to the host whole (sentinels outside the views)."""
    dts = W.tensor_dtypes(spec)
    dev = {n: gpuutil.to_device(bufs[n], dts[n]) for n in W.load_names(spec) + W.store_names(spec)}
    views = _views(spec, tags, dev)
    scal = T.spec_scalars(spec, tags)
    plan = kernel.plan(views, scal)
    kernel.launch(views, scal)
    kernel.sync()
    torch.cuda.synchronize()
    return {n: dev[n].cpu().numpy().view(specutil.NP[dts[n]]) for n in W.store_names(spec)}, plan


@pytest.mark.parametrize("spec,path", [
    (W.strided_bf16(320, 264, 272), "tile2d"),   # the executor that uses the error word
    (W.chain_f32((1 << 16) + 5), "contig"),
    (W.wide_dag(4099), "contig"),
], ids=lambda x: x["name"] if isinstance(x, dict) else x)
def test_static_scratch_kernel_matches_the_oracle_and_the_regular_kernel(spec, path):
    """Two calls in a row of a kernel from the allocation-free entry point:
    every element equals the oracle and the kernel from cmd_compile (the
    tolerance of every parity test: bit-exact, <= 1 ulp for 16-bit floats)."""
    bufs = specutil.host_buffers(spec)
    dts = W.tensor_dtypes(spec)
    want = gpuutil.oracle_every_element(spec, bufs)
    c, tags = T.command_from_spec(spec)
    regular = c.compile()
    static = T.Kernel(T.cmd_compile_static_scratch(c.handle), dict(c.scalar_dtypes))
    for call in range(2):
        got_r, plan_r = _run(regular, spec, tags, bufs)
        got_s, plan_s = _run(static, spec, tags, bufs)
        assert plan_r["path"] == plan_s["path"] == path
        for n in W.store_names(spec):
            gpuutil.compare(got_s[n], want[n], dts[n], f"static-scratch call {call} vs the oracle: {n}")
            gpuutil.compare(got_s[n], got_r[n], dts[n], f"static-scratch call {call} vs cmd_compile: {n}")


def test_static_scratch_allocates_no_device_memory():
    """The library's own count of its device allocations does not move
    across compile, launch, sync and destroy of a kernel from the
    allocation-free entry point, and moves by one for cmd_compile."""
    spec = W.strided_bf16(128, 128, 136)
    bufs = specutil.host_buffers(spec)
    dts = W.tensor_dtypes(spec)
    c, tags = T.command_from_spec(spec)
    dev = {n: gpuutil.to_device(bufs[n], dts[n]) for n in W.load_names(spec) + W.store_names(spec)}
    views = _views(spec, tags, dev)
    scal = T.spec_scalars(spec, tags)
    torch.cuda.synchronize()
    before = T.cmd_device_allocations()
    static = T.Kernel(T.cmd_compile_static_scratch(c.handle), dict(c.scalar_dtypes))
    for _ in range(3):
        static.launch(views, scal)
    static.sync()
    torch.cuda.synchronize()
    T.cmd_kernel_destroy(static.handle)
    static.handle = None
    assert T.cmd_device_allocations() == before
    regular = c.compile()
    assert T.cmd_device_allocations() == before + 1
    del regular


def test_static_scratch_word_reports_a_timeout():
    """The static word is where the tile executor's status goes: a forced
    wait timeout is reported by cmd_sync_status and cleared, and the kernel
    then runs normally."""
    spec = W.strided_bf16(128, 128, 136)
    bufs = specutil.host_buffers(spec)
    dts = W.tensor_dtypes(spec)
    c, tags = T.command_from_spec(spec)
    static = T.Kernel(T.cmd_compile_static_scratch(c.handle), dict(c.scalar_dtypes))
    dev = {n: gpuutil.to_device(bufs[n], dts[n]) for n in W.load_names(spec) + W.store_names(spec)}
    views = _views(spec, tags, dev)
    scal = T.spec_scalars(spec, tags)
    T.cmd_configure_waits(1_000_000, True)
    try:
        static.launch(views, scal)
        with pytest.raises(T.CmdError) as e:
            static.sync()
        assert e.value.name == "CMD_ERR_DEVICE_TIMEOUT"
    finally:
        T.cmd_configure_waits(2_000_000_000, False)
    static.sync()
    want = gpuutil.oracle_every_element(spec, bufs)
    got, _ = _run(static, spec, tags, bufs)
    for n in W.store_names(spec):
        gpuutil.compare(got[n], want[n], dts[n], n)
