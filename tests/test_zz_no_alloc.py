"""The allocation-free compile entry point, cmd_compile_static_scratch.

It serves callers that cannot call cudaMalloc (code running under CUDA graph
capture in global mode, or programs whose device memory all belongs to their
own pool): its kernels keep their one device error word in a static array of
the library instead of an allocation. This file is collected last so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import gpuutil
import specutil

pytestmark = pytest.mark.gpu


def _launch(kernel, spec, tags, dev):
    views = {tags[n]: T.TensorView(t.data_ptr(), spec["sizes"], spec["views"][n]["strides"]) for n, t in dev.items()}
    scal = T.spec_scalars(spec, tags)
    kernel.launch(views, scal)
    kernel.sync()
    torch.cuda.synchronize()
    return kernel.plan(views, scal)


def test_static_scratch_kernel_matches_the_regular_kernel():
    spec = W.strided_bf16(320, 264, 272)  # the tile executor: the kernel with a device error word
    bufs = specutil.host_buffers(spec)
    dts = W.tensor_dtypes(spec)
    c, tags = T.command_from_spec(spec)
    regular = c.compile()
    static = T.Kernel(T.cmd_compile_static_scratch(c.handle), dict(c.scalar_dtypes))
    names = W.load_names(spec) + W.store_names(spec)
    for call in range(2):
        dev_r = {n: gpuutil.to_device(bufs[n], dts[n]) for n in names}
        dev_s = {n: gpuutil.to_device(bufs[n], dts[n]) for n in names}
        assert _launch(regular, spec, tags, dev_r)["path"] == "tile2d"
        assert _launch(static, spec, tags, dev_s)["path"] == "tile2d"
        for n in W.store_names(spec):
            got = dev_s[n].cpu().numpy().view(specutil.NP[dts[n]])
            want = dev_r[n].cpu().numpy().view(specutil.NP[dts[n]])
            gpuutil.compare(got, want, dts[n], f"static-scratch call {call}: {n}")


def test_static_scratch_word_reports_a_timeout():
    """The static word is where the tile executor's status goes: a forced
    wait timeout is reported by cmd_sync_status and cleared, and the kernel
    then runs normally."""
    spec = W.strided_bf16(128, 128, 136)
    bufs = specutil.host_buffers(spec)
    dts = W.tensor_dtypes(spec)
    c, tags = T.command_from_spec(spec)
    static = T.Kernel(T.cmd_compile_static_scratch(c.handle), dict(c.scalar_dtypes))
    regular = c.compile()
    names = W.load_names(spec) + W.store_names(spec)
    dev = {n: gpuutil.to_device(bufs[n], dts[n]) for n in names}
    views = {tags[n]: T.TensorView(t.data_ptr(), spec["sizes"], spec["views"][n]["strides"]) for n, t in dev.items()}
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
    dev_r = {n: gpuutil.to_device(bufs[n], dts[n]) for n in names}
    _launch(regular, spec, tags, dev_r)
    _launch(static, spec, tags, dev)
    for n in W.store_names(spec):
        gpuutil.compare(dev[n].cpu().numpy().view(specutil.NP[dts[n]]),
                        dev_r[n].cpu().numpy().view(specutil.NP[dts[n]]), dts[n], n)
