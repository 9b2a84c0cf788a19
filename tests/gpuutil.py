"""Helpers for GPU parity tests: run a spec through the CUDA path (via the
C ABI binding) and through the oracle on the same host bytes, and compare."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import specutil

TORCH_OF = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.int16, "i32": torch.int32,
            "b1": torch.int32}
NP_OF = {"f32": np.float32, "f16": np.float16, "bf16": np.int16, "i32": np.int32, "b1": np.int32}


def to_device(arr: np.ndarray, dt: str, dev="cuda:0", offset_elems: int = 0) -> torch.Tensor:
    """Copy a flat host buffer to the device. With offset_elems > 0 the data
    starts that many elements into a larger allocation (a misaligned base)."""
    host = torch.from_numpy(np.ascontiguousarray(arr).view(NP_OF[dt]))
    if offset_elems == 0:
        return host.to(dev)
    big = torch.empty(host.numel() + offset_elems, dtype=host.dtype, device=dev)
    big[offset_elems:].copy_(host)
    return big[offset_elems:]


def run_cuda(spec: dict, bufs: dict, offsets=None, stream=None, kernel=None):
    """Launch spec on the GPU with the host buffers' bytes; return host copies
    of every store buffer (whole physical buffers) and the launch plan."""
    dts = W.tensor_dtypes(spec)
    c, tags = T.command_from_spec(spec)
    k = kernel or c.compile()
    dev = {}
    for name in W.load_names(spec) + W.store_names(spec):
        dev[name] = to_device(bufs[name], dts[name], offset_elems=(offsets or {}).get(name, 0))
    views = {tags[n]: T.TensorView(dev[n].data_ptr(), spec["sizes"], spec["views"][n]["strides"])
             for n in dev}
    scal = T.spec_scalars(spec, tags)
    plan = k.plan(views, scal)
    k.launch(views, scal, stream=stream)
    k.sync(stream)
    torch.cuda.synchronize()
    out = {n: dev[n].cpu().numpy().view(specutil.NP[dts[n]]) for n in W.store_names(spec)}
    return out, plan


def ulp_distance_half(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units in the last place between two arrays of 16-bit float
    encodings (sign-magnitude mapped to a monotone integer line)."""
    def line(x):
        x = x.view(np.uint16).astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(line(a) - line(b))


def compare(got: np.ndarray, want: np.ndarray, dt: str, what: str = ""):
    """Bit-exact for f32 and i32 (NaN payloads aside); within 1 ulp for the
    16-bit float types, and exactly equal there too since both sides round to
    nearest even once. Returns the number of elements compared."""
    ok = specutil.same_bits_nan_as_class(got, want, dt)
    if dt in ("f16", "bf16"):
        d = ulp_distance_half(got, want)
        nan_both = ok & (specutil.bits(got) != specutil.bits(want))
        d = np.where(nan_both, 0, d)
        assert d.max(initial=0) <= 1, f"{what}: {int((d > 1).sum())} elements differ by more than 1 ulp"
    bad = np.flatnonzero(~ok)
    assert bad.size == 0, (f"{what}: {bad.size} of {ok.size} elements differ; first at {bad[0]}: "
                           f"got {hex(int(specutil.bits(got)[bad[0]]))} want {hex(int(specutil.bits(want)[bad[0]]))}")
    return ok.size


def parity(spec: dict, bufs: dict | None = None, offsets=None):
    """Run spec on the GPU and on the oracle over every element; compare whole
    output buffers (so elements outside the views must keep the sentinel)."""
    bufs = bufs or specutil.host_buffers(spec)
    got, plan = run_cuda(spec, bufs, offsets)
    ref = {k: v.copy() for k, v in bufs.items()}
    oracle.OracleCommand(spec, ref).eval_range()
    dts = W.tensor_dtypes(spec)
    for name in W.store_names(spec):
        compare(got[name], ref[name], dts[name], f"{spec['name']}:{name}")
    return plan


def host_cores() -> int:
    """Cores this process may run on."""
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return os.cpu_count() or 1


def element_ranges(n: int, parts: int, align: int = 32) -> list:
    """[0, n) cut into at most `parts` contiguous ranges whose inner
    boundaries are multiples of `align` logical elements (so no two ranges
    write the same 32-element packed-bit word)."""
    step = -(-max(1, -(-n // max(1, parts))) // align) * align
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def oracle_every_element(spec: dict, bufs: dict) -> dict:
    """The oracle over every logical index of spec: fresh copies of the store
    buffers (their sentinels kept outside the views) written by element
    ranges split over the host cores. The C walk runs without the
    interpreter lock, and each range is the plain per-element walk."""
    ref = {n: bufs[n].copy() for n in W.store_names(spec)}
    oc = oracle.OracleCommand(spec, {**bufs, **ref})
    cores = host_cores()
    ranges = element_ranges(W.numel(spec), 4 * cores)
    with ThreadPoolExecutor(cores) as ex:
        list(ex.map(lambda r: oc.eval_range(*r), ranges))
    return ref


def full_parity(spec: dict) -> tuple:
    """Run spec on the GPU at its own size and compare every element of every
    store buffer with the oracle (bit-exact; <= 1 ulp for 16-bit floats, and
    they are in fact exact). Returns (plan, elements compared, max ulp)."""
    bufs = specutil.host_buffers(spec)
    got, plan = run_cuda(spec, bufs, offsets=spec.get("offsets"))
    ref = oracle_every_element(spec, bufs)
    dts = W.tensor_dtypes(spec)
    checked, max_ulp = 0, 0
    for name in W.store_names(spec):
        checked += compare(got[name], ref[name], dts[name], f"{spec['name']}:{name} (every element)")
        if dts[name] in ("f16", "bf16"):
            max_ulp = max(max_ulp, int(ulp_distance_half(got[name], ref[name]).max(initial=0)))
        del got[name], ref[name]
    return plan, checked, max_ulp


def sampled_parity(spec: dict, n_samples: int = 1 << 20, seed: int = 0):
    """Full-size run on the GPU; the oracle computes a sample of logical
    indices (random ones plus the first and last 4096) one by one."""
    bufs = specutil.host_buffers(spec)
    got, plan = run_cuda(spec, bufs)
    n = W.numel(spec)
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([np.arange(min(n, 4096)), np.arange(max(0, n - 4096), n),
                                    rng.integers(0, n, size=min(n, n_samples))]))
    want = oracle.OracleCommand(spec, bufs).eval_points(idx)
    dts = W.tensor_dtypes(spec)
    for name in W.store_names(spec):
        st = spec["views"][name]["strides"]
        sizes = spec["sizes"]
        multi = np.unravel_index(idx, sizes)
        off = sum(m.astype(np.int64) * s for m, s in zip(multi, st))
        if dts[name] == "b1":  # bit `off` of the packed words
            g = ((got[name].view(np.uint32)[off // 32] >> (off % 32).astype(np.uint32)) & 1).astype(np.uint8)
            assert (g == want[name]).all(), f"{spec['name']}:{name} (sampled): {(g != want[name]).sum()} bits differ"
            continue
        compare(got[name][off], want[name], dts[name], f"{spec['name']}:{name} (sampled)")
    return plan, idx.size
