"""Test helpers: host buffers for workload specs and golden hand cases.

Only data handling lives here (allocation, seeded filling, reading fixtures);
no Command arithmetic."""
from __future__ import annotations

import json
import os

import numpy as np

import inputgen
from inputgen import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NP = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "i32": np.int32, "b1": np.uint32}
SENTINEL_BITS = {"f32": 0x7FA5A5A5, "f16": 0x7DA5, "bf16": 0x7FA5, "i32": 0x5A5A5A5A, "b1": 0xA5A5A5A5}


def sentinel_array(dt: str, n: int) -> np.ndarray:
    """An array of n elements of type dt filled with a recognisable pattern."""
    if dt in ("f32", "i32", "b1"):
        return np.full(n, SENTINEL_BITS[dt], dtype=np.uint32).view(NP[dt])
    return np.full(n, SENTINEL_BITS[dt], dtype=np.uint16).view(NP[dt])


def host_buffers(spec: dict, threads: int | None = None) -> dict:
    """Seeded host buffers for every load (inputgen recipe; stream k for the
    k-th load) and sentinel-filled buffers for every store."""
    dts = workloads.tensor_dtypes(spec)
    bufs = {}
    for k, name in enumerate(workloads.load_names(spec)):
        kind, lo, hi = spec["inputs"][name]
        n = spec["views"][name]["alloc"]
        arr = inputgen.generate(kind, spec["seed"], k, n, lo, hi, threads)
        bufs[name] = arr.view(NP[dts[name]])
    for name in workloads.store_names(spec):
        bufs[name] = sentinel_array(dts[name], spec["views"][name]["alloc"])
    return bufs


def bits(arr: np.ndarray) -> np.ndarray:
    return arr.view({4: np.uint32, 2: np.uint16, 1: np.uint8}[arr.dtype.itemsize])


def same_bits_nan_as_class(got: np.ndarray, want: np.ndarray, dt: str) -> np.ndarray:
    """Elementwise bit equality, except that any NaN matches any NaN (payloads
    are not pinned)."""
    gb, wb = bits(got), bits(want)
    eq = gb == wb
    if dt in ("f32", "f16", "bf16"):
        if dt == "f32":
            gn = (gb & 0x7FFFFFFF) > 0x7F800000
            wn = (wb & 0x7FFFFFFF) > 0x7F800000
        elif dt == "f16":
            gn = (gb & 0x7FFF) > 0x7C00
            wn = (wb & 0x7FFF) > 0x7C00
        else:
            gn = (gb & 0x7FFF) > 0x7F80
            wn = (wb & 0x7FFF) > 0x7F80
        eq = eq | (gn & wn)
    return eq


def _float_list(values, dt):
    out = []
    for v in values:
        out.append(float.fromhex(v) if isinstance(v, str) else float(v))
    return np.array(out, dtype=NP[dt])


def golden_cases() -> dict:
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        data = json.load(f)
    return {k: v for k, v in data.items() if not k.startswith("_")}


def golden_spec(case: dict):
    """(spec, host buffers, expected-by-store) for one hand case."""
    ops = case["ops"]
    if ops == "wide_dag":
        ops = workloads.wide_dag(1)["ops"]
    ops = [tuple(o) if o[0] != "exec" else ("exec", [tuple(e[:3]) + ((e[3] if len(e) > 3 else None),)
                                                     for e in o[1]]) for o in ops]
    sizes = tuple(case["sizes"])
    n = int(np.prod(sizes))
    spec = dict(name="golden", seed=0, sizes=sizes, ops=ops, views={}, inputs={})
    dense = workloads._dense(sizes)
    dts = workloads.tensor_dtypes(spec)
    for name in list(workloads.load_names(spec)) + list(workloads.store_names(spec)):
        v = case.get("views", {}).get(name)
        spec["views"][name] = (dict(strides=tuple(v["strides"]), alloc=v["alloc"]) if v
                               else dict(strides=dense[0], alloc=n))
    bufs = {}
    for name in workloads.load_names(spec):
        dt = dts[name]
        if "input_bits" in case and name in case["input_bits"]:
            raw = np.array(case["input_bits"][name], dtype=np.uint16 if dt in ("f16", "bf16") else np.uint32)
            bufs[name] = raw.view(NP[dt])
        elif dt == "i32":
            bufs[name] = np.array(case["inputs"][name], dtype=np.int64).astype(np.int32)
        else:
            bufs[name] = _float_list(case["inputs"][name], dt)
    expect = {}
    for name in workloads.store_names(spec):
        dt = dts[name]
        bufs[name] = sentinel_array(dt, spec["views"][name]["alloc"])
        if "expect_bits" in case:
            raw = np.array(case["expect_bits"][name], dtype=np.uint16 if dt in ("f16", "bf16") else np.uint32)
            expect[name] = raw.view(NP[dt])
        elif dt == "i32":
            expect[name] = np.array(case["expect"][name], dtype=np.int64).astype(np.int32)
        else:
            expect[name] = _float_list(case["expect"][name], dt)
    return spec, bufs, expect
