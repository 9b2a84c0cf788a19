"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

Counter-based SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): element ``i`` of
stream ``(seed, stream)`` depends on nothing else, so the bytes are the same
however the range is split over threads. This package holds none of the
Command method's arithmetic: it draws numbers and describes workloads.

The C source builds into ``_build/libinputgen.so`` on first use (gcc).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "inputgen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libinputgen.so")
_lib = None
_lock = threading.Lock()

# distribution kinds, as numbered in inputgen.c
KINDS = {"u32": 0, "uniform_f32": 1, "normal_f32": 2, "uniform_bf16_trunc": 3}
KIND_DTYPE = {
    "u32": np.uint32,
    "uniform_f32": np.float32,
    "normal_f32": np.float32,
    "uniform_bf16_trunc": np.uint16,
}


def build(force: bool = False) -> str:
    """Compile the generator into a shared library; return its path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
         "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"],
        check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.ig_fill.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                    ctypes.c_double, ctypes.c_double, ctypes.c_void_p,
                                    ctypes.c_int64, ctypes.c_int]
            lib.ig_fill.restype = ctypes.c_int
            lib.ig_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.ig_stream_key.restype = ctypes.c_uint64
            lib.ig_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.ig_bits.restype = ctypes.c_uint64
            _lib = lib
        return _lib


def default_threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def fill_ptr(kind: str, seed: int, stream: int, ptr: int, n: int,
             lo: float = 0.0, hi: float = 0.0, threads: int | None = None) -> None:
    """Fill ``n`` elements at host address ``ptr`` (element type per kind)."""
    rc = _get().ig_fill(KINDS[kind], seed & (2**64 - 1), stream & (2**64 - 1),
                        float(lo), float(hi), ctypes.c_void_p(ptr), int(n),
                        threads or default_threads())
    if rc != 0:
        raise ValueError(f"ig_fill rejected kind={kind} n={n}")


def generate(kind: str, seed: int, stream: int, n: int, lo: float = 0.0,
             hi: float = 0.0, threads: int | None = None) -> np.ndarray:
    """Return a new numpy array of ``n`` elements of the given stream."""
    out = np.empty(int(n), dtype=KIND_DTYPE[kind])
    if n:
        fill_ptr(kind, seed, stream, out.ctypes.data, n, lo, hi, threads)
    return out


def stream_bits(seed: int, stream: int, index: int) -> int:
    """The raw 64-bit draw for one element (for tests of the generator)."""
    lib = _get()
    return int(lib.ig_bits(lib.ig_stream_key(seed, stream), index))
