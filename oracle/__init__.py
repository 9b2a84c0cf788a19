"""CPU oracle for fused Command execution (ctypes wrapper over cmd_oracle.c).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline and reference legs may import this package. The
product path (the CUDA executor and its binding) never does, and the two
share no code.

The oracle walks a Command element by element in tag order, with no
dead-tag elimination, no common-subexpression reuse and no reordering; see
``cmd_oracle.h`` for the pages it follows and the readings it takes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cmd_oracle.c")
_HDR = os.path.join(_HERE, "cmd_oracle.h")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

MAX_RANK = 4
DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3, "b1": 4}
# host buffers: b1 stores are u32 words (32 elements each); eval_points gives b1 as 0/1 bytes
NP_DTYPE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "i32": np.int32, "b1": np.uint32}
POINT_DTYPE = dict(NP_DTYPE, b1=np.uint8)
KINDS = {"load": 0, "scalar": 1, "add": 2, "sub": 3, "mul": 4, "neg": 5, "store": 6,
         "div": 7, "min": 8, "max": 9, "abs": 10, "to_f32": 11, "to_i32": 12,
         "lt": 13, "le": 14, "gt": 15, "ge": 16, "eq": 17, "ne": 18,
         "ult": 19, "ule": 20, "ugt": 21, "uge": 22, "select": 23}


class _Op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("a", ctypes.c_int32), ("b", ctypes.c_int32), ("c", ctypes.c_int32),
                ("ptr", ctypes.c_void_p),
                ("strides", ctypes.c_int64 * MAX_RANK),
                ("scalar_bits", ctypes.c_uint32)]


class _Command(ctypes.Structure):
    _fields_ = [("n_ops", ctypes.c_int32), ("ops", ctypes.POINTER(_Op)),
                ("rank", ctypes.c_int32), ("sizes", ctypes.c_int64 * MAX_RANK)]


def build(force: bool = False) -> str:
    """Compile the oracle with contraction and fast-math off; return the path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
         "-fno-fast-math", "-fno-unsafe-math-optimizations", _SRC, "-o", tmp, "-lm"],
        check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.orc_eval_range.argtypes = [ctypes.POINTER(_Command), ctypes.c_int64, ctypes.c_int64]
            L.orc_eval_range.restype = ctypes.c_int
            L.orc_eval_points.argtypes = [ctypes.POINTER(_Command), ctypes.c_void_p,
                                          ctypes.c_int64, ctypes.c_void_p]
            L.orc_eval_points.restype = ctypes.c_int
            for name in ("orc_fadd", "orc_fsub", "orc_fmul", "orc_iadd", "orc_isub", "orc_imul",
                         "orc_fdiv", "orc_idiv", "orc_fmin", "orc_fmax", "orc_imin", "orc_imax"):
                f = getattr(L, name)
                f.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
                f.restype = ctypes.c_uint32
            L.orc_compare.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint32]
            L.orc_compare.restype = ctypes.c_uint32
            for name in ("orc_fneg", "orc_ineg", "orc_fabs", "orc_iabs", "orc_i2f", "orc_f2i"):
                f = getattr(L, name)
                f.argtypes = [ctypes.c_uint32]
                f.restype = ctypes.c_uint32
            for name in ("orc_f32_to_f16", "orc_f32_to_bf16"):
                f = getattr(L, name)
                f.argtypes = [ctypes.c_uint32]
                f.restype = ctypes.c_uint16
            for name in ("orc_f16_to_f32", "orc_bf16_to_f32"):
                f = getattr(L, name)
                f.argtypes = [ctypes.c_uint16]
                f.restype = ctypes.c_uint32
            for name in ("orc_f32_to_f16_n", "orc_f32_to_bf16_n"):
                f = getattr(L, name)
                f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
                f.restype = None
            _lib = L
        return _lib


def _scalar_bits(dtype: str, value) -> int:
    if dtype == "f32":
        return int(np.array([value], dtype=np.float32).view(np.uint32)[0])
    if dtype == "i32":
        return int(np.array([value], dtype=np.int64).astype(np.uint32)[0]) & 0xFFFFFFFF
    raise ValueError(f"scalar dtype {dtype!r}")


class OracleCommand:
    """A spec (see ``inputgen.workloads``) bound to host numpy buffers.

    ``buffers`` maps every load and store name to a flat numpy array holding
    the tensor's physical elements (bf16 as uint16 bits)."""

    def __init__(self, spec: dict, buffers: dict):
        self.spec = spec
        self.buffers = buffers
        tags: dict = {}
        ops = []
        self.store_order = []
        for op in spec["ops"]:
            kind = op[0]
            if kind == "load":
                _, name, dt = op
                o = _Op(kind=KINDS["load"], dtype=DTYPES[dt], a=-1, b=-1, c=-1)
                buf = buffers[name]
                o.ptr = buf.ctypes.data if buf.size else None
                for k, s in enumerate(spec["views"][name]["strides"]):
                    o.strides[k] = s
                tags[name] = len(ops)
                ops.append(o)
            elif kind == "scalar":
                _, name, dt, value = op
                o = _Op(kind=KINDS["scalar"], dtype=DTYPES[dt], a=-1, b=-1, c=-1,
                        scalar_bits=_scalar_bits(dt, value))
                tags[name] = len(ops)
                ops.append(o)
            elif kind == "exec":
                for e in op[1]:
                    # (eop, name, a, b) or, for select, (eop, name, a, b, cond)
                    eop, name, a, b = e[:4]
                    cond = e[4] if len(e) > 4 else None
                    o = _Op(kind=KINDS[eop], dtype=0, a=tags[a],
                            b=tags[b] if b is not None else -1,
                            c=tags[cond] if cond is not None else -1)
                    tags[name] = len(ops)
                    ops.append(o)
            elif kind == "store":
                _, name, src, dt = op
                o = _Op(kind=KINDS["store"], dtype=DTYPES[dt], a=tags[src], b=-1, c=-1)
                buf = buffers[name]
                o.ptr = buf.ctypes.data if buf.size else None
                for k, s in enumerate(spec["views"][name]["strides"]):
                    o.strides[k] = s
                tags[name] = len(ops)
                ops.append(o)
                self.store_order.append((name, dt))
            else:
                raise ValueError(f"unknown op {kind!r}")
        self._ops = (_Op * max(1, len(ops)))(*ops)
        self._cmd = _Command(n_ops=len(ops), ops=self._ops, rank=len(spec["sizes"]))
        for k, s in enumerate(spec["sizes"]):
            self._cmd.sizes[k] = s
        self.numel = int(np.prod(spec["sizes"], dtype=np.int64)) if spec["sizes"] else 1

    def eval_range(self, begin: int = 0, end: int | None = None) -> None:
        """Write every store for logical indices [begin, end)."""
        end = self.numel if end is None else end
        rc = lib().orc_eval_range(ctypes.byref(self._cmd), int(begin), int(end))
        if rc != 0:
            raise ValueError(f"oracle rejected the command (status {rc})")

    def eval_points(self, lin) -> dict:
        """Values of every store at the given logical (row-major) indices."""
        lin = np.ascontiguousarray(lin, dtype=np.int64)
        outs = {name: np.empty(lin.size, dtype=POINT_DTYPE[dt]) for name, dt in self.store_order}
        ptrs = (ctypes.c_void_p * max(1, len(outs)))(
            *[outs[name].ctypes.data for name, _ in self.store_order])
        rc = lib().orc_eval_points(ctypes.byref(self._cmd), lin.ctypes.data, lin.size,
                                   ctypes.cast(ptrs, ctypes.c_void_p))
        if rc != 0:
            raise ValueError(f"oracle rejected the command or an index (status {rc})")
        return outs


def f32_to_f16_bits(x_bits: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x_bits, dtype=np.uint32)
    out = np.empty(x.size, dtype=np.uint16)
    lib().orc_f32_to_f16_n(x.ctypes.data, out.ctypes.data, x.size)
    return out


def f32_to_bf16_bits(x_bits: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x_bits, dtype=np.uint32)
    out = np.empty(x.size, dtype=np.uint16)
    lib().orc_f32_to_bf16_n(x.ctypes.data, out.ctypes.data, x.size)
    return out
