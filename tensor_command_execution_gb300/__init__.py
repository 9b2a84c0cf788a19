"""Fused tensor Command execution on one GB300 GPU: Python binding.

A thin ctypes layer over ``libcmdexec.so`` (the C ABI declared in
``include/cmd.h``). It only marshals arguments: every step of building,
lowering and executing a Command runs in the library and its CUDA kernels.
PyTorch is used for device memory and streams only.

Functions named ``cmd_*`` mirror the C entry points one to one and raise
``CmdError`` on a non-OK status. ``Command`` and ``Kernel`` wrap them for
convenience, and ``command_from_spec`` builds a Command from a workload spec
(the plain-data description used by the tests and the benchmark).

There is no CPU fallback: if the library cannot be built or loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import _build

CMD_MAX_RANK = 4
DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3, "b1": 4}
DTYPE_NAMES = {v: k for k, v in DTYPES.items()}
EOPS = {"add": 0, "sub": 1, "mul": 2, "neg": 3, "div": 4, "min": 5, "max": 6, "abs": 7, "to_f32": 8,
        "to_i32": 9, "lt": 10, "le": 11, "gt": 12, "ge": 13, "eq": 14, "ne": 15, "ult": 16, "ule": 17,
        "ugt": 18, "uge": 19, "select": 20}
PATHS = {0: "none", 1: "contig", 2: "tile2d", 3: "generic"}
STATUS = {0: "CMD_OK", 1: "CMD_ERR_NULL", 2: "CMD_ERR_BAD_TAG", 3: "CMD_ERR_TYPE", 4: "CMD_ERR_SHAPE",
          5: "CMD_ERR_ALIAS", 6: "CMD_ERR_ALIGN", 7: "CMD_ERR_STATE", 8: "CMD_ERR_LIMIT", 9: "CMD_ERR_CUDA",
          10: "CMD_ERR_DEVICE_TIMEOUT", 11: "CMD_ERR_NOMEM", 12: "CMD_ERR_ARG"}


def CMD_LOCAL(i: int) -> int:
    """Operand referring to the i-th op of the same T_Execute block."""
    return -1 - i


class CmdError(RuntimeError):
    def __init__(self, status: int, func: str, message: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{func}: {self.name}: {message}")


class cmd_xop(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("a", ctypes.c_int32), ("b", ctypes.c_int32), ("c", ctypes.c_int32)]


class cmd_tensor_arg(ctypes.Structure):
    _fields_ = [("tag", ctypes.c_int32), ("rank", ctypes.c_int32), ("ptr", ctypes.c_void_p),
                ("sizes", ctypes.c_int64 * CMD_MAX_RANK), ("strides", ctypes.c_int64 * CMD_MAX_RANK)]


class _scalar_value(ctypes.Union):
    _fields_ = [("f32", ctypes.c_float), ("i32", ctypes.c_int32), ("bits", ctypes.c_uint32)]


class cmd_scalar_arg(ctypes.Structure):
    _fields_ = [("tag", ctypes.c_int32), ("v", _scalar_value)]


class cmd_runtime_args(ctypes.Structure):
    _fields_ = [("tensors", ctypes.POINTER(cmd_tensor_arg)), ("n_tensors", ctypes.c_int32),
                ("scalars", ctypes.POINTER(cmd_scalar_arg)), ("n_scalars", ctypes.c_int32)]


class cmd_program_info(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int32) for k in ("n_live_ops", "n_loads", "n_scalars", "n_stores", "n_slots",
                                              "n_words", "tier", "n_moves", "extended")]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


class cmd_launch_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("merged_rank", ctypes.c_int32),
                ("merged_sizes", ctypes.c_int64 * CMD_MAX_RANK), ("n_elements", ctypes.c_int64),
                ("bytes", ctypes.c_int64), ("n_transposed", ctypes.c_int32),
                ("head_elements", ctypes.c_int64), ("contig_elements", ctypes.c_int64),
                ("shifted_loads", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {"path": PATHS.get(self.path, self.path), "merged_rank": self.merged_rank,
                "merged_sizes": list(self.merged_sizes)[: self.merged_rank],
                "n_elements": self.n_elements, "bytes": self.bytes, "n_transposed": self.n_transposed,
                "head_elements": self.head_elements, "contig_elements": self.contig_elements,
                "shifted_loads": self.shifted_loads}


# Every symbol include/cmd.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "cmd_abi_version": (ctypes.c_int32, []),
    "cmd_status_string": (ctypes.c_char_p, [_I]),
    "cmd_last_error": (ctypes.c_char_p, []),
    "cmd_create": (_I, [ctypes.POINTER(_P)]),
    "cmd_destroy": (None, [_P]),
    "cmd_next_tag": (_I, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "cmd_add_load_tensor": (_I, [_P, _I, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "cmd_add_load_scalar": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int32)]),
    "cmd_add_execute": (_I, [_P, ctypes.POINTER(cmd_xop), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "cmd_add_store": (_I, [_P, ctypes.c_int32, _I, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "cmd_lower": (_I, [_P, ctypes.POINTER(cmd_program_info), ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32]),
    "cmd_compile": (_I, [_P, ctypes.POINTER(_P)]),
    "cmd_lower_kernel": (_I, [_P, ctypes.POINTER(_P)]),
    "cmd_compile_static_scratch": (_I, [_P, ctypes.POINTER(_P)]),
    "cmd_kernel_destroy": (None, [_P]),
    "cmd_kernel_info": (_I, [_P, ctypes.POINTER(cmd_program_info)]),
    "cmd_kernel_dump": (_I, [_P, ctypes.c_char_p, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]),
    "cmd_to_yaml": (_I, [_P, ctypes.c_char_p, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]),
    "cmd_from_yaml": (_I, [ctypes.c_char_p, ctypes.c_int64, ctypes.POINTER(_P)]),
    "cmd_plan_launch": (_I, [_P, ctypes.POINTER(cmd_runtime_args), ctypes.POINTER(cmd_launch_plan)]),
    "cmd_launch": (_I, [_P, ctypes.POINTER(cmd_runtime_args), _P]),
    "cmd_sync_status": (_I, [_P, _P]),
    "cmd_configure_waits": (_I, [ctypes.c_uint64, ctypes.c_int32]),
    "cmd_device_allocations": (ctypes.c_int64, []),
}

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """Load libcmdexec.so, building it first when it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA executor library missing at {path}")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
        return _lib


def _check(status: int, func: str) -> None:
    if status != 0:
        msg = lib().cmd_last_error()
        raise CmdError(status, func, msg.decode() if msg else "")


# ---- one-to-one wrappers of the C entry points ------------------------------

def cmd_abi_version() -> int:
    return lib().cmd_abi_version()


def cmd_create() -> int:
    h = _P()
    _check(lib().cmd_create(ctypes.byref(h)), "cmd_create")
    return h.value


def cmd_destroy(cmd: int) -> None:
    lib().cmd_destroy(cmd)


def cmd_next_tag(cmd: int) -> int:
    t = ctypes.c_int32()
    _check(lib().cmd_next_tag(cmd, ctypes.byref(t)), "cmd_next_tag")
    return t.value


def cmd_add_load_tensor(cmd: int, dtype: str, rank: int) -> int:
    t = ctypes.c_int32()
    _check(lib().cmd_add_load_tensor(cmd, DTYPES[dtype], rank, ctypes.byref(t)), "cmd_add_load_tensor")
    return t.value


def cmd_add_load_scalar(cmd: int, dtype: str) -> int:
    t = ctypes.c_int32()
    _check(lib().cmd_add_load_scalar(cmd, DTYPES[dtype], ctypes.byref(t)), "cmd_add_load_scalar")
    return t.value


def cmd_add_execute(cmd: int, ops) -> list:
    """ops: sequence of (eop name, a, b) with b None for the one-operand ops,
    or ("select", a, b, c) for c ? a : b; returns tags."""
    arr = (cmd_xop * len(ops))()
    for i, op in enumerate(ops):
        eop, a, b = op[:3]
        c = op[3] if len(op) > 3 else None
        arr[i].op = EOPS[eop]
        arr[i].a = a
        arr[i].b = -1 if b is None else b
        arr[i].c = -1 if c is None else c
    out = (ctypes.c_int32 * len(ops))()
    _check(lib().cmd_add_execute(cmd, arr, len(ops), out), "cmd_add_execute")
    return list(out)


def cmd_add_store(cmd: int, src: int, dtype: str, rank: int) -> int:
    t = ctypes.c_int32()
    _check(lib().cmd_add_store(cmd, src, DTYPES[dtype], rank, ctypes.byref(t)), "cmd_add_store")
    return t.value


def cmd_lower(cmd: int):
    info = cmd_program_info()
    words = (ctypes.c_uint32 * 512)()
    _check(lib().cmd_lower(cmd, ctypes.byref(info), words, 512), "cmd_lower")
    return info.as_dict(), list(words)[: info.n_words]


def cmd_compile(cmd: int) -> int:
    h = _P()
    _check(lib().cmd_compile(cmd, ctypes.byref(h)), "cmd_compile")
    return h.value


def cmd_compile_static_scratch(cmd: int) -> int:
    """cmd_compile without any device allocation (see include/cmd.h)."""
    h = _P()
    _check(lib().cmd_compile_static_scratch(cmd, ctypes.byref(h)), "cmd_compile_static_scratch")
    return h.value


def cmd_lower_kernel(cmd: int) -> int:
    h = _P()
    _check(lib().cmd_lower_kernel(cmd, ctypes.byref(h)), "cmd_lower_kernel")
    return h.value


def cmd_kernel_destroy(k: int) -> None:
    lib().cmd_kernel_destroy(k)


def cmd_kernel_info(k: int) -> dict:
    info = cmd_program_info()
    _check(lib().cmd_kernel_info(k, ctypes.byref(info)), "cmd_kernel_info")
    return info.as_dict()


def cmd_kernel_dump(k: int) -> str:
    need = ctypes.c_int64()
    _check(lib().cmd_kernel_dump(k, None, 0, ctypes.byref(need)), "cmd_kernel_dump")
    buf = ctypes.create_string_buffer(need.value)
    _check(lib().cmd_kernel_dump(k, buf, need.value, None), "cmd_kernel_dump")
    return buf.value.decode()


def cmd_to_yaml(cmd: int) -> str:
    need = ctypes.c_int64()
    _check(lib().cmd_to_yaml(cmd, None, 0, ctypes.byref(need)), "cmd_to_yaml")
    buf = ctypes.create_string_buffer(need.value)
    _check(lib().cmd_to_yaml(cmd, buf, need.value, None), "cmd_to_yaml")
    return buf.value.decode()


def cmd_from_yaml(text: str) -> int:
    data = text.encode()
    h = _P()
    _check(lib().cmd_from_yaml(data, len(data), ctypes.byref(h)), "cmd_from_yaml")
    return h.value


def cmd_plan_launch(k: int, args: cmd_runtime_args) -> dict:
    plan = cmd_launch_plan()
    _check(lib().cmd_plan_launch(k, ctypes.byref(args), ctypes.byref(plan)), "cmd_plan_launch")
    return plan.as_dict()


def cmd_launch(k: int, args: cmd_runtime_args, stream: int | None) -> None:
    _check(lib().cmd_launch(k, ctypes.byref(args), stream or None), "cmd_launch")


def cmd_sync_status(k: int, stream: int | None) -> None:
    _check(lib().cmd_sync_status(k, stream or None), "cmd_sync_status")


def cmd_configure_waits(timeout_ns: int, force_timeout: bool = False) -> None:
    _check(lib().cmd_configure_waits(int(timeout_ns), 1 if force_timeout else 0), "cmd_configure_waits")


def cmd_device_allocations() -> int:
    return int(lib().cmd_device_allocations())


# ---- argument marshalling ----------------------------------------------------

class TensorView:
    """A raw view: base address, logical sizes and element strides."""

    def __init__(self, ptr: int, sizes, strides):
        self.ptr = int(ptr)
        self.sizes = tuple(int(s) for s in sizes)
        self.strides = tuple(int(s) for s in strides)


def _as_view(x) -> TensorView:
    if isinstance(x, TensorView):
        return x
    # a torch tensor (device memory); its own sizes and element strides
    return TensorView(x.data_ptr(), tuple(x.shape), tuple(x.stride()))


def make_runtime_args(tensors: dict, scalars: dict, scalar_dtypes: dict):
    """tensors: tag -> torch tensor or TensorView; scalars: tag -> value."""
    tarr = (cmd_tensor_arg * max(1, len(tensors)))()
    for i, (tag, x) in enumerate(tensors.items()):
        v = _as_view(x)
        tarr[i].tag = tag
        tarr[i].rank = len(v.sizes)
        tarr[i].ptr = v.ptr
        for d, (s, st) in enumerate(zip(v.sizes, v.strides)):
            tarr[i].sizes[d] = s
            tarr[i].strides[d] = st
    sarr = (cmd_scalar_arg * max(1, len(scalars)))()
    for i, (tag, val) in enumerate(scalars.items()):
        sarr[i].tag = tag
        if scalar_dtypes.get(tag, "f32") == "i32":
            sarr[i].v.i32 = int(val)
        else:
            sarr[i].v.f32 = float(val)
    args = cmd_runtime_args(tarr, len(tensors), sarr, len(scalars))
    args._keep = (tarr, sarr)
    return args


# ---- convenience classes -----------------------------------------------------

class Command:
    """Builder for one Command (owns a cmd_command_t)."""

    def __init__(self, handle: int | None = None):
        self.handle = handle if handle is not None else cmd_create()
        self.scalar_dtypes: dict = {}

    def to_yaml(self) -> str:
        """The Command's text form (see cmd.h)."""
        return cmd_to_yaml(self.handle)

    @classmethod
    def from_yaml(cls, text: str) -> "Command":
        c = cls(cmd_from_yaml(text))
        # scalar types, for launch arguments: from the canonical text form
        for m in re.finditer(r"kind: load_scalar, tag: (\d+), dtype: (\w+)", c.to_yaml()):
            c.scalar_dtypes[int(m.group(1))] = m.group(2)
        return c

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            try:
                cmd_destroy(h)
            except Exception:
                pass
            self.handle = None

    def load_tensor(self, dtype: str, rank: int) -> int:
        return cmd_add_load_tensor(self.handle, dtype, rank)

    def load_scalar(self, dtype: str) -> int:
        t = cmd_add_load_scalar(self.handle, dtype)
        self.scalar_dtypes[t] = dtype
        return t

    def execute(self, ops) -> list:
        return cmd_add_execute(self.handle, ops)

    def store(self, src: int, dtype: str, rank: int) -> int:
        return cmd_add_store(self.handle, src, dtype, rank)

    def lower(self):
        return cmd_lower(self.handle)

    def compile(self) -> "Kernel":
        return Kernel(cmd_compile(self.handle), dict(self.scalar_dtypes))

    def lower_kernel(self) -> "Kernel":
        """A kernel handle lowered on the host only (plan/inspect, no launch)."""
        return Kernel(cmd_lower_kernel(self.handle), dict(self.scalar_dtypes))


class Kernel:
    """A compiled Command (owns a cmd_kernel_t)."""

    def __init__(self, handle: int, scalar_dtypes: dict):
        self.handle = handle
        self.scalar_dtypes = scalar_dtypes

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            try:
                cmd_kernel_destroy(h)
            except Exception:
                pass
            self.handle = None

    def info(self) -> dict:
        return cmd_kernel_info(self.handle)

    def dump(self) -> str:
        return cmd_kernel_dump(self.handle)

    def args(self, tensors: dict, scalars: dict | None = None):
        return make_runtime_args(tensors, scalars or {}, self.scalar_dtypes)

    def plan(self, tensors: dict, scalars: dict | None = None) -> dict:
        return cmd_plan_launch(self.handle, self.args(tensors, scalars))

    def launch(self, tensors: dict, scalars: dict | None = None, stream=None) -> None:
        """Enqueue one pass; stream is a torch.cuda.Stream, a raw handle, or
        None for torch's current stream."""
        if stream is None:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        elif hasattr(stream, "cuda_stream"):
            stream = stream.cuda_stream
        cmd_launch(self.handle, self.args(tensors, scalars), stream)

    def launch_args(self, args: cmd_runtime_args, stream: int | None) -> None:
        """Launch with pre-built arguments (no per-call marshalling)."""
        cmd_launch(self.handle, args, stream)

    def sync(self, stream=None) -> None:
        if hasattr(stream, "cuda_stream"):
            stream = stream.cuda_stream
        cmd_sync_status(self.handle, stream)


def command_from_spec(spec: dict):
    """Build a Command from a workload spec; return (Command, tags by name)."""
    c = Command()
    tags: dict = {}
    rank = len(spec["sizes"])
    for op in spec["ops"]:
        kind = op[0]
        if kind == "load":
            tags[op[1]] = c.load_tensor(op[2], rank)
        elif kind == "scalar":
            tags[op[1]] = c.load_scalar(op[2])
        elif kind == "exec":
            # entries (eop, name, a, b), or (eop, name, a, b, cond) for select
            block = op[1]
            local = {e[1]: i for i, e in enumerate(block)}

            def ref(x, i):
                if x is None:
                    return None
                j = local.get(x)
                if j is not None and j < i:
                    return CMD_LOCAL(j)
                return tags[x]
            res = c.execute([(e[0], ref(e[2], i), ref(e[3], i), ref(e[4] if len(e) > 4 else None, i))
                             for i, e in enumerate(block)])
            for e, t in zip(block, res):
                tags[e[1]] = t
        elif kind == "store":
            tags[op[1]] = c.store(tags[op[2]], op[3], rank)
        else:
            raise ValueError(f"unknown op kind {kind!r}")
    return c, tags


def spec_scalars(spec: dict, tags: dict) -> dict:
    return {tags[op[1]]: op[3] for op in spec["ops"] if op[0] == "scalar"}
