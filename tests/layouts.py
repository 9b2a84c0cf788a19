"""Random Commands over random 1-D and 2-D layouts (plain data: a spec, its
host buffers and the element offset of each tensor in its allocation), for
the GPU parity tests and the host tests of how launches split."""
from __future__ import annotations

import numpy as np

import specutil


def values(rng, dt, n):
    if dt == "i32":
        return rng.integers(-2**31, 2**31, size=n).astype(np.int32)
    f = (rng.standard_normal(n) * 3).astype(np.float32)
    if dt == "f32":
        return f
    if dt == "f16":
        return f.astype(np.float16)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def random_layout_case(seed):
    """A random Command (1 to 12 loads, up to 24 ops, 1 to 3 stores, mixed
    float widths or int32) over random 1-D or 2-D layouts: each tensor at a
    random element offset into its allocation, 2-D rows padded by random
    amounts (some loads read one row for every row). Whichever executor the
    planner picks (dense, shifted, rows, tiles, per element), every element
    and the bytes around the views must match the oracle."""
    rng = np.random.default_rng(10_000 + seed)
    two_d = rng.random() < 0.5
    if two_d:
        rows = int(rng.integers(2, 40))
        cols = int(rng.choice([512, 1024, 768, 1000, 1536, 2048]))
        sizes = (rows, cols)
    else:
        sizes = (int(rng.choice([600, 1037, 4099, 20_011, 70_001])),)
    is_int = rng.random() < 0.25
    n_loads = int(rng.integers(1, 13))
    ops, views, bufs, vals, offsets = [], {}, {}, [], {}

    def layout(allow_bcast):
        if not two_d:
            return (1,), sizes[0]
        r, c = sizes
        if allow_bcast and rng.random() < 0.15:
            return (0, 1), c
        ld = c + int(rng.choice([0, 0, 4, 8, 64, 4, 8, 3]))
        return (ld, 1), (r - 1) * ld + c

    for i in range(n_loads):
        dt = "i32" if is_int else str(rng.choice(["f32", "f16", "bf16"]))
        name = f"L{i}"
        ops.append(("load", name, dt))
        st, n = layout(True)
        views[name] = dict(strides=st, alloc=n)
        bufs[name] = values(rng, dt, n)
        offsets[name] = int(rng.integers(0, 4)) if rng.random() < (0.15 if two_d else 0.6) else 0
        vals.append(name)
    block = []
    for i in range(int(rng.integers(1, 25))):
        eop = str(rng.choice(["add", "sub", "mul", "neg"]))
        a = str(rng.choice(vals))
        b = None if eop == "neg" else str(rng.choice(vals))
        block.append((eop, f"E{i}", a, b))
        vals.append(f"E{i}")
    ops.append(("exec", block))
    store_off = int(rng.integers(0, 4)) if rng.random() < (0.1 if two_d else 0.5) else 0
    for i in range(int(rng.integers(1, 4))):
        src = vals[-1 - int(rng.integers(0, min(4, len(vals))))]
        dt = "i32" if is_int else str(rng.choice(["f32", "f16", "bf16"]))
        name = f"O{i}"
        ops.append(("store", name, src, dt))
        st, n = layout(False)
        views[name] = dict(strides=st, alloc=n)
        bufs[name] = specutil.sentinel_array(dt, n)
        offsets[name] = store_off if rng.random() < 0.9 else int(rng.integers(0, 4))
    spec = dict(name=f"layout{seed}", seed=seed, sizes=sizes, ops=ops, views=views, inputs={})
    return spec, bufs, offsets


def padded_spec(name, rows, cols, loads, stores, block, scalars=(), seed=0):
    """loads: {name: (dtype, row stride)}; stores: {name: (source tag, dtype,
    row stride)}; a row stride of 0 reads one row for every row."""
    ops = [("load", n, dt) for n, (dt, _) in loads.items()]
    ops += [("scalar", n, dt, v) for n, dt, v in scalars]
    ops += [("exec", block)] + [("store", n, src, dt) for n, (src, dt, _) in stores.items()]
    views = {}
    for n, (dt, ld) in loads.items():
        views[n] = dict(strides=(ld, 1), alloc=(rows - 1) * ld + cols)
    for n, (_, dt, ld) in stores.items():
        views[n] = dict(strides=(ld, 1), alloc=(rows - 1) * ld + cols)
    spec = dict(name=name, seed=seed, sizes=(rows, cols), ops=ops, views=views, inputs={})
    rng = np.random.default_rng(seed)
    bufs = {n: values(rng, dt, views[n]["alloc"]) for n, (dt, _) in loads.items()}
    for n, (_, dt, _) in stores.items():
        bufs[n] = specutil.sentinel_array(dt, views[n]["alloc"])
    return spec, bufs
