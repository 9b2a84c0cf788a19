"""Host-side tests of the C ABI: the library loads and exports every declared
symbol, Command building rejects bad input, lowering has the expected
structure, and launch planning validates arguments and picks executors. No
GPU is used (kernels come from cmd_lower_kernel; pointers are never read)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import tensor_command_execution_gb300 as T
from inputgen import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "cmd.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cmd_[a-z_]+)\s*\(", text)) - {"CMD_LOCAL"})


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 18
    L = ctypes.CDLL(T.library_path() if os.path.exists(T.library_path()) else T._build.build())
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(T.SIGNATURES), set(names) ^ set(T.SIGNATURES)
    assert T.cmd_abi_version() == 3


def test_status_strings():
    L = T.lib()
    assert L.cmd_status_string(0) == b"CMD_OK"
    assert L.cmd_status_string(5) == b"CMD_ERR_ALIAS"


# ---- builder errors ------------------------------------------------------------

def _err(fn, *a):
    with pytest.raises(T.CmdError) as e:
        fn(*a)
    return e.value.name


def test_builder_rejects_bad_input():
    c = T.Command()
    x = c.load_tensor("f32", 1)
    i = c.load_tensor("i32", 1)
    assert _err(c.load_tensor, "f32", 5) == "CMD_ERR_SHAPE"
    assert _err(c.load_scalar, "f16") == "CMD_ERR_TYPE"
    # int/float mix
    assert _err(c.execute, [("add", x, i)]) == "CMD_ERR_TYPE"
    # reference to a tag that does not exist yet
    assert _err(c.execute, [("add", x, 99)]) == "CMD_ERR_BAD_TAG"
    # local reference to a later op of the block
    assert _err(c.execute, [("add", x, T.CMD_LOCAL(0))]) == "CMD_ERR_BAD_TAG"
    # a failed block adds nothing
    before = T.cmd_next_tag(c.handle)
    assert _err(c.execute, [("add", x, x), ("add", x, i)]) == "CMD_ERR_TYPE"
    assert T.cmd_next_tag(c.handle) == before
    y, z = c.execute([("mul", x, x), ("neg", T.CMD_LOCAL(0), None)])
    assert (y, z) == (before, before + 1)
    s = c.store(z, "bf16", 1)
    # a store has no value
    assert _err(c.execute, [("neg", s, None)]) == "CMD_ERR_BAD_TAG"
    # int value stored as float and float stored as int
    assert _err(c.store, i, "f32", 1) == "CMD_ERR_TYPE"
    assert _err(c.store, y, "i32", 1) == "CMD_ERR_TYPE"
    assert _err(c.execute, []) == "CMD_ERR_ARG"


def test_tag_limit():
    c = T.Command()
    x = c.load_tensor("f32", 1)
    for _ in range(W_LIMIT - 1):
        c.execute([("neg", x, None)])
    assert _err(c.execute, [("neg", x, None)]) == "CMD_ERR_LIMIT"


W_LIMIT = 128


def test_mixed_ranks_rejected_at_lowering():
    c = T.Command()
    x = c.load_tensor("f32", 2)
    c.store(x, "f32", 1)
    assert _err(c.lower) == "CMD_ERR_SHAPE"


# ---- lowering structure ---------------------------------------------------------

def test_lowering_of_the_workloads():
    expect = {  # live E ops, loads, slots, tier, moves
        "add_f32": (1, 2, 2, 0, 0),
        "chain_f32": (4, 3, 3, 1, 0),
        "wrap_i32": (3, 4, 4, 1, 0),
        "strided_bf16": (3, 2, 2, 0, 0),
        "wide_dag": (15, 6, 7, 2, 3),
        "batched_transpose": (2, 2, 2, 0, 0),
        "div_clamp_i32": (5, 1, 1, 0, 0),
        "threshold_u32": (1, 1, 1, 0, 0),
        "threshold_bits": (1, 1, 1, 0, 0),
        "chain_bf16": (4, 3, 3, 1, 0),
    }
    small = {"strided_bf16": (64, 64, 64), "batched_transpose": (2, 64, 64)}
    for name, f in W.FULL.items():
        c, _ = T.command_from_spec(f(*small[name]) if name in small else f(1024))
        info, words = c.lower()
        got = (info["n_live_ops"], info["n_loads"], info["n_slots"], info["tier"], info["n_moves"])
        assert got == expect[name], (name, info)
        assert info["n_words"] == len(words) == info["n_live_ops"] + info["n_moves"] + info["n_stores"] + 1


def test_dead_tags_and_reuse():
    c = T.Command()
    a = c.load_tensor("f32", 1)
    b = c.load_tensor("f32", 1)
    dead_load = c.load_tensor("f32", 1)
    s = c.load_scalar("f32")
    t = c.execute([("add", a, b), ("add", b, a), ("mul", T.CMD_LOCAL(0), T.CMD_LOCAL(1)),
                   ("sub", dead_load, a), ("mul", a, s), ("mul", s, a), ("sub", T.CMD_LOCAL(4), T.CMD_LOCAL(5))])
    c.store(t[2], "f32", 1)
    c.store(t[6], "f32", 1)
    info, _ = c.lower()
    # b+a reuses a+b; s*a reuses a*s; the sub of the dead load is dropped
    assert info["n_loads"] == 2
    assert info["n_live_ops"] == 4
    assert info["n_scalars"] == 1


def test_sub_is_not_treated_as_commutative():
    c = T.Command()
    a = c.load_tensor("f32", 1)
    b = c.load_tensor("f32", 1)
    t = c.execute([("sub", a, b), ("sub", b, a)])
    c.store(t[0], "f32", 1)
    c.store(t[1], "f32", 1)
    info, _ = c.lower()
    assert info["n_live_ops"] == 2


def test_extended_flag_and_new_op_reuse():
    """A live division marks the program for the executors' extended
    variant; a dead one does not. min/max commute (so reuse merges the
    swapped form), div does not."""
    c = T.Command()
    a = c.load_tensor("f32", 1)
    b = c.load_tensor("f32", 1)
    i = c.load_tensor("i32", 1)
    t = c.execute([("min", a, b), ("min", b, a), ("max", a, b), ("div", a, b), ("div", b, a),
                   ("to_f32", a, None), ("to_i32", i, None), ("abs", i, None)])
    c.store(t[0], "f32", 1)
    c.store(t[1], "f32", 1)
    c.store(t[2], "f32", 1)
    c.store(t[5], "f32", 1)
    c.store(t[6], "i32", 1)
    info, _ = c.lower()
    assert info["extended"] == 0  # both divisions are dead
    assert info["n_live_ops"] == 4  # min (once), max and the two (identity) conversions
    c.store(t[4], "f32", 1)
    info, _ = c.lower()
    assert info["extended"] == 1 and info["n_live_ops"] == 5
    for name, f in W.FULL.items():
        c2, _ = T.command_from_spec(f(2, 64, 64) if name == "batched_transpose"
                                    else f(64, 64, 64) if name == "strided_bf16" else f(64))
        assert c2.lower()[0]["extended"] == (name in ("div_clamp_i32", "threshold_u32", "threshold_bits"))


def test_mixed_classes_rejected():
    c = T.Command()
    a = c.load_tensor("f32", 1)
    i = c.load_tensor("i32", 1)
    with pytest.raises(T.CmdError):
        c.execute([("min", a, i)])


@pytest.mark.parametrize("n_loads,tier", [(12, 4), (16, 3)])
def test_wide_programs_use_the_16_and_32_slot_tiers(n_loads, tier):
    # n loads all live until the end: 9 to 16 slots run the 16-slot tier
    # (tier number 4), more the 32-slot one (tier number 3)
    c = T.Command()
    xs = [c.load_tensor("f32", 1) for _ in range(n_loads)]
    ops = [("add", xs[0], xs[-1])] + [("add", T.CMD_LOCAL(i), xs[(i + 1) % n_loads]) for i in range(n_loads - 1)]
    ops += [("mul", xs[k], xs[k]) for k in range(n_loads)]
    t = c.execute(ops)
    c.store(t[n_loads - 1], "f32", 1)
    for k in range(n_loads, n_loads + 7):
        c.store(t[k], "f32", 1)
    info, words = c.lower()
    assert info["tier"] == tier and info["n_slots"] > 8
    assert (info["n_slots"] <= 16) == (tier == 4)
    # the wide encoding: the end word is kind 31 in the top byte
    assert words[-1] >> 24 == 31


def test_store_of_loads_and_scalars_only():
    c = T.Command()
    x = c.load_tensor("f16", 1)
    s = c.load_scalar("f32")
    c.store(x, "f32", 1)
    c.store(s, "bf16", 1)
    info, _ = c.lower()
    assert info["n_live_ops"] == 0 and info["n_stores"] == 2


def test_dump_lists_the_program():
    c, _ = T.command_from_spec(W.chain_f32(1024))
    text = c.lower_kernel().dump()
    assert "fmul    r1, r0" in text and "store   out0 <- r1 (f32" in text


# ---- launch planning (host only) -------------------------------------------------

BASE = 1 << 30  # fake, 16-byte-aligned device addresses; never dereferenced


def _plan(spec, ptrs=None, overrides=None):
    c, tags = T.command_from_spec(spec)
    k = c.lower_kernel()
    views = {}
    addr = BASE
    for name in W.load_names(spec) + W.store_names(spec):
        v = spec["views"][name]
        p = (ptrs or {}).get(name, addr)
        views[tags[name]] = T.TensorView(p, spec["sizes"], v["strides"])
        addr += (v["alloc"] * 4 + 4096) // 4096 * 4096
    for name, view in (overrides or {}).items():
        views[tags[name]] = view
    return k.plan(views, T.spec_scalars(spec, tags))


def test_plans_of_the_workloads():
    assert _plan(W.add_f32(1 << 20))["path"] == "contig"
    assert _plan(W.chain_f32(1000))["path"] == "contig"  # ragged length still contiguous
    p = _plan(W.strided_bf16(256, 192, 200))
    assert p["path"] == "tile2d" and p["n_transposed"] == 1 and p["merged_sizes"] == [256, 192]
    assert p["bytes"] == 256 * 192 * 6
    p = _plan(W.wide_dag(1 << 20))
    assert p["path"] == "contig" and p["bytes"] == 30 << 20
    p = _plan(W.batched_transpose(4, 128, 64))
    assert p["path"] == "tile2d" and p["merged_sizes"] == [4, 128, 64] and p["n_transposed"] == 1
    p = _plan(W.div_clamp_i32(1 << 20))
    assert p["path"] == "contig" and p["bytes"] == 12 << 20


def test_dims_merge_to_contiguous():
    spec = W.add_f32(24)
    spec["sizes"] = (2, 3, 4)
    for k in spec["views"]:
        spec["views"][k] = dict(strides=(12, 4, 1), alloc=24)
    p = _plan(spec)
    assert p["path"] == "contig" and p["merged_rank"] == 1 and p["merged_sizes"] == [24]


def test_padded_rows_and_permutations_use_the_tile_path():
    spec = W.add_f32(0)
    spec["sizes"] = (64, 64)
    spec["views"] = {"x": dict(strides=(72, 1), alloc=64 * 72), "y": dict(strides=(64, 1), alloc=4096),
                     "out": dict(strides=(64, 1), alloc=4096)}
    assert _plan(spec)["path"] == "tile2d"
    spec["sizes"] = (4, 8, 16)
    spec["views"] = {"x": dict(strides=(1, 64, 4), alloc=512), "y": dict(strides=(128, 16, 1), alloc=512),
                     "out": dict(strides=(128, 16, 1), alloc=512)}
    # the last two dims merge for every view: a 4 x 128 transposed read
    p = _plan(spec)
    assert p["path"] == "tile2d" and p["merged_sizes"] == [4, 128] and p["n_transposed"] == 1
    # a rank-3 permutation tiles over (dim 0, dim 2) with dim 1 as the batch
    spec["views"]["x"] = dict(strides=(1, 4, 32), alloc=512)
    p = _plan(spec)
    assert p["path"] == "tile2d" and p["merged_rank"] == 3 and p["n_transposed"] == 1
    # a view with no unit stride at all cannot be staged as a tile
    spec["views"]["x"] = dict(strides=(2, 8, 64), alloc=1024)
    p = _plan(spec)
    assert p["path"] == "generic" and p["merged_rank"] == 3


def test_padded_rows_whole_chunks_long_take_the_contiguous_executor():
    """Two merged dims, every view unit-stride along the columns, row starts
    on 4-element boundaries, and rows a whole number of warp chunks long
    (512 elements for the two-input add's 2-slot tier): contiguous, merged
    rank 2. A row length that is not, a row stride off the boundary, a
    transposed load or a packed-bit store keep the other paths."""
    spec = W.add_f32(0)
    spec["sizes"] = (64, 1024)
    spec["views"] = {"x": dict(strides=(1032, 1), alloc=64 * 1032), "y": dict(strides=(1024 + 64, 1), alloc=64 * 1088),
                     "out": dict(strides=(1028, 1), alloc=64 * 1028)}
    p = _plan(spec)
    assert p["path"] == "contig" and p["merged_rank"] == 2 and p["merged_sizes"] == [64, 1024]
    spec["views"]["y"] = dict(strides=(0, 1), alloc=1024)       # one row read for every row
    assert _plan(spec)["path"] == "contig"
    spec["sizes"] = (64, 768)                                     # 1.5 chunks per row
    assert _plan(spec)["path"] == "tile2d"
    spec["sizes"] = (64, 1024)
    spec["views"]["x"] = dict(strides=(1030, 1), alloc=64 * 1030)  # rows 8 bytes off the 16-byte boundary
    assert _plan(spec)["path"] == "generic"
    spec["views"]["x"] = dict(strides=(1, 64), alloc=64 * 1024)    # transposed
    assert _plan(spec)["path"] == "tile2d"
    # the chain Command's 4-slot tier has 256-element chunks
    ch = W.chain_f32(0)
    ch["sizes"] = (10, 768)
    ch["views"] = {k: dict(strides=(800, 1), alloc=10 * 800) for k in ("a", "b", "c", "out")}
    p = _plan(ch)
    assert p["path"] == "contig" and p["merged_rank"] == 2
    # rows not a whole number of chunks: aligned views take the tile path, rows
    # at an offset from the vector alignment (which tiles cannot start at) the
    # row walk with shifted loads and their first and last columns per element
    spec["sizes"] = (64, 8200)
    spec["views"] = {"x": dict(strides=(8208, 1), alloc=64 * 8208), "y": dict(strides=(8204, 1), alloc=64 * 8204),
                     "out": dict(strides=(8200, 1), alloc=64 * 8200)}
    assert _plan(spec)["path"] == "tile2d"
    p = _plan(spec, ptrs={"x": BASE + 4})
    assert p["path"] == "contig" and p["merged_rank"] == 2
    spec["sizes"] = (64, 700)                                     # a fifth of each row per element
    assert _plan(spec, ptrs={"x": BASE + 4})["path"] == "generic"
    bits = W.threshold_bits(0)
    bits["sizes"] = (8, 1024)
    bits["views"] = {"x": dict(strides=(1040, 1), alloc=8 * 1040), "bits": dict(strides=(1024, 1), alloc=256)}
    assert _plan(bits)["path"] != "contig"


def test_loads_off_the_stores_alignment_take_the_shifted_contiguous_path():
    """1-D unit-stride views whose loads sit off the stores' vector alignment
    by other element counts run contiguous (shifted loads) once the launch
    is longer than its head (up to 7 elements), one warp chunk and 4 more;
    shorter, in the 32-slot tier, with two stores at different offsets,
    packed bits or a non-unit stride, per element."""
    x_off = {"x": BASE + (1 << 28) + 4}                      # x one element past a 16-byte boundary
    p = _plan(W.add_f32(4096), ptrs=x_off)
    assert p["path"] == "contig" and p["merged_rank"] == 1
    assert _plan(W.add_f32(512 + 11), ptrs=x_off)["path"] == "contig"
    assert _plan(W.add_f32(512 + 6), ptrs=x_off)["path"] == "generic"   # shorter than head + chunk + 4
    out_off = {"out": BASE + 2 * (1 << 28) + 8}                # the store two elements in: head 2 + 4
    assert _plan(W.add_f32(4096), ptrs=out_off)["path"] == "contig"
    assert _plan(W.wide_dag(4096), ptrs={"a": BASE + 4})["path"] == "contig"     # 8-slot tier
    div = W.wide_dag(4096)   # with a division: the extended 8-slot tier, dense ranges only
    i = next(k for k, o in enumerate(div["ops"]) if o[0] == "exec")
    div["ops"][i] = ("exec", list(div["ops"][i][1]) + [("div", "t17", "t16", "t4")])
    div["ops"] = [("store", "out0", "t17", "f32") if (o[0] == "store" and o[1] == "out0") else o for o in div["ops"]]
    assert _plan(div)["path"] == "contig"
    assert _plan(div, ptrs={"a": BASE + 4})["path"] == "generic"
    wide = W.wide32_f32(4096)
    c, _ = T.command_from_spec(wide)
    assert c.lower()[0]["tier"] == 4                                             # 16 slots
    assert _plan(wide, ptrs={"x0": BASE + 4})["path"] == "contig"
    two = W.add_f32(4096)
    two["ops"] = two["ops"] + [("store", "out2", "z", "f32")]
    two["views"]["out2"] = dict(strides=(1,), alloc=4096)
    assert _plan(two)["path"] == "contig"
    assert _plan(two, ptrs={"x": BASE + 4, "out2": BASE + 3 * (1 << 28) + 4})["path"] == "generic"  # stores apart
    stride2 = W.add_f32(4096)
    stride2["views"]["x"] = dict(strides=(2,), alloc=8191)
    assert _plan(stride2)["path"] == "generic"


def test_launch_validation_errors():
    spec = W.add_f32(1024)
    with pytest.raises(T.CmdError) as e:
        _plan(spec, ptrs={"x": BASE + 2})
    assert e.value.name == "CMD_ERR_ALIGN"
    with pytest.raises(T.CmdError) as e:
        _plan(spec, overrides={"y": T.TensorView(BASE, (1000,), (1,))})
    assert e.value.name == "CMD_ERR_SHAPE"
    with pytest.raises(T.CmdError) as e:
        _plan(spec, overrides={"out": T.TensorView(BASE + 8, (1024,), (1,))})  # overlaps x
    assert e.value.name == "CMD_ERR_ALIAS"
    with pytest.raises(T.CmdError) as e:
        _plan(spec, overrides={"out": T.TensorView(BASE + (1 << 29), (1024,), (0,))})  # not injective
    assert e.value.name == "CMD_ERR_ALIAS"
    with pytest.raises(T.CmdError) as e:
        _plan(spec, overrides={"out": T.TensorView(0, (1024,), (1,))})
    assert e.value.name == "CMD_ERR_NULL"
    # an identical view read and written in place is allowed
    p = _plan(spec, overrides={"out": T.TensorView(BASE, (1024,), (1,))})
    assert p["path"] == "contig"


def test_missing_and_unknown_arguments():
    spec = W.chain_f32(64)
    c, tags = T.command_from_spec(spec)
    k = c.lower_kernel()
    views = {tags[n]: T.TensorView(BASE + i * 4096, (64,), (1,)) for i, n in enumerate(["a", "b", "c", "out"])}
    with pytest.raises(T.CmdError) as e:
        k.plan(views, {})
    assert e.value.name == "CMD_ERR_ARG"  # scalar s missing
    with pytest.raises(T.CmdError) as e:
        k.plan({**views, tags["r"]: T.TensorView(BASE, (64,), (1,))}, {tags["s"]: 0.75})
    assert e.value.name == "CMD_ERR_BAD_TAG"  # an E result is not a tensor argument
    # a dead load's argument may be omitted; zero elements plan to nothing
    empty = {t: T.TensorView(BASE, (0,), (1,)) for t in views}
    assert k.plan(empty, {tags["s"]: 0.75})["path"] == "none"


def test_lowered_kernel_cannot_launch():
    c, tags = T.command_from_spec(W.add_f32(64))
    k = c.lower_kernel()
    views = {tags[n]: T.TensorView(BASE + i * 4096, (64,), (1,)) for i, n in enumerate(["x", "y", "out"])}
    with pytest.raises(T.CmdError) as e:
        k.launch(views, stream=0)
    assert e.value.name == "CMD_ERR_STATE"


def test_host_only_calls_allocate_no_device_memory():
    """Building, lowering, inspecting and planning never allocate device
    memory (the library's own count stays put)."""
    before = T.cmd_device_allocations()
    c, tags = T.command_from_spec(W.strided_bf16(128, 72, 80))
    k = c.lower_kernel()
    k.info()
    k.dump()
    del k
    assert T.cmd_device_allocations() == before


def test_configure_waits_validates():
    with pytest.raises(T.CmdError) as e:
        T.cmd_configure_waits(0)
    assert e.value.name == "CMD_ERR_ARG"
    T.cmd_configure_waits(2_000_000_000, False)


def test_compare_select_and_packed_bits_lowering():
    """Slot-slot comparisons and selects read a staging slot above the
    program's values (one more slot, a wider tier when needed); scalar
    comparisons do not. All of them, and packed-bit stores, select the
    extended executor variant."""
    c = T.Command()
    a = c.load_tensor("f32", 1)
    b = c.load_tensor("f32", 1)
    t = c.execute([("lt", a, b), ("add", a, b)])  # a and b live past the comparison
    c.store(t[0], "i32", 1)
    c.store(t[1], "f32", 1)
    info, _ = c.lower()
    assert info["extended"] == 1 and info["n_slots"] == 4 and info["tier"] == 1  # a, b, result, staging
    c = T.Command()
    x = c.load_tensor("i32", 1)
    s = c.load_scalar("i32")
    t = c.execute([("uge", x, s)])
    c.store(t[0], "b1", 1)
    info, _ = c.lower()
    assert info["extended"] == 1 and info["n_slots"] == 1 and info["tier"] == 0
    c = T.Command()
    x = c.load_tensor("f32", 1)
    y = c.load_tensor("f32", 1)
    k = c.load_tensor("i32", 1)
    t = c.execute([("select", x, y, k)])
    c.store(t[0], "f32", 1)
    info, words = c.lower()
    assert info["extended"] == 1 and info["tier"] == 1 and info["n_words"] == len(words)
    c = T.Command()
    x = c.load_tensor("i32", 1)
    t = c.execute([("add", x, x)])
    c.store(t[0], "i32", 1)
    assert c.lower()[0]["extended"] == 0


def test_compare_select_and_packed_bit_type_rules():
    c = T.Command()
    f = c.load_tensor("f32", 1)
    i = c.load_tensor("i32", 1)
    with pytest.raises(T.CmdError):
        c.execute([("ult", f, f)])          # unsigned comparisons take ints
    with pytest.raises(T.CmdError):
        c.execute([("select", f, f, f)])    # the condition must be int
    with pytest.raises(T.CmdError):
        c.execute([("select", f, i, i)])    # a and b of one class
    with pytest.raises(T.CmdError):
        c.store(f, "b1", 1)                 # packed bits store int values
    with pytest.raises(T.CmdError):
        c.load_tensor("b1", 1)              # b1 is a store type only
    t = c.execute([("gt", f, f), ("select", i, i, T.CMD_LOCAL(0))])
    c.store(t[0], "b1", 1)
    c.store(t[1], "i32", 1)
    assert c.lower()[0]["n_live_ops"] == 2


def test_division_by_a_scalar_lowers_to_derived_constants():
    """x / s with a tensor x and a scalar s uses constants derived from s at
    launch (two scalar slots for floats, three for ints, shared by every
    division by the same scalar); s / x and x / y take the general form;
    with the scalar table full the general form is used too."""
    c = T.Command()
    x = c.load_tensor("f32", 1)
    i = c.load_tensor("i32", 1)
    s = c.load_scalar("f32")
    k = c.load_scalar("i32")
    t = c.execute([("div", x, s), ("div", T.CMD_LOCAL(0), s), ("div", i, k), ("div", s, x), ("div", x, x)])
    for j, dt in enumerate(("f32", "f32", "i32", "f32", "f32")):
        c.store(t[j], dt, 1)
    dump = c.lower_kernel().dump()
    assert dump.count("fdivs") == 2 and dump.count("idivs") == 1
    assert dump.count("fdivs   r2, s0  ; through s2..s3, derived from s0") == 2  # one shared pair
    assert "idivs   r1, s1  ; through s4..s6, derived from s1" in dump           # the int triple
    assert "frdiv   r1, s0" in dump and "fdiv    r0, r0" in dump                 # s / x, x / x: general
    # 16 scalars in the table: no room for derived constants
    c = T.Command()
    x = c.load_tensor("f32", 1)
    ss = [c.load_scalar("f32") for _ in range(16)]
    ops = [("add", x, ss[0])] + [("add", T.CMD_LOCAL(j), ss[j + 1]) for j in range(15)] + [("div", T.CMD_LOCAL(15), ss[0])]
    t = c.execute(ops)
    c.store(t[-1], "f32", 1)
    dump = c.lower_kernel().dump()
    assert "fdivs" not in dump and "fdiv" in dump
