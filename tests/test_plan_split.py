"""How contiguous launches split, on the host (plans only, no GPU).

Over random 1-D and 2-D layouts and programs (element offsets, padded and
broadcast rows), each plan on the contiguous executor is checked against
what keeps its accesses inside the views: the contiguous kernel's range is
whole warp chunks inside the row or range; a launch that may read shifted
(its head is 4 elements or more) leaves at least 4 elements after that
range, so the aligned vectors read up to 3 elements before a shifted load's
first element and up to 3 past the range's last stay inside; every load
counted as shifted sits 1..3 elements off; otherwise the head is under one
vector and what follows the range under one chunk (none in a row walk)."""
from __future__ import annotations

import pytest

import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import layouts

BASE = 1 << 30
# elements per slot per thread of the contiguous executor by tier
VEC = {0: 16, 1: 8, 2: 8, 3: 2, 4: 4}


def _plan(spec, offsets):
    c, tags = T.command_from_spec(spec)
    k = c.lower_kernel()
    dts = W.tensor_dtypes(spec)
    views, addr = {}, BASE
    for n in W.load_names(spec) + W.store_names(spec):
        es = 2 if dts[n] in ("f16", "bf16") else 4
        views[tags[n]] = T.TensorView(addr + offsets.get(n, 0) * es, spec["sizes"], spec["views"][n]["strides"])
        addr += 1 << 32
    return k.plan(views, T.spec_scalars(spec, tags)), c.lower()[0], dts


@pytest.mark.parametrize("seed", range(400))
def test_contiguous_split_keeps_reads_inside_the_views(seed):
    spec, _, offsets = layouts.random_layout_case(seed)
    p, info, dts = _plan(spec, offsets)
    if p["path"] != "contig":
        assert p["head_elements"] == p["contig_elements"] == p["shifted_loads"] == 0
        return
    rows_walk = p["merged_rank"] == 2
    cols = p["merged_sizes"][-1] if rows_walk else p["n_elements"]
    head, main = p["head_elements"], p["contig_elements"]
    half2 = all(dts[n] in ("f16", "bf16") for n in W.load_names(spec))
    may_shift = head >= 4
    v = 16 if (info["tier"] == 1 and not info["extended"] and half2 and not may_shift) else VEC[info["tier"]]
    chunk = 32 * v
    assert main % chunk == 0 and 0 <= head and head + main <= cols, p
    if info["tier"] == 2 and info["extended"]:   # built with the dense-range kernel only
        assert not rows_walk and not may_shift, p
    if p["shifted_loads"]:
        assert may_shift, p
    if may_shift:
        assert head <= 7 and cols - head - main >= 4 and main > 0, p
        assert info["tier"] != 3, p   # the 32-slot tier never reads shifted
    elif rows_walk:
        assert head == 0 and main == cols, p
    else:
        assert head < 4 and cols - head - main < chunk, p


def test_split_of_a_known_shifted_launch():
    """4099 elements of the 2-slot tier (512-element chunks). x one element
    in, y and out aligned: a head of 4, 3584 elements (7 chunks), 511 after.
    Aligned: 4096 elements, 3 after. All three 3 elements in: a head of 1."""
    spec = W.add_f32(4099)
    p, _, _ = _plan(spec, {"x": 1})
    assert (p["path"], p["head_elements"], p["contig_elements"], p["shifted_loads"]) == ("contig", 4, 3584, 1)
    p, _, _ = _plan(spec, {})
    assert (p["head_elements"], p["contig_elements"], p["shifted_loads"]) == (0, 4096, 0)
    p, _, _ = _plan(spec, {"x": 3, "y": 3, "out": 3})   # one offset for all: a head of 1
    assert (p["head_elements"], p["contig_elements"], p["shifted_loads"]) == (1, 4096, 0)


def _with_division(spec):
    """spec with a division appended to its T_Execute block and stored by its
    first store: the extended variant of whatever tier the program lands in."""
    ops = [list(o) if o[0] == "exec" else o for o in spec["ops"]]
    i = next(k for k, o in enumerate(ops) if o[0] == "exec")
    block = list(ops[i][1])
    last = block[-1][1]
    first_load = next(o[1] for o in ops if o[0] == "load")
    block.append(("div", "Ediv", last, first_load))
    ops[i] = ("exec", block)
    j = next(k for k, o in enumerate(ops) if o[0] == "store")
    ops[j] = ("store", ops[j][1], "Ediv", ops[j][3])
    return dict(spec, ops=[tuple(o) for o in ops])


@pytest.mark.parametrize("seed", range(200))
def test_contiguous_split_with_extended_programs(seed):
    """The same checks with a division in every program (the extended
    variants; the extended 8-slot tier is built with the dense-range kernel
    only, so it never plans a row walk or shifted loads)."""
    spec, _, offsets = layouts.random_layout_case(seed)
    spec = _with_division(spec)
    p, info, dts = _plan(spec, offsets)
    assert info["extended"] == 1
    if p["path"] != "contig":
        return
    rows_walk = p["merged_rank"] == 2
    cols = p["merged_sizes"][-1] if rows_walk else p["n_elements"]
    head, main = p["head_elements"], p["contig_elements"]
    chunk = 32 * VEC[info["tier"]]
    assert main % chunk == 0 and head + main <= cols, p
    if info["tier"] == 2:
        assert not rows_walk and head < 4, p
    if head >= 4:
        assert head <= 7 and cols - head - main >= 4, p
