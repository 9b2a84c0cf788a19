"""The oracle split over host threads by element ranges (the checker of the
full-size GPU parity tests) writes exactly what the plain single-threaded
walk writes, packed-bit words and sentinels outside the views included."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from inputgen import workloads as W
import gpuutil
import specutil


@pytest.mark.parametrize("spec", [
    W.chain_f32((1 << 16) + 5),
    W.wrap_i32(4099),
    W.wide_dag(3001),
    W.strided_bf16(130, 72, 80),
    W.threshold_bits((1 << 12) + 17),
    W.batched_transpose(3, 40, 24),
    W.tile4_f32(68, 40),
    W.wide32_f32(1000),
], ids=lambda s: s["name"])
def test_split_oracle_equals_single_walk(spec):
    bufs = specutil.host_buffers(spec)
    split = gpuutil.oracle_every_element(spec, bufs)
    whole = {n: bufs[n].copy() for n in W.store_names(spec)}
    oracle.OracleCommand(spec, {**bufs, **whole}).eval_range()
    for n in W.store_names(spec):
        assert split[n].tobytes() == whole[n].tobytes(), n
        # the inputs' own store buffers are untouched (fresh copies were written)
        assert (specutil.bits(bufs[n]) == specutil.bits(specutil.sentinel_array(
            W.tensor_dtypes(spec)[n], bufs[n].size))).all()


def test_element_ranges_cover_once_on_word_boundaries():
    for n in (0, 1, 31, 32, 33, 1000, 1 << 20):
        for parts in (1, 3, 16, 64):
            r = gpuutil.element_ranges(n, parts)
            assert sum(b - a for a, b in r) == n
            assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
            assert all(a % 32 == 0 for a, _ in r)
            assert len(r) <= max(1, parts)
            if n:
                assert r[0][0] == 0 and r[-1][1] == n
            assert np.all([a < b for a, b in r])
