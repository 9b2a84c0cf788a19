"""The seeded input generator: published SplitMix64 outputs, independence
from thread count, and the ranges of each distribution. CPU only."""
import numpy as np

import inputgen


def _splitmix64_reference(state: int, count: int):
    """SplitMix64 as published (Steele, Lea, Flood 2014): advance the state by
    the golden gamma, then mix; written here with Python integers."""
    out = []
    M = (1 << 64) - 1
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & M
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
        out.append(z ^ (z >> 31))
    return out


def test_counter_form_equals_sequential_splitmix64():
    lib = inputgen._get()
    key = lib.ig_stream_key(5, 3)
    seq = _splitmix64_reference(key, 50)
    got = [int(lib.ig_bits(key, i)) for i in range(50)]
    assert got == seq


def test_known_first_output_of_state_zero():
    # SplitMix64 started from state 0 first returns 0xE220A8397B1DCDAF
    lib = inputgen._get()
    assert int(lib.ig_bits(0, 0)) == 0xE220A8397B1DCDAF


def test_thread_count_does_not_change_bytes():
    n = 3 * 65536 * 4 + 17
    for kind in inputgen.KINDS:
        a = inputgen.generate(kind, 7, 2, n, -4.0, 4.0, threads=1)
        b = inputgen.generate(kind, 7, 2, n, -4.0, 4.0, threads=4)
        assert a.tobytes() == b.tobytes()


def test_streams_and_seeds_differ():
    a = inputgen.generate("u32", 1, 0, 1000)
    b = inputgen.generate("u32", 1, 1, 1000)
    c = inputgen.generate("u32", 2, 0, 1000)
    assert (a != b).mean() > 0.99 and (a != c).mean() > 0.99


def test_distribution_ranges():
    n = 1 << 20
    u = inputgen.generate("uniform_f32", 0, 0, n, -1.0, 1.0)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(float(u.mean())) < 0.01
    g = inputgen.generate("normal_f32", 1, 0, n)
    assert abs(float(g.mean())) < 0.01 and abs(float(g.std()) - 1.0) < 0.01
    i = inputgen.generate("u32", 2, 0, n).view(np.int32)
    assert i.min() < -2**31 + 2**24 and i.max() > 2**31 - 2**24
    h = inputgen.generate("uniform_bf16_trunc", 3, 0, n, -4.0, 4.0)
    f = (h.astype(np.uint32) << 16).view(np.float32)
    assert f.min() >= -4.0 and f.max() < 4.0
