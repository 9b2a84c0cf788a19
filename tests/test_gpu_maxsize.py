"""Maximum sizes: more logical elements than 32-bit indexes reach.

Each executor at a size past 2^32 elements (contiguous, generic) or past
2^31 (tile, 2-D), with inputs filled on the device from closed forms and
the results checked at the index boundaries (around 2^31 and 2^32, the
last elements) and at random samples: int32 results against the exact
integer formula reduced modulo 2^32, the bf16 tile result against fp32
operations done one by one by torch on the same device and rounded once to
bfloat16. These catch index arithmetic that wraps at 32 bits."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tensor_command_execution_gb300 as T

pytestmark = pytest.mark.gpu

CH = 1 << 28


def _fill_formula(t: torch.Tensor, mul: int, add: int):
    """t[i] = (i * mul + add) mod 2^32 as int32 bits, chunk by chunk (the
    int64 product may wrap modulo 2^64, which leaves its low 32 bits right)."""
    n = t.numel()
    for a in range(0, n, CH):
        b = min(n, a + CH)
        v = (torch.arange(a, b, dtype=torch.int64, device=t.device) * mul + add) & 0xFFFFFFFF
        t[a:b] = (v - ((v >> 31) << 32)).to(torch.int32)  # [2^31, 2^32) to the negative int32s


def _sample(n: int, rng) -> np.ndarray:
    edges = [np.arange(max(0, c - 8), min(n, c + 8)) for c in (0, 2**31, 2**32, n - 8)]
    return np.unique(np.concatenate(edges + [rng.integers(0, n, 100000)]))


def _formula(idx: np.ndarray, mul: int, add: int) -> np.ndarray:
    return (idx.astype(object) * mul + add) % 2**32


def _int_case(n: int, offset: int, path: str, z2_offset=None):
    """z = x * y + x with x `offset` elements into its allocation; with
    z2_offset, a second store of the same value that many elements in."""
    torch.cuda.empty_cache()
    big = torch.empty(n + offset, dtype=torch.int32, device="cuda")
    x = big[offset:]
    y = torch.empty(n, dtype=torch.int32, device="cuda")
    z = torch.empty(n, dtype=torch.int32, device="cuda")
    _fill_formula(x, 1, 12345)
    _fill_formula(y, 2654435761, 7)
    c = T.Command()
    tx, ty = c.load_tensor("i32", 1), c.load_tensor("i32", 1)
    t = c.execute([("mul", tx, ty), ("add", T.CMD_LOCAL(0), tx)])
    tz = c.store(t[1], "i32", 1)
    args = {tx: x, ty: y, tz: z}
    outs = [z]
    if z2_offset is not None:
        big2 = torch.empty(n + z2_offset, dtype=torch.int32, device="cuda")
        z2 = big2[z2_offset:]
        args[c.store(t[1], "i32", 1)] = z2
        outs.append(z2)
    k = c.compile()
    assert k.plan(args)["path"] == path
    k.launch(args)
    k.sync()
    torch.cuda.synchronize()
    idx = _sample(n, np.random.default_rng(n))
    xv, yv = _formula(idx, 1, 12345), _formula(idx, 2654435761, 7)
    want = np.array([int(a * b + a) % 2**32 for a, b in zip(xv, yv)], dtype=np.int64)
    for out in outs:
        got = out[torch.from_numpy(idx).cuda()].cpu().numpy().astype(np.int64) % 2**32
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, (path, int(idx[bad[0]]), int(got[bad[0]]), int(want[bad[0]]))
    del big, y, z, outs, args
    torch.cuda.empty_cache()


def test_contiguous_past_2_32_elements():
    _int_case((1 << 32) + 37, 0, "contig")


def test_shifted_loads_past_2_32_elements():
    # x one element past its allocation's start, y and z aligned: the
    # contiguous executor with x's loads shifted
    _int_case((1 << 32) + 5, 1, "contig")


def test_generic_past_2_32_elements():
    # two stores at different offsets from the vector alignment: per element
    _int_case((1 << 32) + 5, 1, "generic", z2_offset=1)


def test_tile_past_2_31_elements():
    """out = A*B^T - A + 0.5 (the strided workload's Command) with A and B
    50000 x 50000 bf16: 2.5e9 logical elements on the tile executor."""
    torch.cuda.empty_cache()
    m = n = 50000
    A = torch.empty(m * n, dtype=torch.int16, device="cuda")
    B = torch.empty(m * n, dtype=torch.int16, device="cuda")
    out = torch.empty(m * n, dtype=torch.int16, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    for a in range(0, m * n, CH):  # bf16 values of uniform[-4, 4) (upper halves of fp32)
        b = min(m * n, a + CH)
        A[a:b] = ((torch.rand(b - a, device="cuda", generator=g) * 8 - 4).view(torch.int32) >> 16).to(torch.int16)
        B[a:b] = ((torch.rand(b - a, device="cuda", generator=g) * 8 - 4).view(torch.int32) >> 16).to(torch.int16)
    c = T.Command()
    ta, tb = c.load_tensor("bf16", 2), c.load_tensor("bf16", 2)
    h = c.load_scalar("f32")
    t = c.execute([("mul", ta, tb), ("sub", T.CMD_LOCAL(0), ta), ("add", T.CMD_LOCAL(1), h)])
    to = c.store(t[2], "bf16", 2)
    k = c.compile()
    views = {ta: T.TensorView(A.data_ptr(), (m, n), (n, 1)), tb: T.TensorView(B.data_ptr(), (m, n), (1, m)),
             to: T.TensorView(out.data_ptr(), (m, n), (n, 1))}
    assert k.plan(views, {h: 0.5})["path"] == "tile2d"
    k.launch(views, {h: 0.5})
    k.sync()
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    lin = np.unique(np.concatenate([np.arange(2**31 - 8, 2**31 + 8), np.arange(m * n - 8, m * n),
                                    rng.integers(0, m * n, 100000)]))
    i, j = lin // n, lin % n
    li = torch.from_numpy(lin).cuda()
    a = (A[li].to(torch.int32) << 16).view(torch.float32)
    bt = (B[torch.from_numpy(j * m + i).cuda()].to(torch.int32) << 16).view(torch.float32)
    p = a * bt
    q = p - a
    r = q + 0.5
    want = r.to(torch.bfloat16).view(torch.int16)
    got = out[li]
    bad = (got != want).nonzero()
    assert bad.numel() == 0, (int(lin[bad[0, 0].item()]), int(got[bad[0, 0]]), int(want[bad[0, 0]]))
    del A, B, out
    torch.cuda.empty_cache()
