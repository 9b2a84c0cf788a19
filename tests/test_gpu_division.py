"""Division by a scalar, exhaustively over the dividends, on the GPU.

A tensor divided by a Load_Scalar runs through constants the host derives
per launch: binary32 by a correctly rounded reciprocal and two FMA
corrections of the quotient (Markstein's method), int32 by a multiply-high
constant and shift (Granlund and Montgomery, "Division by invariant integers
using multiplication", PLDI 1994, section 5), with the general division for
what falls outside their range. These tests run every one of the 2^32
dividends for a set of divisors and compare with the GPU's own IEEE / C
division (torch on the same device): bit for bit for ints, and for floats
too, NaNs as a class."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tensor_command_execution_gb300 as T

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


def _kernel(dt: str):
    c = T.Command()
    x = c.load_tensor(dt, 1)
    k = c.load_scalar(dt)
    t = c.execute([("div", x, k)])
    y = c.store(t[0], dt, 1)
    info, _ = c.lower()
    assert info["extended"] == 1 and "divs" in c.lower_kernel().dump()  # the scalar form
    return c.compile(), x, k, y


def _all_values(start: int, n: int, dtype) -> torch.Tensor:
    """The 32-bit patterns start .. start + n - 1 (an int32 range) as dtype."""
    return torch.arange(start, start + n, dtype=torch.int64, device="cuda").to(torch.int32).view(dtype)


INT_DIVISORS = [1, 2, 3, 5, 7, 10, 16, 641, 1 << 16, 1 << 30, 2**31 - 1, -2, -3, -7, -16, -(1 << 30),
                -2**31, -2**31 + 1, 12345, -99999, 3 << 20, 6700417]


@pytest.mark.parametrize("d", INT_DIVISORS)
def test_int_division_by_scalar_all_dividends(d):
    k_, x, k, y = _kernel("i32")
    out = torch.empty(CHUNK, dtype=torch.int32, device="cuda")
    for start in range(-2**31, 2**31, CHUNK):
        xs = _all_values(start, CHUNK, torch.int32)
        k_.launch({x: xs, y: out}, {k: d})
        want = torch.div(xs, d, rounding_mode="trunc")
        bad = (out != want).nonzero()
        assert bad.numel() == 0, (d, int(xs[bad[0, 0]]), int(out[bad[0, 0]]), int(want[bad[0, 0]]))


def test_int_division_by_zero_and_minus_one():
    """The divisors the constants do not cover: x / 0 = -1, x / -1 = 0 - x
    (INT_MIN / -1 = INT_MIN), on the general path."""
    k_, x, k, y = _kernel("i32")
    xs = torch.tensor([0, 1, -1, 7, -7, 2**31 - 1, -2**31], dtype=torch.int32, device="cuda")
    out = torch.empty_like(xs)
    k_.launch({x: xs, y: out}, {k: 0})
    assert out.tolist() == [-1] * 7
    k_.launch({x: xs, y: out}, {k: -1})
    assert out.tolist() == [0, -1, 1, -7, 7, -(2**31 - 1), -2**31]


FLOAT_DIVISORS = [0.0074, 3.0, 1.0 / 3.0, 3.14159265, -2.5, 7.0, 0.1, 1e-3, 65504.0, 2.0 ** -60, 2.0 ** 60,
                  2.0 ** -61, 1e-20, 7e30, -1.0, 1.0, 2.0 ** -149, 0.0, float("inf"), float("nan")]


@pytest.mark.parametrize("s", FLOAT_DIVISORS, ids=lambda v: repr(v))
def test_float_division_by_scalar_all_dividends(s):
    """Every binary32 pattern divided by s: subnormal, huge, zero, infinite
    and NaN dividends and the divisors outside [2^-60, 2^60] take the general
    division; the rest the reciprocal form; all must equal IEEE division."""
    k_, x, k, y = _kernel("f32")
    out = torch.empty(CHUNK, dtype=torch.float32, device="cuda")
    sv = torch.tensor(s, dtype=torch.float32, device="cuda")
    for start in range(-2**31, 2**31, CHUNK):
        xs = _all_values(start, CHUNK, torch.float32)
        k_.launch({x: xs, y: out}, {k: float(np.float32(s))})
        want = xs / sv
        ob, wb = out.view(torch.int32), want.view(torch.int32)
        same = (ob == wb) | (torch.isnan(out) & torch.isnan(want))
        bad = (~same).nonzero()
        assert bad.numel() == 0, (s, hex(int(xs.view(torch.int32)[bad[0, 0]]) & 0xFFFFFFFF),
                                  hex(int(ob[bad[0, 0]]) & 0xFFFFFFFF), hex(int(wb[bad[0, 0]]) & 0xFFFFFFFF))
