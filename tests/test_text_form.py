"""The text form of a Command (cmd_to_yaml / cmd_from_yaml): rocRoller,
"Design Overview", section "Serialization" (a Command converts to and from
YAML, for saving and caching kernel definitions). Round trips over every
workload and the random Commands of the GPU tests, a hand-written golden
file, and the reader's errors. CPU only (lowering needs no GPU)."""
from __future__ import annotations

import os

import pytest

import tensor_command_execution_gb300 as T
from inputgen import workloads as W
import specutil
import test_gpu_parity as G

SMALL = {"strided_bf16": (64, 64, 72), "batched_transpose": (2, 64, 64)}


def _workload_specs():
    for name, f in W.FULL.items():
        yield f(*SMALL[name]) if name in SMALL else f(1000)


def _random_specs():
    for seed in range(60):
        yield G.random_case(seed)[0]
    for seed in range(80):
        yield G.random_mixed_case(seed)[0]
    for seed in range(100):
        yield G.random_cmp_case(seed)[0]


def _round_trip(spec):
    c, _ = T.command_from_spec(spec)
    text = c.to_yaml()
    c2 = T.Command.from_yaml(text)
    assert c2.to_yaml() == text
    info, words = c.lower()
    info2, words2 = c2.lower()
    assert info == info2 and words == words2
    return text


@pytest.mark.parametrize("spec", list(_workload_specs()), ids=lambda s: s["name"])
def test_workloads_round_trip(spec):
    text = _round_trip(spec)
    assert text.startswith("# tensor Command") and "version: 1\n" in text


def test_random_commands_round_trip():
    n = 0
    for spec in _random_specs():
        _round_trip(spec)
        n += 1
    assert n == 240


def test_blocks_and_scalars_survive():
    c = T.Command()
    x = c.load_tensor("f32", 2)
    s = c.load_scalar("i32")
    k = c.load_scalar("f32")
    t1 = c.execute([("mul", x, k), ("neg", T.CMD_LOCAL(0), None)])
    t2 = c.execute([("gt", t1[1], x), ("select", t1[0], x, T.CMD_LOCAL(0)), ("ult", s, s)])
    c.store(t2[1], "bf16", 2)
    c.store(t2[0], "b1", 2)
    c.store(t2[2], "i32", 2)
    text = c.to_yaml()
    assert text.count("kind: execute") == 2
    assert "{tag: 6, op: select, a: 3, b: 0, c: 5}" in text
    c2 = T.Command.from_yaml(text)
    assert c2.scalar_dtypes == {1: "i32", 2: "f32"}
    assert c2.to_yaml() == text


def test_golden_hand_written_file():
    with open(os.path.join(specutil.GOLDEN, "chain_f32.cmd.yaml")) as f:
        text = f.read()
    c = T.Command.from_yaml(text)
    ref, _ = T.command_from_spec(W.chain_f32(1000))
    assert c.to_yaml() == ref.to_yaml()
    assert c.lower() == ref.lower()


BASE = """version: 1
operations:
  - {kind: load_tensor, tag: 0, dtype: f32, rank: 1}
  - kind: execute
    ops:
      - {tag: 1, op: neg, a: 0}
  - {kind: store_tensor, tag: 2, src: 1, dtype: f32, rank: 1}
"""


@pytest.mark.parametrize("text,status,line,words", [
    (BASE.replace("version: 1", "version: 2"), "CMD_ERR_ARG", 1, "version"),
    (BASE.replace("version: 1\n", ""), "CMD_ERR_ARG", 1, "version"),
    (BASE.replace("tag: 1, op: neg", "tag: 3, op: neg"), "CMD_ERR_ARG", 6, "out of order"),
    (BASE.replace("op: neg, a: 0", "op: negate, a: 0"), "CMD_ERR_ARG", 6, "unknown E op"),
    (BASE.replace("op: neg, a: 0", "op: neg, a: 0, b: 0"), "CMD_ERR_ARG", 6, "one operand"),
    (BASE.replace("op: neg, a: 0", "op: add, a: 0"), "CMD_ERR_ARG", 6, "missing key 'b'"),
    (BASE.replace("op: neg, a: 0", "op: neg, a: 1"), "CMD_ERR_ARG", 6, "earlier"),
    (BASE.replace("dtype: f32, rank: 1}\n  - kind", "dtype: f64, rank: 1}\n  - kind"), "CMD_ERR_ARG", 3, "dtype"),
    (BASE.replace("src: 1, dtype: f32", "src: 1, dtype: i32"), "CMD_ERR_TYPE", 7, "cannot store"),
    (BASE.replace("src: 1", "src: 9"), "CMD_ERR_BAD_TAG", 7, "store source"),
    (BASE.replace("rank: 1}\n  - kind", "rank: 9}\n  - kind"), "CMD_ERR_SHAPE", 3, "rank"),
    (BASE.replace("{kind: store_tensor", "{kind: save_tensor"), "CMD_ERR_ARG", 7, "unknown kind"),
    (BASE.replace("    ops:\n", ""), "CMD_ERR_ARG", 4, "ops:"),
    (BASE.replace("tag: 0, dtype", "tag: 0 dtype"), "CMD_ERR_ARG", 3, "expected ','"),
    (BASE.replace("  - {kind: store", "   - {kind: store"), "CMD_ERR_ARG", 7, "line up"),
    (BASE.replace("rank: 1}\n  - kind", "rank: 1, color: red}\n  - kind"), "CMD_ERR_ARG", 3, "unexpected key"),
    (BASE + "\tx\n", "CMD_ERR_ARG", 8, "tabs"),
])
def test_reader_errors(text, status, line, words):
    with pytest.raises(T.CmdError) as e:
        T.Command.from_yaml(text)
    assert e.value.name == status, str(e.value)
    assert f"line {line}:" in str(e.value) and words in str(e.value), str(e.value)


def test_unsigned_compare_of_floats_is_rejected_with_its_line():
    text = BASE.replace("op: neg, a: 0", "op: ult, a: 0, b: 0").replace("dtype: f32, rank: 1}\n\n", "")
    with pytest.raises(T.CmdError) as e:
        T.Command.from_yaml(text)
    assert e.value.name == "CMD_ERR_TYPE" and "line 4:" in str(e.value)
