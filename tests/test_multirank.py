"""The benchmark's multi-process path on CPU, world size 2 over gloo.

The hot path has no exchange step: each rank runs its own replica of the
workload, and the job's time is the slowest rank's (max over ranks). These
tests check that reduction and the whole-job throughput with two gloo
processes, and the reference arm under torchrun, where rank 0 alone runs the
oracle and prints the line while rank 1 exits 0 without work."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        local_ms = [2.5, 4.0][rank]
        ms = bench.max_over_ranks(local_ms, world)
        gbs = bench.whole_job_gbs(1 << 30, world, ms)
        # a second reduction in a different order of magnitudes
        ms2 = bench.max_over_ranks([1e-3, 7.25][rank], world)
        out.put((rank, ms, gbs, ms2))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, gbs, ms2 in res:
        assert ms == 4.0 and ms2 == 7.25          # every rank sees the slowest rank's time
        assert gbs == pytest.approx((1 << 30) * 2 / 4.0e-3 / 1e9)  # both replicas' bytes over it


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_gbs(10**9, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_prints_on_rank_0_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload", "chain_f32", "--cpu-seconds", "0.05"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["metric"].startswith("fused Command throughput")
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_range_split_keeps_packed_words_apart():
    sys.path.insert(0, ROOT)
    import bench
    for m, parts in [(0, 4), (1, 8), (31, 3), (1000, 8), (4097, 7), (10**6 + 3, 16)]:
        r = bench.split_ranges(m, parts)
        assert [a for a, _ in r[1:]] == [b for _, b in r[:-1]]          # contiguous
        assert (r[0][0] if r else 0) == 0 and (r[-1][1] if r else m) == m
        assert all(a % 32 == 0 for a, _ in r) and len(r) <= max(1, parts)


@pytest.mark.parametrize("name,n", [("threshold_bits", 5003), ("chain_f32", 4099), ("strided_bf16", 0)])
def test_threaded_oracle_leg_matches_one_thread(name, n):
    """The multi-core oracle timing writes what one thread writes, packed-bit
    tail included."""
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np

    import bench
    import oracle
    import specutil
    from inputgen import workloads as W
    spec = W.FULL[name](*(() if n == 0 else (n,))) if name != "strided_bf16" else W.strided_bf16(40, 72, 80)
    total = W.numel(spec)
    one, many = specutil.host_buffers(spec), specutil.host_buffers(spec)
    oracle.OracleCommand(spec, one).eval_range(0, total)
    res = bench.oracle_threads(oracle.OracleCommand(spec, many), total, 1.0, 1e12, 1.0)
    assert res["cores"] >= 1 and res["value"] > 0
    for s in W.store_names(spec):
        assert np.array_equal(one[s].view(np.uint8), many[s].view(np.uint8)), s
