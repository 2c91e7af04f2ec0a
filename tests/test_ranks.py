"""The N > 1 path of the benchmark on CPU: two gloo ranks on 127.0.0.1.

Each rank reports its own step times; max_over_ranks must give every rank the
slowest rank's times, and the whole-job value counts both ranks' tokens over
that time.  The reference arm runs on rank 0 only (other ranks return
nothing).  No GPU and no data-path collective are involved.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.5 + rank, 10.0 - rank, 0.25 * (rank + 1)]   # step ms, e2e ms, attention ms
        got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        value = bench.aggregate_tokens_per_s(world, 8192, got[0])
        ref_arm = bench.run_reference(None, rank, world) if rank != 0 else "skipped"
        out.put((rank, got, value, ref_arm))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_by_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, got, value, ref_arm = q.get(timeout=120)
        res[rank] = (got, value, ref_arm)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        got, value, _ = res[rank]
        assert got == [2.5, 10.0, 0.5]
        assert value == pytest.approx(2 * 8192 / 2.5e-3)
    assert res[1][2] is None   # the reference arm does no work on rank 1


def test_reference_arm_line_on_cpu():
    """The reference arm (the oracle on the host cores, a bounded sample of the
    8K workload per step) prints the benchmark's line: same metric and unit,
    impl = reference, a cpu_baseline describing the run, and an e2e object
    with no host-device copies."""
    import types
    sys.path.insert(0, ROOT)
    import bench
    res = bench.run_reference(types.SimpleNamespace(steps=1, warmup=0), 0, 1)
    assert res["impl"] == "reference" and res["metric"] == bench.METRIC and res["unit"] == "tokens/s"
    assert res["higher_is_better"] is True and res["value"] > 0
    cb = res["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == res["value"] and cb["cores"] >= 1 and cb["sample"]
    assert res["e2e"] == {"value": res["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
    assert res["config"]["workload"] == "c2_csa_prefill_8k"
    # the same config dict as the GPU arm prints, and the sample size stated
    assert res["config"] == bench.bench_config(1)
    assert cb["rows_sampled"] >= 1 and str(cb["rows_sampled"]) in cb["sample"]
