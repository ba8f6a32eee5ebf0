"""The multi-GPU form of the benchmark is replicas only: one process per GPU,
a barrier around the timed region, the time taken as the maximum over ranks
and the units as the sum over ranks.  These tests run that host logic as two
gloo ranks on the CPU (no GPU, no collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, out):
    os.environ.update({"WORLD_SIZE": str(ws), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    r, local, w = bench.dist_setup("gloo")
    try:
        bench.barrier(w)
        t_max = bench.max_over_ranks(1.5 + r, w)          # per-rank timed region
        units = bench.sum_over_ranks(1000.0 * (r + 1), w)  # per-rank units
        ref = bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1"]), r, w) \
            if r != 0 else "skipped"
        out.put((r, local, w, t_max, units, ref))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_aggregate_as_replicas():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=90) for _ in range(ws))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for r, (rank, local, w, t_max, units, ref) in enumerate(results):
        assert (rank, local, w) == (r, r, ws)
        assert t_max == 2.5            # the slowest rank's time
        assert units == 3000.0         # all ranks' units
    # the reference arm runs on rank 0 alone; other ranks return without work
    assert results[1][5] is None


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    bench.barrier(1)


def test_cpu_baseline_reports_single_core_rate_and_cpu_model():
    """The oracle's host timing names the CPU and gives the one-core rate beside the all-cores one."""
    rate, info = bench.cpu_oracle_rate("tiny", 0.2, 1)
    assert rate > 0 and info["cores"] >= 1
    assert info["single_core_value"] > 0
    assert isinstance(info["cpu_model"], str) and info["cpu_model"]
    _, info2 = bench.cpu_oracle_rate("tiny", 0.0, 1, single_core=False)
    assert "single_core_value" not in info2
