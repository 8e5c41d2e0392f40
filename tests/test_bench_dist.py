"""The multi-rank plumbing of bench.py on CPU: two gloo ranks, each with its own row
count and time, must agree on the whole-job value (all rows over the slowest rank's
time); rank 0 alone reports.  No GPU and no data-path collective are involved."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, rows, secs, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.dist_barrier()
    value, slowest = bench.aggregate(rows[rank], secs[rank])
    out.put((rank, value, slowest))
    bench.dist_barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_rows_over_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    rows, secs = [64, 64], [0.010, 0.025]
    procs = [ctx.Process(target=_rank, args=(r, 2, port, rows, secs, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(out.get(timeout=5) for _ in range(2))
    for rank, value, slowest in res:
        assert slowest == 0.025
        assert abs(value - 128 / 0.025) < 1e-6


def test_single_process_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    value, slowest = bench.aggregate(64, 0.02)
    assert slowest == 0.02 and abs(value - 3200.0) < 1e-9


def test_stored_traffic_files_are_consistent():
    """Each stored ncu traffic figure is read + write, and is reported only for the kernel
    sources it was captured on."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    with open(bench.TRAFFIC_FILE) as f:
        tr = json.load(f)
    for w, e in tr["workloads"].items():
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"], w
        got = bench.stored_traffic(w)
        assert got is None or got == e["dram_bytes_per_launch"]
        assert (got is None) == (tr["kernel_source_hash"] != bench.kernel_source_hash())
    assert bench.stored_traffic("no such workload") is None
    with open(bench.KSTORE_TRAFFIC_FILE) as f:
        ks = json.load(f)
    assert ks["dram_bytes_per_launch"] == ks["dram_bytes_read"] + ks["dram_bytes_write"]
    got = bench.stored_kstore_traffic()
    assert (got is None) == (ks["kernel_source_hash"] != bench.source_hash(bench.KSTORE_DEPS))
