"""The multi-rank host path of bench.py on CPU, world size 2 over gloo.

The path does not shard (one replica per GPU, no collective on the data path), so the
only cross-rank steps are the barriers around the timed region and the max over ranks
of the timed milliseconds.  These tests run those steps in two processes, and run the
reference arm under torchrun, where rank 0 alone prints the contract line."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench

    r, w, dist = bench.dist_init()
    try:
        bench.barrier(dist)
        value, ms = bench.job_throughput(local_ms[rank], 1e9, 4, w, dist, "cpu")
        bench.barrier(dist)
        q.put((r, w, value, ms))
    finally:
        dist.destroy_process_group()


def test_job_throughput_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")  # no fork of a process that may hold threads
    q = ctx.Queue()
    port = _free_port()
    local_ms = [40.0, 50.0]  # rank 1 is slower
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, value, ms) in enumerate(got):
        assert (rank, world) == (r, 2)
        # 2 ranks x 1e9 units x 4 steps in the slowest rank's 50 ms
        assert abs(value - 2 * 1e9 * 4 / 0.050) < 1e-3 * value
        assert abs(ms - 12.5) < 1e-9


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    value, ms = bench.job_throughput(30.0, 2e9, 3, 1, None, "cpu")
    assert abs(value - 2e9 * 3 / 0.030) < 1e-6 * value and abs(ms - 10.0) < 1e-12


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--impl", "reference", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
