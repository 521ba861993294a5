"""Multi-process host logic of bench.py, on CPU: two gloo ranks on 127.0.0.1.

Each GPU runs an independent replica of the path (no data-path collective);
the timed region is bracketed by barriers and its duration is the maximum
over ranks, and the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_info()
    dist = bench.init_dist(w, "gloo")
    dist.barrier()
    # a slower rank 1: every rank must report rank 1's time
    ms = bench.max_over_ranks(dist, 1.0 + 2.5 * r, "cpu")
    dist.barrier()
    q.put((r, w, local, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert [(r, w, local) for r, w, local, _ in res] == [(0, 2, 0), (1, 2, 1)]
    assert [ms for *_, ms in res] == [3.5, 3.5]


def test_single_process_needs_no_process_group():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 1.25, "cpu") == 1.25


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
