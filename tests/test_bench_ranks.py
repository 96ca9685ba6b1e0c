"""The multi-GPU bench path (independent replicas, one process per GPU) on CPU:
the whole-job aggregation over world_size 2 with the gloo backend, and the
reference arm's non-zero ranks leaving without work."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [10.0, 12.5][rank]
        tokens = [100, 150][rank]
        e2e = [11.0, 13.0][rank]
        out[rank] = bench.reduce_over_ranks(elapsed, tokens, e2e, "cpu")
        out[2 + rank] = bench.reduce_over_ranks(elapsed, tokens, None, "cpu")
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    # slowest rank's time, all ranks' tokens, slowest e2e step
    assert res[0] == res[1] == (12.5, 250, 13.0)
    assert res[2] == res[3] == (12.5, 250, None)


def test_single_process_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.0, 7, 4.0, "cpu") == (3.0, 7, 4.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_gpu_count_must_match_the_launcher():
    """Under a launcher, --gpus N must equal WORLD_SIZE (a mismatch would report
    the wrong job size); the run stops with a non-zero code before any work."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="3", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "WORLD_SIZE 3" in r.stderr
