"""bench.py's multi-process path on the CPU (gloo, world size 2): the job's time per step is the
slowest rank's, the job's throughput counts every rank's tokens, and the reference arm runs on
rank 0 only."""
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


def _rank_main(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=2)
    own = [1.25, 2.5][rank]
    ms = bench.slowest_rank_ms(own, 2, "cpu")
    q.put((rank, ms, bench.job_tokens_per_s(2, 8, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in out] == [0, 1]
    for _, ms, value in out:
        assert ms == 2.5
        assert abs(value - 2 * 8 / 2.5e-3) < 1e-6


def test_single_rank_keeps_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(3.0, 1, "cpu") == 3.0
    assert bench.job_tokens_per_s(1, 512, 0.5) == 512 / 0.5e-3


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
