"""bench.py with N > 1 replicas (torchrun): the job's time is the slowest rank's and its
rate counts every replica's weights; the reference arm does its work on rank 0 only.
Two gloo ranks on the CPU."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.slowest_rank_seconds(1.0 + rank, world, "cpu")      # rank 1 is the slower one
    rate = bench.job_rate_mweights(world, 10, 4096 * 4096, t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, t, rate))


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, rate in out:
        assert t == 2.0
        assert abs(rate - 2 * 10 * 4096 * 4096 / 2.0 / 1e6) < 1e-9


def test_single_replica_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_seconds(1.25, 1, "cpu") == 1.25
    assert bench.job_rate_mweights(1, 4, 1000, 2.0) == 4 * 1000 / 2.0 / 1e6


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(bench.argparse.Namespace(workload="llama_4096_g128", layer=0, steps=1, warmup=1, gpus=2,
                                                 threads=None, tokens=None))
    assert capsys.readouterr().out == ""
