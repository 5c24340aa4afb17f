"""Host logic of the benchmark's multi-rank path, on CPU: world size 2 over
gloo (every rank runs its own copy of the workload; the job's time is the
slowest rank's)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, times, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(times[rank])
    v = bench.whole_job_gbs(10 ** 9, world, t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, t, v))


def test_max_over_ranks_and_whole_job_value():
    world, port = 2, _free_port()
    times = [0.004, 0.005]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == max(times)
        assert v == pytest.approx(2 * 1e9 / 0.005 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.whole_job_gbs(2 * 10 ** 9, 1, 0.5) == pytest.approx(4.0)


def test_reference_arm_other_ranks_exit(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(workload="tiny", steps=1, warmup=0, gpus=2)
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
