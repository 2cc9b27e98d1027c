"""The N > 1 path of bench.py on CPU: two gloo ranks, replica timing logic
(barrier, max over ranks, whole-job value = ranks x work / slowest time)."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    r, w, local = bench.dist_setup(None)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    t = bench.max_over_ranks(1.0 + rank, w)   # rank 1 is the slower one
    out[rank] = t
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.0, 1: 2.0}


def test_reference_arm_other_ranks_exit_without_work(capsys):
    import argparse

    import bench
    args = argparse.Namespace(workload=bench.DEFAULT_WORKLOAD, steps=3, warmup=3)
    bench.reference_arm(args, rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_flop_count_matches_definition():
    import bench
    assert bench.attention_flops(4, 16, 4096, 4096, 128, False) == 4.0 * 4 * 16 * 4096 * 4096 * 128
    assert bench.attention_flops(1, 64, 32768, 32768, 128, True) == 2.0 * 64 * 32768 ** 2 * 128


def test_bench_rejects_too_few_warmups():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
