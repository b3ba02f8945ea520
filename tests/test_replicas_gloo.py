"""The multi-rank (replica) host logic of bench.py on CPU with gloo, world
size 2: every rank serves its own seeded batch, the job time is the slowest
rank's, and the job rate counts all ranks' bytes. No data-path collective
exists: ranks only exchange their timings."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = synth.decode_config("qwen3_4b", seed=bench.rank_seed(rank), layers=1)
    my_ms = 10.0 + 5.0 * rank
    ms = bench.max_over_ranks(my_ms, dist)
    total = bench.sum_over_ranks(cfg.kv_bytes_step(), dist)
    rate = bench.job_rate(total, ms)
    q.put((rank, ms, rate, cfg.kv_bytes_step(), int(cfg.seq_len.sum()), total))
    dist.destroy_process_group()


def test_replica_timing_reduction_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    assert res[0][1] == res[1][1] == 15.0          # slowest rank's time on both
    assert res[0][2] == pytest.approx(res[1][2])   # same job rate reported
    assert res[0][4] != res[1][4]                  # each rank decodes its own batch
    assert res[0][5] == res[1][5] == res[0][3] + res[1][3]   # bytes of all ranks
    assert res[0][2] == pytest.approx((res[0][3] + res[1][3]) / 15e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.sum_over_ranks(7.0, None) == 7.0
    assert bench.job_rate(10 ** 9, 1000.0) == pytest.approx(1.0)
