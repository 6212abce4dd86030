"""The N > 1 path of bench.py on CPU: two gloo ranks combine their timings
(max over ranks) and the job-wide value counts every rank's units."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = [1.0 + rank, 2.0 - rank, 0.5 * (rank + 1), 0.25]
    got = bench.combine_ranks(times)
    stats = dict(ms=got[0], e2e_ms=got[1], dec_ms=got[2], app_ms=got[3], dec_b=1e9, app_b=1e6,
                 kv_tokens=1e6, h2d=10, d2h=20, clocks=None, fill_s=0.0, L=2, B=4, lens=[], ws_bytes=0)

    class A:
        workload = "qwen2.5-7b-32k"
        steps = 3
        warmup = 3
        layers = 2
    line = bench.report_ours(A, stats, world, None)
    q.put((rank, got, line["value"], line["n_gpus"], line["scaling"]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value, n, scaling in res:
        assert got == [2.0, 2.0, 1.0, 0.25]
        # value = both ranks' bytes over the slowest rank's step time
        assert value == pytest.approx(2 * (1e9 + 1e6) / (2.0e-3) / 1e9, rel=1e-3)
        assert n == 2 and scaling == "weak"
