"""The N > 1 host logic of bench.py on CPU: two gloo ranks (world size 2).

The decode path does not shard: `bench.py --gpus N` runs N independent replicas,
each routing its own tokens, and reports the whole job's bytes over the slowest
rank's time.  These ranks run that bookkeeping with the gloo backend; no GPU and
no kernel is involved.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    import bench
    from rotated_codebook_quantized_gb300 import workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(torch, times[rank], world, torch.device("cpu"))
        logits = wl.router_logits(bench.rank_seed(rank), 3, bench.E)
        q.put((rank, t, bench.job_gbs(world, 50, 114720768, t), logits))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_route_their_own_tokens():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [3.25, 4.5]  # ms: rank 1 is the slower
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(2):
            r, t, v, logits = q.get(timeout=120)
            got[r] = (t, v, logits)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for r in range(2):
        t, v, _ = got[r]
        assert t == 4.5  # every rank sees the job time: the max over ranks
        assert v == pytest.approx(2 * 50 * 114720768 / 4.5e-3 / 1e9)  # both ranks' bytes over it
    # each replica routes its own tokens, deterministically
    assert not np.array_equal(got[0][2], got[1][2])
    import bench
    from rotated_codebook_quantized_gb300 import workloads as wl

    np.testing.assert_array_equal(got[1][2], wl.router_logits(bench.rank_seed(1), 3, bench.E))


def test_one_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(torch, 2.5, 1, torch.device("cpu")) == 2.5
    assert bench.job_gbs(1, 10, 1000, 1.0) == pytest.approx(10 * 1000 / 1e-3 / 1e9)
