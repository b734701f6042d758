"""The replicas-only multi-GPU path of ``bench.py``, on CPU with two gloo ranks.

A decode step does not shard: each GPU runs an independent replica, and the only
cross-rank steps are host-side. The timed region ends with a barrier, ``value`` is the
tokens of all ranks over the slowest rank's time, and rank 0 alone prints. Two ``gloo``
ranks run the same helpers that the torchrun launch uses: the environment read, the
max-reduction of the step time, the sum of the tokens and the barrier.
"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, w, lr = bench.dist_env()
        slowest = bench.max_over_ranks(1.5 + rank, w)          # per-rank step times
        tokens = bench.sum_over_ranks(10.0 * (rank + 1), w)     # per-rank tokens
        bench.barrier(w)
        q.put((rank, r, w, lr, slowest, tokens))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, r, w, lr, slowest, tokens in results:
        assert (r, w, lr) == (rank, 2, rank)
        assert slowest == 2.5      # the max over the ranks, on every rank
        assert tokens == 30.0      # the sum over the ranks, on every rank


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    bench.barrier(1)   # no process group: a no-op
