"""The multi-rank host path of bench.py on CPU: two gloo ranks, as torchrun would launch them on
two GPUs.  Each rank builds its own batch of the workload (distinct seeds, same shape), the ranks
agree on the maximum of their timings, and nothing else is exchanged."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from pkv_inputs import workloads as W

        cfg = W.CONFIGS[3]
        step = W.make_step(cfg, bench.rank_seed(cfg, rank))
        elapsed = 1.0 + rank  # stand-in for each rank's measured time
        worst = bench.reduce_max(elapsed, world)
        q.put((rank, bench.rank_seed(cfg, rank), step.kv_bytes(), int(step.seq_len.sum()), worst))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_build_distinct_batches_and_agree_on_the_max_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    (r0, seed0, kv0, tok0, worst0), (r1, seed1, kv1, tok1, worst1) = res
    assert seed0 != seed1 and tok0 != tok1, "each rank must own a distinct batch"
    assert worst0 == worst1 == 2.0
    from pkv_inputs import workloads as W

    assert seed0 == W.SEED_BASE + 3  # rank 0 runs the standard workload
