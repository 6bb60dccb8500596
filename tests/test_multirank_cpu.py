"""The benchmark's multi-rank bookkeeping on CPU ranks (gloo, world size 2):
every rank draws its own batch (distinct seeds, distinct inputs: the units
shard with no exchange) and every rank ends up with the slowest rank's step
time, from which the whole-job rate is formed."""
import os
import socket

import torch
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        from kimi_delta_attention_rule_gb300 import inputs
        ms = bench.max_over_ranks(1.5 + rank, WORLD, "cpu")  # rank 1 is the slow one
        seed = bench.rank_seed(bench.PREFILL["seed"], rank)
        x = inputs.prefill_inputs([64], H=2, io="bf16", seed=seed)
        units = 2 * 64 * WORLD  # every rank's head-tokens
        q.put((rank, ms, seed, float(x.q.float().sum()), units / (ms * 1e-3) / 1e6))
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks_shard_and_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in range(WORLD))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, s0, sum0, rate0), (r1, ms1, s1, sum1, rate1) = res
    assert (r0, r1) == (0, 1)
    assert ms0 == ms1 == 2.5                # both see the slowest rank's time
    assert s0 != s1 and sum0 != sum1        # independent batches
    assert rate0 == rate1 == 2 * 64 * 2 / 2.5e-3 / 1e6


def test_one_rank_is_its_own_maximum():
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.rank_seed(5, 0) == 5
