"""The multi-rank host logic of bench.py, on CPU with two gloo ranks.

Streams are independent, so under torchrun every rank runs its own streams (weak
scaling) with no collective on the data path; the only collectives are the barrier and
the max-over-ranks of the timed region.  Checked here: the ranks draw different inputs,
their streams partition the global batch (each (b, h) exactly once), every rank sees the
slowest rank's time, and the whole-job rate counts the units of all ranks over that time.
"""

import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    import bench
    import sdm_inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = sdm_inputs.CONFIGS["tiny"]
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        d = sdm_inputs.make_inputs(cfg, seed=bench.rank_seed(cfg, rank))
        # every rank's share of the global streams, gathered on every rank
        B, H = 3, 2
        mine = torch.tensor(bench.rank_streams(B, H, rank, world), dtype=torch.int64)
        parts = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        allst = sorted(tuple(x) for p_ in parts for x in p_.tolist())
        out.put((rank, ms, float(d["q_w"].double().sum()), float(d["k_val"].double().sum()), allst))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_shard_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    (r0, ms0, qw0, kv0, st0), (r1, ms1, qw1, kv1, st1) = got
    assert (r0, r1) == (0, 1)
    # the two ranks' streams cover the global batch's (b, h) exactly once
    assert st0 == st1 == [(b, h) for b in range(2 * 3) for h in range(2)]
    assert ms0 == ms1 == 15.0                      # the slowest rank's time, on every rank
    assert qw0 != qw1 and kv0 != kv1               # each rank runs its own streams


def test_whole_job_rate_counts_every_rank():
    import bench
    assert bench.whole_job_rate(8192, 2, 4.0) == 8192 * 2 / 4e-3
    assert bench.max_over_ranks(3.5, None, torch.device("cpu")) == 3.5
    import sdm_inputs
    cfg = sdm_inputs.CONFIGS["layer"]
    assert len({bench.rank_seed(cfg, r) for r in range(8)}) == 8
