"""The benchmark's multi-GPU path on the CPU: two ranks over gloo.

`bench.py --gpus N` runs one independent replica per rank (weak scaling, no
collective on the data path); ranks meet only to take the slowest rank's time.
These tests run that host logic with world_size 2 on 127.0.0.1."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        slowest = bench.max_over_ranks(1.5 + r, w)               # per-rank "milliseconds"
        cfg = bench.replica_cfg(synth.CONFIGS["tiny_w4a16"], r)
        ids, _ = synth.generate_routing(cfg)
        got = torch.tensor([float(ids.sum())], dtype=torch.float64)
        gathered = [torch.zeros(1, dtype=torch.float64) for _ in range(w)]
        dist.all_gather(gathered, got)
        q.put((r, w, local, slowest, cfg.seed, [float(g.item()) for g in gathered]))
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def test_ranks_see_their_environment(two_ranks):
    assert [(r, w, l) for r, w, l, *_ in two_ranks] == [(0, 2, 0), (1, 2, 1)]


def test_job_time_is_the_slowest_rank(two_ranks):
    assert [t[3] for t in two_ranks] == [2.5, 2.5]


def test_replicas_draw_independent_batches(two_ranks):
    seeds = [t[4] for t in two_ranks]
    assert seeds == [0, 1]
    sums = two_ranks[0][5]
    assert sums[0] != sums[1]            # different routing per rank


def test_whole_job_throughput_counts_every_rank():
    assert bench.tokens_per_s(1, 8, 0.5) == pytest.approx(16000.0)
    assert bench.tokens_per_s(4, 8, 0.5) == pytest.approx(64000.0)
    assert bench.max_over_ranks(3.0, 1) == 3.0
