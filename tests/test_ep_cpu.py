"""Expert parallelism on the CPU: the partition of the experts over ranks and
the one exchange step (an all-reduce of fp32 partial outputs), run as two
gloo ranks on 127.0.0.1.

Each rank evaluates the oracle on its own expert range only (routes to other
experts dropped, as the library's routing plan drops them); the ranks sum
their exact partials through ep_step's all-reduce, and the sum must equal
the oracle over all experts."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_scaled_fp4_sort_gb300.ep import ep_step, expert_range


@pytest.mark.parametrize("E,world", [(8, 2), (256, 8), (7, 3), (3, 4), (1, 1)])
def test_expert_ranges_partition_the_experts(E, world):
    seen = []
    for r in range(world):
        off, cnt = expert_range(E, world, r)
        assert cnt in (E // world, E // world + 1)
        seen += list(range(off, off + cnt))
    assert seen == list(range(E))


def test_expert_range_rejects_bad_ranks():
    with pytest.raises(ValueError):
        expert_range(8, 2, 2)
    with pytest.raises(ValueError):
        expert_range(8, 0, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, cfg_name, E, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import synth
        cfg = synth.CONFIGS[cfg_name].with_(E=E)
        inp = synth.generate(cfg)
        off, cnt = expert_range(cfg.E, world, rank)
        # the rank holds only its experts' weights (local expert l = global off + l)
        import dataclasses
        sl = slice(off, off + cnt)
        local = dataclasses.replace(inp, w1=inp.w1[sl], w1_sf=inp.w1_sf[sl], w2=inp.w2[sl],
                                    w2_sf=inp.w2_sf[sl], w1_alpha=inp.w1_alpha[sl],
                                    w2_alpha=inp.w2_alpha[sl])
        orc = oracle.OracleMoE.from_inputs(local, T=16, E_local=cnt, offset=off)
        _, exact_local, _ = orc.forward(rsf=0.5)
        got = {}

        def local_partial():
            return torch.from_numpy(exact_local.copy())

        def combine(t):
            got["sum"] = t.numpy().copy()

        ep_step(local_partial, lambda t: dist.all_reduce(t, op=dist.ReduceOp.SUM), combine)
        if rank == 0:
            full_bits, full_exact, _ = oracle.OracleMoE.from_inputs(inp, T=16).forward(rsf=0.5)
            q.put((got["sum"], full_exact, full_bits, exact_local))
        else:
            q.put(None)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("E", [8, 5])
def test_two_ranks_sum_to_the_full_forward(E):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, "tiny_w4a16", E, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    summed, full_exact, full_bits, part0 = next(r for r in res if r is not None)
    # each rank holds only part of the result; the all-reduced sum is the
    # whole forward (double sums in another order: equal to rounding)
    assert np.abs(part0 - full_exact).max() > 1e-3
    assert np.allclose(summed, full_exact, rtol=1e-12, atol=1e-15)
    # rounded once to BF16 it is the oracle's output
    rounded = torch.from_numpy(summed).to(torch.float32).to(torch.bfloat16)
    bits = rounded.view(torch.int16).numpy().view(np.uint16)
    assert np.mean(bits == full_bits) > 0.999
