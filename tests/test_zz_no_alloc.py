"""The allocation-free routing entry point, through the C ABI (GPU).

moe_route_sort_noalloc serves callers that cannot allocate device memory;
its scratch lives in a static device array inside the library.  Its results
must equal moe_route_sort's bit for bit (indices), on two calls in a row with
different routings, so that nothing left in the shared array from one call
leaks into the next.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp4_sort_gb300 as fm
from block_scaled_fp4_sort_gb300.buffers import MoEBuffers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_scaled_fp4_sort_gb300 import build
    build.build()


def _ids(M, E, k, seed, hot=False):
    rng = np.random.default_rng(seed)
    ids = np.argsort(rng.random((M, E)), axis=1)[:, :k].astype(np.int32)
    if hot:
        ids[: M // 4, 0] = 3
    return torch.from_numpy(np.ascontiguousarray(ids)).cuda()


def _noalloc(p, B, ids, error_flag=None):
    R = p.num_tokens * p.top_k
    out = dict(e2p=torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda"),
               p2e=torch.full((B.S,), -7, dtype=torch.int32, device="cuda"),
               te=torch.full((B.tiles,), -7, dtype=torch.int32, device="cuda"),
               tm=torch.full((B.tiles,), -7, dtype=torch.int32, device="cuda"),
               nt=torch.zeros(4, dtype=torch.int32, device="cuda"),
               cnt=torch.zeros(p.num_local_experts or p.num_experts, dtype=torch.int32, device="cuda"))
    fm.moe_route_sort_noalloc(p, ids, out["e2p"], out["p2e"], out["te"], out["tm"], out["nt"],
                              out["cnt"], error_flag)
    return out


def _same(B, o, R):
    assert int(o["nt"][0]) == int(B.num_tiles[0])
    assert torch.equal(o["e2p"][:R], B.e2p[:R])
    assert torch.equal(o["p2e"], B.p2e)
    assert torch.equal(o["te"], B.tile_expert)
    assert torch.equal(o["tm"], B.tile_mn)
    assert torch.equal(o["cnt"], B.counts)


@pytest.mark.parametrize("M,E,k,T", [(20000, 256, 8, 64), (8, 256, 8, 16)])
def test_noalloc_route_sort_matches_workspace_version_twice(M, E, k, T):
    p = fm.problem(M, 256, 256, E, k, route_tile=T)
    for seed in (1, 2):                       # two calls in a row, different routings
        ids = _ids(M, E, k, seed, hot=seed == 2)
        B = MoEBuffers(p)
        B.route(ids)
        o = _noalloc(p, B, ids)
        torch.cuda.synchronize()
        _same(B, o, M * k)
        assert fm.read_error(B.route_ws) == 0


def test_noalloc_reports_bad_ids_and_rejects_oversized_problems():
    p = fm.problem(3, 256, 256, 8, 2)
    ids = torch.tensor([[0, 1], [7, 9], [-1, 2]], dtype=torch.int32, device="cuda")
    flag = torch.full((4,), 123, dtype=torch.int32, device="cuda")
    B = MoEBuffers(p)
    o = _noalloc(p, B, ids, flag)
    torch.cuda.synchronize()
    assert int(flag[0]) == fm.ERR_DEVICE
    e2p = o["e2p"][:6].cpu().numpy()
    assert e2p[3] == -1 and e2p[4] == -1
    big = fm.problem(2_000_000, 256, 256, 2048, 8, route_tile=128)   # 3907 chunks x 2048 experts
    with pytest.raises(fm.Fp4MoeError) as ei:
        fm.moe_route_sort_noalloc(big, ids, o["e2p"], o["p2e"], o["te"], o["tm"], o["nt"])
    assert ei.value.status == fm.ERR_UNSUPPORTED
