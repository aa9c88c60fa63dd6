"""Host logic of the gather-locality measurement (`bench.py --locality`, the
pages' M1/M2 table of distinct 2 MiB pages of x touched per GEMM1 tile): page
counting, per-expert route groups and the arrival-order model, on small
routing plans from the oracle (no GPU)."""
import numpy as np

import bench
import oracle


def _plan(M=64, E=8, k=2, T=16, seed=1):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(M)]).astype(np.int32)
    r = oracle.route_plan(M, E, k, T, ids)
    plan = dict(p2e=r["permuted_idx_to_expanded_idx"], tile_expert=r["tile_idx_to_expert"],
                tile_mn=r["tile_idx_to_mn_limit"], num_tiles=r["num_non_exiting_tiles"])
    return ids, plan


def test_pages_per_tile_hand_cases():
    page = 1 << 12
    top_k = 2
    # slots holding routes 0..7 -> tokens 0..3; rows of page/4 bytes: one page
    g = np.arange(8, dtype=np.int32)
    assert list(bench.pages_per_tile([g], top_k, page // 4, page)) == [1]
    # tokens 0 and 8 with rows of page/4 bytes: pages 0 and 2
    g = np.array([0, 16, -1, -1], dtype=np.int32)
    assert list(bench.pages_per_tile([g], top_k, page // 4, page)) == [2]
    # a row of 3/4 page starting at 3/4 page straddles pages 0 and 1 and reaches page 1 only
    g = np.array([2], dtype=np.int32)     # token 1
    assert list(bench.pages_per_tile([g], top_k, 3 * page // 4, page)) == [2]
    # groups holding only padding are skipped
    assert bench.pages_per_tile([np.array([-1, -1], dtype=np.int32)], top_k, 64, page).size == 0


def test_expert_groups_partition_each_experts_routes():
    ids, plan = _plan()
    p2e, te, tm, nt = plan["p2e"], plan["tile_expert"], plan["tile_mn"], int(plan["num_tiles"])
    groups = bench.expert_groups(p2e, te, tm, nt, 16, 5)
    seen = np.concatenate(groups)
    # every valid route exactly once, no padding
    assert np.array_equal(np.sort(seen), np.arange(ids.size))
    for g in groups:
        assert 1 <= g.size <= 5
        experts = ids.reshape(-1)[g]
        assert np.all(experts == experts[0])       # one expert per group
        assert np.all(np.diff(g) > 0)              # stable order kept


def test_arrival_model_permutes_within_experts_only():
    ids, plan = _plan(M=96)
    p2e, te, tm, nt = plan["p2e"], plan["tile_expert"], plan["tile_mn"], int(plan["num_tiles"])
    sh = bench.shuffled_within_experts(p2e, te, tm, nt, 16, seed=3)
    assert np.array_equal(sh[p2e < 0], p2e[p2e < 0])          # padding untouched
    flat = ids.reshape(-1)
    for e in np.unique(flat):
        mine = p2e >= 0
        a = p2e[mine & (flat[np.maximum(p2e, 0)] == e)]
        b = sh[mine & (flat[np.maximum(p2e, 0)] == e)]
        assert np.array_equal(np.sort(a), np.sort(b))          # same routes per expert
        assert np.all(flat[b] == e)
    assert not np.array_equal(sh, p2e)                         # something moved
    again = bench.shuffled_within_experts(p2e, te, tm, nt, 16, seed=3)
    assert np.array_equal(sh, again)                           # seeded
