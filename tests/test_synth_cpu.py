"""The seeded synthetic workloads match the recipe they are documented with:
routing statistics of every configuration at seed 0, the route tile the
benchmarks pick, and the model-load NVFP4 / MXFP4 quantisers checked code by
code with the oracle's own E2M1 / E4M3 / E8M0 decoders (no GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.moe_inputs import generate_routing, quantize_mxfp4, quantize_nvfp4, route_tile_for


def _counts(cfg):
    ids, w = generate_routing(cfg)
    assert ids.shape == (cfg.M, cfg.top_k) and w.shape == (cfg.M, cfg.top_k)
    assert ids.dtype == np.int32 and w.dtype == np.float32
    assert ids.min() >= 0 and ids.max() < cfg.E
    # top-k picks distinct experts; the weights are a positive partition of 1
    assert all(len(set(r)) == cfg.top_k for r in ids.tolist())
    assert (w > 0).all() and np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    return np.bincount(ids.ravel(), minlength=cfg.E)


@pytest.mark.parametrize("name", sorted(synth.CONFIGS))
def test_routing_draw_is_valid_and_seeded(name):
    cfg = synth.CONFIGS[name]
    a = generate_routing(cfg)
    b = generate_routing(cfg)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    c = generate_routing(cfg.with_(seed=1))
    assert not np.array_equal(a[0], c[0])
    _counts(cfg)


def test_workload_statistics():
    dec = _counts(synth.CONFIGS["decode_w4a16"])
    assert (dec > 0).sum() == 60                          # experts touched by 8 tokens x 8
    sk = _counts(synth.CONFIGS["skewed_w4a16"])
    assert (sk == 0).sum() == 8 and sk.max() == 875       # 8 experts never win
    assert abs(np.sort(sk)[::-1][:13].sum() / sk.sum() - 0.52) < 0.01
    lg = _counts(synth.CONFIGS["large_w4a16"])
    mean = lg.sum() / lg.size                             # 4096 routes per expert
    assert mean == 4096 and np.abs(lg - mean).max() < 0.06 * mean
    pf = _counts(synth.CONFIGS["prefill_w4a4"])
    assert (pf > 0).all()


def test_route_tiles():
    got = {n: route_tile_for(c) for n, c in synth.CONFIGS.items()}
    # the benchmarks' tile is the library's automatic choice
    import block_scaled_fp4_sort_gb300 as fm
    from block_scaled_fp4_sort_gb300.buffers import problem_for
    for n, c in synth.CONFIGS.items():
        assert fm.route_tile(problem_for(c, 0)) == got[n], n
    assert got == {"tiny_w4a16": 16, "decode_w4a16": 16, "prefill_w4a4": 128, "skewed_w4a16": 128,
                   "prefill_w4a8": 128, "large_w4a16": 128}


def _half_spacing(a):
    # half the distance to the neighbouring E2M1 magnitudes around |v| <= 6
    return np.where(a < 2.0, 0.25, np.where(a < 4.0, 0.5, 1.0))


def test_nvfp4_model_load_quantiser():
    g = torch.Generator().manual_seed(7)
    w = torch.randn(24, 128, generator=g) * 0.02
    w[3, 16:32] = 0.0                                     # an all-zero block
    q, sf, gs = quantize_nvfp4(w)
    gs = float(gs)
    assert abs(gs - 2688.0 / float(w.abs().max())) <= 1e-6 * gs
    wn = w.numpy().astype(np.float64)
    qn, sfn = q.numpy(), sf.numpy()
    for r in range(w.shape[0]):
        for b in range(w.shape[1] // 16):
            blk = wn[r, 16 * b:16 * b + 16]
            s = oracle.e4m3_value(int(sfn[r, b]))
            # the block scale is E4M3(amax_blk / 6 * gs), the product taken in fp32
            # as the generator takes it, rounded to E4M3 as the oracle rounds
            pre = np.float32(np.float32(np.abs(blk).max()) / np.float32(6.0)) * np.float32(gs)
            assert s == oracle.round_e4m3(float(pre))
            for i in range(16):
                k = 16 * b + i
                code = int(qn[r, k // 2] >> (4 * (k % 2))) & 15
                v = oracle.e2m1_value(code)
                if s == 0:
                    assert v == 0.0
                    continue
                target = min(abs(blk[i] * gs / s), 6.0)
                assert abs(abs(v) - target) <= _half_spacing(target) + 1e-6
                assert v == 0.0 or np.sign(v) == np.sign(blk[i])


def test_mxfp4_model_load_quantiser():
    g = torch.Generator().manual_seed(8)
    w = torch.randn(8, 128, generator=g) * 0.05
    q, e8 = quantize_mxfp4(w)
    wn = w.numpy().astype(np.float64)
    qn, en = q.numpy(), e8.numpy()
    for r in range(w.shape[0]):
        for b in range(w.shape[1] // 32):
            blk = wn[r, 32 * b:32 * b + 32]
            s = oracle.ue8m0_value(int(en[r, b]))
            # 2^(floor(log2 amax) - 2): the block maximum lands in [4, 8)
            assert 4.0 <= np.abs(blk).max() / s < 8.0
            for i in range(32):
                k = 32 * b + i
                code = int(qn[r, k // 2] >> (4 * (k % 2))) & 15
                target = min(abs(blk[i] / s), 6.0)
                assert abs(abs(oracle.e2m1_value(code)) - target) <= _half_spacing(target) + 1e-6
