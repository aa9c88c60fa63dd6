"""Pins of the CPU oracle against things other than itself (no GPU needed).

What pins what:
  codecs       E2M1 table (OCP MX spec, tests/golden), E4M3 and bf16 decode
               against torch's float8_e4m3fn / bfloat16 conversions (all codes),
               rounding against torch's RNE conversions and hand RNE cases.
  quantiser    round trips, amax = 0 blocks, saturation, a hand-worked block.
  route sort   histogram (np.bincount), bijection, stable order, tile formulas,
               brute force with Python's stable sorted() on tiny inputs.
  forward      dense per-token evaluation with numpy matmuls over weights
               decoded by the test itself (P4), the E=1/top_k=1 dense MLP via
               torch.matmul (P5), accumulate=False == zero seed bit for bit and
               an expert-parallel split (P6), SwiGLU against scipy's expit.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

from ref_decode import (E2M1_TABLE, _golden, bf16_np, dequant_np, e4m3_np,  # noqa: F401
                        to_bf16_torch)


# ---------------------------------------------------------------- P1: codecs

def test_e2m1_values_match_ocp_table():
    for code, val in _golden("e2m1_values.txt"):
        got = oracle.e2m1_value(int(code))
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)


def test_e4m3_all_codes_match_torch():
    ref = e4m3_np(np.arange(256, dtype=np.uint8))
    for c in range(256):
        got = oracle.e4m3_value(c)
        if np.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_bf16_all_codes_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_np(bits)
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _fp32_samples(rng, n):
    exps = rng.integers(-140, 128, n)
    mant = rng.random(n) + 1.0
    v = (mant * np.exp2(exps.astype(np.float64))).astype(np.float32)
    v *= np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    # exact bf16 midpoints (ties) and their neighbours
    mids = (np.arange(1000, dtype=np.uint32) * 7919 % 0x7F00 << 16 | 0x8000).view(np.float32)
    return np.concatenate([v, mids, np.nextafter(mids, np.float32(np.inf))])


def test_round_bf16_matches_torch_rne():
    rng = np.random.default_rng(1)
    v = _fp32_samples(rng, 20000)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(x)) for x in v])
    assert np.array_equal(got, ref)
    bits = np.array([oracle.bf16_bits(float(x)) for x in v], np.uint32).astype(np.uint16)
    ref_bits = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref_bits)


def test_round_e4m3_matches_torch_rne_in_range():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, 20000))).astype(np.float32)
    v = v[np.abs(v) < 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.round_e4m3(float(x)) for x in v])
    assert np.array_equal(got, ref)
    # satfinite: clamp to the largest finite magnitude; 464 is the 448/480 tie -> 448 (even)
    for x, want in [(449.0, 448.0), (464.0, 448.0), (1e9, 448.0), (-1e9, -448.0), (2.0 ** -10, 0.0),
                    (3 * 2.0 ** -11, 2.0 ** -9)]:
        assert oracle.round_e4m3(x) == want, x
    for c in range(0x7F):
        assert oracle.e4m3_code(oracle.e4m3_value(c)) == c


def test_e2m1_rne_cases():
    for x, want in _golden("e2m1_rne_cases.txt"):
        assert oracle.round_e2m1(x) == want, (x, oracle.round_e2m1(x), want)
    for c in range(16):
        if c == 8:
            continue
        assert oracle.e2m1_code(oracle.e2m1_value(c)) == c


def test_e2m1_times_e4m3_is_exact_in_bf16():
    """Every E2M1*E4M3 product is a BF16 value, so a decode to BF16 loses nothing."""
    e2 = E2M1_TABLE[:8]
    e4 = e4m3_np(np.arange(0x7F, dtype=np.uint8))
    prods = np.outer(e2, e4).ravel()
    assert np.array_equal(to_bf16_torch(prods), prods)


# ---------------------------------------------------------------- P2: quantiser

def test_nvfp4_quantizer_hand_block():
    # amax 6 at s = 1: sf = E4M3(6/6) = 1.0 (code 0x38); codes are the values themselves
    h = np.array([6, -3, 1.5, 0.5, 0, 2, 4, -6, 1, -1, 0.25, 0.75, 5, 3.5, -2.5, 1.25], np.float32)
    q, sf = oracle.nvfp4_quantize_f32(h, 1.0)
    assert sf[0] == 0x38
    vals = dequant_np(q, sf)
    want = [6, -3, 1.5, 0.5, 0, 2, 4, -6, 1, -1, 0, 1, 4, 4, -2, 1]   # RNE ties -> even codes
    assert list(vals) == want


def test_nvfp4_quantizer_zero_block_and_saturation():
    q, sf = oracle.nvfp4_quantize_f32(np.zeros(16, np.float32), 4.0)
    assert sf[0] == 0 and np.all(q == 0)
    # amax*s/6 beyond 448 saturates the scale to 448
    h = np.full(16, 1e6, np.float32)
    q, sf = oracle.nvfp4_quantize_f32(h, 1.0)
    assert oracle.e4m3_value(int(sf[0])) == 448.0
    assert np.all(dequant_np(q, sf) == 6 * 448.0)


def test_nvfp4_quantizer_roundtrip_on_grid():
    rng = np.random.default_rng(3)
    for _ in range(50):
        codes = rng.integers(0, 16, 16)
        codes[rng.integers(0, 16)] = 7          # amax exactly 6 * scale
        scale_code = int(rng.integers(0x20, 0x70))
        s = oracle.e4m3_value(scale_code)
        h = (E2M1_TABLE[codes] * s).astype(np.float32)
        q, sf = oracle.nvfp4_quantize_f32(h, 1.0)
        assert int(sf[0]) == scale_code
        assert np.array_equal(dequant_np(q, sf), h.astype(np.float64))


# ---------------------------------------------------------------- P3: routing

def _route(ids, E, k, T, E_local=None, offset=0):
    M = ids.shape[0]
    E_local = E if E_local is None else E_local
    o = oracle.OracleMoE(M, 128, 128, E, k, ids, np.ones_like(ids, np.float32),
                         np.zeros((E_local, 256, 64), np.uint8), np.zeros((E_local, 256, 8), np.uint8),
                         np.ones(E_local, np.float32), np.zeros((E_local, 128, 64), np.uint8),
                         np.zeros((E_local, 128, 8), np.uint8), np.ones(E_local, np.float32),
                         x=np.zeros((M, 128), np.uint16), E_local=E_local, offset=offset, T=T)
    return o.route_sort()


def _check_plan(plan, ids, E, T, E_local=None, offset=0):
    E_local = E if E_local is None else E_local
    flat = ids.ravel()
    R = flat.size
    local = (flat >= offset) & (flat < offset + E_local)
    loc = np.where(local, flat - offset, -1)
    cnt = np.bincount(loc[local], minlength=E_local)
    assert np.array_equal(plan["expert_counts"], cnt)               # histogram
    pad = -(-cnt // T) * T
    off = np.concatenate([[0], np.cumsum(pad)])
    assert plan["num_non_exiting_tiles"] * T == off[-1]
    S = oracle.max_permuted_slots(R, E_local, T)
    assert S >= off[-1] and S % T == 0
    e2p = plan["expanded_idx_to_permuted_idx"].ravel()
    p2e = plan["permuted_idx_to_expanded_idx"]
    assert p2e.size == S
    assert np.all(e2p[~local] == -1)
    valid = e2p[local]
    assert np.unique(valid).size == valid.size                        # injective
    assert np.array_equal(p2e[valid], np.nonzero(local)[0])           # inverse maps agree
    assert np.sum(p2e >= 0) == local.sum()                            # nothing else is valid
    for e in range(E_local):
        rows = p2e[off[e]:off[e] + cnt[e]]
        assert np.all(loc[rows] == e) and np.all(np.diff(rows) > 0)  # own expert, stable order
        assert np.all(p2e[off[e] + cnt[e]:off[e + 1]] == -1)         # padding
        for tt in range(off[e] // T, off[e + 1] // T):
            assert plan["tile_idx_to_expert"][tt] == e
            assert plan["tile_idx_to_mn_limit"][tt] == min(tt * T + T, off[e] + cnt[e])
    nt = plan["num_non_exiting_tiles"]
    assert np.all(plan["tile_idx_to_expert"][nt:] == -1)


@pytest.mark.parametrize("M,E,k,T,seed", [(16, 8, 2, 16, 0), (8, 256, 8, 16, 1), (300, 32, 4, 32, 2),
                                          (1000, 64, 6, 128, 3), (1, 1, 1, 16, 4), (50, 4, 4, 64, 5)])
def test_route_sort_invariants(M, E, k, T, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    _check_plan(_route(ids, E, k, T), ids, E, T)


def test_route_sort_skewed_and_duplicates():
    rng = np.random.default_rng(7)
    ids = rng.zipf(1.5, size=(500, 4)).astype(np.int32) % 16     # duplicates within a token too
    _check_plan(_route(ids, 16, 4, 16), ids, 16, 16)
    ids = np.zeros((100, 3), np.int32)                               # everything on expert 0
    _check_plan(_route(ids, 4, 3, 32), ids, 4, 32)


def test_route_sort_expert_parallel_and_invalid():
    rng = np.random.default_rng(8)
    ids = rng.integers(0, 32, (200, 4)).astype(np.int32)
    plan = _route(ids, 32, 4, 16, E_local=8, offset=12)
    _check_plan(plan, ids, 32, 16, E_local=8, offset=12)
    assert not plan["bad"]
    bad_ids = ids.copy()
    bad_ids[3, 1] = 32
    bad_ids[7, 0] = -5
    plan = _route(bad_ids, 32, 4, 16)
    assert plan["bad"]
    assert plan["expanded_idx_to_permuted_idx"][3, 1] == -1
    assert plan["expanded_idx_to_permuted_idx"][7, 0] == -1


def test_route_sort_bruteforce_tiny():
    rng = np.random.default_rng(9)
    for trial in range(20):
        M, E, k, T = int(rng.integers(1, 12)), int(rng.integers(1, 6)), 0, 16
        k = int(rng.integers(1, E + 1))
        ids = rng.integers(0, E, (M, k)).astype(np.int32)
        plan = _route(ids, E, k, T)
        order = sorted(range(M * k), key=lambda r: (ids.ravel()[r], r))    # stable by expert
        got = [int(r) for r in plan["permuted_idx_to_expanded_idx"] if r >= 0]
        assert got == order


def test_max_permuted_slots_bound():
    # the bound must hold for every routing of R routes over E experts
    for R, E, T in [(64, 256, 16), (32768, 256, 128), (8192, 128, 64), (5, 3, 16), (1, 1, 128)]:
        S = oracle.max_permuted_slots(R, E, T)
        worst = min(E, R) * (T - 1) + R           # each non-empty expert wastes < T slots
        assert S >= worst and S % T == 0 and S - worst < T


# ---------------------------------------------------------------- P4/P5/P6: forward

def _small_inputs(mode="w4a16", **kw):
    base = synth.CONFIGS["tiny_w4a16"] if mode == "w4a16" else synth.CONFIGS["prefill_w4a4"]
    cfg = base.with_(**kw) if kw else base
    if mode == "w4a4" and not kw:
        cfg = cfg.with_(M=16, H=256, I=128, E=8, top_k=2, sample=0)
    return synth.generate(cfg)


def _dense_reference(inp, orc, tokens):
    """numpy float64 evaluation, per token, with its own decode (P4)."""
    cfg = inp.cfg
    H, I = cfg.H, cfg.I
    w1 = dequant_np(inp.w1.numpy(), inp.w1_sf.numpy())      # [E, 2I, H]
    w2 = dequant_np(inp.w2.numpy(), inp.w2_sf.numpy())      # [E, H, I]
    a1 = inp.w1_alpha.double().numpy()
    a2 = inp.w2_alpha.double().numpy()
    ids = inp.token_selected_experts.numpy()
    wts = inp.token_final_scales.numpy().astype(np.float64)
    if inp.x is not None:
        X = inp.x.to(torch.float64).numpy()
    else:
        X = dequant_np(inp.x_q.numpy(), inp.x_sf.numpy())
    outs = []
    for t in tokens:
        acc = np.zeros(H)
        for j in range(cfg.top_k):
            e = ids[t, j]
            gu = a1[e] * (w1[e] @ X[t])
            g, u = gu[:I], gu[I:]
            h = g / (1.0 + np.exp(-g)) * u
            if inp.x is not None:
                hin = to_bf16_torch(h)
            else:
                st = orc.expert_ffn(e, t)       # quantiser pinned separately
                hin = dequant_np(st["hq"][None], st["hsf"][None])[0]
            acc += float(wts[t, j]) * (a2[e] * (w2[e] @ hin))
        outs.append(acc)
    return np.array(outs)


def test_forward_matches_dense_numpy_w4a16():
    inp = _small_inputs()
    orc = oracle.OracleMoE.from_inputs(inp)
    toks = np.arange(inp.cfg.M)
    bits, exact, bad = orc.forward(toks)
    ref = _dense_reference(inp, orc, toks)
    assert not bad
    # the two evaluations differ only in summation order and, rarely, in the
    # double-vs-(double->fp32->bf16) rounding of h; both are far below 1e-9 here
    np.testing.assert_allclose(exact, ref, rtol=1e-9, atol=1e-12)
    assert np.array_equal(bf16_np(bits), to_bf16_torch(exact)) or np.mean(
        bf16_np(bits) != to_bf16_torch(exact)) < 1e-3


def test_forward_matches_dense_numpy_w4a4():
    inp = _small_inputs("w4a4")
    orc = oracle.OracleMoE.from_inputs(inp)
    toks = np.arange(inp.cfg.M)
    _, exact, _ = orc.forward(toks)
    ref = _dense_reference(inp, orc, toks)
    np.testing.assert_allclose(exact, ref, rtol=1e-9, atol=1e-12)


def test_staged_values_swiglu_and_quantiser():
    inp = _small_inputs("w4a4")
    orc = oracle.OracleMoE.from_inputs(inp)
    from scipy.special import expit
    st = orc.expert_ffn(3, 5)
    np.testing.assert_allclose(st["h_pre"], st["g"] * expit(st["g"]) * st["u"], rtol=1e-13, atol=1e-300)
    q, sf = oracle.nvfp4_quantize_f32(st["h_pre"].astype(np.float32), float(inp.fc2_input_scale[0]))
    assert np.array_equal(q, st["hq"]) and np.array_equal(sf, st["hsf"])
    np.testing.assert_array_equal(st["h_in"], dequant_np(q[None], sf[None])[0])
    xh = orc.xhat(5)
    np.testing.assert_array_equal(xh, dequant_np(inp.x_q.numpy()[5:6], inp.x_sf.numpy()[5:6])[0])
    # bf16 activations: xhat is x itself
    inp16 = _small_inputs()
    o16 = oracle.OracleMoE.from_inputs(inp16)
    np.testing.assert_array_equal(o16.xhat(2), inp16.x[2].double().numpy())
    st16 = o16.expert_ffn(1, 2)
    np.testing.assert_array_equal(st16["h_in"], to_bf16_torch(st16["h_pre"]))


def test_single_expert_is_dense_mlp():
    """P5: E=1, top_k=1, weight 1 reduces to bf16(W2 R(silu(G x) * U x)) -- torch.matmul in float64."""
    cfg = synth.CONFIGS["tiny_w4a16"].with_(E=1, top_k=1, M=8)
    inp = synth.generate(cfg)
    inp.token_final_scales[:] = 1.0
    orc = oracle.OracleMoE.from_inputs(inp)
    _, exact, _ = orc.forward()
    W1 = torch.from_numpy(dequant_np(inp.w1.numpy()[0], inp.w1_sf.numpy()[0])) * float(inp.w1_alpha[0])
    W2 = torch.from_numpy(dequant_np(inp.w2.numpy()[0], inp.w2_sf.numpy()[0])) * float(inp.w2_alpha[0])
    X = inp.x.to(torch.float64)
    gu = torch.matmul(X, W1.T)
    g, u = gu[:, :cfg.I], gu[:, cfg.I:]
    h = torch.nn.functional.silu(g) * u
    h = h.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    ref = torch.matmul(h, W2.T).numpy()
    np.testing.assert_allclose(exact, ref, rtol=1e-9, atol=1e-12)


def test_accumulate_false_equals_zero_seed_bitwise_and_ep_split():
    inp = _small_inputs()
    cfg = inp.cfg
    orc = oracle.OracleMoE.from_inputs(inp)
    a, _, _ = orc.forward(rsf=0.75, accumulate=False)
    b, _, _ = orc.forward(rsf=0.75, accumulate=True, out_old=np.zeros((cfg.M, cfg.H), np.uint16))
    assert np.array_equal(a, b)
    # expert parallel: two disjoint halves, the second seeded with the first's output
    half = cfg.E // 2

    def part(off):
        o = oracle.OracleMoE(cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k,
                             inp.token_selected_experts.numpy(), inp.token_final_scales.numpy(),
                             inp.w1.numpy()[off:off + half], inp.w1_sf.numpy()[off:off + half],
                             inp.w1_alpha.numpy()[off:off + half], inp.w2.numpy()[off:off + half],
                             inp.w2_sf.numpy()[off:off + half], inp.w2_alpha.numpy()[off:off + half],
                             x=inp.x.view(torch.int16).numpy().view(np.uint16), E_local=half,
                             offset=off)
        return o
    p0, _, _ = part(0).forward(rsf=0.75)
    p1, ex1, _ = part(half).forward(rsf=0.75, accumulate=True, out_old=p0)
    _, full, _ = orc.forward(rsf=0.75)
    # equal up to the two extra bf16 roundings (of the first half's partial
    # sum and of the final value), each within u = 2^-8 relative (bf16, p = 8)
    bound = 2.0 ** -8 * (np.abs(bf16_np(p0)) + np.abs(bf16_np(p1))) + 1e-30
    assert np.all(np.abs(bf16_np(p1) - full) <= bound)
    # a plain sum with rsf folds linearly
    c, ec, _ = orc.forward(rsf=1.5)
    _, ea, _ = orc.forward(rsf=0.75)
    np.testing.assert_allclose(ec, 2 * ea, rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- GEMM2 from arbitrary FC1 codes

def test_expert_down_from_codes_matches_numpy():
    """The oracle's GEMM2 on caller-given FC1 codes (what the GEMM2-only GPU
    parity checks compare against) equals alpha2 * (W2_e @ decode(codes)) with
    W2 and the codes decoded by the tests' own table and torch's E4M3: random
    NVFP4 codes under random signed E4M3 scales (NaN bytes excluded), with an
    all-zero-scale block."""
    inp = _small_inputs("w4a4")
    orc = oracle.OracleMoE.from_inputs(inp)
    I = inp.cfg.I
    rng = np.random.default_rng(11)
    W2 = dequant_np(inp.w2.numpy(), inp.w2_sf.numpy())
    a2 = inp.w2_alpha.double().numpy()
    for e in (0, 5):
        hq = rng.integers(0, 256, I // 2, dtype=np.uint8)
        hsf = rng.integers(0, 256, I // 16, dtype=np.uint8)
        hsf[(hsf & 0x7F) == 0x7F] = 0x38                  # no NaN scales
        hsf[2] = 0x80                                     # a negative-zero scale
        ref = a2[e] * (W2[e] @ dequant_np(hq[None], hsf[None])[0])
        np.testing.assert_allclose(orc.expert_down_codes(e, hq, hsf), ref, rtol=1e-12, atol=1e-15)


def test_expert_down_from_mxfp8_codes_matches_numpy():
    """The same for w4a8: MXFP8 FC1 codes (E4M3 elements, E8M0 block-32 scales)
    against MXFP4 weights, both decoded here."""
    cfg = synth.CONFIGS["tiny_w4a16"].with_(mode="w4a8")
    inp = synth.generate(cfg, device="cpu")
    orc = oracle.OracleMoE.from_inputs(inp)
    I = cfg.I
    rng = np.random.default_rng(12)
    q2, s2 = inp.w2.numpy(), inp.w2_sf.numpy().astype(np.int64)
    lo, hi = E2M1_TABLE[q2 & 15], E2M1_TABLE[q2 >> 4]
    W2 = np.stack([lo, hi], -1).reshape(q2.shape[:-1] + (q2.shape[-1] * 2,)) * np.exp2(
        np.repeat(s2 - 127, 32, axis=-1).astype(np.float64))
    a2 = inp.w2_alpha.double().numpy()
    for e in (1, 6):
        hq = rng.integers(0, 256, I, dtype=np.uint8)
        hq[(hq & 0x7F) == 0x7F] = 0x30                    # no NaN elements
        hsf = rng.integers(118, 136, I // 32, dtype=np.uint8)
        hin = e4m3_np(hq) * np.exp2(np.repeat(hsf.astype(np.int64) - 127, 32).astype(np.float64))
        ref = a2[e] * (W2[e] @ hin)
        np.testing.assert_allclose(orc.expert_down_codes(e, hq, hsf), ref, rtol=1e-12, atol=1e-15)
