"""Pins of the oracle's w4a8 formats (FlashInfer PR #4440: MXFP8 activations,
E4M3 with linear block-32 E8M0 scales; MXFP4 weights, E2M1 with block-32 E8M0
scales; an MXFP8 FC1 intermediate), against the OCP MX scale definition,
torch's own float8_e4m3fn rounding and numpy brute force."""
import math

import numpy as np
import torch

import oracle
import synth
from ref_decode import E2M1_TABLE, e4m3_np


def test_e8m0_values():
    assert oracle.ue8m0_value(127) == 1.0
    assert oracle.ue8m0_value(128) == 2.0
    assert oracle.ue8m0_value(0) == 2.0 ** -127
    assert oracle.ue8m0_value(254) == 2.0 ** 127
    assert math.isnan(oracle.ue8m0_value(255))


def _torch_e4m3(v):
    """E4M3 RNE by torch (values already inside +-448)."""
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_mxfp8_quantiser_against_torch_rounding():
    rng = np.random.default_rng(5)
    n = 32 * 512
    mags = np.exp2(rng.integers(-30, 30, n // 32)).repeat(32)
    h = (rng.standard_normal(n) * mags).astype(np.float32)
    q, sf = oracle.mxfp8_quantize_f32(h)
    blocks = h.reshape(-1, 32)
    for b in range(blocks.shape[0]):
        amax = np.abs(blocks[b]).max()
        X = math.floor(math.log2(amax)) - 8
        assert sf[b] == X + 127
        scaled = blocks[b] * np.float32(2.0 ** -X)
        want = _torch_e4m3(np.clip(scaled, -448, 448))
        assert np.array_equal(q[b * 32:(b + 1) * 32], want), b


def test_mxfp8_quantiser_special_blocks():
    h = np.zeros(32 * 4, np.float32)
    # block 0: zeros -> X = -127, codes 0
    # block 1: amax 500 = 1.95 * 2^8 -> X = 0, 500 saturates to 448 (0x7E)
    h[32] = 500.0
    h[33] = -1.0
    # block 2: a NaN -> code 255, NaN elements
    h[64] = np.nan
    # block 3: an exact MXFP8 block round-trips (amax 1.75 * 2^-6: the recipe
    # maps it to 448 exactly; a block whose amax mantissa exceeds 1.75 would
    # saturate, the recipe putting amax in [256, 512))
    codes = np.concatenate([[0x06], np.arange(0x08, 0x27)]).astype(np.uint8)   # 32 normal codes
    vals = e4m3_np(codes) * 2.0 ** -3
    h[96:128] = vals
    q, sf = oracle.mxfp8_quantize_f32(h)
    assert sf[0] == 0 and not q[:32].any()
    assert sf[1] == 127 and q[32] == 0x7E and q[33] == 0xB8
    assert sf[2] == 255 and np.all(q[64:96] == 0x7F)
    amax = vals.max()
    assert sf[3] == math.floor(math.log2(amax)) - 8 + 127
    back = e4m3_np(q[96:128]) * 2.0 ** (int(sf[3]) - 127)
    assert np.array_equal(back, vals)


def test_w4a8_ffn_matches_numpy_brute_force():
    cfg = synth.CONFIGS["tiny_w4a16"].with_(mode="w4a8")
    inp = synth.generate(cfg, device="cpu")
    orc = oracle.OracleMoE.from_inputs(inp)
    H, I = cfg.H, cfg.I
    # MXFP8 activations: E4M3 (torch) times 2^(e - 127)
    xq = inp.x_q.numpy()
    xs = inp.x_sf.numpy().astype(np.int64)
    xh = e4m3_np(xq) * np.exp2(np.repeat(xs - 127, 32, axis=1).astype(np.float64))
    for t in range(3):
        assert np.array_equal(orc.xhat(t), xh[t])
    # MXFP4 weights: E2M1 (golden table) times 2^(e - 127) per 32
    def dec(q, sf):
        lo, hi = E2M1_TABLE[q & 15], E2M1_TABLE[q >> 4]
        v = np.stack([lo, hi], -1).reshape(q.shape[:-1] + (q.shape[-1] * 2,))
        return v * np.exp2(np.repeat(sf.astype(np.int64) - 127, 32, axis=-1).astype(np.float64))
    W1 = dec(inp.w1.numpy(), inp.w1_sf.numpy())
    W2 = dec(inp.w2.numpy(), inp.w2_sf.numpy())
    ids = inp.token_selected_experts.numpy()
    for t in range(3):
        for j in range(cfg.top_k):
            e = ids[t, j]
            st = orc.expert_ffn(int(e), t)
            g = W1[e, :I] @ xh[t]
            u = W1[e, I:] @ xh[t]
            assert np.allclose(st["g"], g, rtol=1e-12, atol=1e-15)
            assert np.allclose(st["u"], u, rtol=1e-12, atol=1e-15)
            # h_in is the MXFP8 round trip of the fp32 activation output
            q, sf = oracle.mxfp8_quantize_f32(st["h_pre"].astype(np.float32))
            hin = e4m3_np(q) * np.exp2(np.repeat(sf.astype(np.int64) - 127, 32).astype(np.float64))
            assert np.array_equal(st["h_in"], hin)
            assert np.array_equal(st["hq"], q) and np.array_equal(st["hsf"], sf)
            assert np.allclose(st["y"], W2[e] @ hin, rtol=1e-12, atol=1e-15)
