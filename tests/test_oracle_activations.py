"""Pins of the oracle's FC1 activation variants and per-token input scale
(cute_dsl_fused_moe: activation_type, swiglu_alpha/beta/limit, situ_beta,
situ_linear_beta, per_token_scale), each against something other than the
oracle's own formula: reductions to the default SwiGLU, limits, saturation
invariants, an independent GELU, and numpy brute force."""
import numpy as np
import pytest
import torch

import oracle
import synth
from ref_decode import bf16_np, dequant_np

TINY = synth.CONFIGS["tiny_w4a16"]


def _inputs(act="swiglu", x_scale=1.0, **cfg_kw):
    cfg = TINY.with_(act=act, **cfg_kw)
    inp = synth.generate(cfg, device="cpu")
    if x_scale != 1.0 and inp.x is not None:
        inp.x = (inp.x.float() * x_scale).to(torch.bfloat16)   # exact: a power of two
    return cfg, inp


def _staged(orc, cfg, inp, t_max=6):
    """(g, u, h_pre) of the first routes, stacked."""
    rows = {"g": [], "u": [], "h_pre": []}
    ids = inp.token_selected_experts.numpy()
    for t in range(t_max):
        for j in range(cfg.top_k):
            st = orc.expert_ffn(int(ids[t, j]), t)
            for k in rows:
                rows[k].append(st[k])
    return {k: np.concatenate(v) for k, v in rows.items()}


def _oracle(cfg, inp, act_type=None, act_params=None, **kw):
    o = oracle.OracleMoE.from_inputs(inp)
    if act_type is None and act_params is None and not kw:
        return o
    t, p = synth.activation_spec(cfg)
    a = inp
    host = lambda v: None if v is None else v.detach().cpu().numpy()
    x = None if a.x is None else a.x.view(torch.int16).numpy().view(np.uint16)
    return oracle.OracleMoE(cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k, host(a.token_selected_experts),
                            host(a.token_final_scales), host(a.w1), host(a.w1_sf), host(a.w1_alpha),
                            host(a.w2), host(a.w2_sf), host(a.w2_alpha), x=x, x_q=host(a.x_q),
                            x_sf=host(a.x_sf), fc2_input_scale=host(a.fc2_input_scale),
                            act_type=t if act_type is None else act_type,
                            act_params=p if act_params is None else act_params, **kw)


def test_swiglu_oai_at_default_parameters_is_swiglu():
    cfg, inp = _inputs()
    base = _staged(_oracle(cfg, inp), cfg, inp)
    oai = _staged(_oracle(cfg, inp, act_params={"swiglu_alpha": 1.0, "swiglu_beta": 0.0,
                                                "swiglu_limit": float("inf")}), cfg, inp)
    assert np.allclose(oai["h_pre"], base["h_pre"], rtol=1e-13, atol=0)


def test_swiglu_oai_clamps_gate_and_up():
    # once every pre-activation is beyond the limit, scaling x further changes nothing
    cfg, inp_a = _inputs("swiglu_oai", x_scale=2.0 ** 12)
    _, inp_b = _inputs("swiglu_oai", x_scale=2.0 ** 14)
    a = _staged(_oracle(cfg, inp_a), cfg, inp_a)
    b = _staged(_oracle(cfg, inp_b), cfg, inp_b)
    L = synth.ACTIVATIONS["swiglu_oai"][1]["swiglu_limit"]
    sat = (a["g"] > L) & (np.abs(a["u"]) > L)
    assert sat.sum() > 50
    assert np.array_equal(a["h_pre"][sat], b["h_pre"][sat])
    # and the default SwiGLU is not bounded that way
    d = _staged(_oracle(cfg, inp_b, act_type=0, act_params={}), cfg, inp_b)
    assert np.abs(d["h_pre"][sat]).max() > 10 * np.abs(b["h_pre"][sat]).max()


def test_situ_tends_to_swiglu_for_large_beta():
    cfg, inp = _inputs()
    base = _staged(_oracle(cfg, inp), cfg, inp)
    situ = _staged(_oracle(cfg, inp, act_params={"situ_beta": 1e9}), cfg, inp)
    assert np.allclose(situ["h_pre"], base["h_pre"], rtol=1e-9, atol=1e-300)
    lin = _staged(_oracle(cfg, inp, act_params={"situ_beta": 1e9, "situ_linear_beta": 1e9}), cfg, inp)
    assert np.allclose(lin["h_pre"], base["h_pre"], rtol=1e-9, atol=1e-300)


def test_situ_gate_and_up_are_bounded_by_their_betas():
    cfg, inp = _inputs("situ_linear", x_scale=2.0 ** 8)
    st = _staged(_oracle(cfg, inp), cfg, inp)
    p = synth.ACTIVATIONS["situ_linear"][1]
    assert np.all(np.abs(st["h_pre"]) <= p["situ_beta"] * p["situ_linear_beta"] * (1 + 1e-12))
    cfg, inp = _inputs("situ", x_scale=2.0 ** 8)
    st = _staged(_oracle(cfg, inp), cfg, inp)
    assert np.all(np.abs(st["h_pre"]) <= synth.ACTIVATIONS["situ"][1]["situ_beta"] * np.abs(st["u"]) * (1 + 1e-12))


def test_geglu_tanh_is_close_to_the_erf_gelu():
    special = pytest.importorskip("scipy.special")
    cfg, inp = _inputs("geglu_tanh", x_scale=4.0)
    st = _staged(_oracle(cfg, inp), cfg, inp)
    m = np.abs(st["u"]) > 1e-3
    gate = st["h_pre"][m] / st["u"][m]
    g = st["g"][m]
    gelu = 0.5 * g * (1.0 + special.erf(g / np.sqrt(2.0)))
    assert np.max(np.abs(gate - gelu)) < 1e-3
    assert np.abs(g).max() > 1.5                       # the test reaches the curved part


def test_relu2_matches_numpy_brute_force():
    cfg, inp = _inputs("relu2")
    assert inp.w1.shape[1] == cfg.I                  # non-gated: no gate rows
    st = _staged(_oracle(cfg, inp), cfg, inp, t_max=4)
    W1 = dequant_np(inp.w1.numpy(), inp.w1_sf.numpy())            # [E, I, H] float64
    xh = bf16_np(inp.x.view(torch.int16).numpy().view(np.uint16))  # [M, H]
    ids = inp.token_selected_experts.numpy()
    a1 = inp.w1_alpha.numpy().astype(np.float64)
    want_u, want_h = [], []
    for t in range(4):
        for j in range(cfg.top_k):
            e = ids[t, j]
            u = a1[e] * (W1[e] @ xh[t])
            want_u.append(u)
            want_h.append(np.maximum(u, 0.0) ** 2)
    assert np.allclose(st["u"], np.concatenate(want_u), rtol=1e-12, atol=1e-15)
    assert np.allclose(st["h_pre"], np.concatenate(want_h), rtol=1e-11, atol=1e-18)
    assert (np.concatenate(want_u) < 0).mean() > 0.3


def test_per_token_scale_equals_scaling_the_activation_scales():
    # w4a4: a per-token scale of 1/2 equals halving every E4M3 scale byte of x
    # (exponent - 1, exact for the normal codes the generator produces)
    cfg, inp = _inputs(mode="w4a4")
    sf = inp.x_sf.numpy()
    assert np.all((sf & 0x78) >= 0x10) and np.all((sf & 0x80) == 0)   # stays normal when halved
    half = np.full(cfg.M, 0.5, np.float32)
    a = _oracle(cfg, inp, per_token_scale=half)
    inp2 = synth.MoEInputs(**{**inp.__dict__, "x_sf": torch.from_numpy(sf - 8)})
    b = oracle.OracleMoE.from_inputs(inp2)
    _, ea, _ = a.forward()
    _, eb, _ = b.forward()
    _, e1, _ = oracle.OracleMoE.from_inputs(inp).forward()
    assert np.array_equal(ea, eb)
    assert not np.array_equal(ea, e1)
