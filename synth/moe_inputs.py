"""Seeded synthetic workloads for the NVFP4 fused-MoE forward pass.

The five workloads follow the problem statement of the fused-MoE API pages
(flashinfer.fused_moe.cute_dsl_fused_moe, "Parameters": x / x_sf /
token_selected_experts / token_final_scales / w1_weight [E, 2I, H/2] /
w2_weight [E, H, I/2] / alphas) with the shapes of the DeepSeek-like
H=7168/E=256/k=8 case and the H=6144 large-batch case of the route-window
table on the flashinfer PR #4440 page.

What is drawn here (input preparation, shared by both sides):
  * routing: numpy PCG64 streams spawned from SeedSequence(seed).
  * activations and weights: torch's Philox generator on the target device
    (weights one expert at a time), then the standard NVFP4 model-load
    quantiser: global scale gs = 448*6/amax, E4M3 block-16 scales
    RNE(amax_blk/6*gs), E2M1 codes RNE(v*gs/scale), alpha = 1/gs.
    This is what a checkpoint converter does before the forward pass runs;
    the forward pass's own FC1 re-quantisation (w4a4) is NOT taken from here.

Packed layout: element 2i of a row sits in the low nibble of byte i,
element 2i+1 in the high nibble.  Scales are linear row-major [rows, K/16].
Gate rows are w1[:, :I], up rows are w1[:, I:].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

# --------------------------------------------------------------------------
# workload table
# --------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    M: int          # tokens
    H: int          # hidden
    I: int          # intermediate (per gate / up half)
    E: int          # experts (all local)
    top_k: int
    mode: str       # "w4a16", "w4a4" or "w4a8"
    routing: str    # "softmax", "skewed" or "uniform"
    sample: int = 0  # 0: check every token; else number of sampled tokens
    seed: int = 0
    act: str = "swiglu"           # FC1 activation, see ACTIVATIONS
    per_token_scale: bool = False  # draw a per-token input row scale (w4a4)

    @property
    def routes(self) -> int:
        return self.M * self.top_k

    def flops(self) -> float:
        """Algorithmic flops of the routed work: 6*R*H*I (GEMM1 4RHI, GEMM2 2RHI)."""
        return 6.0 * self.routes * self.H * self.I

    def with_(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


# FC1 activations of the tests: name -> (type, parameters).  Type 0 = the
# SwiGLU family, 1 = GeGLU with tanh, 2 = non-gated ReLU^2; parameter values
# are picked so that the clamps and the tanh saturation are reached at the
# tests' pre-activation scale (g, u ~ N(0, 0.02^2 H / gs^2), |g| up to ~1).
ACTIVATIONS = {
    "swiglu": (0, {}),
    "swiglu_oai": (0, {"swiglu_alpha": 1.702, "swiglu_beta": 1.0, "swiglu_limit": 0.25}),
    "situ": (0, {"situ_beta": 0.3}),
    "situ_linear": (0, {"situ_beta": 0.3, "situ_linear_beta": 0.2}),
    "geglu_tanh": (1, {}),
    "relu2": (2, {}),
}


def activation_spec(cfg: "MoEConfig"):
    """(type, parameter dict) of cfg's FC1 activation (configuration only)."""
    return ACTIVATIONS[cfg.act]


CONFIGS = {
    "tiny_w4a16": MoEConfig("tiny_w4a16", M=16, H=256, I=256, E=8, top_k=2,
                            mode="w4a16", routing="softmax"),
    "decode_w4a16": MoEConfig("decode_w4a16", M=8, H=7168, I=2048, E=256, top_k=8,
                              mode="w4a16", routing="softmax"),
    "prefill_w4a4": MoEConfig("prefill_w4a4", M=4096, H=7168, I=2048, E=256, top_k=8,
                              mode="w4a4", routing="softmax", sample=1024),
    "skewed_w4a16": MoEConfig("skewed_w4a16", M=2048, H=4096, I=1536, E=128, top_k=4,
                              mode="w4a16", routing="skewed"),
    "prefill_w4a8": MoEConfig("prefill_w4a8", M=4096, H=7168, I=2048, E=256, top_k=8,
                              mode="w4a8", routing="softmax", sample=1024),
    "large_w4a16": MoEConfig("large_w4a16", M=131072, H=6144, I=2048, E=256, top_k=8,
                             mode="w4a16", routing="uniform", sample=1024),
}


def route_tile_for(cfg: MoEConfig) -> int:
    """Route tile the benchmarks use (the library's automatic choice): the
    average routes per expert -- doubled above 16 for BF16 activations, whose
    GEMMs size each MMA to a tile's valid slots -- rounded up to a power of
    two and clamped to [16, 128]."""
    avg = max(1, -(-cfg.routes // cfg.E))
    if cfg.mode == "w4a16" and avg > 16:
        avg *= 2
    t = 16
    while t < avg and t < 128:
        t *= 2
    return t


@dataclasses.dataclass
class MoEInputs:
    cfg: MoEConfig
    token_selected_experts: torch.Tensor   # int32 [M, k]   (cpu)
    token_final_scales: torch.Tensor       # fp32  [M, k]   (cpu)
    x: Optional[torch.Tensor]              # bf16 [M, H]         (w4a16)
    x_q: Optional[torch.Tensor]            # uint8 [M, H/2]      (w4a4)
    x_sf: Optional[torch.Tensor]           # uint8 e4m3 [M, H/16](w4a4)
    w1: torch.Tensor                       # uint8 [E, 2I, H/2]  (ReLU^2: [E, I, H/2])
    w1_sf: torch.Tensor                    # uint8 [E, 2I, H/16] (ReLU^2: [E, I, H/16])
    w1_alpha: torch.Tensor                 # fp32 [E]
    w2: torch.Tensor                       # uint8 [E, H, I/2]
    w2_sf: torch.Tensor                    # uint8 [E, H, I/16]
    w2_alpha: torch.Tensor                 # fp32 [E]
    fc2_input_scale: Optional[torch.Tensor]  # fp32 [1] (w4a4)
    sample_tokens: np.ndarray              # int64 sorted token ids to check
    per_token_scale: Optional[torch.Tensor] = None  # fp32 [M] or None

    def to(self, device) -> "MoEInputs":
        def mv(t):
            return None if t is None else t.to(device)
        return dataclasses.replace(
            self, x=mv(self.x), x_q=mv(self.x_q), x_sf=mv(self.x_sf), w1=mv(self.w1),
            w1_sf=mv(self.w1_sf), w1_alpha=mv(self.w1_alpha), w2=mv(self.w2),
            w2_sf=mv(self.w2_sf), w2_alpha=mv(self.w2_alpha),
            fc2_input_scale=mv(self.fc2_input_scale), per_token_scale=mv(self.per_token_scale))


# --------------------------------------------------------------------------
# model-load NVFP4 quantiser (input preparation)
# --------------------------------------------------------------------------

_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Round fp32 values to E2M1 (nearest, ties to the even code, saturating)."""
    a = v.abs()
    mids = torch.tensor(_E2M1_MID, dtype=torch.float32, device=v.device)
    idx = torch.bucketize(a, mids, right=False)            # ties go to the lower code
    up = (a == 0.75) | (a == 1.75) | (a == 3.5)             # ...unless the upper one is even
    idx = idx + up.to(idx.dtype)
    sign = torch.signbit(v).to(idx.dtype)
    return (idx | (sign << 3)).to(torch.uint8)


def _pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    lo = codes[..., 0::2]
    hi = codes[..., 1::2]
    return (lo | (hi << 4)).to(torch.uint8)


def quantize_nvfp4(w: torch.Tensor, gs: Optional[torch.Tensor] = None):
    """NVFP4-quantise a fp32 matrix [rows, K] along K (block 16).

    Returns (packed uint8 [rows, K/2], e4m3 scale bytes [rows, K/16], gs).
    """
    rows, K = w.shape
    assert K % 16 == 0
    if gs is None:
        amax = w.abs().amax().clamp_min(1e-30)
        gs = (448.0 * 6.0) / amax
    blk = w.reshape(rows, K // 16, 16)
    bmax = blk.abs().amax(dim=-1)
    sf = (bmax / 6.0 * gs).to(torch.float8_e4m3fn)
    sf_val = sf.to(torch.float32)
    safe = torch.where(sf_val > 0, sf_val, torch.ones_like(sf_val))
    scaled = blk * gs / safe.unsqueeze(-1)
    scaled = torch.where(sf_val.unsqueeze(-1) > 0, scaled, torch.zeros_like(scaled))
    codes = _e2m1_codes(scaled.reshape(rows, K))
    return _pack_nibbles(codes), sf.view(torch.uint8), gs


def _mx_exponents(w: torch.Tensor, emax: int) -> torch.Tensor:
    """OCP MX shared exponents of [rows, K] along K (block 32): floor(log2 amax) -
    emax, clamped to [-127, 127]; -127 for an all-zero block."""
    rows, K = w.shape
    amax = w.reshape(rows, K // 32, 32).abs().amax(dim=-1)
    _, e = torch.frexp(amax)                                # amax = m 2^e, m in [0.5, 1)
    X = (e.to(torch.int32) - 1) - emax
    X = torch.where(amax > 0, X, torch.full_like(X, -127))
    return X.clamp(-127, 127)


def quantize_mxfp4(w: torch.Tensor):
    """MXFP4-quantise [rows, K] along K: E2M1 codes with E8M0 block-32 scales
    2^X, X = floor(log2 amax) - 2.  Returns (packed uint8 [rows, K/2], e8m0 [rows, K/32])."""
    rows, K = w.shape
    X = _mx_exponents(w, 2)
    scaled = w.reshape(rows, K // 32, 32) * torch.exp2(-X.to(torch.float32)).unsqueeze(-1)
    codes = _e2m1_codes(scaled.reshape(rows, K))
    return _pack_nibbles(codes), (X + 127).to(torch.uint8)


def quantize_mxfp8(x: torch.Tensor):
    """MXFP8-quantise [rows, K] along K: E4M3 elements (saturating) with E8M0
    block-32 scales 2^X, X = floor(log2 amax) - 8.  Returns (e4m3 [rows, K], e8m0 [rows, K/32])."""
    rows, K = x.shape
    X = _mx_exponents(x, 8)
    scaled = x.reshape(rows, K // 32, 32) * torch.exp2(-X.to(torch.float32)).unsqueeze(-1)
    q = scaled.clamp(-448.0, 448.0).reshape(rows, K).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), (X + 127).to(torch.uint8)


# --------------------------------------------------------------------------
# routing draws
# --------------------------------------------------------------------------


def _softmax_topk(logits: np.ndarray, k: int):
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]      # ties go to the lower id
    sel = np.take_along_axis(p, order, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def _routing(cfg: MoEConfig, rng: np.random.Generator):
    M, E, k = cfg.M, cfg.E, cfg.top_k
    if cfg.routing == "softmax":
        return _softmax_topk(rng.standard_normal((M, E)), k)
    if cfg.routing == "skewed":
        # N(0,1) logits plus a log-Zipf bias over a seeded expert ranking;
        # the 8 lowest-ranked experts never win (bias -inf).
        perm = rng.permutation(E)
        ranks = np.arange(1, E + 1, dtype=np.float64)
        bias_by_rank = -0.4 * 1.2 * np.log(ranks)
        bias_by_rank[-8:] = -np.inf
        bias = np.empty(E)
        bias[perm] = bias_by_rank
        logits = rng.standard_normal((M, E)) + bias[None, :]
        return _softmax_topk(logits, k)
    if cfg.routing == "uniform":
        noise = rng.random((M, E))
        ids = np.argpartition(noise, k, axis=1)[:, :k].astype(np.int32)
        u = rng.random((M, k))
        g = -np.log1p(-u)                      # Exp(1) draws -> Dirichlet(1) weights
        w = (g / g.sum(axis=1, keepdims=True)).astype(np.float32)
        return ids, w
    raise ValueError(cfg.routing)


# --------------------------------------------------------------------------
# whole workload
# --------------------------------------------------------------------------


def generate_routing(cfg: MoEConfig):
    """Routing draw of `cfg` alone: (ids int32 [M, k], weights fp32 [M, k]) as numpy."""
    ss_route = np.random.SeedSequence(cfg.seed).spawn(5)[0]
    return _routing(cfg, np.random.Generator(np.random.PCG64(ss_route)))


def _torch_seed(ss: np.random.SeedSequence) -> int:
    return int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 62) - 1))


def generate(cfg: MoEConfig, device="cpu", experts: Optional[int] = None) -> MoEInputs:
    """Draw the workload `cfg` (seed cfg.seed) with weights on `device`.

    `experts` limits weight generation to the first n experts (only for tests
    that route to a subset); routing always uses cfg.E.
    """
    device = torch.device(device)
    ss_route, ss_x, ss_w1, ss_w2, ss_sample = np.random.SeedSequence(cfg.seed).spawn(5)
    ids, w = _routing(cfg, np.random.Generator(np.random.PCG64(ss_route)))

    M, H, I, E = cfg.M, cfg.H, cfg.I, cfg.E
    gx = torch.Generator(device=device)
    gx.manual_seed(_torch_seed(ss_x))
    xf = torch.randn(M, H, generator=gx, device=device, dtype=torch.float32)
    x = x_q = x_sf = None
    gs_x = None
    if cfg.mode == "w4a16":
        x = xf.to(torch.bfloat16)
    elif cfg.mode == "w4a8":
        x_q, x_sf = quantize_mxfp8(xf)
    else:
        x_q, x_sf, gs_x = quantize_nvfp4(xf)
    del xf

    n_gen = E if experts is None else experts
    rows1 = I if activation_spec(cfg)[0] == 2 else 2 * I   # ReLU^2 has no gate rows
    sb = 32 if cfg.mode == "w4a8" else 16                  # MXFP4 / NVFP4 scale block
    w1 = torch.empty(E, rows1, H // 2, dtype=torch.uint8, device=device)
    w1_sf = torch.empty(E, rows1, H // sb, dtype=torch.uint8, device=device)
    w2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
    w2_sf = torch.empty(E, H, I // sb, dtype=torch.uint8, device=device)
    gs1 = torch.ones(E, dtype=torch.float32, device=device)
    gs2 = torch.ones(E, dtype=torch.float32, device=device)
    base1, base2 = _torch_seed(ss_w1), _torch_seed(ss_w2)
    g = torch.Generator(device=device)
    for e in range(n_gen):
        g.manual_seed(base1 + e)
        W = torch.randn(rows1, H, generator=g, device=device, dtype=torch.float32) * 0.02
        if cfg.mode == "w4a8":
            w1[e], w1_sf[e] = quantize_mxfp4(W)
        else:
            w1[e], w1_sf[e], gs1[e] = quantize_nvfp4(W)
        g.manual_seed(base2 + e)
        W = torch.randn(H, I, generator=g, device=device, dtype=torch.float32) * 0.02
        if cfg.mode == "w4a8":
            w2[e], w2_sf[e] = quantize_mxfp4(W)
        else:
            w2[e], w2_sf[e], gs2[e] = quantize_nvfp4(W)
        del W
    if n_gen < E:
        for t in (w1, w1_sf, w2, w2_sf):
            t[n_gen:].zero_()

    fc2 = None
    if cfg.mode in ("w4a16", "w4a8"):   # MX formats carry no global scale: gs = 1
        a1 = 1.0 / gs1
        a2 = 1.0 / gs2
    else:
        # fc2_input_scale: a power of two fixed by the generation distribution
        # (g, u ~ N(0, 0.02^2 H); a 16-block of h = silu(g)*u stays below
        # ~25 sigma^2), chosen so that s*amax/6 of such a block fits E4M3.
        sigma2 = 0.02 * 0.02 * H
        s = 2.0 ** math.floor(math.log2(448.0 * 6.0 / (2.0 * 25.0 * sigma2)))
        fc2 = torch.tensor([s], dtype=torch.float32, device=device)
        a1 = 1.0 / (gs_x * gs1)
        a2 = 1.0 / (s * gs2)

    srng = np.random.Generator(np.random.PCG64(ss_sample))
    if cfg.sample and cfg.sample < M:
        sample = np.sort(srng.choice(M, size=cfg.sample, replace=False)).astype(np.int64)
    else:
        sample = np.arange(M, dtype=np.int64)
    pts = None
    if cfg.per_token_scale:
        # per-token row scales 2^U(-1, 1), from their own sub-stream of x's seed
        prng = np.random.Generator(np.random.PCG64(ss_x.spawn(1)[0]))
        pts = torch.from_numpy(np.exp2(prng.uniform(-1.0, 1.0, M)).astype(np.float32)).to(device)

    return MoEInputs(
        cfg=cfg,
        token_selected_experts=torch.from_numpy(ids),
        token_final_scales=torch.from_numpy(w),
        x=x, x_q=x_q, x_sf=x_sf,
        w1=w1, w1_sf=w1_sf, w1_alpha=a1.to(torch.float32).contiguous(),
        w2=w2, w2_sf=w2_sf, w2_alpha=a2.to(torch.float32).contiguous(),
        fc2_input_scale=fc2, sample_tokens=sample, per_token_scale=pts)
