"""Device buffers for one fused-MoE problem (torch is used for memory only).

`MoEBuffers` owns the routing-plan arrays, the prepared weights and the
workspaces, sized by the library's own size queries, and calls the C ABI
through the binding.  No arithmetic of the forward pass happens here.
"""
from __future__ import annotations

import torch

from . import (ACT_RELU2, W4A4, W4A8, W4A16, FINALIZE_DETERMINISTIC, activation,
               domain_weight_size, fused_moe_forward, fused_moe_forward_localized,
               gemm_workspace_size, localized, localized_workspace_size, max_permuted_slots,
               moe_finalize, moe_gemm1_swiglu, moe_gemm2, moe_permute, moe_route_sort,
               prepare_domain_weights, prepare_weights, prepared_weight_size, problem, route_tile,
               route_workspace_size, workspace_size)


def _empty(n, dtype, device):
    return torch.empty(max(int(n), 1), dtype=dtype, device=device)


def _zeros(n, dtype, device):
    # workspaces start zeroed: their first word is the sticky device error word
    return torch.zeros(max(int(n), 1), dtype=dtype, device=device)


class MoEBuffers:
    """Plan, prepared weights and workspaces for `p` on `device`."""

    def __init__(self, p, device="cuda"):
        self.p = p
        self.device = torch.device(device)
        self.T = route_tile(p)
        self.S = max_permuted_slots(p)
        self.tiles = self.S // self.T
        M, k = p.num_tokens, p.top_k
        E_local = p.num_local_experts or p.num_experts
        d = self.device
        i32 = torch.int32
        # the plan starts empty (zero tiles) until route() writes it
        self.e2p = _zeros(M * k, i32, d)
        self.p2e = _zeros(self.S, i32, d)
        self.tile_expert = _zeros(self.tiles, i32, d)
        self.tile_mn = _zeros(self.tiles, i32, d)
        self.num_tiles = _zeros(4, i32, d)
        self.counts = _zeros(E_local, i32, d)
        self.route_ws = _zeros(route_workspace_size(p), torch.uint8, d)
        self.gemm1_ws = _zeros(gemm_workspace_size(p, 1), torch.uint8, d)
        self.gemm2_ws = _zeros(gemm_workspace_size(p, 2), torch.uint8, d)
        self.fused_ws = None
        self.local_ws = None
        self.w1p = None
        self.w2p = None
        self.w1d = None     # per-domain prepared shards (prepare_domains)
        self.w2d = None

    # -- weights
    def prepare(self, w1, w1_sf, w2, w2_sf, stream=None):
        p, d = self.p, self.device
        self.w1p = _empty(prepared_weight_size(p, 1), torch.uint8, d)
        self.w2p = _empty(prepared_weight_size(p, 2), torch.uint8, d)
        prepare_weights(p, 1, w1, w1_sf, self.w1p, stream)
        prepare_weights(p, 2, w2, w2_sf, self.w2p, stream)
        return self

    def prepare_domains(self, w1, w1_sf, w2, w2_sf):
        """Split the linear weights into the two locality domains' shards
        (FC1 on I: gate rows then the matching up rows; FC2 on H) and prepare
        each, on the current stream."""
        p, d = self.p, self.device
        I, H = p.inter, p.hidden
        self.w1d, self.w2d = [], []
        for k in range(2):
            half = torch.arange(k * I // 2, (k + 1) * I // 2, device=w1.device)
            rows = half if p.activation.type == ACT_RELU2 else torch.cat([half, half + I])
            w1s = w1.index_select(1, rows).contiguous()
            w1s_sf = w1_sf.index_select(1, rows).contiguous()
            w2s = w2[:, k * H // 2:(k + 1) * H // 2].contiguous()
            w2s_sf = w2_sf[:, k * H // 2:(k + 1) * H // 2].contiguous()
            p1 = _empty(domain_weight_size(p, 1), torch.uint8, d)
            p2 = _empty(domain_weight_size(p, 2), torch.uint8, d)
            prepare_domain_weights(p, 1, w1s, w1s_sf, p1)
            prepare_domain_weights(p, 2, w2s, w2s_sf, p2)
            self.w1d.append(p1)
            self.w2d.append(p2)
        return self

    def ensure_fused_ws(self):
        if self.fused_ws is None:
            self.fused_ws = _zeros(workspace_size(self.p), torch.uint8, self.device)
        return self.fused_ws

    # -- staged path
    def route(self, ids, stream=None):
        moe_route_sort(self.p, ids, self.e2p, self.p2e, self.tile_expert, self.tile_mn,
                       self.num_tiles, self.counts, self.route_ws, stream)

    def _rows(self, K):
        """Zeroed [S, K] activation rows and scales in the problem's format."""
        p, d, S = self.p, self.device, self.S
        if p.mode == W4A16:
            return torch.zeros(S, K, dtype=torch.bfloat16, device=d), None
        if p.mode == W4A8:   # MXFP8: E4M3 bytes + E8M0 block-32 scales
            return (torch.zeros(S, K, dtype=torch.uint8, device=d),
                    torch.zeros(S, K // 32, dtype=torch.uint8, device=d))
        return (torch.zeros(S, K // 2, dtype=torch.uint8, device=d),     # NVFP4
                torch.zeros(S, K // 16, dtype=torch.uint8, device=d))

    def alloc_permuted(self):
        """Buffers for x in slot order (moe_permute's output)."""
        return self._rows(self.p.hidden)

    def alloc_h(self):
        """Buffers for GEMM1's output h."""
        return self._rows(self.p.inter)

    def permute(self, x, x_sf=None, stream=None):
        px, psf = self.alloc_permuted()
        moe_permute(self.p, x, x_sf, self.p2e, self.num_tiles, px, psf, stream)
        return px, psf

    def gemm1(self, a, a_sf, w1_alpha, fc2_input_scale=None, gather=True, stream=None,
              per_token_scale=None):
        p = self.p
        h, hsf = self.alloc_h()
        moe_gemm1_swiglu(p, a, a_sf, self.p2e if gather else None, self.w1p, w1_alpha,
                         fc2_input_scale, self.tile_expert, self.tile_mn, self.num_tiles, h, hsf,
                         self.gemm1_ws, stream, per_token_scale=per_token_scale)
        return h, hsf

    def gemm2(self, h, hsf, w2_alpha, stream=None):
        p = self.p
        y = torch.zeros(self.S, p.hidden, dtype=torch.float32, device=self.device)
        moe_gemm2(p, h, hsf, self.w2p, w2_alpha, self.tile_expert, self.tile_mn, self.num_tiles, y,
                  self.gemm2_ws, stream)
        return y

    def finalize(self, y, token_final_scales, out, rsf=1.0, accumulate=False, stream=None):
        moe_finalize(self.p, y, self.e2p, token_final_scales, rsf, accumulate, out, stream)
        return out

    # -- fused path
    def forward(self, x, x_sf, ids, token_final_scales, w1_alpha, w2_alpha, out,
                fc2_input_scale=None, rsf=1.0, accumulate=False,
                finalize_mode=FINALIZE_DETERMINISTIC, stream=None, per_token_scale=None):
        ws = self.ensure_fused_ws()
        fused_moe_forward(self.p, x, x_sf, ids, token_final_scales, self.w1p, w1_alpha,
                          fc2_input_scale, self.w2p, w2_alpha, rsf, accumulate, finalize_mode, out,
                          ws, stream, per_token_scale=per_token_scale)
        return out

    def forward_localized(self, x, x_sf, ids, token_final_scales, w1_alpha, w2_alpha, out, streams,
                          sm_count=0, memset_stream=None, fc2_input_scale=None, rsf=1.0,
                          accumulate=False, finalize_mode=FINALIZE_DETERMINISTIC, stream=None,
                          per_token_scale=None):
        if self.local_ws is None:
            self.local_ws = _zeros(localized_workspace_size(self.p), torch.uint8, self.device)
        loc = localized(self.w1d, self.w2d, streams, sm_count, memset_stream)
        fused_moe_forward_localized(self.p, x, x_sf, ids, token_final_scales, loc, w1_alpha,
                                    fc2_input_scale, w2_alpha, rsf, accumulate, finalize_mode, out,
                                    self.local_ws, stream, per_token_scale=per_token_scale)
        return out


def problem_for(cfg, route_tile_=0, num_local_experts=0, local_expert_offset=0):
    """fp4moe_problem for a synth.MoEConfig (its activation included)."""
    import synth
    kind, params = synth.activation_spec(cfg)
    return problem(cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k, num_local_experts, local_expert_offset,
                   route_tile_, {"w4a16": W4A16, "w4a4": W4A4, "w4a8": W4A8}[cfg.mode],
                   activation(kind, **params))
