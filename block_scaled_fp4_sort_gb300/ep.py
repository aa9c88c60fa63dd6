"""Expert parallelism over ranks (cute_dsl_fused_moe: num_local_experts,
local_expert_offset; cutlass_fused_moe: ep_size, ep_rank).

Rank g of G owns a contiguous range of experts.  Every rank sees the same
tokens (x, ids and routing weights replicated); each runs the fused forward
over its own experts only -- routes to other experts are dropped by the
routing plan -- with the fp32 partial finalize, the ranks sum their partials
with one all-reduce, and moe_combine rounds the sum into the BF16 output.
The only collective is that all-reduce; everything else is the single-GPU
path on a smaller expert set.

Argument marshalling and the collective call only: the arithmetic runs in
the library's kernels (the fused forward, moe_combine) and in the
collective backend.
"""
from __future__ import annotations

import torch

from . import FINALIZE_PARTIAL_F32, moe_combine, problem
from .buffers import MoEBuffers


def expert_range(num_experts: int, world: int, rank: int):
    """(offset, count) of rank's experts: contiguous ranges, sizes differing
    by at most one, covering [0, num_experts) exactly once."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank %d of %d" % (rank, world))
    base, extra = divmod(num_experts, world)
    count = base + (1 if rank < extra else 0)
    offset = rank * base + min(rank, extra)
    return offset, count


def ep_step(local_partial, all_reduce, combine):
    """One expert-parallel forward: this rank's partial sums, their sum over
    the ranks (in place), then the rounding into the output."""
    part = local_partial()
    all_reduce(part)
    combine(part)
    return part


class ExpertParallelMoE:
    """One rank's share of an expert-parallel fused MoE forward.

    p_full: the problem over all experts (its num_local_experts and
    local_expert_offset are ignored); the rank's local problem restricts it
    to expert_range(E, world, rank)."""

    def __init__(self, p_full, world: int, rank: int, device="cuda", group=None):
        self.world, self.rank, self.group = world, rank, group
        E = p_full.num_experts
        self.offset, self.count = expert_range(E, world, rank)
        self.hidden = p_full.hidden
        self.device = torch.device(device)
        self.p = problem(p_full.num_tokens, p_full.hidden, p_full.inter, E, p_full.top_k,
                         self.count, self.offset, p_full.route_tile, p_full.mode,
                         p_full.activation) if self.count else None
        self.buffers = MoEBuffers(self.p, self.device) if self.count else None
        self._partial = None

    def prepare(self, w1, w1_sf, w2, w2_sf):
        """Prepare this rank's experts from the full weight tensors [E, ...]."""
        if self.count:
            sl = slice(self.offset, self.offset + self.count)
            self.buffers.prepare(w1[sl].clone(), w1_sf[sl].clone(), w2[sl].clone(),
                                 w2_sf[sl].clone())
        return self

    def local_alphas(self, w1_alpha, w2_alpha):
        # copies: a slice of the [E] tensors may start off a 16-byte boundary
        sl = slice(self.offset, self.offset + self.count)
        return w1_alpha[sl].clone(), w2_alpha[sl].clone()

    def local_partial(self, x, x_sf, ids, token_final_scales, w1_alpha, w2_alpha,
                      fc2_input_scale=None, rsf=1.0, stream=None, per_token_scale=None):
        """fp32 [M, H]: this rank's routes' weighted terms in route order
        (zero where a token has none of this rank's experts).  w1_alpha and
        w2_alpha are the full [E] tensors."""
        M, H = ids.shape[0], self.hidden
        if self._partial is None or self._partial.shape != (M, H):
            self._partial = torch.empty(M, H, dtype=torch.float32, device=self.device)
        if not self.count:
            self._partial.zero_()
            return self._partial
        a1, a2 = self.local_alphas(w1_alpha, w2_alpha)
        self.buffers.forward(x, x_sf, ids, token_final_scales, a1, a2, self._partial,
                             fc2_input_scale, rsf, False, finalize_mode=FINALIZE_PARTIAL_F32,
                             stream=stream, per_token_scale=per_token_scale)
        return self._partial

    def combine(self, partial, out, accumulate=False, stream=None):
        """out = bf16(partial [+ out]): the all-reduced partials into the output."""
        p = self.p if self.p is not None else self._any_problem(partial)
        moe_combine(p, partial, accumulate, out, stream)
        return out

    def forward(self, x, x_sf, ids, token_final_scales, w1_alpha, w2_alpha, out,
                fc2_input_scale=None, rsf=1.0, accumulate=False, stream=None,
                per_token_scale=None, all_reduce=None):
        """The whole expert-parallel forward on this rank; `all_reduce` sums a
        tensor over the ranks in place (default: torch.distributed over the
        group this object was made with)."""
        if all_reduce is None:
            def all_reduce(t):
                torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM, group=self.group)
        return ep_step(
            lambda: self.local_partial(x, x_sf, ids, token_final_scales, w1_alpha, w2_alpha,
                                       fc2_input_scale, rsf, stream, per_token_scale),
            all_reduce, lambda part: self.combine(part, out, accumulate, stream))

    def _any_problem(self, partial):
        # a rank without experts still rounds the summed partial: any valid
        # problem of the same M and H does
        M, H = partial.shape
        return problem(M, H, 128, 1, 1)
