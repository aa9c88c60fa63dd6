"""Python binding of libfp4moe (the GB300 NVFP4 fused-MoE forward).

Argument marshalling only: every function here forwards torch tensors'
device pointers and sizes to the C ABI of include/fp4moe.h and raises
Fp4MoeError on a non-OK status.  There is no fallback: if the CUDA library is
not built, importing the functions raises.  Build it with
`python -m block_scaled_fp4_sort_gb300.build` (or __graft_entry__.build()).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp4moe.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_DEVICE, ERR_DEVICE_TIMEOUT = range(7)
W4A16, W4A4, W4A8 = 0, 1, 2
FINALIZE_DETERMINISTIC, FINALIZE_ATOMIC, FINALIZE_PARTIAL_F32 = 0, 1, 2

ABI_FUNCTIONS = (
    "fp4moe_status_string", "fp4moe_route_tile", "fp4moe_max_permuted_slots",
    "fp4moe_route_workspace_size", "fp4moe_gemm_workspace_size", "fp4moe_workspace_size",
    "fp4moe_prepared_weight_size", "fp4moe_read_error", "fp4moe_clear_error",
    "fp4moe_prepare_weights", "moe_route_sort", "moe_route_sort_noalloc", "moe_permute", "moe_gemm1_swiglu", "moe_gemm2",
    "moe_finalize", "fused_moe_forward", "moe_combine", "fp4moe_debug_quantize_nvfp4",
    "fp4moe_debug_quantize_mxfp8", "fp4moe_debug_decode_prepared", "fp4moe_debug_wait_timeout",
    "fp4moe_domain_weight_size", "fp4moe_prepare_domain_weights",
    "fp4moe_localized_workspace_size", "fused_moe_forward_localized", "fp4moe_domains_create",
    "fp4moe_domains_stream", "fp4moe_domains_destroy",
)


class Fp4MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


ACT_SWIGLU, ACT_GEGLU_TANH, ACT_RELU2 = 0, 1, 2
ACT_F_SWIGLU_OAI, ACT_F_SITU, ACT_F_SITU_LINEAR = 1, 2, 4


class Activation(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("swiglu_alpha", ctypes.c_float), ("swiglu_beta", ctypes.c_float),
                ("swiglu_limit", ctypes.c_float), ("situ_beta", ctypes.c_float),
                ("situ_linear_beta", ctypes.c_float)]


class Problem(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("num_local_experts", ctypes.c_int32),
                ("local_expert_offset", ctypes.c_int32), ("route_tile", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("activation", Activation)]


class Localized(ctypes.Structure):
    """fp4moe_localized: the two domains' prepared shards and streams."""
    _fields_ = [("w1_prepared", ctypes.c_void_p * 2), ("w2_prepared", ctypes.c_void_p * 2),
                ("streams", ctypes.c_void_p * 2), ("sm_count", ctypes.c_int32),
                ("memset_stream", ctypes.c_void_p)]


def activation(type=ACT_SWIGLU, swiglu_alpha=None, swiglu_beta=None, swiglu_limit=None,
               situ_beta=None, situ_linear_beta=None) -> Activation:
    """The FC1 activation; swiglu_* parameters select swiglu_oai (defaults 1, 0,
    +inf), situ_beta selects SiTU, situ_linear_beta adds its up-branch clamp."""
    a = Activation(type, 0, 1.0, 0.0, float("inf"), 0.0, 0.0)
    if swiglu_alpha is not None or swiglu_beta is not None or swiglu_limit is not None:
        a.flags |= ACT_F_SWIGLU_OAI
        a.swiglu_alpha = 1.0 if swiglu_alpha is None else swiglu_alpha
        a.swiglu_beta = 0.0 if swiglu_beta is None else swiglu_beta
        a.swiglu_limit = float("inf") if swiglu_limit is None else swiglu_limit
    if situ_beta is not None:
        a.flags |= ACT_F_SITU
        a.situ_beta = situ_beta
    if situ_linear_beta is not None:
        a.flags |= ACT_F_SITU_LINEAR
        a.situ_linear_beta = situ_linear_beta
    return a


def problem(num_tokens, hidden, inter, num_experts, top_k, num_local_experts=0,
            local_expert_offset=0, route_tile=0, mode=W4A16, act=None) -> Problem:
    return Problem(num_tokens, hidden, inter, num_experts, top_k, num_local_experts,
                   local_expert_offset, route_tile, mode, act if act is not None else Activation())


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libfp4moe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libfp4moe.so is not built (%s); run "
                               "`python -m block_scaled_fp4_sort_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        P = ctypes.POINTER(Problem)
        sig = {
            "fp4moe_status_string": (ctypes.c_char_p, [i32]),
            "fp4moe_route_tile": (i32, [P]),
            "fp4moe_max_permuted_slots": (i64, [P]),
            "fp4moe_route_workspace_size": (sz, [P]),
            "fp4moe_gemm_workspace_size": (sz, [P, i32]),
            "fp4moe_workspace_size": (sz, [P]),
            "fp4moe_prepared_weight_size": (sz, [P, i32]),
            "fp4moe_read_error": (i32, [vp, ctypes.POINTER(i32), vp]),
            "fp4moe_clear_error": (i32, [vp, vp]),
            "fp4moe_prepare_weights": (i32, [P, i32, vp, vp, vp, vp]),
            "moe_route_sort": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "moe_route_sort_noalloc": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "moe_permute": (i32, [P, vp, vp, vp, vp, vp, vp, vp]),
            "moe_gemm1_swiglu": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                       vp]),
            "moe_gemm2": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "moe_finalize": (i32, [P, vp, vp, vp, f32, i32, vp, vp]),
            "fused_moe_forward": (i32, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, vp,
                                        vp, sz, vp]),
            "moe_combine": (i32, [P, vp, i32, vp, vp]),
            "fp4moe_debug_quantize_nvfp4": (i32, [vp, i64, vp, vp, vp, vp]),
            "fp4moe_debug_quantize_mxfp8": (i32, [vp, i64, vp, vp, vp]),
            "fp4moe_debug_decode_prepared": (i32, [P, i32, vp, vp, vp]),
            "fp4moe_debug_wait_timeout": (i32, [i64, vp, vp]),
            "fp4moe_domain_weight_size": (sz, [P, i32]),
            "fp4moe_prepare_domain_weights": (i32, [P, i32, vp, vp, vp, vp]),
            "fp4moe_localized_workspace_size": (sz, [P]),
            "fused_moe_forward_localized": (i32, [P, vp, vp, vp, vp, ctypes.POINTER(Localized), vp,
                                                  vp, vp, vp, f32, i32, i32, vp, vp, sz, vp]),
            "fp4moe_domains_create": (i32, [i32, i32, ctypes.POINTER(vp)]),
            "fp4moe_domains_stream": (i32, [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(i32)]),
            "fp4moe_domains_destroy": (i32, [vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fp4moe_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise Fp4MoeError(status, where)


def _p(t) -> Optional[int]:
    """Device pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    return t.data_ptr()


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- queries

def route_tile(p: Problem) -> int:
    v = lib().fp4moe_route_tile(ctypes.byref(p))
    if v < 0:
        raise Fp4MoeError(-v, "fp4moe_route_tile")
    return v


def max_permuted_slots(p: Problem) -> int:
    v = lib().fp4moe_max_permuted_slots(ctypes.byref(p))
    if v < 0:
        raise Fp4MoeError(-v, "fp4moe_max_permuted_slots")
    return v


def route_workspace_size(p: Problem) -> int:
    return lib().fp4moe_route_workspace_size(ctypes.byref(p))


def gemm_workspace_size(p: Problem, which: int) -> int:
    return lib().fp4moe_gemm_workspace_size(ctypes.byref(p), which)


def workspace_size(p: Problem) -> int:
    return lib().fp4moe_workspace_size(ctypes.byref(p))


def prepared_weight_size(p: Problem, which: int) -> int:
    return lib().fp4moe_prepared_weight_size(ctypes.byref(p), which)


def read_error(workspace, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(lib().fp4moe_read_error(_p(workspace), ctypes.byref(code), _stream(stream)),
           "fp4moe_read_error")
    return code.value


def clear_error(workspace, stream=None):
    _check(lib().fp4moe_clear_error(_p(workspace), _stream(stream)), "fp4moe_clear_error")


# ---------------------------------------------------------------- entry points

def prepare_weights(p: Problem, which: int, w, w_sf, prepared, stream=None):
    _check(lib().fp4moe_prepare_weights(ctypes.byref(p), which, _p(w), _p(w_sf), _p(prepared),
                                        _stream(stream)), "fp4moe_prepare_weights")


def moe_route_sort(p: Problem, token_selected_experts, expanded_idx_to_permuted_idx,
                   permuted_idx_to_expanded_idx, tile_idx_to_expert, tile_idx_to_mn_limit,
                   num_non_exiting_tiles, expert_counts, workspace, stream=None):
    _check(lib().moe_route_sort(ctypes.byref(p), _p(token_selected_experts),
                                _p(expanded_idx_to_permuted_idx), _p(permuted_idx_to_expanded_idx),
                                _p(tile_idx_to_expert), _p(tile_idx_to_mn_limit),
                                _p(num_non_exiting_tiles), _p(expert_counts), _p(workspace),
                                _nbytes(workspace), _stream(stream)), "moe_route_sort")


def moe_route_sort_noalloc(p: Problem, token_selected_experts, expanded_idx_to_permuted_idx,
                           permuted_idx_to_expanded_idx, tile_idx_to_expert, tile_idx_to_mn_limit,
                           num_non_exiting_tiles, expert_counts=None, error_flag=None, stream=None):
    """moe_route_sort without a workspace: the library keeps its scratch in a
    static device array (for callers that cannot allocate device memory)."""
    _check(lib().moe_route_sort_noalloc(ctypes.byref(p), _p(token_selected_experts),
                                        _p(expanded_idx_to_permuted_idx),
                                        _p(permuted_idx_to_expanded_idx), _p(tile_idx_to_expert),
                                        _p(tile_idx_to_mn_limit), _p(num_non_exiting_tiles),
                                        _p(expert_counts), _p(error_flag), _stream(stream)),
           "moe_route_sort_noalloc")


def moe_permute(p: Problem, x, x_sf, permuted_idx_to_expanded_idx, num_non_exiting_tiles,
                permuted_x, permuted_x_sf=None, stream=None):
    _check(lib().moe_permute(ctypes.byref(p), _p(x), _p(x_sf), _p(permuted_idx_to_expanded_idx),
                             _p(num_non_exiting_tiles), _p(permuted_x), _p(permuted_x_sf),
                             _stream(stream)), "moe_permute")


def moe_gemm1_swiglu(p: Problem, a, a_sf, gather_rows, w1_prepared, w1_alpha, fc2_input_scale,
                     tile_idx_to_expert, tile_idx_to_mn_limit, num_non_exiting_tiles, h, h_sf,
                     workspace, stream=None, per_token_scale=None):
    _check(lib().moe_gemm1_swiglu(ctypes.byref(p), _p(a), _p(a_sf), _p(gather_rows),
                                  _p(w1_prepared), _p(w1_alpha), _p(fc2_input_scale),
                                  _p(per_token_scale), _p(tile_idx_to_expert), _p(tile_idx_to_mn_limit),
                                  _p(num_non_exiting_tiles), _p(h), _p(h_sf), _p(workspace),
                                  _nbytes(workspace), _stream(stream)), "moe_gemm1_swiglu")


def moe_gemm2(p: Problem, h, h_sf, w2_prepared, w2_alpha, tile_idx_to_expert,
              tile_idx_to_mn_limit, num_non_exiting_tiles, y, workspace, stream=None):
    _check(lib().moe_gemm2(ctypes.byref(p), _p(h), _p(h_sf), _p(w2_prepared), _p(w2_alpha),
                           _p(tile_idx_to_expert), _p(tile_idx_to_mn_limit),
                           _p(num_non_exiting_tiles), _p(y), _p(workspace), _nbytes(workspace),
                           _stream(stream)), "moe_gemm2")


def moe_finalize(p: Problem, y, expanded_idx_to_permuted_idx, token_final_scales,
                 routed_scaling_factor, accumulate, out, stream=None):
    _check(lib().moe_finalize(ctypes.byref(p), _p(y), _p(expanded_idx_to_permuted_idx),
                              _p(token_final_scales), float(routed_scaling_factor),
                              int(bool(accumulate)), _p(out), _stream(stream)), "moe_finalize")


def fused_moe_forward(p: Problem, x, x_sf, token_selected_experts, token_final_scales,
                      w1_prepared, w1_alpha, fc2_input_scale, w2_prepared, w2_alpha,
                      routed_scaling_factor, accumulate, finalize_mode, out, workspace,
                      stream=None, per_token_scale=None):
    _check(lib().fused_moe_forward(ctypes.byref(p), _p(x), _p(x_sf), _p(token_selected_experts),
                                   _p(token_final_scales), _p(w1_prepared), _p(w1_alpha),
                                   _p(fc2_input_scale), _p(per_token_scale), _p(w2_prepared),
                                   _p(w2_alpha),
                                   float(routed_scaling_factor), int(bool(accumulate)),
                                   int(finalize_mode), _p(out), _p(workspace), _nbytes(workspace),
                                   _stream(stream)), "fused_moe_forward")


def moe_combine(p: Problem, partial, accumulate, out, stream=None):
    _check(lib().moe_combine(ctypes.byref(p), _p(partial), int(bool(accumulate)), _p(out),
                             _stream(stream)), "moe_combine")


def debug_quantize_mxfp8(x, q, sf, stream=None):
    _check(lib().fp4moe_debug_quantize_mxfp8(_p(x), x.numel(), _p(q), _p(sf), _stream(stream)),
           "fp4moe_debug_quantize_mxfp8")


def debug_quantize_nvfp4(x, scale, q, sf, stream=None):
    _check(lib().fp4moe_debug_quantize_nvfp4(_p(x), x.numel(), _p(scale), _p(q), _p(sf),
                                             _stream(stream)), "fp4moe_debug_quantize_nvfp4")


def debug_wait_timeout(limit_ns: int, workspace, stream=None):
    _check(lib().fp4moe_debug_wait_timeout(int(limit_ns), _p(workspace), _stream(stream)),
           "fp4moe_debug_wait_timeout")


def debug_decode_prepared(p: Problem, which: int, prepared, out, stream=None):
    _check(lib().fp4moe_debug_decode_prepared(ctypes.byref(p), which, _p(prepared), _p(out),
                                              _stream(stream)), "fp4moe_debug_decode_prepared")


# ------------------------------------------------ two locality domains

def domain_weight_size(p: Problem, which: int) -> int:
    return lib().fp4moe_domain_weight_size(ctypes.byref(p), which)


def localized_workspace_size(p: Problem) -> int:
    return lib().fp4moe_localized_workspace_size(ctypes.byref(p))


def prepare_domain_weights(p: Problem, which: int, w_shard, w_sf_shard, prepared, stream=None):
    _check(lib().fp4moe_prepare_domain_weights(ctypes.byref(p), which, _p(w_shard), _p(w_sf_shard),
                                               _p(prepared), _stream(stream)),
           "fp4moe_prepare_domain_weights")


def localized(w1_prepared, w2_prepared, streams, sm_count=0, memset_stream=None) -> Localized:
    """Localized from two prepared shards per GEMM and two streams (torch
    streams or raw cudaStream_t handles)."""
    raw = lambda st: None if st is None else (st if isinstance(st, int) else st.cuda_stream)
    L = Localized()
    for d in range(2):
        L.w1_prepared[d] = _p(w1_prepared[d])
        L.w2_prepared[d] = _p(w2_prepared[d])
        L.streams[d] = raw(streams[d])
    L.sm_count = int(sm_count)
    L.memset_stream = raw(memset_stream)
    return L


def fused_moe_forward_localized(p: Problem, x, x_sf, token_selected_experts, token_final_scales,
                                loc: Localized, w1_alpha, fc2_input_scale, w2_alpha,
                                routed_scaling_factor, accumulate, finalize_mode, out, workspace,
                                stream=None, per_token_scale=None):
    _check(lib().fused_moe_forward_localized(
        ctypes.byref(p), _p(x), _p(x_sf), _p(token_selected_experts), _p(token_final_scales),
        ctypes.byref(loc), _p(w1_alpha), _p(fc2_input_scale), _p(per_token_scale), _p(w2_alpha),
        float(routed_scaling_factor), int(bool(accumulate)), int(finalize_mode), _p(out),
        _p(workspace), _nbytes(workspace), _stream(stream)), "fused_moe_forward_localized")


class Domains:
    """Two green-context locality domains of one device (fp4moe_domains_*)."""

    def __init__(self, device: int = 0, min_sm_count: int = 0):
        h = ctypes.c_void_p()
        _check(lib().fp4moe_domains_create(int(device), int(min_sm_count), ctypes.byref(h)),
               "fp4moe_domains_create")
        self._h = h
        self.streams = []
        self.sm_count = 0
        for i in range(2):
            st, n = ctypes.c_void_p(), ctypes.c_int32()
            _check(lib().fp4moe_domains_stream(h, i, ctypes.byref(st), ctypes.byref(n)),
                   "fp4moe_domains_stream")
            self.streams.append(int(st.value))
            self.sm_count = int(n.value)

    def close(self):
        if self._h is not None:
            _check(lib().fp4moe_domains_destroy(self._h), "fp4moe_domains_destroy")
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
