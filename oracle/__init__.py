"""CPU oracle for the NVFP4 fused-MoE forward -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this package.  The product path (block_scaled_fp4_sort_gb300) never
does.  The C source (fp4moe_oracle.c) is built with gcc on first use (or by
__graft_entry__.build()), with -ffp-contract=off so no multiply-add fuses.

Parity status of each function (what pins it) is listed in the test file
tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4moe_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liborc_fp4moe.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, plain C11)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "fp4moe_oracle.h"))):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


class Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("M", "H", "I", "E", "top_k", "E_local", "offset", "T", "mode", "act_type",
                 "act_flags")] + [(n, ctypes.c_double) for n in
                                  ("swiglu_alpha", "swiglu_beta", "swiglu_limit", "situ_beta",
                                   "situ_linear_beta")]


class Inputs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("x_q", ctypes.c_void_p), ("x_sf", ctypes.c_void_p),
                ("ids", ctypes.c_void_p), ("wts", ctypes.c_void_p),
                ("w1", ctypes.c_void_p), ("w1_sf", ctypes.c_void_p), ("w1_alpha", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_sf", ctypes.c_void_p), ("w2_alpha", ctypes.c_void_p),
                ("fc2_input_scale", ctypes.c_void_p), ("per_token_scale", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            d, u32, i32, i64, vp = (ctypes.c_double, ctypes.c_uint32, ctypes.c_int32,
                                    ctypes.c_int64, ctypes.c_void_p)
            for name in ("orc_e2m1_value", "orc_e4m3_value", "orc_bf16_value"):
                getattr(L, name).restype = d
                getattr(L, name).argtypes = [u32]
            for name in ("orc_round_bf16", "orc_round_e4m3_satfinite", "orc_round_e2m1_satfinite"):
                getattr(L, name).restype = d
                getattr(L, name).argtypes = [d]
            for name in ("orc_bf16_bits", "orc_e4m3_code_satfinite", "orc_e2m1_code_satfinite"):
                getattr(L, name).restype = u32
                getattr(L, name).argtypes = [d]
            L.orc_nvfp4_quantize_f32.restype = None
            L.orc_nvfp4_quantize_f32.argtypes = [vp, i64, ctypes.c_float, vp, vp]
            L.orc_ue8m0_value.restype = d
            L.orc_ue8m0_value.argtypes = [u32]
            L.orc_mxfp8_quantize_f32.restype = None
            L.orc_mxfp8_quantize_f32.argtypes = [vp, i64, vp, vp]
            L.orc_max_permuted_slots.restype = i64
            L.orc_max_permuted_slots.argtypes = [i64, i32, i32]
            L.orc_route_sort.restype = i32
            L.orc_route_sort.argtypes = [ctypes.POINTER(Problem), vp, vp, vp, vp, vp, vp, vp]
            L.orc_expert_ffn.restype = None
            L.orc_expert_ffn.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Inputs), i32, vp,
                                         vp, vp, vp, vp, vp, vp, vp]
            L.orc_expert_down_nvfp4.restype = None
            L.orc_expert_down_nvfp4.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Inputs),
                                                i32, vp, vp, vp]
            L.orc_xhat.restype = None
            L.orc_xhat.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Inputs), i64, vp]
            L.orc_moe_tokens.restype = i32
            L.orc_moe_tokens.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Inputs), vp, i64,
                                         ctypes.c_float, i32, vp, vp, vp, i32]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------------------
# numpy-level wrappers
# ---------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(bits)


def round_bf16(v: float) -> float:
    return lib().orc_round_bf16(v)


def bf16_bits(v: float) -> int:
    return lib().orc_bf16_bits(v)


def round_e4m3(v: float) -> float:
    return lib().orc_round_e4m3_satfinite(v)


def e4m3_code(v: float) -> int:
    return lib().orc_e4m3_code_satfinite(v)


def round_e2m1(v: float) -> float:
    return lib().orc_round_e2m1_satfinite(v)


def e2m1_code(v: float) -> int:
    return lib().orc_e2m1_code_satfinite(v)


def nvfp4_quantize_f32(h: np.ndarray, s: float):
    """fp32 NVFP4 quantiser of the w4a4 FC1 output.  h: float32 [..., n]."""
    h = np.ascontiguousarray(h, dtype=np.float32)
    n = h.size
    q = np.zeros(n // 2, np.uint8)
    sf = np.zeros(n // 16, np.uint8)
    lib().orc_nvfp4_quantize_f32(_ptr(h), n, ctypes.c_float(s), _ptr(q), _ptr(sf))
    return q.reshape(h.shape[:-1] + (h.shape[-1] // 2,)), sf.reshape(h.shape[:-1] + (h.shape[-1] // 16,))


def ue8m0_value(code: int) -> float:
    return lib().orc_ue8m0_value(code)


def mxfp8_quantize_f32(h: np.ndarray):
    """fp32 MXFP8 quantiser of the w4a8 FC1 output.  h: float32 [..., n], n % 32 == 0."""
    h = np.ascontiguousarray(h, dtype=np.float32)
    n = h.size
    q = np.zeros(n, np.uint8)
    sf = np.zeros(n // 32, np.uint8)
    lib().orc_mxfp8_quantize_f32(_ptr(h), n, _ptr(q), _ptr(sf))
    return q.reshape(h.shape), sf.reshape(h.shape[:-1] + (h.shape[-1] // 32,))


def max_permuted_slots(routes: int, E_local: int, T: int) -> int:
    return int(lib().orc_max_permuted_slots(routes, E_local, T))


class OracleMoE:
    """Holds host copies (numpy) of one workload and evaluates the oracle on it."""

    def __init__(self, M, H, I, E, top_k, ids, wts, w1, w1_sf, w1_alpha, w2, w2_sf, w2_alpha,
                 x=None, x_q=None, x_sf=None, fc2_input_scale=None, E_local=None, offset=0, T=16,
                 act_type=0, act_params=None, per_token_scale=None, mode=None):
        """act_type / act_params: the FC1 activation (0 SwiGLU family with optional
        swiglu_alpha/beta/limit or situ_beta/situ_linear_beta, 1 GeGLU-tanh,
        2 non-gated ReLU^2); per_token_scale: fp32 [M] or None."""
        c = np.ascontiguousarray
        self.arrays = dict(
            x=None if x is None else c(x, dtype=np.uint16),
            x_q=None if x_q is None else c(x_q, dtype=np.uint8),
            x_sf=None if x_sf is None else c(x_sf, dtype=np.uint8),
            ids=c(ids, dtype=np.int32), wts=c(wts, dtype=np.float32),
            w1=c(w1, dtype=np.uint8), w1_sf=c(w1_sf, dtype=np.uint8),
            w1_alpha=c(w1_alpha, dtype=np.float32),
            w2=c(w2, dtype=np.uint8), w2_sf=c(w2_sf, dtype=np.uint8),
            w2_alpha=c(w2_alpha, dtype=np.float32),
            fc2_input_scale=None if fc2_input_scale is None else c(fc2_input_scale, dtype=np.float32),
            per_token_scale=None if per_token_scale is None else c(per_token_scale, dtype=np.float32))
        if mode is None:                     # 0 w4a16, 1 w4a4, 2 w4a8 (MXFP8 x, MXFP4 weights)
            mode = 0 if x is not None else 1
        E_local = E if E_local is None else E_local
        ap = dict(act_params or {})
        flags = 0
        if {"swiglu_alpha", "swiglu_beta", "swiglu_limit"} & set(ap):
            flags |= 1
        if "situ_beta" in ap:
            flags |= 2
        if "situ_linear_beta" in ap:
            flags |= 4
        self.p = Problem(M, H, I, E, top_k, E_local, offset, T, mode, act_type, flags,
                         float(ap.get("swiglu_alpha", 1.0)), float(ap.get("swiglu_beta", 0.0)),
                         float(ap.get("swiglu_limit", float("inf"))), float(ap.get("situ_beta", 0.0)),
                         float(ap.get("situ_linear_beta", 0.0)))
        self.inp = Inputs(**{k: _ptr(v) for k, v in self.arrays.items()})

    @classmethod
    def from_inputs(cls, inp, T=16, E_local=None, offset=0):
        """Build from a synth.MoEInputs (tensors anywhere; copied to host)."""
        cfg = inp.cfg

        def h(t):
            if t is None:
                return None
            t = t.detach().cpu().contiguous()
            if t.dtype == _bf16():
                return t.view(_i16()).numpy().view(np.uint16)
            return t.numpy()
        import synth
        act_type, act_params = synth.activation_spec(cfg)
        return cls(cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k, h(inp.token_selected_experts),
                   h(inp.token_final_scales), h(inp.w1), h(inp.w1_sf), h(inp.w1_alpha), h(inp.w2),
                   h(inp.w2_sf), h(inp.w2_alpha), x=h(inp.x), x_q=h(inp.x_q), x_sf=h(inp.x_sf),
                   fc2_input_scale=h(inp.fc2_input_scale), E_local=E_local, offset=offset, T=T,
                   act_type=act_type, act_params=act_params,
                   per_token_scale=h(getattr(inp, "per_token_scale", None)),
                   mode={"w4a16": 0, "w4a4": 1, "w4a8": 2}[cfg.mode])

    @property
    def H(self):
        return self.p.H

    @property
    def I(self):
        return self.p.I

    def route_sort(self):
        p = self.p
        R = p.M * p.top_k
        S = max_permuted_slots(R, p.E_local, p.T)
        e2p = np.zeros(R, np.int32)
        p2e = np.zeros(S, np.int32)
        te = np.zeros(S // p.T, np.int32)
        tm = np.zeros(S // p.T, np.int32)
        nt = np.zeros(1, np.int32)
        cnt = np.zeros(p.E_local, np.int32)
        bad = lib().orc_route_sort(ctypes.byref(p), _ptr(self.arrays["ids"]), _ptr(e2p), _ptr(p2e),
                                   _ptr(te), _ptr(tm), _ptr(nt), _ptr(cnt))
        return dict(expanded_idx_to_permuted_idx=e2p.reshape(p.M, p.top_k),
                    permuted_idx_to_expanded_idx=p2e, tile_idx_to_expert=te,
                    tile_idx_to_mn_limit=tm, num_non_exiting_tiles=int(nt[0]), expert_counts=cnt,
                    bad=bool(bad))

    def xhat(self, t):
        out = np.zeros(self.p.H, np.float64)
        lib().orc_xhat(ctypes.byref(self.p), ctypes.byref(self.inp), int(t), _ptr(out))
        return out

    def expert_ffn(self, e_local, t):
        """Staged values for token t through local expert e_local."""
        p = self.p
        xh = self.xhat(t)
        g = np.zeros(p.I); u = np.zeros(p.I); hp = np.zeros(p.I); hi = np.zeros(p.I)
        y = np.zeros(p.H)
        mx = p.mode == 2                      # w4a8: MXFP8 codes of h
        hq = np.zeros(p.I if mx else p.I // 2, np.uint8)
        hsf = np.zeros(p.I // (32 if mx else 16), np.uint8)
        lib().orc_expert_ffn(ctypes.byref(p), ctypes.byref(self.inp), int(e_local), _ptr(xh),
                             _ptr(g), _ptr(u), _ptr(hp), _ptr(hi), _ptr(hq), _ptr(hsf), _ptr(y))
        return dict(g=g, u=u, h_pre=hp, h_in=hi, hq=hq, hsf=hsf, y=y)

    def expert_down_codes(self, e_local, hq, hsf):
        """GEMM2 alone from FC1 codes: NVFP4 (w4a4: hq [I/2], hsf [I/16]) or MXFP8
        (w4a8: hq [I], hsf [I/32])."""
        y = np.zeros(self.p.H)
        hq = np.ascontiguousarray(hq, np.uint8)
        hsf = np.ascontiguousarray(hsf, np.uint8)
        lib().orc_expert_down_nvfp4(ctypes.byref(self.p), ctypes.byref(self.inp), int(e_local),
                                    _ptr(hq), _ptr(hsf), _ptr(y))
        return y

    def forward(self, tokens=None, rsf=1.0, accumulate=False, out_old=None, nthreads=1):
        """Oracle rows for `tokens`: (bf16 bits uint16 [n, H], exact double [n, H], bad)."""
        p = self.p
        toks = np.arange(p.M, dtype=np.int64) if tokens is None else np.ascontiguousarray(
            tokens, dtype=np.int64)
        n = toks.size
        out = np.zeros((n, p.H), np.uint16)
        ex = np.zeros((n, p.H), np.float64)
        old = None
        if accumulate:
            old = np.ascontiguousarray(out_old, dtype=np.uint16)
            assert old.shape == (n, p.H)
        bad = lib().orc_moe_tokens(ctypes.byref(p), ctypes.byref(self.inp), _ptr(toks), n,
                                   ctypes.c_float(rsf), int(bool(accumulate)), _ptr(old), _ptr(out),
                                   _ptr(ex), int(nthreads))
        return out, ex, bool(bad)


def route_plan(M, E, top_k, T, ids, E_local=None, offset=0):
    """Oracle routing plan for ids [M, top_k] (no weights needed)."""
    E_local = E if E_local is None else E_local
    z = np.zeros
    o = OracleMoE(M, 128, 128, E, top_k, np.asarray(ids, np.int32).reshape(M, top_k),
                  z((M, top_k), np.float32), z((1, 256, 64), np.uint8), z((1, 256, 8), np.uint8),
                  z(1, np.float32), z((1, 128, 64), np.uint8), z((1, 128, 8), np.uint8),
                  z(1, np.float32), x=z((max(M, 1), 128), np.uint16), E_local=E_local,
                  offset=offset, T=T)
    return o.route_sort()


def _bf16():
    import torch
    return torch.bfloat16


def _i16():
    import torch
    return torch.int16


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of bf16 bit patterns (vectorised; bf16 -> fp32 is a shift)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
