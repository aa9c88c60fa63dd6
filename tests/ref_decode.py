"""Reference decoding used by the tests, independent of the oracle and of the
CUDA library: E2M1 values from the golden OCP table, E4M3 and bf16 through
torch's own float8_e4m3fn / bfloat16 conversions."""
import os

import numpy as np
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(v) for v in line.split()])
    return rows


# ---------------------------------------------------------------- decoding helpers
# independent of the oracle: E2M1 from the golden table, E4M3 via torch

E2M1_TABLE = np.array([v for _, v in _golden("e2m1_values.txt")], np.float64)
E2M1_TABLE[8] = -0.0


def e4m3_np(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).double().numpy()


def dequant_np(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """[..., K/2] packed + [..., K/16] scales -> float64 [..., K]."""
    lo = E2M1_TABLE[q & 15]
    hi = E2M1_TABLE[q >> 4]
    vals = np.stack([lo, hi], axis=-1).reshape(q.shape[:-1] + (q.shape[-1] * 2,))
    s = np.repeat(e4m3_np(sf), 16, axis=-1)
    return vals * s


def bf16_np(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def to_bf16_torch(v: np.ndarray) -> np.ndarray:
    """double -> bf16 via torch (double -> fp32 -> bf16, both RNE)."""
    return torch.from_numpy(v).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()




# ---------------------------------------------------------------- FC1 re-quantisation flips
# Where the GPU's FC1 codes differ from the oracle's, the staged check of the
# w4a4 and w4a8 forwards requires the oracle's pre-quantisation value to sit
# within `rel` (relative) of a rounding boundary: fp32 accumulation on the GPU
# and double accumulation in the oracle may then round to neighbouring codes.

def _midpoints(vals):
    v = np.unique(np.abs(vals[np.isfinite(vals)]))
    return (v[1:] + v[:-1]) / 2.0


E2M1_MIDPOINTS = _midpoints(E2M1_TABLE)                                 # 0.25 .. 5
E4M3_MIDPOINTS = _midpoints(e4m3_np(np.arange(256, dtype=np.uint8)))    # 2^-10 .. 416


def near_boundary(v, mids, rel=1e-3):
    """True if |v| lies within rel * b of one of the rounding boundaries b."""
    a = abs(float(v))
    return bool(np.any(np.abs(a - mids) <= rel * mids))


def unexplained_nvfp4_flips(h_pre, s, gpu_q, gpu_sf, orc_q, orc_sf, rel=1e-3):
    """NVFP4 FC1 output of one slot (h_pre double [I], fc2_input_scale s):
    indices of 16-blocks whose differing scale byte, or of elements whose
    differing code, is not explained by a rounding boundary of the oracle's
    pre-quantisation value (scale: amax*s/6 against the E4M3 midpoints; code:
    h*s/scale against the E2M1 midpoints; a zero of either sign is a zero)."""
    bad = []
    hs = np.asarray(h_pre, np.float64) * s
    codes_g = np.stack([gpu_q & 15, gpu_q >> 4], -1).reshape(-1)
    codes_o = np.stack([orc_q & 15, orc_q >> 4], -1).reshape(-1)
    for b in range(len(orc_sf)):
        blk = slice(16 * b, 16 * b + 16)
        if gpu_sf[b] != orc_sf[b]:
            if not near_boundary(np.abs(hs[blk]).max() / 6.0, E4M3_MIDPOINTS, rel):
                bad.append(("scale", b))
            continue
        dec = float(e4m3_np(np.array([orc_sf[b]], np.uint8))[0])
        for i in np.nonzero(codes_g[blk] != codes_o[blk])[0]:
            n = 16 * b + int(i)
            if (codes_g[n] & 7) == 0 and (codes_o[n] & 7) == 0:
                continue                      # +0 against -0
            if dec == 0.0 or not near_boundary(hs[n] / dec, E2M1_MIDPOINTS, rel):
                bad.append(("code", n))
    return bad


def unexplained_mxfp8_flips(h_pre, gpu_q, gpu_sf, orc_q, orc_sf, rel=1e-3):
    """MXFP8 FC1 output of one slot (h_pre double [I]): as above, with the
    OCP MX scale X = floor(log2 amax) - 8 per 32-block (boundary: amax at a
    power of two) and E4M3 elements h * 2^-X (boundaries: E4M3 midpoints)."""
    bad = []
    h = np.asarray(h_pre, np.float64)
    for b in range(len(orc_sf)):
        blk = slice(32 * b, 32 * b + 32)
        if gpu_sf[b] != orc_sf[b]:
            amax = np.abs(h[blk]).max()
            p2 = 2.0 ** np.round(np.log2(amax)) if amax > 0 else 0.0
            if not (amax > 0 and abs(amax - p2) <= rel * p2):
                bad.append(("scale", b))
            continue
        x = int(orc_sf[b]) - 127
        for i in np.nonzero(gpu_q[blk] != orc_q[blk])[0]:
            n = 32 * b + int(i)
            if (gpu_q[n] & 0x7F) == 0 and (orc_q[n] & 0x7F) == 0:
                continue                      # +0 against -0
            if not near_boundary(h[n] * 2.0 ** (-x), E4M3_MIDPOINTS, rel):
                bad.append(("code", n))
    return bad
