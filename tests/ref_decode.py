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


