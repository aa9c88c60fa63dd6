"""The staged FC1 gate of the w4a4 / w4a8 parity tests, checked on the CPU.

The GPU tests accept an FC1 code or scale that differs from the oracle's only
where the oracle's pre-quantisation value lies within 1e-3 (relative) of a
rounding boundary.  Here the gate itself is pinned: flips planted into the
oracle's own codes are accepted at a boundary and rejected away from one.
"""
import numpy as np

import oracle
from ref_decode import (E2M1_MIDPOINTS, E4M3_MIDPOINTS, e4m3_np, unexplained_mxfp8_flips,
                        unexplained_nvfp4_flips)


def _nibble_set(q, n, code):
    q = q.copy()
    b = q[n // 2]
    q[n // 2] = (b & 0xF0) | code if n % 2 == 0 else (b & 0x0F) | (code << 4)
    return q


def _nibble(q, n):
    return (q[n // 2] >> (4 * (n % 2))) & 15


def test_boundary_tables():
    assert np.allclose(E2M1_MIDPOINTS, [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    # E4M3: smallest subnormal 2^-9 -> first midpoint 2^-10; last finite pair 416, 448
    assert E4M3_MIDPOINTS[0] == 2.0 ** -10 and E4M3_MIDPOINTS[-1] == 432.0


def test_nvfp4_gate_accepts_boundary_flips_only():
    s = 4.0
    h = np.linspace(-0.9, 1.3, 32).astype(np.float32)
    q, sf = oracle.nvfp4_quantize_f32(h, s)
    dec = float(e4m3_np(sf[:1])[0])
    assert not unexplained_nvfp4_flips(h.astype(np.float64), s, q, sf, q, sf)
    # element 3 placed just above the 1.25 midpoint (code 3 = 1.5), flipped to code 2 (1.0)
    h2 = h.astype(np.float64).copy()
    h2[3] = 1.25 * (1 + 4e-4) * dec / s
    q2, sf2 = oracle.nvfp4_quantize_f32(h2.astype(np.float32), s)
    assert np.array_equal(sf2, sf) and _nibble(q2, 3) == 3
    flipped = _nibble_set(q2, 3, 2)
    assert not unexplained_nvfp4_flips(h2, s, flipped, sf2, q2, sf2)
    # the same flip on an element far from every boundary is rejected
    far = [n for n in range(16) if min(abs(abs(h2[n] * s / dec) - E2M1_MIDPOINTS)) > 0.1]
    n = far[0]
    c = _nibble(q2, n)
    bad = unexplained_nvfp4_flips(h2, s, _nibble_set(q2, n, c ^ 1), sf2, q2, sf2)
    assert bad == [("code", n)]
    # +0 against -0 is a zero either way
    z = np.zeros(16)
    qz, sfz = oracle.nvfp4_quantize_f32(z.astype(np.float32), s)
    assert not unexplained_nvfp4_flips(z, s, _nibble_set(qz, 5, 8), sfz, qz, sfz)


def test_nvfp4_gate_scale_flip():
    s = 1.0
    # amax * s / 6 just above the E4M3 midpoint 1.0625 (between 1.0 and 1.125)
    h = np.full(16, 0.5)
    h[7] = 6.0 * 1.0625 * (1 + 5e-4)
    q, sf = oracle.nvfp4_quantize_f32(h.astype(np.float32), s)
    other = sf.copy()
    other[0] = 0x38                      # E4M3 1.0, the neighbour below
    assert not unexplained_nvfp4_flips(h, s, q, other, q, sf)
    h[7] = 6.0 * 1.1                     # far from a boundary
    q, sf = oracle.nvfp4_quantize_f32(h.astype(np.float32), s)
    other = sf.copy()
    other[0] ^= 1
    assert unexplained_nvfp4_flips(h, s, q, other, q, sf) == [("scale", 0)]


def test_mxfp8_gate():
    rng = np.random.default_rng(3)
    h = rng.standard_normal(64)
    q, sf = oracle.mxfp8_quantize_f32(h.astype(np.float32))
    assert not unexplained_mxfp8_flips(h, q, sf, q, sf)
    # an element far from an E4M3 boundary, flipped by one code: rejected
    x = int(sf[0]) - 127
    n = next(i for i in range(32)
             if min(abs(abs(h[i] * 2.0 ** -x) - E4M3_MIDPOINTS) / E4M3_MIDPOINTS) > 0.01)
    q2 = q.copy()
    q2[n] ^= 1
    assert unexplained_mxfp8_flips(h, q2, sf, q, sf) == [("code", n)]
    # block amax just below a power of two: a scale flip is explained
    h3 = h.copy()
    h3[:32] *= 0.5 / np.abs(h3[:32]).max()
    h3[0] = 0.5 * (1 - 3e-4)
    q3, sf3 = oracle.mxfp8_quantize_f32(h3.astype(np.float32))
    other = sf3.copy()
    other[0] += 1
    assert not unexplained_mxfp8_flips(h3, q3, other, q3, sf3)
    other = sf3.copy()
    other[1] += 1                        # second block: amax not at a power of two
    assert unexplained_mxfp8_flips(h3, q3, other, q3, sf3) == [("scale", 1)]
