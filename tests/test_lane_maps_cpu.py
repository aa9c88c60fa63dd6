"""Index arithmetic of the atomic-finalize epilogues, checked on the CPU.

The two-tile and native GEMM2 epilogues hold, in lane L of a warp, the fp32
accumulators of feature row L for 16 consecutive slot columns.  Before the
16-byte atomic adds, each quad of lanes (features 4g..4g+3) transposes every
4 x 4 block: in round r lane q (= L % 4) sends its column (q + r) % 4 and reads
lane 4g + (q - r) % 4, so after four rounds lane q holds the four features of
slot column 4c + q.  These tests replay that schedule with the warp shuffle
modelled as "read the sender's chosen value", and check the 16-byte alignment
of every add's target.
"""
import numpy as np
import pytest


def quad_transpose(v):
    """v[lane][col] for 32 lanes and 16 columns -> b[lane][c][k], the value the
    kernel leaves in lane `lane` for sub-block c, element k."""
    lanes = np.arange(32)
    b = np.full((32, 4, 4), np.nan)
    for c in range(4):
        for r in range(4):
            q = lanes & 3
            send = v[lanes, 4 * c + ((q + r) & 3)]       # each lane's outgoing value
            k = (q - r) & 3
            src = (lanes & ~3) | k                       # __shfl_sync source lane
            b[lanes, c, k] = send[src]
    return b


def test_quad_transpose_gives_each_lane_one_slot_four_features():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((32, 16))
    b = quad_transpose(v)
    for lane in range(32):
        g, q = lane >> 2, lane & 3
        for c in range(4):
            # lane q of quad g: slot column 4c + q, features 4g .. 4g + 3
            assert np.array_equal(b[lane, c], v[4 * g: 4 * g + 4, 4 * c + q])


def test_every_value_is_added_exactly_once():
    v = np.arange(32 * 16, dtype=np.float64).reshape(32, 16)
    b = quad_transpose(v)
    assert sorted(b.ravel().tolist()) == sorted(v.ravel().tolist())


@pytest.mark.parametrize("H,out_ld", [(256, 256), (6144, 6144), (7168, 7168)])
def test_atomic_targets_are_16_byte_aligned(H, out_ld):
    # feature n = f * 256 + tile * 128 + row (two-tile kernel) or f * 128 + row
    # (native kernel), row = 32 * lane_quarter + lane; the add starts at n - q
    for f in range(H // 256):
        for tile in range(2):
            for row in range(128):
                n = f * 256 + tile * 128 + row
                q = (row & 31) & 3
                for t in (0, 1, 7):
                    byte = 4 * (t * out_ld + n - q)
                    assert byte % 16 == 0
