"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and validates arguments on the host (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import block_scaled_fp4_sort_gb300 as fm
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4moe.h")


def _declared():
    src = open(HEADER).read()
    return re.findall(r"^FP4MOE_API [^(]*?\b([a-z_0-9]+)\(", src, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    from block_scaled_fp4_sort_gb300 import build
    build.build()
    return fm.lib()


def test_header_declares_the_six_entry_points():
    names = set(_declared())
    for n in ("moe_route_sort", "moe_permute", "moe_gemm1_swiglu", "moe_gemm2", "moe_finalize",
              "fused_moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared()
    assert names and set(names) == set(fm.ABI_FUNCTIONS)
    raw = ctypes.CDLL(fm.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_product_does_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "block_scaled_fp4_sort_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fp4moe_oracle" not in text and "orc_" not in text, f


@pytest.mark.parametrize("M,E,k,T", [(8, 256, 8, 16), (4096, 256, 8, 128), (2048, 128, 4, 64),
                                     (131072, 256, 8, 128), (16, 8, 2, 16), (1, 1, 1, 32), (0, 4, 2, 16),
                                     (8, 256, 8, 8), (131072, 256, 8, 256), (2048, 128, 4, 256)])
def test_slot_bound_matches_oracle(lib, M, E, k, T):
    p = fm.problem(M, 256, 256, E, k, route_tile=T)
    assert fm.max_permuted_slots(p) == oracle.max_permuted_slots(M * k, E, T)
    assert fm.route_tile(p) == T


def test_auto_route_tile(lib):
    assert fm.route_tile(fm.problem(8, 7168, 2048, 256, 8)) == 16
    assert fm.route_tile(fm.problem(4096, 7168, 2048, 256, 8)) == 128
    assert fm.route_tile(fm.problem(2048, 4096, 1536, 128, 4)) == 128   # BF16: twice the average
    assert fm.route_tile(fm.problem(2048, 4096, 1536, 128, 4, mode=fm.W4A4)) == 64
    assert fm.route_tile(fm.problem(128, 256, 256, 8, 2)) == 64            # average 32, doubled
    assert fm.route_tile(fm.problem(64, 256, 256, 8, 2)) == 16             # average 16: as it is
    assert fm.route_tile(fm.problem(131072, 6144, 2048, 256, 8)) == 128


def test_sizes(lib):
    p = fm.problem(8, 7168, 2048, 256, 8)
    assert fm.workspace_size(p) > 0
    assert fm.prepared_weight_size(p, 1) == 256 * 16 * 56 * 18432      # I/128 blocks x H/128 chunks
    assert fm.prepared_weight_size(p, 2) == 256 * 28 * 16 * 18432      # H/256 blocks x I/128 chunks
    assert fm.gemm_workspace_size(p, 1) >= 256
    assert fm.prepared_weight_size(p, 3) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(hidden=200), fm.ERR_INVALID_ARG),
    (dict(inter=100), fm.ERR_INVALID_ARG),
    (dict(top_k=0), fm.ERR_INVALID_ARG),
    (dict(route_tile=7), fm.ERR_INVALID_ARG),
    (dict(route_tile=12), fm.ERR_INVALID_ARG),
    (dict(route_tile=24), fm.ERR_UNSUPPORTED),
    (dict(route_tile=512), fm.ERR_UNSUPPORTED),
    (dict(route_tile=8, mode=fm.W4A4), fm.ERR_UNSUPPORTED),
    (dict(route_tile=256, mode=fm.W4A4), fm.ERR_UNSUPPORTED),
    (dict(route_tile=256, mode=fm.W4A8), fm.ERR_UNSUPPORTED),
    (dict(num_local_experts=300), fm.ERR_INVALID_ARG),
    (dict(num_local_experts=16, local_expert_offset=250), fm.ERR_INVALID_ARG),
    (dict(mode=5), fm.ERR_INVALID_ARG),
])
def test_invalid_problems_are_rejected_on_the_host(lib, kw, status):
    base = dict(num_tokens=8, hidden=256, inter=256, num_experts=256, top_k=8)
    base.update(kw)
    p = fm.problem(**base)
    with pytest.raises(fm.Fp4MoeError) as ei:
        fm.route_tile(p)
    assert ei.value.status == status
    assert fm.workspace_size(p) == 0


def test_null_pointers_rejected_before_any_launch(lib):
    p = fm.problem(8, 256, 256, 8, 2)

    class Fake:
        def __init__(self, n):
            self.n = n

        def data_ptr(self):
            return 0

        def numel(self):
            return self.n

        def element_size(self):
            return 1
    ws = Fake(1 << 20)
    with pytest.raises(fm.Fp4MoeError) as ei:
        fm.fused_moe_forward(p, None, None, None, None, None, None, None, None, None, 1.0, False, 0,
                             None, ws, stream=0)
    assert ei.value.status == fm.ERR_INVALID_ARG
    with pytest.raises(fm.Fp4MoeError) as ei:
        fm.moe_route_sort(p, None, None, None, None, None, None, None, ws, stream=0)
    assert ei.value.status == fm.ERR_INVALID_ARG
    assert fm.status_string(fm.ERR_DEVICE_TIMEOUT).startswith("device error")


@pytest.mark.parametrize("act", [
    dict(type=3),                                                  # unknown type
    dict(type=fm.ACT_GEGLU_TANH, flags=fm.ACT_F_SITU, situ_beta=1.0),  # flags only with SwiGLU
    dict(flags=fm.ACT_F_SWIGLU_OAI | fm.ACT_F_SITU, situ_beta=1.0, swiglu_limit=1.0),
    dict(flags=fm.ACT_F_SITU_LINEAR, situ_linear_beta=1.0),         # linear clamp needs SiTU
    dict(flags=fm.ACT_F_SITU, situ_beta=0.0),
    dict(flags=fm.ACT_F_SITU | fm.ACT_F_SITU_LINEAR, situ_beta=1.0, situ_linear_beta=float("inf")),
    dict(flags=fm.ACT_F_SWIGLU_OAI, swiglu_alpha=float("nan"), swiglu_limit=1.0),
    dict(flags=fm.ACT_F_SWIGLU_OAI, swiglu_limit=0.0),
    dict(flags=8),
])
def test_invalid_activations_are_rejected(lib, act):
    a = fm.Activation()
    for k, v in act.items():
        setattr(a, k, v)
    p = fm.problem(8, 256, 256, 8, 2, act=a)
    with pytest.raises(fm.Fp4MoeError) as ei:
        fm.route_tile(p)
    assert ei.value.status == fm.ERR_INVALID_ARG


def test_activation_helper_and_relu2_sizes(lib):
    assert fm.activation().flags == 0
    a = fm.activation(swiglu_alpha=1.702, swiglu_beta=1.0, swiglu_limit=7.0)
    assert a.flags == fm.ACT_F_SWIGLU_OAI
    a = fm.activation(situ_beta=2.0, situ_linear_beta=1.0)
    assert a.flags == fm.ACT_F_SITU | fm.ACT_F_SITU_LINEAR
    for T in (16, 32):
        p = fm.problem(8, 7168, 2048, 256, 8, route_tile=T, act=fm.activation(fm.ACT_RELU2))
        assert fm.route_tile(p) == T
        assert fm.prepared_weight_size(p, 1) == 256 * 8 * 56 * 18432     # I/256 blocks, no gate rows
        p = fm.problem(8, 7168, 384, 256, 8, route_tile=T, act=fm.activation(fm.ACT_RELU2))
        assert fm.prepared_weight_size(p, 1) == 256 * 2 * 56 * 18432     # a half-empty last block
        g = fm.problem(8, 7168, 2048, 256, 8, route_tile=T, act=fm.activation(fm.ACT_GEGLU_TANH))
        assert fm.prepared_weight_size(g, 1) == 256 * 16 * 56 * 18432


def test_per_token_scale_needs_the_slot_map(lib):
    p = fm.problem(8, 256, 256, 8, 2, mode=fm.W4A4)

    class Fake:
        def __init__(self, addr, n):
            self.addr, self.n = addr, n

        def data_ptr(self):
            return self.addr

        def numel(self):
            return self.n

        def element_size(self):
            return 1
    dev = Fake(1 << 20, 1 << 24)                      # an aligned address; never dereferenced
    with pytest.raises(fm.Fp4MoeError) as ei:
        fm.moe_gemm1_swiglu(p, dev, dev, None, dev, dev, dev, dev, dev, dev, dev, dev, dev,
                            stream=0, per_token_scale=dev)
    assert ei.value.status == fm.ERR_INVALID_ARG


def test_domain_shard_sizes(lib):
    # FC1 shard: I/2 h columns; FC2 shard: H/2 output rows over the full I
    for T in (16, 32):
        p = fm.problem(8, 7168, 2048, 256, 8, route_tile=T)
        assert 2 * fm.domain_weight_size(p, 1) == fm.prepared_weight_size(p, 1)
        assert 2 * fm.domain_weight_size(p, 2) == fm.prepared_weight_size(p, 2)
        # the fused workspace plus an fp32 [M, H] accumulator (and, for the
        # warp-MMA route tile, a second K-split scratch)
        assert fm.localized_workspace_size(p) >= fm.workspace_size(p) + 8 * 7168 * 4
    r = fm.problem(8, 7168, 2048, 256, 8, route_tile=32, act=fm.activation(fm.ACT_RELU2))
    assert fm.domain_weight_size(r, 1) == 256 * 4 * 56 * 18432        # I/2 rows, no gate rows
    m = fm.problem(8, 6144, 2048, 256, 8, route_tile=32, mode=fm.W4A8)
    assert 2 * fm.domain_weight_size(m, 2) == fm.prepared_weight_size(m, 2)
    # I or H not a multiple of 256 does not split
    for I, H in ((384, 7168), (2048, 384)):
        q = fm.problem(8, H, I, 256, 8)
        assert fm.domain_weight_size(q, 1) == 0 and fm.domain_weight_size(q, 2) == 0
        assert fm.localized_workspace_size(q) == 0


def test_localized_forward_rejected_on_the_host(lib):
    class Fake:
        def __init__(self, addr, n):
            self.addr, self.n = addr, n

        def data_ptr(self):
            return self.addr

        def numel(self):
            return self.n

        def element_size(self):
            return 1
    dev = Fake(1 << 20, 1 << 24)                      # an aligned address; never dereferenced
    small_ws = Fake(1 << 20, 1024)
    p = fm.problem(8, 256, 256, 8, 2, route_tile=32)
    shards = [dev, dev]

    def call(p, loc, ws=small_ws, fc2=None, mode=0):
        with pytest.raises(fm.Fp4MoeError) as ei:
            fm.fused_moe_forward_localized(p, dev, dev, dev, dev, loc, dev, fc2, dev, 1.0, False,
                                           mode, dev, ws, stream=0)
        return ei.value.status
    assert call(p, fm.Localized()) == fm.ERR_INVALID_ARG                  # null shards
    loc = fm.localized(shards, shards, [0, 0])
    assert call(p, loc, mode=7) == fm.ERR_INVALID_ARG                      # finalize mode
    bad = fm.localized(shards, [dev, Fake((1 << 20) + 8, 1)], [0, 0])
    assert call(p, bad) == fm.ERR_INVALID_ARG                              # misaligned shard
    neg = fm.localized(shards, shards, [0, 0], sm_count=-1)
    assert call(p, neg) == fm.ERR_INVALID_ARG
    assert call(fm.problem(8, 256, 384, 8, 2, route_tile=32), loc) == fm.ERR_UNSUPPORTED   # I % 256
    assert call(p, loc) == fm.ERR_WORKSPACE_TOO_SMALL
    # w4a4 needs fc2_input_scale; w4a8 takes none
    assert call(fm.problem(8, 256, 256, 8, 2, route_tile=32, mode=fm.W4A4), loc) == fm.ERR_INVALID_ARG
    assert call(fm.problem(8, 256, 256, 8, 2, route_tile=32, mode=fm.W4A8), loc,
                fc2=dev) == fm.ERR_INVALID_ARG
    with pytest.raises(fm.Fp4MoeError) as ei:
        fm.prepare_domain_weights(fm.problem(8, 256, 384, 8, 2), 1, dev, dev, dev, stream=0)
    assert ei.value.status == fm.ERR_UNSUPPORTED
