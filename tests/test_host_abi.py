"""Host-side checks of the C ABI (no GPU): the library builds, loads, exports
every declared entry point, and rejects bad arguments before any launch.

The argument checks pass fake device addresses that only a host-side
rejection keeps from ever reaching a kernel.  On a machine with a GPU a
regression there would launch kernels on those addresses, so those tests run
only where no CUDA device is present (the CPU suite)."""
import ctypes
import re

import pytest
import torch

from routing_grouped_expert_router_gb300 import binding as mb
from routing_grouped_expert_router_gb300 import build as mbuild
from routing_grouped_expert_router_gb300.configs import CONFIGS


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return mb.load()


def test_exports_every_declared_symbol(lib):
    names = mb.declared_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(mb._SIGS), set(names) ^ set(mb._SIGS)


def test_version_and_status_strings(lib):
    assert "sm_103a" in mb.moe_version()
    for code in range(7):
        s = mb.status_string(code)
        assert s.startswith("MOE_")
    assert mb.status_string(mb.MOE_ERR_DEVICE_INDEX).startswith("MOE_ERR_DEVICE_INDEX")
    assert mb.status_string(99) == "unknown moe_status"


def test_status_codes_match_the_header():
    src = open(mb.HEADER).read()
    codes = dict((n, int(v)) for n, v in re.findall(r"\b(MOE_(?:OK|ERR_\w+)) = (\d+)", src))
    assert len(codes) == 7
    for name, value in codes.items():
        assert getattr(mb, name) == value, name


FAKE = 1 << 20          # aligned, non-null address; never dereferenced
MISALIGNED = FAKE + 8
# calls with FAKE pointers: only where no device can run a kernel on them
no_device = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="fake device addresses: host-only check")


def _d(**kw):
    base = dict(T=64, h=128, f=256, E=8, k=2, has_bias=0)
    base.update(kw)
    return mb.moe_dims(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(k=0), mb.MOE_ERR_INVALID_ARG),
    (dict(k=9, E=16), mb.MOE_ERR_UNSUPPORTED),
    (dict(k=5, E=4), mb.MOE_ERR_INVALID_ARG),
    (dict(E=65), mb.MOE_ERR_UNSUPPORTED),
    (dict(h=100), mb.MOE_ERR_UNSUPPORTED),
    # h = 8 meets the ABI's h % 8 == 0, but the matmuls' 64-wide K blocks need
    # h and h_ffn to be multiples of 64: declined, not computed wrongly
    (dict(h=8), mb.MOE_ERR_UNSUPPORTED),
    (dict(h=32), mb.MOE_ERR_UNSUPPORTED),
    (dict(f=72), mb.MOE_ERR_UNSUPPORTED),
    (dict(T=-1), mb.MOE_ERR_INVALID_ARG),
    (dict(T=1 << 29, k=8), mb.MOE_ERR_UNSUPPORTED),
    (dict(capacity=-1), mb.MOE_ERR_INVALID_ARG),
])
@no_device
def test_bad_dims_rejected(lib, kw, code):
    d = _d(**kw)
    st = lib.moe_route(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE, 1 << 30, None)
    assert st == code
    assert lib.moe_workspace_bytes(ctypes.byref(d), mb.OP_LAYER_FWD) == 0
    assert lib.moe_saved_bytes(ctypes.byref(d)) == 0


def test_null_dims(lib):
    assert lib.moe_route(None, FAKE, FAKE, None, FAKE, FAKE, FAKE, 1 << 30, None) \
        == mb.MOE_ERR_INVALID_ARG


def test_null_and_misaligned_pointers(lib):
    d = _d()
    big = 1 << 40
    assert lib.moe_route(ctypes.byref(d), None, FAKE, None, FAKE, FAKE, FAKE, big, None) \
        == mb.MOE_ERR_INVALID_ARG
    assert lib.moe_route(ctypes.byref(d), MISALIGNED, FAKE, None, FAKE, FAKE, FAKE, big, None) \
        == mb.MOE_ERR_INVALID_ARG
    d.has_bias = 1
    assert lib.moe_route(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE, big, None) \
        == mb.MOE_ERR_INVALID_ARG
    d.has_bias = 0
    # workspace must be 256-byte aligned
    assert lib.moe_route(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE + 16, big, None) \
        == mb.MOE_ERR_INVALID_ARG
    args = [FAKE] * 12
    args[3] = None
    assert lib.moe_layer_bwd(ctypes.byref(d), *args, FAKE, big, None) == mb.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(d), FAKE, FAKE, None, FAKE, None) == mb.MOE_ERR_INVALID_ARG
    assert lib.moe_unpermute(ctypes.byref(d), FAKE, MISALIGNED, FAKE, None) \
        == mb.MOE_ERR_INVALID_ARG


@no_device
@pytest.mark.parametrize("op", range(7))
def test_workspace_too_small(lib, op):
    d = _d()
    need = lib.moe_workspace_bytes(ctypes.byref(d), op)
    assert need >= 256
    P = FAKE
    calls = {
        mb.OP_ROUTE: lambda n: lib.moe_route(ctypes.byref(d), P, P, None, P, P, P, n, None),
        mb.OP_PERMUTE: lambda n: lib.moe_permute(ctypes.byref(d), P, None, P, P, P, P, None, P,
                                                 n, None),
        mb.OP_EXPERT_FFN_FWD: lambda n: lib.moe_expert_ffn_fwd(ctypes.byref(d), *([P] * 10), P,
                                                               n, None),
        mb.OP_EXPERT_FFN_BWD: lambda n: lib.moe_expert_ffn_bwd(ctypes.byref(d), *([P] * 17), P,
                                                               n, None),
        mb.OP_ROUTER_BWD: lambda n: lib.moe_router_bwd(ctypes.byref(d), *([P] * 11), P, n, None),
        mb.OP_LAYER_FWD: lambda n: lib.moe_layer_fwd(ctypes.byref(d), P, P, None, P, P, P, P, P,
                                                     P, n, None),
        mb.OP_LAYER_BWD: lambda n: lib.moe_layer_bwd(ctypes.byref(d), *([P] * 12), P, n, None),
    }
    assert calls[op](need - 1) == mb.MOE_ERR_WORKSPACE


def test_sizes_cover_tensors(lib):
    for cfg in CONFIGS.values():
        d = mb.dims_of(cfg)
        R = cfg.T * cfg.k
        saved = lib.moe_saved_bytes(ctypes.byref(d))
        acts = R * (cfg.h * 2 * 2 + cfg.f * 2 * 3) + R * 16
        assert saved >= acts
        bw = lib.moe_workspace_bytes(ctypes.byref(d), mb.OP_LAYER_BWD)
        assert bw >= R * (cfg.h * 2 + cfg.f * 4 + cfg.h * 4)
        # views are inside the buffer, in declaration order, 256-byte aligned
        offs = [mb.moe_saved_view(d, FAKE, n) - FAKE for n in
                ("topk_idx", "gates", "counts", "offsets", "perm_src", "perm_dst", "x_perm",
                 "A", "B", "H", "O")]
        assert offs == sorted(offs) and offs[0] == 0 and offs[-1] < saved
        assert all(o % 256 == 0 for o in offs)
    with pytest.raises(mb.MoeError):
        mb.moe_saved_view(_d(), FAKE, "nope")


@pytest.mark.parametrize("lo,hi,ok", [(0, 8, True), (3, 4, True), (-1, 4, False), (4, 4, False),
                                      (5, 3, False), (0, 9, False)])
@no_device
def test_permute_local_range_checked(lib, lo, hi, ok):
    d = _d()
    need = lib.moe_workspace_bytes(ctypes.byref(d), mb.OP_PERMUTE)
    P = FAKE
    # a valid range with a too-small workspace stops at the workspace check,
    # so nothing is launched either way
    st = lib.moe_permute_local(ctypes.byref(d), P, lo, hi, None, P, P, P, P, None, P, need - 1,
                               None)
    assert st == (mb.MOE_ERR_WORKSPACE if ok else mb.MOE_ERR_INVALID_ARG)


def test_capacity_for(lib):
    assert mb.capacity_for(16384, 2, 8, 1.0) == 4096
    assert mb.capacity_for(10, 3, 4, 1.25) == 10   # ceil(9.375)
    assert mb.capacity_for(0, 2, 8, 1.0) == 0
    assert lib.moe_capacity_for(10, 0, 4, 1.0) == -1
    assert lib.moe_capacity_for(10, 2, 0, 1.0) == -1
    assert lib.moe_capacity_for(10, 2, 4, 0.0) == -1
    assert lib.moe_capacity_for(1 << 30, 8, 1, 4.0) == -1      # past int32
    with pytest.raises(mb.MoeError):
        mb.capacity_for(10, 2, 4, -1.0)
    assert mb.dims(4, 64, 64, 4, 2, capacity=3).capacity == 3
    assert mb.dims(4, 64, 64, 4, 2).capacity == 0


@no_device
def test_status_word_without_workspace_needs_a_device(lib):
    """moe_read_device_status(NULL) reads the per-device word of the calls
    without a workspace: with no device it reports MOE_ERR_CUDA, and a
    misaligned workspace is an argument error."""
    assert lib.moe_read_device_status(None, None) == mb.MOE_ERR_CUDA
    assert lib.moe_clear_device_status(None, None) == mb.MOE_ERR_CUDA
    assert lib.moe_read_device_status(FAKE + 16, None) == mb.MOE_ERR_INVALID_ARG


def test_saved_bytes_follow_sar_formula(lib):
    """moe_saved_bytes against the activation-memory formula at n = 1: the
    MoE terms 2k + 3kf (x_perm, O; A, B, H) before selective activation
    rematerialisation and 2kf (A, B) after, in units of T*h bf16 elements."""
    for cfg in CONFIGS.values():
        R, T, h, f, k = cfg.T * cfg.k, cfg.T, cfg.h, cfg.f, cfg.k
        maps = sum(-(-n // 256) * 256 for n in (R * 4, R * 4, cfg.E * 4, (cfg.E + 1) * 4,
                                                 R * 4, R * 4))
        fr = f / h
        for sar, units in ((0, 2 * k + 3 * k * fr), (1, 2 * k * fr)):
            d = mb.dims_of(cfg, sar=sar)
            acts = lib.moe_saved_bytes(ctypes.byref(d)) - maps
            assert abs(acts - 2 * units * T * h) < 256 * 5, (cfg.name, sar)
        d = mb.dims_of(cfg, sar=True)
        for name in ("x_perm", "H", "O"):
            assert lib.moe_saved_view(ctypes.byref(d), FAKE, name.encode()) is None
        for name in ("A", "B", "offsets"):
            assert lib.moe_saved_view(ctypes.byref(d), FAKE, name.encode())
    d = _d(sar=2)
    assert lib.moe_saved_bytes(ctypes.byref(d)) == 0


@no_device
def test_fp8_shape_and_argument_checks(lib):
    d = _d(h=192)                                # h not a multiple of 128
    assert lib.moe_fp8_weight_bytes(ctypes.byref(d)) == 0
    assert lib.moe_quantize_weights_fp8(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, None) \
        == mb.MOE_ERR_UNSUPPORTED
    d = _d(h=256, f=384, E=4)
    need = lib.moe_fp8_weight_bytes(ctypes.byref(d))
    assert need >= 4 * (2 * 384 * 256 + 256 * 384) + 4 * 4 * (384 * 2 + 256)
    assert lib.moe_quantize_weights_fp8(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE + 16, None) \
        == mb.MOE_ERR_INVALID_ARG
    offs = [mb.moe_fp8_weight_view(d, FAKE, n) - FAKE for n in ("W13q", "W2q", "s1", "s3", "s2")]
    assert offs == sorted(offs) and offs[-1] < need and all(o % 256 == 0 for o in offs)
    ws = lib.moe_workspace_bytes(ctypes.byref(d), mb.OP_LAYER_FWD_FP8)
    assert ws >= lib.moe_workspace_bytes(ctypes.byref(d), mb.OP_LAYER_FWD) + 64 * 2 * (256 + 384)
    assert lib.moe_layer_fwd_fp8(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, ws - 1,
                                 None) == mb.MOE_ERR_WORKSPACE
    assert lib.moe_quantize_rows_fp8(FAKE, 4, 24, None, 1, 4, FAKE, FAKE, None) \
        == mb.MOE_ERR_INVALID_ARG           # n not a multiple of 16
    assert lib.moe_quantize_rows_fp8(FAKE, 8, 32, None, 1, 4, FAKE, FAKE, None) \
        == mb.MOE_ERR_INVALID_ARG           # rows beyond the source without idx


@no_device
def test_selftest_arguments_checked(lib):
    assert lib.moe_selftest_wait_timeout(None, 10, None) == mb.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(FAKE + 16, 10, None) == mb.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(FAKE, 0, None) == mb.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(FAKE, 2000000, None) == mb.MOE_ERR_INVALID_ARG


def test_profile_hook_without_events(lib):
    assert mb.moe_profile_events(None, 0) == 0
    assert mb.moe_profile_kernel_name(-1) == ""


def test_launch_failure_hook_is_host_only(lib):
    """The failure-injection hook only sets a host-side counter: setting and
    clearing it needs no device and launches nothing."""
    before = lib.moe_kernel_launches()
    mb.moe_test_fail_launch_after(5)
    mb.moe_test_fail_launch_after(0)
    mb.moe_test_fail_launch_after(-3)
    assert lib.moe_kernel_launches() == before
