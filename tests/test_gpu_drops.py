"""GPU parity of the dispatch variants with the oracle: per-expert capacity
(token dropping) through the whole layer, and the local expert range of the
all-gather path's "scatter & drop".

Bit-exact: counts, offsets, the placed part of perm_src, perm_dst (with -1 on
dropped assignments) and the permuted rows.  Floating point as in the dropless
parity tests: y, dx relative L2 <= 5e-3; weight and router gradients <= 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.cref as ref
from routing_grouped_expert_router_gb300 import binding as mb
from routing_grouped_expert_router_gb300 import build as mbuild
from tests.gpu_runner import LayerRun, workspace
from tests.helpers import conditioned_inputs, rel_l2, small_config

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]

TOL_Y = 5e-3
TOL_W = 1e-2

CASES = {
    # name: (layer shape, capacity factor)
    "mixtral_mid_cf1": (dict(T=1024, h=512, f=1024, E=8, k=2, seed=2), 1.0),
    "internal_zipf_cf125": (dict(T=1024, h=384, f=448, E=32, k=3, seed=3, zipf_s=1.2), 1.25),
    "deepseek_cf05": (dict(T=512, h=256, f=192, E=64, k=6, seed=1), 0.5),
    "ragged_cap1": (dict(T=777, h=192, f=320, E=5, k=3, seed=8), None),  # capacity 1
    "cap_above_max": (dict(T=256, h=128, f=256, E=8, k=2, seed=0), 100.0),
}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    return mb.load()


def _to(inp, device):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _case(name):
    shape, factor = CASES[name]
    cfg = small_config(name=name, **shape)
    cap = 1 if factor is None else mb.capacity_for(cfg.T, cfg.k, cfg.E, factor)
    return cfg, conditioned_inputs(cfg), cap


@pytest.mark.parametrize("name", list(CASES))
def test_layer_with_capacity_matches_oracle(lib, name):
    cfg, inp, cap = _case(name)
    y, ctx = ref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"],
                              cfg.k, capacity=cap)
    g = ref.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    n = int(ctx["offsets"][-1])
    if name != "cap_above_max":
        assert n < cfg.T * cfg.k, "the case must drop assignments"
    else:
        assert n == cfg.T * cfg.k
    d = mb.dims_of(cfg, has_bias=cfg.zipf_s > 0, capacity=cap)
    run = LayerRun(d)
    dev = _to(inp, "cuda")
    run.fwd(dev)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    out = run.outputs()
    np.testing.assert_array_equal(out["topk_idx"].numpy(), ctx["topk_idx"])
    np.testing.assert_array_equal(out["counts"].numpy(), ctx["counts"])
    np.testing.assert_array_equal(out["offsets"].numpy(), ctx["offsets"])
    np.testing.assert_array_equal(out["perm_src"].numpy()[:n], ctx["perm_src"])
    np.testing.assert_array_equal(out["perm_dst"].numpy(), ctx["perm_dst"])
    np.testing.assert_array_equal(out["x_perm"][:n].double().numpy(), ctx["x_perm"])
    assert rel_l2(out["O"][:n].double().numpy(), ctx["O"]) <= TOL_Y
    assert rel_l2(out["y"].double().numpy(), y) <= TOL_Y
    assert rel_l2(out["dx"].double().numpy(), g["dx"]) <= TOL_Y
    for key in ("dW1", "dW3", "dW2", "dWg"):
        assert rel_l2(out[key].numpy(), g[key]) <= TOL_W, key
    # a token all of whose slots were dropped gets y = 0 exactly
    dropped_all = np.all(ctx["perm_dst"].reshape(cfg.T, cfg.k) < 0, axis=1)
    if dropped_all.any():
        assert torch.all(out["y"][torch.from_numpy(dropped_all)] == 0)


def test_capacity_above_max_is_bitwise_dropless(lib):
    cfg, inp, cap = _case("cap_above_max")
    dev = _to(inp, "cuda")
    outs = []
    for c in (0, cap):
        run = LayerRun(mb.dims_of(cfg, has_bias=False, capacity=c))
        run.fwd(dev)
        run.bwd(dev)
        torch.cuda.synchronize()
        outs.append(run.outputs())
    for key in outs[0]:
        a, b = outs[0][key], outs[1][key]
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b), key


def _local(d, idx, lo, hi, x, R, h):
    EL = hi - lo
    i32 = dict(dtype=torch.int32, device="cuda")
    counts = torch.full((EL,), -7, **i32)
    offsets = torch.full((EL + 1,), -7, **i32)
    psrc = torch.full((R,), -7, **i32)
    pdst = torch.full((R,), -7, **i32)
    xp = torch.zeros(R, h, dtype=torch.bfloat16, device="cuda")
    mb.moe_permute_local(d, idx, lo, hi, x, counts, offsets, psrc, pdst, xp,
                         workspace(d, mb.OP_PERMUTE))
    return counts, offsets, psrc, pdst, xp


@pytest.mark.parametrize("E,k,ranges,cap", [
    (8, 2, [(0, 3), (3, 8)], 0),
    (32, 3, [(0, 5), (5, 6), (6, 32)], 0),
    (64, 6, [(0, 8), (8, 16), (56, 64)], 0),
    (16, 4, [(0, 4), (4, 16)], 40),
])
def test_permute_local_matches_oracle(lib, E, k, ranges, cap):
    cfg = small_config(name="local", T=900, h=128, f=128, E=E, k=k, seed=40 + E)
    inp = conditioned_inputs(cfg)
    idx_np, _, _ = ref.route(inp["x"], inp["Wg"], inp["b"], k)
    d = mb.dims_of(cfg, has_bias=False, capacity=cap)
    R = cfg.T * k
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int32)).cuda()
    x = inp["x"].cuda()
    for lo, hi in ranges:
        counts, offsets, psrc, pdst = ref.dispatch(idx_np, E, cap or None, (lo, hi))
        g = _local(d, idx, lo, hi, x, R, cfg.h)
        torch.cuda.synchronize()
        n = int(offsets[-1])
        np.testing.assert_array_equal(g[0].cpu().numpy(), counts)
        np.testing.assert_array_equal(g[1].cpu().numpy(), offsets)
        np.testing.assert_array_equal(g[2].cpu().numpy()[:n], psrc)
        np.testing.assert_array_equal(g[3].cpu().numpy(), pdst)
        np.testing.assert_array_equal(g[4][:n].cpu().double().numpy(),
                                      ref.permute_rows(oracle.as_f64(inp["x"]), psrc, k))
        # rows past the placed ones are left alone
        assert torch.all(g[4][n:] == 0)


def test_local_expert_ranges_sum_to_layer(lib):
    """Scatter & drop per expert range, the local GroupedGEMMs and a partial
    combine on each range; the partials summed in fp32 match the oracle."""
    cfg = small_config(name="local_sum", T=1024, h=256, f=512, E=8, k=4, seed=77)
    inp = conditioned_inputs(cfg)
    y_ref, ctx = ref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                                  inp["W2"], cfg.k)
    dev = _to(inp, "cuda")
    T, h, f, k = cfg.T, cfg.h, cfg.f, cfg.k
    R = T * k
    d = mb.dims_of(cfg, has_bias=False)
    idx = torch.from_numpy(np.ascontiguousarray(ctx["topk_idx"], dtype=np.int32)).cuda()
    gates = torch.from_numpy(np.asarray(ctx["gates"], dtype=np.float32)).cuda()
    total = torch.zeros(T, h, dtype=torch.float32, device="cuda")
    for lo, hi in [(0, 2), (2, 3), (3, 8)]:
        counts, offsets, psrc, pdst, _ = _local(d, idx, lo, hi, None, R, h)
        dl = mb.dims(T, h, f, hi - lo, k)
        A = torch.empty(R, f, dtype=torch.bfloat16, device="cuda")
        B, H = torch.empty_like(A), torch.empty_like(A)
        O = torch.empty(R, h, dtype=torch.bfloat16, device="cuda")
        mb.moe_expert_ffn_fwd(dl, dev["x"], psrc, offsets, dev["W1"][lo:hi], dev["W3"][lo:hi],
                              dev["W2"][lo:hi], A, B, H, O, workspace(dl, mb.OP_EXPERT_FFN_FWD))
        part = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
        mb.moe_combine(d, O, gates, pdst, part)
        total += part.float()
    torch.cuda.synchronize()
    assert rel_l2(total.cpu().double().numpy(), y_ref) <= TOL_Y


def test_noalloc_with_capacity_equals_permute(lib):
    cfg = small_config(name="na", T=2000, h=64, f=64, E=16, k=2, seed=13)
    inp = conditioned_inputs(cfg)
    idx_np, _, _ = ref.route(inp["x"], inp["Wg"], inp["b"], cfg.k)
    cap = mb.capacity_for(cfg.T, cfg.k, cfg.E, 0.9)
    d = mb.dims_of(cfg, has_bias=False, capacity=cap)
    R = cfg.T * cfg.k
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int32)).cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    a = [torch.empty(cfg.E, **i32), torch.empty(cfg.E + 1, **i32), torch.empty(R, **i32),
         torch.empty(R, **i32)]
    b = [torch.empty_like(t) for t in a]
    mb.moe_permute(d, idx, None, *a, None, workspace(d, mb.OP_PERMUTE))
    mb.moe_permute_noalloc(d, idx, None, *b, None)
    torch.cuda.synchronize()
    counts, offsets, psrc, pdst = ref.dispatch(idx_np, cfg.E, cap)
    n = int(offsets[-1])
    assert n < R
    for got in (a, b):
        np.testing.assert_array_equal(got[0].cpu().numpy(), counts)
        np.testing.assert_array_equal(got[1].cpu().numpy(), offsets)
        np.testing.assert_array_equal(got[2].cpu().numpy()[:n], psrc)
        np.testing.assert_array_equal(got[3].cpu().numpy(), pdst)
