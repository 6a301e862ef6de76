"""Parity of the CUDA layer (through the C ABI) with the CPU oracle.

Bit-exact: routing indices, counts, offsets, both permutation maps and every
row move.  Floating point (relative L2 over the whole tensor, float64):
y, dx <= 5e-3; weight and router gradients <= 1e-2; gates max |diff| <= 1e-5
(exactly 1 for k = 1).  Shapes span several tiles with ragged tails in every
GEMM dimension, plus the degenerate cases (E > T, one token, k = 8, every
token on one expert, experts without tokens, T = 0).
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.cref as ref
from routing_grouped_expert_router_gb300 import binding as mb
from routing_grouped_expert_router_gb300 import build as mbuild
from routing_grouped_expert_router_gb300 import synth
from tests.gpu_runner import LayerRun, workspace
from tests.helpers import conditioned_inputs, rel_l2, small_config

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]

TOL_Y = 5e-3
TOL_W = 1e-2
TOL_GATE = 1e-5

CASES = {
    "tiny": dict(T=256, h=128, f=256, E=8, k=2, seed=0),
    "deepseek_mid": dict(T=512, h=256, f=192, E=64, k=6, seed=1),
    "mixtral_mid": dict(T=1024, h=512, f=1024, E=8, k=2, seed=2),
    "internal_mid_zipf": dict(T=1024, h=384, f=448, E=32, k=3, seed=3, zipf_s=1.2),
    "hunyuan_mid": dict(T=2048, h=320, f=576, E=16, k=1, seed=4),
    "experts_gt_tokens": dict(T=20, h=64, f=64, E=32, k=4, seed=5),
    "k8": dict(T=100, h=128, f=128, E=16, k=8, seed=6),
    "one_token": dict(T=1, h=64, f=128, E=4, k=2, seed=7),
    "ragged": dict(T=777, h=192, f=320, E=5, k=3, seed=8),
    # E <= 8 with h > 4096: the router's chunked kernel and its select kernel
    "wide_h": dict(T=300, h=4160, f=192, E=6, k=2, seed=9),
    # degenerate routings: one expert (a plain SwiGLU FFN, every gate 1) and
    # every token to every expert (k = E, the gates the full softmax)
    "single_expert": dict(T=300, h=128, f=128, E=1, k=1, seed=10),
    "k_equals_E": dict(T=200, h=128, f=192, E=4, k=4, seed=11),
}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    return mb.load()


def _inputs(name, **over):
    kw = dict(CASES[name])
    kw.update(over)
    cfg = small_config(name=name, **kw)
    inp = conditioned_inputs(cfg)
    return cfg, inp


def _to(inp, device):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _oracle(cfg, inp):
    y, ctx = ref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"],
                              cfg.k)
    g = ref.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    return y, ctx, g


def _check_routing(cfg, out, ctx):
    np.testing.assert_array_equal(out["topk_idx"].numpy(), ctx["topk_idx"])
    gates = out["gates"].double().numpy()
    assert np.max(np.abs(gates - ctx["gates"])) <= TOL_GATE
    if cfg.k == 1:
        assert torch.all(out["gates"] == 1.0)
    np.testing.assert_array_equal(out["counts"].numpy(), ctx["counts"])
    np.testing.assert_array_equal(out["offsets"].numpy(), ctx["offsets"])
    np.testing.assert_array_equal(out["perm_src"].numpy(), ctx["perm_src"])
    np.testing.assert_array_equal(out["perm_dst"].numpy(), ctx["perm_dst"])


@pytest.mark.parametrize("name", list(CASES))
def test_layer_matches_oracle(lib, name):
    cfg, inp = _inputs(name)
    d = mb.dims_of(cfg, has_bias=cfg.zipf_s > 0)
    y, ctx, g = _oracle(cfg, inp)
    run = LayerRun(d)
    dev = _to(inp, "cuda")
    run.fwd(dev)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    out = run.outputs()
    _check_routing(cfg, out, ctx)
    np.testing.assert_array_equal(out["x_perm"].double().numpy(), ctx["x_perm"])
    for key in ("A", "B", "H", "O"):
        assert rel_l2(out[key].double().numpy(), ctx[key]) <= TOL_Y, key
    errs = {"y": rel_l2(out["y"].double().numpy(), y),
            "dx": rel_l2(out["dx"].double().numpy(), g["dx"])}
    for key in ("dW1", "dW3", "dW2", "dWg"):
        errs[key] = rel_l2(out[key].numpy(), g[key])
    assert errs["y"] <= TOL_Y and errs["dx"] <= TOL_Y, errs
    for key in ("dW1", "dW3", "dW2", "dWg"):
        assert errs[key] <= TOL_W, errs
    if cfg.k == 1:
        assert torch.all(out["dWg"] == 0)
    # experts that received no token get exact zeros
    for e in np.nonzero(ctx["counts"] == 0)[0]:
        assert torch.all(out["dW1"][e] == 0) and torch.all(out["dW2"][e] == 0)


def test_all_tokens_on_one_expert(lib):
    cfg = small_config(name="one_expert", T=300, h=128, f=192, E=6, k=2, seed=9)
    inp = synth.make_layer(cfg)
    inp["b"] = torch.tensor([0, 0, 0, 40.0, 0, 0])
    inp["x"], _ = oracle.condition_router_margins(
        inp["x"], inp["Wg"], inp["b"], cfg.k,
        lambda r, a: synth.replacement_x_rows(cfg, r, a))
    d = mb.dims_of(cfg, has_bias=True)
    y, ctx, g = _oracle(cfg, inp)
    assert ctx["counts"][3] == cfg.T
    run = LayerRun(d)
    dev = _to(inp, "cuda")
    run.fwd(dev)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    out = run.outputs()
    _check_routing(cfg, out, ctx)
    assert rel_l2(out["y"].double().numpy(), y) <= TOL_Y
    assert rel_l2(out["dx"].double().numpy(), g["dx"]) <= TOL_Y
    for key in ("dW1", "dW3", "dW2", "dWg"):
        assert rel_l2(out[key].numpy(), g[key]) <= TOL_W, key


@pytest.mark.parametrize("E,k,h", [(8, 2, 256), (16, 3, 192), (64, 6, 128), (8, 2, 4160)])
def test_zero_upstream_gradient_gives_exact_zeros(lib, E, k, h):
    """dy = 0: every gradient is exactly zero (dx, dWg and all expert weight
    gradients; the gate gradients and the router backward vanish too), for
    each router kernel family (E = 8 with h <= 4096 and h > 4096, E = 16..64)."""
    cfg = small_config(name="dy0", T=333, h=h, f=192, E=E, k=k, seed=21)
    inp = conditioned_inputs(cfg)
    inp["dy"] = torch.zeros_like(inp["dy"])
    run = LayerRun(mb.dims_of(cfg, has_bias=False))
    dev = _to(inp, "cuda")
    for t in (run.dx, run.dWg, run.dW1, run.dW3, run.dW2):
        t.fill_(7)
    run.fwd(dev)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    for name in ("dx", "dWg", "dW1", "dW3", "dW2"):
        assert torch.all(getattr(run, name) == 0), name


@pytest.mark.parametrize("E,k,h", [(8, 2, 256), (16, 3, 192), (64, 6, 128), (8, 2, 4160)])
def test_zero_tokens_tie_to_the_lowest_experts(lib, E, k, h):
    """x = 0 (no bias): every logit is exactly 0, so every token ties across all
    E experts.  Ties go to the lower id: every token takes experts 0..k-1 in
    that order with gates exactly 1/k, the dispatch is the identity order
    within each of those experts, and y = 0 exactly (A = B = H = 0)."""
    cfg = small_config(name="x0", T=257, h=h, f=192, E=E, k=k, seed=22)
    inp = conditioned_inputs(cfg)
    inp["x"] = torch.zeros_like(inp["x"])
    run = LayerRun(mb.dims_of(cfg, has_bias=False))
    dev = _to(inp, "cuda")
    run.fwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    T = cfg.T
    idx = run.saved_view("topk_idx").cpu()
    assert torch.equal(idx, torch.arange(k, dtype=torch.int32).repeat(T, 1))
    gates = run.saved_view("gates").cpu()
    np.testing.assert_array_equal(gates.numpy(), np.full((T, k), np.float32(1.0) / np.float32(k)))
    counts = run.saved_view("counts").cpu()
    assert torch.equal(counts[:k], torch.full((k,), T, dtype=torch.int32))
    assert torch.all(counts[k:] == 0)
    # within expert j the rows are the tokens in order: perm_src[j T + t] = t k + j
    psrc = run.saved_view("perm_src").cpu().view(k, T)
    want = torch.arange(T, dtype=torch.int32)[None, :] * k + torch.arange(k, dtype=torch.int32)[:, None]
    assert torch.equal(psrc, want)
    assert torch.all(run.y == 0)


def _layer_outputs(cfg, inp):
    run = LayerRun(mb.dims_of(cfg, has_bias=False))
    run.fwd(inp)
    run.bwd(inp)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    return run


@pytest.mark.parametrize("name", ["mixtral_mid", "deepseek_mid"])
def test_exact_scaling(lib, name):
    """Power-of-two scalings commute with every rounding on the path: W2 -> 2 W2
    gives y -> 2 y exactly, and dy -> 2 dy gives every gradient times 2
    exactly (the fp32 sums see exactly doubled terms)."""
    cfg, inp = _inputs(name)
    dev = _to(inp, "cuda")
    base = _layer_outputs(cfg, dev)
    w2 = dict(dev)
    w2["W2"] = dev["W2"] * 2
    assert torch.equal((w2["W2"].float() / 2).to(torch.bfloat16), dev["W2"])
    run = _layer_outputs(cfg, w2)
    assert torch.equal(run.y.float(), 2 * base.y.float())
    dy2 = dict(dev)
    dy2["dy"] = dev["dy"] * 2
    run = _layer_outputs(cfg, dy2)
    assert torch.equal(run.y, base.y)
    for key in ("dx", "dWg", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(run, key).float(), 2 * getattr(base, key).float()), key


@pytest.mark.parametrize("name", ["mixtral_mid", "hunyuan_mid"])
def test_token_permutation_permutes_rows_exactly(lib, name):
    """Permuting the tokens permutes y and dx rows bitwise: a row's router
    logits, its expert rows' dot products and its combine all run in an order
    that does not depend on the row's position in the batch."""
    cfg, inp = _inputs(name)
    dev = _to(inp, "cuda")
    base = _layer_outputs(cfg, dev)
    perm = torch.randperm(cfg.T, generator=torch.Generator().manual_seed(5)).cuda()
    pd = dict(dev)
    pd["x"] = dev["x"][perm].contiguous()
    pd["dy"] = dev["dy"][perm].contiguous()
    run = _layer_outputs(cfg, pd)
    assert torch.equal(run.y.view(torch.int16), base.y[perm].view(torch.int16))
    assert torch.equal(run.dx.view(torch.int16), base.dx[perm].view(torch.int16))
    assert torch.equal(run.saved_view("topk_idx"), base.saved_view("topk_idx")[perm])


def test_empty_batch(lib):
    d = mb.dims(0, 128, 128, 8, 2)
    run = LayerRun(d)
    W = synth.make_layer(small_config(T=1, h=128, f=128, E=8, k=2), "cuda")
    dev = dict(W)
    dev["x"] = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    dev["dy"] = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    run.dW1.fill_(7)
    run.dWg.fill_(7)
    run.fwd(dev)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    assert torch.all(run.saved_view("offsets") == 0)
    assert torch.all(run.dW1 == 0) and torch.all(run.dWg == 0)


def test_deterministic_bitwise(lib):
    cfg, inp = _inputs("internal_mid_zipf")
    d = mb.dims_of(cfg, has_bias=True)
    dev = _to(inp, "cuda")
    outs = []
    for _ in range(2):
        run = LayerRun(d)
        run.fwd(dev)
        run.bwd(dev)
        torch.cuda.synchronize()
        outs.append(run.outputs())
    for key in outs[0]:
        a, b = outs[0][key], outs[1][key]
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b), key


# ------------------------------------------------------ stage entry points ---

@pytest.mark.parametrize("name", ["mixtral_mid", "internal_mid_zipf", "deepseek_mid"])
def test_stage_entry_points(lib, name):
    cfg, inp = _inputs(name)
    d = mb.dims_of(cfg, has_bias=cfg.zipf_s > 0)
    y, ctx, g = _oracle(cfg, inp)
    dev = _to(inp, "cuda")
    T, h, f, E, k = cfg.T, cfg.h, cfg.f, cfg.E, cfg.k
    R = T * k
    i32 = dict(dtype=torch.int32, device="cuda")

    # route
    idx = torch.empty(T, k, **i32)
    gates = torch.empty(T, k, dtype=torch.float32, device="cuda")
    mb.moe_route(d, dev["x"], dev["Wg"], dev["b"], idx, gates, workspace(d, mb.OP_ROUTE))
    np.testing.assert_array_equal(idx.cpu().numpy(), ctx["topk_idx"])
    assert np.max(np.abs(gates.cpu().double().numpy() - ctx["gates"])) <= TOL_GATE

    # permute (maps + rows) and unpermute
    counts = torch.empty(E, **i32)
    offsets = torch.empty(E + 1, **i32)
    psrc = torch.empty(R, **i32)
    pdst = torch.empty(R, **i32)
    xp = torch.empty(R, h, dtype=torch.bfloat16, device="cuda")
    mb.moe_permute(d, idx, dev["x"], counts, offsets, psrc, pdst, xp,
                   workspace(d, mb.OP_PERMUTE))
    np.testing.assert_array_equal(counts.cpu().numpy(), ctx["counts"])
    np.testing.assert_array_equal(offsets.cpu().numpy(), ctx["offsets"])
    np.testing.assert_array_equal(psrc.cpu().numpy(), ctx["perm_src"])
    np.testing.assert_array_equal(pdst.cpu().numpy(), ctx["perm_dst"])
    np.testing.assert_array_equal(xp.cpu().double().numpy(), ctx["x_perm"])
    back = torch.empty(R, h, dtype=torch.bfloat16, device="cuda")
    mb.moe_unpermute(d, pdst, xp, back)
    assert torch.equal(back.view(T, k, h).cpu(), inp["x"][:, None, :].expand(T, k, h))

    # expert FFN forward from the oracle's dispatch
    psrc_o = torch.from_numpy(ctx["perm_src"]).cuda()
    off_o = torch.from_numpy(ctx["offsets"]).cuda()
    A = torch.empty(R, f, dtype=torch.bfloat16, device="cuda")
    B, H = torch.empty_like(A), torch.empty_like(A)
    O = torch.empty(R, h, dtype=torch.bfloat16, device="cuda")
    mb.moe_expert_ffn_fwd(d, dev["x"], psrc_o, off_o, dev["W1"], dev["W3"], dev["W2"], A, B, H, O,
                          workspace(d, mb.OP_EXPERT_FFN_FWD))
    for key, t in (("A", A), ("B", B), ("H", H), ("O", O)):
        assert rel_l2(t.cpu().double().numpy(), ctx[key]) <= TOL_Y, key

    # combine of an independent synthetic O
    O_syn = synth.normal(99, 1, (R, h), 1.0, torch.bfloat16)
    g32 = torch.from_numpy(ctx["gates"]).float()
    y_syn = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    mb.moe_combine(d, O_syn.cuda(), g32.cuda(), torch.from_numpy(ctx["perm_dst"]).cuda(), y_syn)
    y_ref = ref.combine(oracle.as_f64(O_syn), g32.double().numpy(), ctx["perm_dst"], T, k)
    assert rel_l2(y_syn.cpu().double().numpy(), y_ref) <= 3e-3

    # expert FFN backward from the oracle's activations (rounded to bf16)
    bf = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()
    dX = torch.empty(R, h, dtype=torch.float32, device="cuda")
    dg = torch.empty(R, dtype=torch.float32, device="cuda")
    dW1 = torch.empty(E, h, f, dtype=torch.float32, device="cuda")
    dW3, dW2 = torch.empty_like(dW1), torch.empty(E, f, h, dtype=torch.float32, device="cuda")
    mb.moe_expert_ffn_bwd(d, dev["x"], dev["dy"], g32.cuda(), psrc_o, off_o, dev["W1"], dev["W3"],
                          dev["W2"], bf(ctx["A"]), bf(ctx["B"]), bf(ctx["H"]), bf(ctx["O"]), dX,
                          dg, dW1, dW3, dW2, workspace(d, mb.OP_EXPERT_FFN_BWD))
    assert rel_l2(dX.cpu().numpy(), g["dX_perm"]) <= TOL_Y
    assert rel_l2(dg.cpu().double().numpy().reshape(T, k), g["dg"]) <= TOL_W
    for key, t in (("dW1", dW1), ("dW3", dW3), ("dW2", dW2)):
        assert rel_l2(t.cpu().numpy(), g[key]) <= TOL_W, key

    # router backward + token gradient from the oracle's dg and dX_perm
    dxo = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dWg = torch.empty(h, E, dtype=torch.float32, device="cuda")
    mb.moe_router_bwd(d, dev["x"], dev["Wg"], torch.from_numpy(ctx["topk_idx"]).cuda(),
                      g32.cuda(), torch.from_numpy(g["dg"].ravel()).float().cuda(),
                      torch.from_numpy(g["dX_perm"]).float().cuda(), psrc_o,
                      torch.from_numpy(ctx["perm_dst"]).cuda(), off_o, dxo, dWg,
                      workspace(d, mb.OP_ROUTER_BWD))
    assert rel_l2(dxo.cpu().double().numpy(), g["dx"]) <= TOL_Y
    assert rel_l2(dWg.cpu().numpy(), g["dWg"]) <= TOL_W
    torch.cuda.synchronize()
