"""GPU parity of the FP8 (e4m3, per-token scale) expert forward with the
oracle's FP8 forward.

Bit-exact: every weight code and scale (moe_quantize_weights_fp8) and every
code and scale of the permuted token rows (moe_quantize_rows_fp8), since both
come from exact bf16 inputs.  Floating point: A, B, H, O, y relative L2
<= 5e-3 against the oracle run with the same quantisation (the remaining
differences are fp32 summation order and bf16 storage); the bf16 backward on
the FP8 activations at the default tolerances (dx <= 5e-3, weight and router
gradients <= 1e-2).
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
    "tiny": dict(T=256, h=128, f=256, E=8, k=2, seed=0),
    "deepseek_mid": dict(T=512, h=256, f=256, E=64, k=6, seed=1),
    "mixtral_mid": dict(T=1024, h=512, f=1024, E=8, k=2, seed=2),
    "internal_mid_zipf": dict(T=1024, h=384, f=512, E=32, k=3, seed=3, zipf_s=1.2),
    "hunyuan_mid": dict(T=2048, h=384, f=640, E=16, k=1, seed=4),
    "one_token": dict(T=1, h=128, f=128, E=4, k=2, seed=7),
    "ragged_tokens": dict(T=777, h=256, f=384, E=5, k=3, seed=8),
}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    return mb.load()


def _to(inp, device):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _codes(t: torch.Tensor) -> np.ndarray:
    """e4m3 bytes -> their exact values."""
    return t.cpu().view(torch.float8_e4m3fn).float().double().numpy()


def _view(d, qw, name, shape, dtype):
    off = mb.moe_fp8_weight_view(d, qw, name) - qw.data_ptr()
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    return qw[off:off + n].view(dtype).view(shape)


def _quant_weights(d, dev):
    qw = torch.zeros(mb.moe_fp8_weight_bytes(d), dtype=torch.uint8, device="cuda")
    mb.moe_quantize_weights_fp8(d, dev["W1"], dev["W3"], dev["W2"], qw)
    return qw


# f = 8320: W2's contraction dimension is above 8192, where the weight
# quantiser switches from 64- to 32-column slabs
@pytest.mark.parametrize("f", [640, 8320])
def test_weight_codes_and_scales_bit_exact(lib, f):
    cfg = small_config(name="wq", T=8, h=384, f=f, E=3, k=2, seed=21)
    inp = conditioned_inputs(cfg)
    d = mb.dims_of(cfg, has_bias=False)
    qw = _quant_weights(d, _to(inp, "cuda"))
    torch.cuda.synchronize()
    E, h, f = cfg.E, cfg.h, cfg.f
    W1q, s1 = ref.quantize_cols_e4m3(oracle.as_f64(inp["W1"]))
    W3q, s3 = ref.quantize_cols_e4m3(oracle.as_f64(inp["W3"]))
    W2q, s2 = ref.quantize_cols_e4m3(oracle.as_f64(inp["W2"]))
    np.testing.assert_array_equal(_view(d, qw, "s1", (E, f), torch.float32).cpu().numpy(), s1)
    np.testing.assert_array_equal(_view(d, qw, "s3", (E, f), torch.float32).cpu().numpy(), s3)
    np.testing.assert_array_equal(_view(d, qw, "s2", (E, h), torch.float32).cpu().numpy(), s2)
    W13 = _codes(_view(d, qw, "W13q", (E, f // 128, 2, 128, h), torch.uint8))
    np.testing.assert_array_equal(W13[:, :, 0].reshape(E, f, h), np.transpose(W1q, (0, 2, 1)))
    np.testing.assert_array_equal(W13[:, :, 1].reshape(E, f, h), np.transpose(W3q, (0, 2, 1)))
    W2 = _codes(_view(d, qw, "W2q", (E, h, f), torch.uint8))
    np.testing.assert_array_equal(W2, np.transpose(W2q, (0, 2, 1)))


# row lengths: a block row of 256 x 16-byte pieces or less, a ragged second
# piece per thread, and rows above the register-held limit (16384 values)
@pytest.mark.parametrize("h", [512, 2112, 17408])
def test_row_codes_and_scales_bit_exact(lib, h):
    cfg = small_config(name="xq", T=333, h=h, f=128, E=8, k=2, seed=22)
    inp = conditioned_inputs(cfg)
    inp["x"][17] = 0                               # a zero row: scale 1, codes 0
    _, ctx = ref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"],
                              cfg.k)
    R = cfg.T * cfg.k
    q = torch.empty(R, cfg.h, dtype=torch.uint8, device="cuda")
    sc = torch.empty(R, dtype=torch.float32, device="cuda")
    psrc = torch.from_numpy(ctx["perm_src"]).cuda()
    mb.moe_quantize_rows_fp8(inp["x"].cuda(), R, cfg.h, psrc, cfg.k, cfg.T, q, sc)
    torch.cuda.synchronize()
    Xq, sx = ref.quantize_rows_e4m3(ctx["x_perm"])
    np.testing.assert_array_equal(sc.cpu().numpy(), sx)
    np.testing.assert_array_equal(_codes(q), Xq)
    assert np.sum(sx == 1.0) == cfg.k


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_layer_matches_fp8_oracle(lib, name):
    cfg = small_config(name=name, **CASES[name])
    inp = conditioned_inputs(cfg)
    y, ctx = ref.layer_fwd_fp8(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                                  inp["W2"], cfg.k)
    g = ref.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    dev = _to(inp, "cuda")
    d = mb.dims_of(cfg, has_bias=cfg.zipf_s > 0)
    qw = _quant_weights(d, dev)
    run = LayerRun(d)
    ws = workspace(d, mb.OP_LAYER_FWD_FP8)
    mb.moe_layer_fwd_fp8(d, dev["x"], dev["Wg"], dev["b"] if d.has_bias else None, qw, run.y,
                         run.saved, ws)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert mb.moe_read_device_status(ws) == mb.MOE_OK and run.status() == mb.MOE_OK
    out = run.outputs()
    np.testing.assert_array_equal(out["topk_idx"].numpy(), ctx["topk_idx"])
    np.testing.assert_array_equal(out["perm_src"].numpy(), ctx["perm_src"])
    np.testing.assert_array_equal(out["x_perm"].double().numpy(), ctx["x_perm"])
    for key in ("A", "B", "H", "O"):
        assert rel_l2(out[key].double().numpy(), ctx[key]) <= TOL_Y, key
    assert rel_l2(out["y"].double().numpy(), y) <= TOL_Y
    assert rel_l2(out["dx"].double().numpy(), g["dx"]) <= TOL_Y
    for key in ("dW1", "dW3", "dW2", "dWg"):
        assert rel_l2(out[key].numpy(), g[key]) <= TOL_W, key


def test_fp8_layer_with_capacity(lib):
    cfg = small_config(name="fp8_cap", T=1024, h=512, f=1024, E=8, k=2, seed=2)
    inp = conditioned_inputs(cfg)
    cap = mb.capacity_for(cfg.T, cfg.k, cfg.E, 1.0)
    y, ctx = ref.layer_fwd_fp8(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                                  inp["W2"], cfg.k, capacity=cap)
    g = ref.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    assert int(ctx["offsets"][-1]) < cfg.T * cfg.k
    dev = _to(inp, "cuda")
    d = mb.dims_of(cfg, has_bias=False, capacity=cap)
    qw = _quant_weights(d, dev)
    run = LayerRun(d)
    ws = workspace(d, mb.OP_LAYER_FWD_FP8)
    mb.moe_layer_fwd_fp8(d, dev["x"], dev["Wg"], None, qw, run.y, run.saved, ws)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert mb.moe_read_device_status(ws) == mb.MOE_OK and run.status() == mb.MOE_OK
    out = run.outputs()
    assert rel_l2(out["y"].double().numpy(), y) <= TOL_Y
    assert rel_l2(out["dx"].double().numpy(), g["dx"]) <= TOL_Y
    for key in ("dW1", "dW3", "dW2", "dWg"):
        assert rel_l2(out[key].numpy(), g[key]) <= TOL_W, key
    # the sar context does not combine with the FP8 forward
    ds = mb.dims_of(cfg, has_bias=False, capacity=cap, sar=True)
    with pytest.raises(mb.MoeError) as err:
        mb.moe_layer_fwd_fp8(ds, dev["x"], dev["Wg"], None, qw, run.y, run.saved, ws)
    assert err.value.status == mb.MOE_ERR_UNSUPPORTED


def test_fp8_fullsize_sampled(lib):
    """The FP8 forward at the full Mixtral-shaped size, in the bench's launch
    configuration: routing and maps bit-exact; every code and scale of two
    experts' quantised weights bit-exact; A, B and y rows of tokens routed to
    those two experts against the FP8 oracle run on just those rows and
    experts (row scales are per row, column scales per expert, so the
    sampled computation is the full one restricted)."""
    from routing_grouped_expert_router_gb300 import synth
    from routing_grouped_expert_router_gb300.configs import CONFIGS
    cfg = CONFIGS["mixtral8x7b"]
    T, h, f, E, k = cfg.T, cfg.h, cfg.f, cfg.E, cfg.k
    inp = synth.make_layer(cfg, "cuda")
    x_cpu, _ = oracle.condition_router_margins(
        inp["x"].cpu(), inp["Wg"].cpu(), inp["b"].cpu(), k,
        lambda r, a: synth.replacement_x_rows(cfg, r, a))
    inp["x"] = x_cpu.cuda()
    d = mb.dims_of(cfg)
    qw = _quant_weights(d, inp)
    run = LayerRun(d)
    ws = workspace(d, mb.OP_LAYER_FWD_FP8)
    mb.moe_layer_fwd_fp8(d, inp["x"], inp["Wg"], None, qw, run.y, run.saved, ws)
    run.bwd(inp)
    torch.cuda.synchronize()
    assert mb.moe_read_device_status(ws) == mb.MOE_OK and run.status() == mb.MOE_OK

    idx, gates, _ = ref.route(x_cpu, inp["Wg"].cpu(), inp["b"].cpu(), k)
    counts, offsets, psrc, pdst = ref.dispatch(idx, E)
    np.testing.assert_array_equal(run.saved_view("topk_idx").cpu().numpy(), idx)
    np.testing.assert_array_equal(run.saved_view("perm_src").cpu().numpy(), psrc)

    pair = (0, 1)
    both = np.nonzero(np.all(np.isin(idx, pair), axis=1))[0]
    assert both.size >= 4
    toks = both[np.linspace(0, both.size - 1, 4).astype(int)]
    W13 = _view(d, qw, "W13q", (E, f // 128, 2, 128, h), torch.uint8)
    W2v = _view(d, qw, "W2q", (E, h, f), torch.uint8)
    s1v = _view(d, qw, "s1", (E, f), torch.float32).cpu().numpy()
    s3v = _view(d, qw, "s3", (E, f), torch.float32).cpu().numpy()
    s2v = _view(d, qw, "s2", (E, h), torch.float32).cpu().numpy()
    x64 = oracle.as_f64(x_cpu)
    O_rows = {}
    A_gpu = run.saved_view("A")
    B_gpu = run.saved_view("B")
    for e in pair:
        rows = [(int(t), j) for t in toks for j in range(k) if idx[t, j] == e]
        X = x64[[t for t, _ in rows]]
        f8 = ref.expert_ffn_fwd_fp8(X, np.array([0, len(rows)]), inp["W1"][e:e + 1].cpu(),
                                       inp["W3"][e:e + 1].cpu(), inp["W2"][e:e + 1].cpu())
        # the expert's quantised weights, every code and scale
        np.testing.assert_array_equal(s1v[e], f8["s1"][0])
        np.testing.assert_array_equal(s3v[e], f8["s3"][0])
        np.testing.assert_array_equal(s2v[e], f8["s2"][0])
        Wg = _codes(W13[e])
        np.testing.assert_array_equal(Wg[:, 0].reshape(f, h), f8["W1q"][0].T)
        np.testing.assert_array_equal(Wg[:, 1].reshape(f, h), f8["W3q"][0].T)
        np.testing.assert_array_equal(_codes(W2v[e]), f8["W2q"][0].T)
        prow = [int(pdst[t * k + j]) for t, j in rows]
        assert rel_l2(A_gpu[prow].double().cpu().numpy(), f8["A"]) <= 5e-3
        assert rel_l2(B_gpu[prow].double().cpu().numpy(), f8["B"]) <= 5e-3
        for i, key in enumerate(rows):
            O_rows[key] = f8["O"][i]
    y_ref = np.stack([sum(gates[t, j] * O_rows[(int(t), j)] for j in range(k)) for t in toks])
    assert rel_l2(run.y[torch.from_numpy(toks)].double().cpu().numpy(), y_ref) <= 5e-3


# --------------------------------------------------------- FP8 data gradients

def _bwd_weights(d, dev):
    qwb = torch.zeros(mb.moe_fp8_bwd_weight_bytes(d), dtype=torch.uint8, device="cuda")
    mb.moe_quantize_weights_fp8_bwd(d, dev["W1"], dev["W3"], qwb)
    return qwb


def _bview(d, qwb, name, shape, dtype):
    off = mb.moe_fp8_bwd_weight_view(d, qwb, name) - qwb.data_ptr()
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    return qwb[off:off + n].view(dtype).view(shape)


@pytest.mark.parametrize("f", [640, 4224, 16512])
def test_bwd_weight_codes_and_scales_bit_exact(lib, f):
    cfg = small_config(name="wqb", T=8, h=384, f=f, E=3, k=2, seed=23)
    inp = conditioned_inputs(cfg)
    d = mb.dims_of(cfg, has_bias=False)
    qwb = _bwd_weights(d, _to(inp, "cuda"))
    torch.cuda.synchronize()
    E, h, f = cfg.E, cfg.h, cfg.f
    W1r = _codes(_bview(d, qwb, "W1r", (E, h, f), torch.uint8))
    W3r = _codes(_bview(d, qwb, "W3r", (E, h, f), torch.uint8))
    s13r = _bview(d, qwb, "s13r", (E, h), torch.float32).cpu().numpy()
    for e in range(E):
        q1, q3, s13 = ref.quantize_rows_joint_e4m3(oracle.as_f64(inp["W1"][e]),
                                                      oracle.as_f64(inp["W3"][e]))
        np.testing.assert_array_equal(W1r[e], q1)
        np.testing.assert_array_equal(W3r[e], q3)
        np.testing.assert_array_equal(s13r[e], s13)


@pytest.mark.parametrize("name,fwd8", [("tiny", False), ("mixtral_mid", True),
                                       ("internal_mid_zipf", False), ("deepseek_mid", True),
                                       ("hunyuan_mid", True), ("one_token", False),
                                       ("ragged_tokens", True)])
def test_fp8_backward_matches_fp8_oracle(lib, name, fwd8):
    cfg = small_config(name=name, **CASES[name])
    inp = conditioned_inputs(cfg)
    fwd = ref.layer_fwd_fp8 if fwd8 else ref.layer_fwd
    y, ctx = fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], cfg.k)
    g = ref.layer_bwd_fp8(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    dev = _to(inp, "cuda")
    d = mb.dims_of(cfg, has_bias=cfg.zipf_s > 0)
    run = LayerRun(d)
    b = dev["b"] if d.has_bias else None
    if fwd8:
        qw = _quant_weights(d, dev)
        mb.moe_layer_fwd_fp8(d, dev["x"], dev["Wg"], b, qw, run.y, run.saved,
                             workspace(d, mb.OP_LAYER_FWD_FP8))
    else:
        run.fwd(dev)
    qwb = _bwd_weights(d, dev)
    wsb = workspace(d, mb.OP_LAYER_BWD_FP8)
    mb.moe_layer_bwd_fp8(d, dev["x"], dev["dy"], dev["Wg"], dev["W2"], qwb, run.saved, run.dx,
                         run.dWg, run.dW1, run.dW3, run.dW2, wsb)
    torch.cuda.synchronize()
    assert mb.moe_read_device_status(wsb) == mb.MOE_OK and run.status() == mb.MOE_OK
    out = run.outputs()
    assert rel_l2(out["y"].double().numpy(), y) <= TOL_Y
    assert rel_l2(out["dx"].double().numpy(), g["dx"]) <= TOL_Y
    for key in ("dW1", "dW3", "dW2", "dWg"):
        assert rel_l2(out[key].numpy(), g[key]) <= TOL_W, key
    if cfg.k == 1:
        assert torch.all(out["dWg"] == 0)


def test_fp8_backward_rejects_sar(lib):
    cfg = small_config(name="sarb", T=64, h=128, f=128, E=4, k=2, seed=3)
    d = mb.dims_of(cfg, has_bias=False, sar=True)
    dev = _to(conditioned_inputs(cfg), "cuda")
    run = LayerRun(d)
    qwb = _bwd_weights(mb.dims_of(cfg, has_bias=False), dev)
    with pytest.raises(mb.MoeError) as err:
        mb.moe_layer_bwd_fp8(d, dev["x"], dev["dy"], dev["Wg"], dev["W2"], qwb, run.saved,
                             run.dx, run.dWg, run.dW1, run.dW3, run.dW2,
                             workspace(mb.dims_of(cfg, has_bias=False), mb.OP_LAYER_BWD_FP8))
    assert err.value.status == mb.MOE_ERR_UNSUPPORTED


def test_fp8_backward_fullsize_sampled(lib):
    """The FP8 backward (e4m3 FC1 dgrad) at the full Mixtral-shaped size, after
    the bf16 forward, in the bench's launch configuration (`--fp8-dgrad`).

    Bit-exact: the row codes and scales of W1/W3 for two experts.  A token
    sample S (the first and last tokens, the edge rows of every expert, random
    tokens): each token's dx row depends on that token alone, so the oracle's
    expert forward and FP8 expert backward run on S's rows only, one expert
    at a time, and the router side of dx follows from them.  A second
    backward with dy zeroed outside S gives weight gradients from S alone,
    which the oracle computes in full for every expert S reaches."""
    from routing_grouped_expert_router_gb300 import synth
    from routing_grouped_expert_router_gb300.configs import CONFIGS
    cfg = CONFIGS["mixtral8x7b"]
    T, h, f, E, k = cfg.T, cfg.h, cfg.f, cfg.E, cfg.k
    inp = synth.make_layer(cfg, "cuda")
    x_cpu, _ = oracle.condition_router_margins(
        inp["x"].cpu(), inp["Wg"].cpu(), inp["b"].cpu(), k,
        lambda r, a: synth.replacement_x_rows(cfg, r, a))
    inp["x"] = x_cpu.cuda()
    d = mb.dims_of(cfg)
    run = LayerRun(d)
    run.fwd(inp)
    qwb = _bwd_weights(d, inp)
    wsb = workspace(d, mb.OP_LAYER_BWD_FP8)

    def bwd(dy):
        mb.moe_layer_bwd_fp8(d, inp["x"], dy, inp["Wg"], inp["W2"], qwb, run.saved, run.dx,
                             run.dWg, run.dW1, run.dW3, run.dW2, wsb)
        torch.cuda.synchronize()
        assert mb.moe_read_device_status(wsb) == mb.MOE_OK and run.status() == mb.MOE_OK

    bwd(inp["dy"])
    Wg_cpu, b_cpu = inp["Wg"].cpu(), inp["b"].cpu()
    idx, gates, _ = ref.route(x_cpu, Wg_cpu, b_cpu, k)
    counts, offsets, psrc, pdst = ref.dispatch(idx, E)
    np.testing.assert_array_equal(run.saved_view("topk_idx").cpu().numpy(), idx)

    # W1/W3 row codes and scales of the largest and the smallest expert
    W1r = _bview(d, qwb, "W1r", (E, h, f), torch.uint8)
    W3r = _bview(d, qwb, "W3r", (E, h, f), torch.uint8)
    s13r = _bview(d, qwb, "s13r", (E, h), torch.float32).cpu().numpy()
    big, small = int(np.argmax(counts)), int(np.argmin(counts))
    for e in {big, small}:
        q1, q3, s13 = ref.quantize_rows_joint_e4m3(oracle.as_f64(inp["W1"][e]),
                                                  oracle.as_f64(inp["W3"][e]))
        np.testing.assert_array_equal(_codes(W1r[e]), q1)
        np.testing.assert_array_equal(_codes(W3r[e]), q3)
        np.testing.assert_array_equal(s13r[e], s13)

    # the token sample
    toks = {0, T - 1}
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for r in (lo, hi - 1, lo + ((hi - lo - 1) // 256) * 256):
            if lo <= r < hi:
                toks.add(int(psrc[r]) // k)
    rng = np.random.default_rng(cfg.seed)
    while len(toks) < 64:
        toks.add(int(rng.integers(0, T)))
    S = np.array(sorted(toks))
    St = torch.from_numpy(S)
    n = len(S)
    dx_S = run.dx[St].cpu()

    # the masked backward: dy zeroed outside S
    mask = torch.zeros(T, 1, dtype=torch.bfloat16, device="cuda")
    mask[St.cuda()] = 1
    bwd(inp["dy"] * mask)

    # the oracle on S, one expert at a time
    xS = x_cpu[St]
    dyS = oracle.as_f64(inp["dy"][St.cuda()].cpu())
    gS = gates[S].astype(np.float64)
    iS = idx[S]
    dg = np.zeros(n * k)
    dX = np.zeros((n * k, h))
    for e in sorted(set(iS.ravel().tolist())):
        slots = np.nonzero(iS.ravel() == e)[0]
        rows = slots // k
        one = np.array([0, len(slots)], np.int32)
        W = (inp["W1"][e:e + 1].cpu(), inp["W3"][e:e + 1].cpu(), inp["W2"][e:e + 1].cpu())
        A, B, H, O = ref.expert_ffn_fwd(xS[torch.from_numpy(rows)], one, *W)
        dg[slots] = np.sum(dyS[rows] * O, axis=1)
        dO = ref.bf16_round(np.float32(gS.ravel()[slots])[:, None] * np.float32(dyS[rows]))
        bw = ref.expert_ffn_bwd_fp8(dO, xS[torch.from_numpy(rows)], one, *W, A, B, H)
        dX[slots] = bw["dX_perm"]
        assert rel_l2(oracle.as_f64(run.dW1[e]), bw["dW1"][0]) <= TOL_W, e
        assert rel_l2(oracle.as_f64(run.dW3[e]), bw["dW3"][0]) <= TOL_W, e
        assert rel_l2(oracle.as_f64(run.dW2[e]), bw["dW2"][0]) <= TOL_W, e
    tg = ref.token_grads(xS, Wg_cpu, iS, gates[S], np.arange(n * k, dtype=np.int32), dg, dX)
    assert rel_l2(dx_S.double().numpy(), tg["dx"]) <= TOL_Y
    for i in range(n):
        assert rel_l2(dx_S[i].double().numpy(), tg["dx"][i]) <= 2e-2, int(S[i])
    assert rel_l2(oracle.as_f64(run.dWg), tg["dWg"]) <= TOL_W
    # the masked run leaves every other dx row exactly zero
    others = torch.ones(T, dtype=torch.bool)
    others[St] = False
    assert torch.all(run.dx.cpu()[others] == 0)
