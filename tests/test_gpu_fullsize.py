"""Parity at the full workload sizes, in the launch configuration the
benchmark times (moe_layer_fwd + moe_layer_bwd on one stream).

Routing and dispatch are compared in full and bit-exactly (the oracle routes
every token).  Outputs the oracle cannot afford in full are sampled: whole
rows of y and dx for a few tokens (each token straight from the definition,
one expert at a time), and whole columns of dW1/dW3 and rows of dW2 for two
experts (from all of the expert's tokens).  dWg is checked exactly (it is 0)
for k = 1; other configs check it in full at reduced size in
test_gpu_parity.
"""
import numpy as np
import pytest
import torch

import oracle
from routing_grouped_expert_router_gb300 import binding as mb
from routing_grouped_expert_router_gb300 import build as mbuild
from routing_grouped_expert_router_gb300 import synth
from routing_grouped_expert_router_gb300.configs import CONFIGS
from tests.gpu_runner import LayerRun
from tests.helpers import rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    return mb.load()


def _f64(t):
    return t.detach().cpu().double().numpy()


@pytest.mark.parametrize("name", ["mixtral8x7b", "deepseekmoe", "internal352b", "hunyuan"])
def test_fullsize_sampled(lib, name):
    _check_fullsize(CONFIGS[name])


@pytest.mark.parametrize("name,factor,sar", [("mixtral8x7b", 0.0, True),
                                             ("internal352b", 1.0, False),
                                             ("deepseekmoe", 1.0, True)])
def test_fullsize_variants(lib, name, factor, sar):
    """The same sampled checks with a per-expert capacity (token dropping) and
    with the selective-rematerialisation context."""
    cfg = CONFIGS[name]
    cap = mb.capacity_for(cfg.T, cfg.k, cfg.E, factor) if factor else 0
    _check_fullsize(cfg, capacity=cap, sar=sar)


def _check_fullsize(cfg, capacity=0, sar=False):
    T, h, f, E, k = cfg.T, cfg.h, cfg.f, cfg.E, cfg.k
    inp = synth.make_layer(cfg, "cuda")
    x_cpu, n_fix = oracle.condition_router_margins(
        inp["x"].cpu(), inp["Wg"].cpu(), inp["b"].cpu(), k,
        lambda r, a: synth.replacement_x_rows(cfg, r, a))
    inp["x"] = x_cpu.cuda()
    d = mb.dims_of(cfg, capacity=capacity, sar=sar)
    run = LayerRun(d)
    run.fwd(inp)
    run.bwd(inp)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK

    # ---- routing and dispatch: every token, bit-exact
    Wg_cpu, b_cpu = inp["Wg"].cpu(), inp["b"].cpu()
    idx, gates, _ = oracle.route(x_cpu, Wg_cpu, b_cpu, k)
    counts, offsets, psrc, pdst = oracle.dispatch(idx, E, capacity or None)
    nkept = int(offsets[-1])
    if capacity:
        assert nkept < T * k, "the capacity must drop assignments"
    np.testing.assert_array_equal(run.saved_view("topk_idx").cpu().numpy(), idx)
    assert np.max(np.abs(_f64(run.saved_view("gates")) - gates)) <= 1e-5
    np.testing.assert_array_equal(run.saved_view("counts").cpu().numpy(), counts)
    np.testing.assert_array_equal(run.saved_view("offsets").cpu().numpy(), offsets)
    np.testing.assert_array_equal(run.saved_view("perm_src").cpu().numpy()[:nkept], psrc)
    np.testing.assert_array_equal(run.saved_view("perm_dst").cpu().numpy(), pdst)
    if cfg.zipf_s > 0 and not capacity:
        assert counts[-1] == 0 and counts[0] > 0.25 * T * k

    # ---- sampled tokens: y and dx rows
    rng = np.random.default_rng(cfg.seed)
    ntok = 4 if k >= 3 else 6
    toks = sorted(set([0, T - 1] + rng.choice(T, ntok - 2, replace=False).tolist()))
    if capacity:  # include tokens with dropped slots
        dropped = np.nonzero(np.any(pdst.reshape(T, k) < 0, axis=1))[0]
        toks = sorted(set(toks) | set(dropped[:: max(1, len(dropped) // 3)][:3].tolist()))
    dy_cpu = inp["dy"].cpu()
    needed = {}
    for t in toks:
        for j in range(k):
            needed.setdefault(int(idx[t, j]), []).append((t, j))
    terms = {}
    for e, pairs in sorted(needed.items()):
        W1e, W3e, W2e = _f64(inp["W1"][e]), _f64(inp["W3"][e]), _f64(inp["W2"][e])
        for (t, j) in pairs:
            terms[(t, j)] = oracle.expert_terms(oracle.as_f64(x_cpu[t]), oracle.as_f64(dy_cpu[t]),
                                                gates[t, j], W1e, W3e, W2e)
        del W1e, W3e, W2e
    y_ref, dx_ref = [], []
    zero = {"o": np.zeros((1, h)), "dg": np.zeros(1), "dx": np.zeros((1, h))}
    for t in toks:
        # a dropped slot adds nothing to y and has dg = 0
        tt = [terms[(t, j)] if pdst[t * k + j] >= 0 else zero for j in range(k)]
        r = oracle.assemble_token(gates[t], idx[t], tt, Wg_cpu)
        y_ref.append(r["y"])
        dx_ref.append(r["dx"])
    y_gpu = _f64(run.y[toks])
    dx_gpu = _f64(run.dx[toks])
    assert rel_l2(y_gpu, np.stack(y_ref)) <= 5e-3
    assert rel_l2(dx_gpu, np.stack(dx_ref)) <= 5e-3

    # ---- sampled weight-gradient columns for two experts
    live = np.nonzero(counts)[0]
    experts = sorted({int(live[np.argmax(counts[live])]), int(live[len(live) // 2])})
    cols = np.array(sorted({0, 1, 127, 128, f // 2, f - 1}))
    g_flat = gates.ravel()
    for e in experts:
        a = psrc[offsets[e]:offsets[e + 1]].astype(np.int64)
        tk = a // k
        X_e = oracle.as_f64(x_cpu[torch.from_numpy(tk)])
        dO_e = g_flat[a][:, None] * oracle.as_f64(dy_cpu[torch.from_numpy(tk)])
        W1c = _f64(inp["W1"][e][:, cols])
        W3c = _f64(inp["W3"][e][:, cols])
        W2r = _f64(inp["W2"][e][cols, :])
        # expert_wgrad_columns indexes its weights by `cols`; hand it the slices
        w = oracle.expert_wgrad_columns(X_e, dO_e, W1c, W3c, W2r, np.arange(len(cols)))
        assert rel_l2(_f64(run.dW1[e][:, cols]), w["dW1"]) <= 1e-2, e
        assert rel_l2(_f64(run.dW3[e][:, cols]), w["dW3"]) <= 1e-2, e
        assert rel_l2(_f64(run.dW2[e][cols, :]), w["dW2"]) <= 1e-2, e
    for e in np.nonzero(counts == 0)[0]:
        assert torch.all(run.dW1[e] == 0) and torch.all(run.dW2[e] == 0)
    if k == 1:
        assert torch.all(run.dWg == 0)
