"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not share code with:
a dense brute-force mixture, torch autograd, central finite differences,
closed forms printed on the pages, library routines (scipy softmax, torch
silu), pure-Python brute force and exact scaling identities.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from routing_grouped_expert_router_gb300 import synth
from routing_grouped_expert_router_gb300.configs import CONFIGS
from tests.helpers import conditioned_inputs, small_config, rel_l2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _run(inp, k, counter=None):
    y, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                              inp["W2"], k, counter)
    g = oracle.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"],
                         inp["W2"], ctx, counter)
    return y, ctx, g


# ------------------------------------------------------------- generator ---

def test_splitmix64_published_first_output():
    # splitmix64 seeded with state 0 first returns 0xE220A8397B1DCDAF.
    assert synth.splitmix64_py(synth.GAMMA) == 0xE220A8397B1DCDAF


def test_generator_deterministic_and_distinct():
    a = synth.normal(5, 1, (64, 32), 1.0, torch.bfloat16)
    b = synth.normal(5, 1, (64, 32), 1.0, torch.bfloat16)
    c = synth.normal(5, 2, (64, 32), 1.0, torch.bfloat16)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a, c)
    r = synth.rows(5, 1, [3, 7], 32, 1.0, torch.bfloat16)
    assert torch.equal(r, a[[3, 7]])
    big = synth.normal(9, 1, (200000,), 1.0, torch.float64).numpy()
    assert abs(big.mean()) < 0.01 and abs(big.std() - 1.0) < 0.01


# ------------------------------------------------------- forward: dense ---

def _dense_mixture(inp, k):
    """Every token through every expert, masked by its gates (no dispatch)."""
    x = oracle.as_f64(inp["x"]); Wg = oracle.as_f64(inp["Wg"]); b = oracle.as_f64(inp["b"])
    W1 = oracle.as_f64(inp["W1"]); W3 = oracle.as_f64(inp["W3"]); W2 = oracle.as_f64(inp["W2"])
    T, E = x.shape[0], Wg.shape[1]
    logits = x @ Wg + b
    y = np.zeros_like(x)
    for t in range(T):
        # pure-Python selection: k largest, ties to the lower id
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        w = np.exp(logits[t, order] - logits[t, order].max())
        w = w / w.sum()
        for e in range(E):
            m = w[order.index(e)] if e in order else 0.0
            a = x[t] @ W1[e]
            hh = a / (1 + np.exp(-a)) * (x[t] @ W3[e])
            y[t] += m * (hh @ W2[e])
    return y


@pytest.mark.parametrize("E,k", [(4, 2), (6, 3), (3, 1), (4, 4), (1, 1)])
def test_forward_equals_dense_bruteforce(E, k):
    cfg = small_config(T=40, h=16, f=24, E=E, k=k, seed=100 + E * 10 + k)
    inp = conditioned_inputs(cfg)
    y, _ = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                            inp["W2"], k)
    np.testing.assert_allclose(y, _dense_mixture(inp, k), rtol=1e-12, atol=1e-12)


def test_e1_k1_is_textbook_swiglu_ffn():
    cfg = small_config(T=32, h=16, f=40, E=1, k=1, seed=7)
    inp = conditioned_inputs(cfg)
    y, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                              inp["W2"], 1)
    x = inp["x"].double()
    ref = (torch.nn.functional.silu(x @ inp["W1"][0].double()) * (x @ inp["W3"][0].double())) \
        @ inp["W2"][0].double()
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(ctx["gates"] == 1.0)


# ------------------------------------------------ backward: torch autograd ---

def _autograd_layer(inp, k):
    """Independent float64 autograd formulation of the same layer."""
    x = inp["x"].double().requires_grad_(True)
    Wg = inp["Wg"].double().requires_grad_(True)
    W1 = inp["W1"].double().requires_grad_(True)
    W3 = inp["W3"].double().requires_grad_(True)
    W2 = inp["W2"].double().requires_grad_(True)
    b = inp["b"].double()
    logits = x @ Wg + b
    sel = torch.topk(logits.detach(), k, dim=1).indices
    p = torch.softmax(logits, dim=1)
    ps = p.gather(1, sel)
    gates = ps / ps.sum(dim=1, keepdim=True)
    gates.retain_grad()
    y = torch.zeros_like(x)
    for j in range(k):
        e = sel[:, j]
        a = torch.einsum("th,thf->tf", x, W1[e])
        bb = torch.einsum("th,thf->tf", x, W3[e])
        o = torch.einsum("tf,tfh->th", torch.nn.functional.silu(a) * bb, W2[e])
        y = y + gates[:, j:j + 1] * o
    loss = (y * inp["dy"].double()).sum()
    loss.backward()
    return dict(y=y.detach(), dx=x.grad, dWg=Wg.grad, dW1=W1.grad, dW3=W3.grad,
                dW2=W2.grad, dg=gates.grad, sel=sel)


@pytest.mark.parametrize("E,k,seed", [(4, 2, 1), (6, 3, 2), (5, 1, 3), (3, 3, 4)])
def test_backward_matches_torch_autograd(E, k, seed):
    cfg = small_config(T=36, h=16, f=24, E=E, k=k, seed=seed)
    inp = conditioned_inputs(cfg)
    y, ctx, g = _run(inp, k)
    ref = _autograd_layer(inp, k)
    np.testing.assert_array_equal(ctx["topk_idx"], ref["sel"].numpy())
    np.testing.assert_allclose(y, ref["y"].numpy(), rtol=1e-12, atol=1e-12)
    for key in ("dx", "dWg", "dW1", "dW3", "dW2", "dg"):
        np.testing.assert_allclose(g[key], ref[key].numpy(), rtol=1e-10, atol=1e-12,
                                   err_msg=key)


# ------------------------------------------------ backward: finite diffs ---

def test_finite_differences():
    k = 2
    cfg = small_config(T=12, h=8, f=16, E=4, k=k, seed=21)
    inp = conditioned_inputs(cfg)
    dyf = oracle.as_f64(inp["dy"])
    y0, ctx, g = _run(inp, k)
    rng = np.random.default_rng(0)

    def loss(vals):
        y, c = oracle.layer_fwd(vals["x"], vals["Wg"], inp["b"], vals["W1"],
                                vals["W3"], vals["W2"], k)
        assert np.array_equal(c["topk_idx"], ctx["topk_idx"])
        return float((y * dyf).sum())

    base = {n: torch.from_numpy(oracle.as_f64(inp[n])) for n in ("x", "Wg", "W1", "W3", "W2")}
    grads = {"x": g["dx"], "Wg": g["dWg"], "W1": g["dW1"], "W3": g["dW3"], "W2": g["dW2"]}
    eps = 1e-5
    for name, grad in grads.items():
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in grad.shape)
            plus = {n: v.clone() for n, v in base.items()}
            minus = {n: v.clone() for n, v in base.items()}
            plus[name][idx] += eps
            minus[name][idx] -= eps
            fd = (loss(plus) - loss(minus)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (name, idx, fd, grad[idx])


# ------------------------------------------------------------- routing ---

def test_routing_decision_matches_float64_bruteforce():
    cfg = small_config(T=400, h=64, f=16, E=16, k=4, seed=31)
    inp = conditioned_inputs(cfg)
    idx, gates, l64 = oracle.route(inp["x"], inp["Wg"], inp["b"], cfg.k)
    for t in range(cfg.T):
        order = sorted(range(cfg.E), key=lambda e: (-l64[t, e], e))[:cfg.k]
        assert list(idx[t]) == order
    np.testing.assert_allclose(gates.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(oracle.router_margin(l64, cfg.k) >= 1e-3)


def test_gates_are_softmax_over_selected_logits():
    from scipy.special import softmax
    cfg = small_config(T=64, h=32, f=16, E=8, k=3, seed=41)
    inp = conditioned_inputs(cfg)
    idx, gates, l64 = oracle.route(inp["x"], inp["Wg"], inp["b"], cfg.k)
    sel = np.take_along_axis(l64, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(gates, softmax(sel, axis=1), rtol=1e-13)
    assert np.all(np.diff(sel, axis=1) < 0)


def test_k_equals_E_gives_full_softmax():
    from scipy.special import softmax
    cfg = small_config(T=32, h=16, f=16, E=5, k=5, seed=51)
    inp = conditioned_inputs(cfg)
    idx, gates, l64 = oracle.route(inp["x"], inp["Wg"], inp["b"], 5)
    full = softmax(l64, axis=1)
    np.testing.assert_allclose(gates, np.take_along_axis(full, idx.astype(np.int64), 1),
                               rtol=1e-13)


def test_ties_go_to_lower_expert_id():
    x = synth.normal(1, 1, (8, 16), 1.0, torch.bfloat16)
    col = synth.normal(1, 2, (16, 1), 0.25, torch.float32)
    other = synth.normal(1, 3, (16, 1), 0.25, torch.float32)
    # experts 1 and 3 share a column; experts 0 and 2 are pushed far below
    Wg = torch.cat([other, col, other, col], dim=1)
    b = torch.tensor([-100.0, 0.0, -100.0, 0.0])
    idx, gates, _ = oracle.route(x, Wg, b, 2)
    assert np.all(idx == np.array([1, 3]))
    np.testing.assert_allclose(gates, 0.5, rtol=0, atol=0)


def test_k1_gates_exactly_one_and_router_grad_zero():
    cfg = small_config(T=40, h=16, f=16, E=6, k=1, seed=61)
    inp = conditioned_inputs(cfg)
    _, ctx, g = _run(inp, 1)
    assert np.all(ctx["gates"] == 1.0)
    assert np.all(g["dWg"] == 0.0) and np.all(g["dl"] == 0.0)


def test_zipf_bias_shapes_load():
    base = CONFIGS["internal352b"]
    cfg = small_config(T=2048, h=512, f=64, E=base.E, k=base.k, seed=base.seed,
                       zipf_s=base.zipf_s)
    inp = synth.make_layer(cfg, with_dy=False)
    idx, _, _ = oracle.route(inp["x"], inp["Wg"], inp["b"], cfg.k)
    counts = np.bincount(idx.ravel(), minlength=cfg.E)
    assert counts[-1] == 0
    share = counts / counts.sum()
    assert 0.25 < share[0] < 0.40
    assert np.all(np.diff(share[:8]) < 0)  # head of the ranking falls monotonically


# ------------------------------------------------------------ dispatch ---

def test_dispatch_matches_python_counting_sort():
    rng = np.random.default_rng(3)
    for T, E, k in [(50, 7, 3), (1, 4, 1), (200, 3, 2), (33, 64, 6)]:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        counts, offsets, psrc, pdst = oracle.dispatch(idx, E)
        flat = idx.ravel().tolist()
        expect = []
        for e in range(E):
            for a, ee in enumerate(flat):
                if ee == e:
                    expect.append(a)
        assert psrc.tolist() == expect
        assert counts.sum() == T * k and offsets[-1] == T * k
        assert offsets.tolist() == [sum(counts[:e]) for e in range(E + 1)]
        assert sorted(pdst.tolist()) == list(range(T * k))
        assert all(psrc[pdst[a]] == a for a in range(T * k))
        x = rng.standard_normal((T, 5))
        xp = oracle.permute_rows(x, psrc, k)
        back = oracle.unpermute_rows(xp, pdst)
        np.testing.assert_array_equal(back.reshape(T, k, 5), np.repeat(x[:, None], k, 1))


# ------------------------------------------------------- scaling / sums ---

def test_exact_scaling_identities():
    k = 2
    cfg = small_config(T=30, h=16, f=24, E=4, k=k, seed=71)
    inp = conditioned_inputs(cfg)
    y, _, g = _run(inp, k)
    inp2 = dict(inp); inp2["W2"] = inp["W2"].double() * 2
    y2, _, _ = _run(inp2, k)
    np.testing.assert_array_equal(y2, 2 * y)
    inp3 = dict(inp); inp3["dy"] = inp["dy"].double() * 2
    _, _, g3 = _run(inp3, k)
    for key in ("dx", "dWg", "dW1", "dW3", "dW2", "dg"):
        np.testing.assert_array_equal(g3[key], 2 * g[key], err_msg=key)
    # permuting tokens permutes y
    perm = torch.randperm(cfg.T, generator=torch.Generator().manual_seed(0))
    inp4 = dict(inp); inp4["x"] = inp["x"][perm]
    y4, _ = oracle.layer_fwd(inp4["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                             inp["W2"], k)
    np.testing.assert_allclose(y4, y[perm.numpy()], rtol=1e-13, atol=1e-13)


def test_mac_counter_matches_closed_form():
    for (T, h, f, E, k) in [(40, 16, 24, 4, 2), (33, 8, 16, 6, 3), (20, 8, 8, 3, 1)]:
        cfg = small_config(T=T, h=h, f=f, E=E, k=k, seed=T)
        inp = conditioned_inputs(cfg)
        c = oracle.moe_oracle.MacCounter()
        _, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                                  inp["W2"], k, c)
        assert c.macs == oracle.gemm_macs_fwd(T, h, f, k) == cfg.gemm_macs_fwd()
        c2 = oracle.moe_oracle.MacCounter()
        oracle.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"],
                         ctx, c2)
        assert c2.macs == 2 * oracle.gemm_macs_fwd(T, h, f, k)


# ------------------------------------------------- sampled / per-token forms ---

def test_token_forms_match_layer():
    k = 3
    cfg = small_config(T=24, h=16, f=32, E=5, k=k, seed=81)
    inp = conditioned_inputs(cfg)
    y, ctx, g = _run(inp, k)
    W1, W3, W2 = (oracle.as_f64(inp[n]) for n in ("W1", "W3", "W2"))
    for t in (0, 5, 23):
        r = oracle.token_fwd_bwd(inp["x"][t], inp["dy"][t], inp["Wg"], inp["b"], k,
                                 lambda e: (W1[e], W3[e], W2[e]))
        np.testing.assert_array_equal(r["topk_idx"], ctx["topk_idx"][t])
        np.testing.assert_allclose(r["y"], y[t], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["dx"], g["dx"][t], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(r["dg"], g["dg"][t], rtol=1e-12, atol=1e-12)
    for e in range(cfg.E):
        lo, hi = ctx["offsets"][e], ctx["offsets"][e + 1]
        cols = [0, 7, 31]
        w = oracle.expert_wgrad_columns(ctx["x_perm"][lo:hi], g["dO"][lo:hi],
                                        W1[e], W3[e], W2[e], cols)
        np.testing.assert_allclose(w["dW1"], g["dW1"][e][:, cols], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(w["dW3"], g["dW3"][e][:, cols], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(w["dW2"], g["dW2"][e][cols, :], rtol=1e-11, atol=1e-12)


def test_margin_conditioning_enforces_margin():
    cfg = small_config(T=3000, h=32, f=8, E=64, k=6, seed=91)
    inp = synth.make_layer(cfg, with_dy=False)
    l64, _ = oracle.router_logits(inp["x"], inp["Wg"], inp["b"])
    assert np.any(oracle.router_margin(l64, cfg.k) < 1e-3)   # raw draws do have near-ties
    c = conditioned_inputs(cfg)
    l64c, _ = oracle.router_logits(c["x"], c["Wg"], c["b"])
    assert c["n_resampled"] > 0
    assert np.all(oracle.router_margin(l64c, cfg.k) >= 1e-3)


# ------------------------------------------------------ printed values ---

def test_pages_worked_byte_values():
    gv = json.load(open(os.path.join(GOLDEN, "digest_worked_values.json")))
    a = gv["activation"]
    assert round(oracle.activation_bytes(a["b"], a["s"], a["h"], a["elem_bytes"]) / 1e6, 1) \
        == a["printed_MB"]
    d = gv["dispatch_per_token"]
    assert oracle.dispatch_bytes_per_token(d["k"], d["h"], d["elem_bytes"]) == d["printed_bytes"]
    th = gv["throughput"]
    from routing_grouped_expert_router_gb300.metrics import tokens_per_s
    v = tokens_per_s(th["seqs_per_step"] * th["seq_len"], th["step_s"] * 1e3)
    assert round(v / 1e6, 2) == th["printed_M_tokens_per_s"]


def test_configs_follow_model_table():
    table = json.load(open(os.path.join(GOLDEN, "model_table.json")))["rows"]
    pairs = {"deepseekmoe": "DeepSeekMoE", "mixtral8x7b": "Mixtral-8x7B",
             "internal352b": "Internal-352B", "hunyuan": "Hunyuan-Large"}
    for name, row in pairs.items():
        c, r = CONFIGS[name], table[row]
        assert (c.h, c.f, c.E, c.k) == (r["h"], r["h_ffn"], r["experts"], r["top_k"])
