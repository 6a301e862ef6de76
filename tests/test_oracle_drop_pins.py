"""Pins of the oracle's dispatch variants (no GPU): per-expert capacity with
deterministic token dropping, and the local expert range of the all-gather
path's "scatter & drop".

Each test checks the oracle against a formulation it shares no code with:
a pure-Python one-pass counter, a dense masked mixture, torch autograd on the
masked mixture, and the identity that the partial outputs of disjoint expert
ranges sum to the whole layer.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import conditioned_inputs, small_config

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _python_keep(flat, E, cap, lo, hi):
    """One pass over the assignments in order; expert e keeps its first `cap`."""
    seen = [0] * E
    kept = []
    for a, e in enumerate(flat):
        if lo <= e < hi and seen[e] < cap:
            seen[e] += 1
            kept.append(a)
    return kept


@pytest.mark.parametrize("T,E,k,cap,rng_lo,rng_hi", [
    (50, 7, 3, 5, 0, 7), (200, 3, 2, 17, 0, 3), (33, 64, 6, 2, 0, 64),
    (40, 8, 2, 1000, 2, 5), (40, 8, 2, 4, 3, 8), (1, 4, 1, 0, 0, 4), (30, 6, 3, None, 6, 6),
])
def test_dispatch_with_drops_matches_python_counter(T, E, k, cap, rng_lo, rng_hi):
    rng = np.random.default_rng(T + E + k)
    # skewed choice so that some experts overflow the capacity
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.5
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)])
    idx = idx.astype(np.int32)
    flat = idx.ravel().tolist()
    c = T * k if cap is None else cap
    counts, offsets, psrc, pdst = oracle.dispatch(idx, E, cap, (rng_lo, rng_hi))
    kept = _python_keep(flat, E, c, rng_lo, rng_hi)
    expect = []
    for e in range(rng_lo, rng_hi):
        expect += [a for a in kept if flat[a] == e]
    assert psrc.tolist() == expect
    assert counts.tolist() == [sum(1 for a in kept if flat[a] == e) for e in range(rng_lo, rng_hi)]
    assert offsets.tolist() == [sum(counts[:i]) for i in range(rng_hi - rng_lo + 1)]
    assert all(cnt <= c for cnt in counts)
    for a in range(T * k):
        if a in kept:
            assert psrc[pdst[a]] == a
        else:
            assert pdst[a] == -1
    # dropped rows come back as zeros, kept ones bit-exactly
    x = rng.standard_normal((T, 5))
    back = oracle.unpermute_rows(oracle.permute_rows(x, psrc, k), pdst).reshape(T, k, 5)
    for a in range(T * k):
        want = x[a // k] if a in kept else np.zeros(5)
        np.testing.assert_array_equal(back[a // k, a % k], want)


def test_large_capacity_and_full_range_are_dropless():
    rng = np.random.default_rng(9)
    idx = np.stack([rng.choice(8, size=2, replace=False) for _ in range(100)]).astype(np.int32)
    ref = oracle.dispatch(idx, 8)
    for cap, ex in [(200, None), (None, (0, 8)), (10 ** 6, (0, 8))]:
        got = oracle.dispatch(idx, 8, cap, ex)
        for r, g in zip(ref, got):
            np.testing.assert_array_equal(r, g)
    assert ref[1][-1] == 200 and np.all(ref[3] >= 0)


def _kept_mask(topk_idx, E, cap):
    """[T, k] 0/1 mask of kept slots, from the pure-Python counter."""
    T, k = topk_idx.shape
    kept = set(_python_keep(topk_idx.ravel().tolist(), E, cap, 0, E))
    return np.array([[1.0 if t * k + j in kept else 0.0 for j in range(k)] for t in range(T)])


def _dense_masked_mixture(inp, k, mask):
    x = oracle.as_f64(inp["x"]); Wg = oracle.as_f64(inp["Wg"]); b = oracle.as_f64(inp["b"])
    W1 = oracle.as_f64(inp["W1"]); W3 = oracle.as_f64(inp["W3"]); W2 = oracle.as_f64(inp["W2"])
    T, E = x.shape[0], Wg.shape[1]
    logits = x @ Wg + b
    y = np.zeros_like(x)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        w = np.exp(logits[t, order] - logits[t, order].max())
        w = w / w.sum()
        for j, e in enumerate(order):
            if mask[t, j] == 0.0:
                continue
            a = x[t] @ W1[e]
            hh = a / (1 + np.exp(-a)) * (x[t] @ W3[e])
            y[t] += w[j] * (hh @ W2[e])
    return y


@pytest.mark.parametrize("E,k,cap", [(4, 2, 9), (6, 3, 7), (3, 1, 5), (4, 2, 1)])
def test_forward_with_drops_equals_dense_masked_mixture(E, k, cap):
    cfg = small_config(T=40, h=16, f=24, E=E, k=k, seed=300 + E * 10 + k)
    inp = conditioned_inputs(cfg)
    y, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                              inp["W2"], k, capacity=cap)
    mask = _kept_mask(ctx["topk_idx"], E, cap)
    assert mask.sum() < 40 * k, "the case must drop something"
    np.testing.assert_allclose(y, _dense_masked_mixture(inp, k, mask), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("E,k,cap,seed", [(4, 2, 10, 1), (6, 3, 8, 2), (5, 1, 4, 3)])
def test_backward_with_drops_matches_torch_autograd(E, k, cap, seed):
    cfg = small_config(T=36, h=16, f=24, E=E, k=k, seed=400 + seed)
    inp = conditioned_inputs(cfg)
    y, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                              inp["W2"], k, capacity=cap)
    g = oracle.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    mask = torch.from_numpy(_kept_mask(ctx["topk_idx"], E, cap))
    assert float(mask.sum()) < 36 * k
    x = inp["x"].double().requires_grad_(True)
    Wg = inp["Wg"].double().requires_grad_(True)
    W1 = inp["W1"].double().requires_grad_(True)
    W3 = inp["W3"].double().requires_grad_(True)
    W2 = inp["W2"].double().requires_grad_(True)
    logits = x @ Wg + inp["b"].double()
    sel = torch.topk(logits.detach(), k, dim=1).indices
    ps = torch.softmax(logits, dim=1).gather(1, sel)
    gates = ps / ps.sum(dim=1, keepdim=True)
    gates.retain_grad()
    out = torch.zeros_like(x)
    for j in range(k):
        e = sel[:, j]
        a = torch.einsum("th,thf->tf", x, W1[e])
        bb = torch.einsum("th,thf->tf", x, W3[e])
        o = torch.einsum("tf,tfh->th", torch.nn.functional.silu(a) * bb, W2[e])
        out = out + (mask[:, j:j + 1] * gates[:, j:j + 1]) * o
    (out * inp["dy"].double()).sum().backward()
    np.testing.assert_allclose(y, out.detach().numpy(), rtol=1e-12, atol=1e-12)
    ref = dict(dx=x.grad, dWg=Wg.grad, dW1=W1.grad, dW3=W3.grad, dW2=W2.grad)
    for key, v in ref.items():
        np.testing.assert_allclose(g[key], v.numpy(), rtol=1e-10, atol=1e-12, err_msg=key)
    # dL/dg is zero on a dropped slot and <dy, o> on a kept one
    np.testing.assert_allclose(g["dg"], gates.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.all(g["dg"][mask.numpy() == 0] == 0.0)


@pytest.mark.parametrize("E,k,ranges", [(8, 2, [(0, 3), (3, 8)]), (6, 3, [(0, 2), (2, 4), (4, 6)]),
                                        (4, 4, [(0, 1), (1, 4)])])
def test_local_ranges_sum_to_the_layer(E, k, ranges):
    """Scatter & drop per expert range, local GroupedGEMM, partial combine: the
    partial outputs of a partition of the experts add up to the whole layer
    (the reduce-scatter of the all-gather path, written as a plain sum)."""
    cfg = small_config(T=30, h=16, f=24, E=E, k=k, seed=500 + E)
    inp = conditioned_inputs(cfg)
    y, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                              inp["W2"], k)
    total = np.zeros_like(y)
    x64 = oracle.as_f64(inp["x"])
    for lo, hi in ranges:
        counts, offsets, psrc, pdst = oracle.dispatch(ctx["topk_idx"], E, None, (lo, hi))
        xp = oracle.permute_rows(x64, psrc, k)
        _, _, _, O = oracle.expert_ffn_fwd(xp, offsets, inp["W1"][lo:hi], inp["W3"][lo:hi],
                                           inp["W2"][lo:hi])
        total += oracle.combine(O, ctx["gates"], pdst, 30, k)
    np.testing.assert_allclose(total, y, rtol=1e-12, atol=1e-12)
