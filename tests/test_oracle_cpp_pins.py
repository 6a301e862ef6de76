"""Pins of the C++ oracle (the oracle of record) to facts outside itself (no GPU).

The C++ oracle runs its templates in two precisions: "f32" (bf16 inputs, fp32
accumulation and intermediates: the record) and "f64" (double throughout, for
finite differences).  Each test checks one of them against something it shares
no code with: a dense brute-force mixture, torch autograd, central finite
differences, library routines (scipy softmax, torch silu, torch's bf16 and
float8_e4m3fn conversions), a pure-Python counting sort and exact identities.
The float64 numpy oracle is a second, independent implementation; the two are
also compared with each other.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.cref as cref
from routing_grouped_expert_router_gb300 import synth
from tests.helpers import conditioned_inputs, rel_l2, small_config
from tests.test_oracle_drop_pins import _dense_masked_mixture, _kept_mask, _python_keep
from tests.test_oracle_pins import _autograd_layer, _dense_mixture

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

# fp32 accumulation over contractions of a few dozen terms: ~1e-7 relative;
# a dropped term, a wrong sign or a swapped operand moves results by O(1)
TOL32 = 1e-5


def _run(inp, k, prec, capacity=None):
    y, ctx = cref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], k,
                            capacity=capacity, prec=prec)
    g = cref.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    return y, ctx, g


# ------------------------------------------------------- forward: dense ---

@pytest.mark.parametrize("E,k", [(4, 2), (6, 3), (3, 1), (4, 4), (1, 1)])
def test_forward_equals_dense_bruteforce(E, k):
    cfg = small_config(T=40, h=16, f=24, E=E, k=k, seed=100 + E * 10 + k)
    inp = conditioned_inputs(cfg)
    ref = _dense_mixture(inp, k)
    y64, _ = cref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], k,
                            prec="f64")
    np.testing.assert_allclose(y64, ref, rtol=1e-12, atol=1e-12)
    y32, _ = cref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], k)
    assert y32.dtype == np.float32
    assert rel_l2(y32, ref) <= TOL32


def test_e1_k1_is_textbook_swiglu_ffn():
    cfg = small_config(T=32, h=16, f=40, E=1, k=1, seed=7)
    inp = conditioned_inputs(cfg)
    x = inp["x"].double()
    ref = (torch.nn.functional.silu(x @ inp["W1"][0].double()) * (x @ inp["W3"][0].double())) \
        @ inp["W2"][0].double()
    for prec, tol in (("f64", 1e-12), ("f32", TOL32)):
        y, ctx = cref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"],
                                1, prec=prec)
        assert rel_l2(y, ref.numpy()) <= tol
        assert np.all(ctx["gates"] == 1.0)


# ------------------------------------------------ backward: torch autograd ---

@pytest.mark.parametrize("E,k,seed", [(4, 2, 1), (6, 3, 2), (5, 1, 3), (3, 3, 4)])
def test_backward_matches_torch_autograd(E, k, seed):
    cfg = small_config(T=36, h=16, f=24, E=E, k=k, seed=seed)
    inp = conditioned_inputs(cfg)
    ref = _autograd_layer(inp, k)
    for prec in ("f64", "f32"):
        y, ctx, g = _run(inp, k, prec)
        np.testing.assert_array_equal(ctx["topk_idx"], ref["sel"].numpy())
        for key in ("dx", "dWg", "dW1", "dW3", "dW2", "dg"):
            r = ref[key].numpy()
            if prec == "f64":
                np.testing.assert_allclose(g[key], r, rtol=1e-10, atol=1e-12, err_msg=key)
            else:
                assert g[key].dtype == np.float32
                if k == 1 and key == "dWg":
                    # 0 exactly here; autograd leaves float64 round-off (~1e-16)
                    assert np.all(g[key] == 0) and np.max(np.abs(r)) < 1e-12
                    continue
                assert rel_l2(g[key], r) <= TOL32, key


def test_backward_with_drops_matches_torch_autograd():
    E, k, cap = 6, 3, 8
    cfg = small_config(T=36, h=16, f=24, E=E, k=k, seed=402)
    inp = conditioned_inputs(cfg)
    y, ctx, g = _run(inp, k, "f64", capacity=cap)
    mask = _kept_mask(ctx["topk_idx"], E, cap)
    assert mask.sum() < 36 * k
    np.testing.assert_allclose(y, _dense_masked_mixture(inp, k, mask), rtol=1e-12, atol=1e-12)
    # gradients: autograd of the masked mixture
    m = torch.from_numpy(mask)
    x = inp["x"].double().requires_grad_(True)
    Wg = inp["Wg"].double().requires_grad_(True)
    W1 = inp["W1"].double().requires_grad_(True)
    W3 = inp["W3"].double().requires_grad_(True)
    W2 = inp["W2"].double().requires_grad_(True)
    logits = x @ Wg + inp["b"].double()
    sel = torch.topk(logits.detach(), k, dim=1).indices
    ps = torch.softmax(logits, dim=1).gather(1, sel)
    gates = ps / ps.sum(dim=1, keepdim=True)
    out = torch.zeros_like(x)
    for j in range(k):
        e = sel[:, j]
        a = torch.einsum("th,thf->tf", x, W1[e])
        bb = torch.einsum("th,thf->tf", x, W3[e])
        o = torch.einsum("tf,tfh->th", torch.nn.functional.silu(a) * bb, W2[e])
        out = out + (m[:, j:j + 1] * gates[:, j:j + 1]) * o
    (out * inp["dy"].double()).sum().backward()
    for key, v in dict(dx=x.grad, dWg=Wg.grad, dW1=W1.grad, dW3=W3.grad, dW2=W2.grad).items():
        np.testing.assert_allclose(g[key], v.numpy(), rtol=1e-10, atol=1e-12, err_msg=key)
    assert np.all(g["dg"][mask == 0] == 0.0)


# ------------------------------------------------ backward: finite diffs ---

def test_finite_differences_f64():
    k = 2
    cfg = small_config(T=12, h=8, f=16, E=4, k=k, seed=21)
    inp = conditioned_inputs(cfg)
    base = {n: oracle.as_f64(inp[n]) for n in ("x", "Wg", "W1", "W3", "W2", "dy", "b")}
    y0, ctx = cref.layer_fwd(base["x"], base["Wg"], base["b"], base["W1"], base["W3"],
                             base["W2"], k, prec="f64")
    g = cref.layer_bwd(base["dy"], base["x"], base["Wg"], base["W1"], base["W3"], base["W2"],
                       ctx)
    rng = np.random.default_rng(0)

    def loss(vals):
        y, c = cref.layer_fwd(vals["x"], vals["Wg"], base["b"], vals["W1"], vals["W3"],
                              vals["W2"], k, prec="f64")
        assert np.array_equal(c["topk_idx"], ctx["topk_idx"])
        return float((y * base["dy"]).sum())

    grads = {"x": g["dx"], "Wg": g["dWg"], "W1": g["dW1"], "W3": g["dW3"], "W2": g["dW2"]}
    eps = 1e-5
    for name, grad in grads.items():
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in grad.shape)
            plus = {n: v.copy() for n, v in base.items()}
            minus = {n: v.copy() for n, v in base.items()}
            plus[name][idx] += eps
            minus[name][idx] -= eps
            fd = (loss(plus) - loss(minus)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (name, idx, fd)


# ------------------------------------------------------------- routing ---

def test_routing_decision_matches_float64_bruteforce():
    cfg = small_config(T=400, h=64, f=16, E=16, k=4, seed=31)
    inp = conditioned_inputs(cfg)
    l64 = oracle.as_f64(inp["x"]) @ oracle.as_f64(inp["Wg"]) + oracle.as_f64(inp["b"])
    for prec in ("f32", "f64"):
        idx, gates, _ = cref.route(inp["x"], inp["Wg"], inp["b"], cfg.k, prec)
        for t in range(cfg.T):
            order = sorted(range(cfg.E), key=lambda e: (-l64[t, e], e))[:cfg.k]
            assert list(idx[t]) == order
        np.testing.assert_allclose(gates.sum(axis=1), 1.0, rtol=0,
                                   atol=1e-6 if prec == "f32" else 1e-12)


def test_gates_are_softmax_over_selected_logits():
    from scipy.special import softmax
    cfg = small_config(T=64, h=32, f=16, E=8, k=3, seed=41)
    inp = conditioned_inputs(cfg)
    l64 = oracle.as_f64(inp["x"]) @ oracle.as_f64(inp["Wg"]) + oracle.as_f64(inp["b"])
    for prec, tol in (("f64", 1e-13), ("f32", 2e-6)):
        idx, gates, logits = cref.route(inp["x"], inp["Wg"], inp["b"], cfg.k, prec)
        sel = np.take_along_axis(l64, idx.astype(np.int64), axis=1)
        np.testing.assert_allclose(gates, softmax(sel, axis=1), rtol=tol, atol=tol)
        assert np.all(np.diff(sel, axis=1) < 0)
        np.testing.assert_allclose(logits, l64, rtol=0, atol=1e-5 if prec == "f32" else 1e-12)


def test_k_equals_E_gives_full_softmax():
    from scipy.special import softmax
    cfg = small_config(T=32, h=16, f=16, E=5, k=5, seed=51)
    inp = conditioned_inputs(cfg)
    idx, gates, l64 = cref.route(inp["x"], inp["Wg"], inp["b"], 5, "f64")
    full = softmax(l64, axis=1)
    np.testing.assert_allclose(gates, np.take_along_axis(full, idx.astype(np.int64), 1),
                               rtol=1e-13)


def test_ties_go_to_lower_expert_id():
    x = synth.normal(1, 1, (8, 16), 1.0, torch.bfloat16)
    col = synth.normal(1, 2, (16, 1), 0.25, torch.float32)
    other = synth.normal(1, 3, (16, 1), 0.25, torch.float32)
    Wg = torch.cat([other, col, other, col], dim=1)
    b = torch.tensor([-100.0, 0.0, -100.0, 0.0])
    for prec in ("f32", "f64"):
        idx, gates, _ = cref.route(x, Wg, b, 2, prec)
        assert np.all(idx == np.array([1, 3]))
        np.testing.assert_array_equal(gates, 0.5)


def test_k1_gates_exactly_one_and_router_grad_zero():
    cfg = small_config(T=40, h=16, f=16, E=6, k=1, seed=61)
    inp = conditioned_inputs(cfg)
    for prec in ("f32", "f64"):
        _, ctx, g = _run(inp, 1, prec)
        assert np.all(ctx["gates"] == 1.0)
        assert np.all(g["dWg"] == 0.0) and np.all(g["dl"] == 0.0)


def test_router_bwd_is_softmax_jacobian():
    """dl = J^T dg with J the Jacobian of softmax over the selected logits
    (torch autograd of torch.softmax)."""
    rng = np.random.default_rng(12)
    l = torch.from_numpy(rng.standard_normal((20, 4))).requires_grad_(True)
    g = torch.softmax(l, dim=1)
    dg = torch.from_numpy(rng.standard_normal((20, 4)))
    (g * dg).sum().backward()
    for prec, tol in (("f64", 1e-14), ("f32", 1e-6)):
        dl = cref.router_bwd(g.detach().numpy(), dg.numpy(), prec)
        np.testing.assert_allclose(dl, l.grad.numpy(), rtol=tol, atol=tol)


# ------------------------------------------------------------ dispatch ---

@pytest.mark.parametrize("T,E,k,cap,lo,hi", [
    (50, 7, 3, None, 0, 7), (200, 3, 2, 17, 0, 3), (33, 64, 6, 2, 0, 64),
    (40, 8, 2, 1000, 2, 5), (40, 8, 2, 4, 3, 8), (1, 4, 1, 0, 0, 4), (30, 6, 3, None, 6, 6),
])
def test_dispatch_matches_python_counter(T, E, k, cap, lo, hi):
    rng = np.random.default_rng(T + E + k)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.5
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)])
    idx = idx.astype(np.int32)
    flat = idx.ravel().tolist()
    c = T * k if cap is None else cap
    counts, offsets, psrc, pdst = cref.dispatch(idx, E, cap, (lo, hi))
    kept = _python_keep(flat, E, c, lo, hi)
    expect = []
    for e in range(lo, hi):
        expect += [a for a in kept if flat[a] == e]
    assert psrc.tolist() == expect
    assert counts.tolist() == [sum(1 for a in kept if flat[a] == e) for e in range(lo, hi)]
    assert offsets.tolist() == [sum(counts[:i]) for i in range(hi - lo + 1)]
    for a in range(T * k):
        assert (psrc[pdst[a]] == a) if a in kept else (pdst[a] == -1)
    # the rows move bit-exactly, and unpermute(permute(x)) repeats every kept row
    x = synth.normal(3, 1, (T, 8), 1.0, torch.bfloat16)
    xp = cref.permute_rows(x, psrc, k)
    back = cref.unpermute_rows(xp, pdst).reshape(T, k, 8)
    xf = x.float().numpy()
    for a in range(T * k):
        want = xf[a // k] if a in kept else np.zeros(8, np.float32)
        np.testing.assert_array_equal(back[a // k, a % k], want)


def test_dispatch_keep_mask_drops_exactly_the_masked_slots():
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(6, size=2, replace=False) for _ in range(40)]).astype(np.int32)
    keep = rng.random((40, 2)) < 0.7
    counts, offsets, psrc, pdst = cref.dispatch(idx, 6, keep=keep)
    flat = idx.ravel()
    kept = [a for a in range(80) if keep.ravel()[a]]
    assert psrc.tolist() == [a for e in range(6) for a in kept if flat[a] == e]
    assert np.all(pdst[~keep.ravel()] == -1)
    with pytest.raises(ValueError):
        cref.dispatch(np.array([[0, 7]], np.int32), 6)


# ------------------------------------------------------- scaling / sums ---

def test_exact_scaling_identities_f32():
    """Doubling W2 doubles y exactly and doubling dy doubles every gradient
    exactly: both only change exponents in fp32."""
    k = 2
    cfg = small_config(T=30, h=16, f=24, E=4, k=k, seed=71)
    inp = conditioned_inputs(cfg)
    y, _, g = _run(inp, k, "f32")
    inp2 = dict(inp); inp2["W2"] = (inp["W2"].float() * 2).to(torch.bfloat16)
    y2, _, _ = _run(inp2, k, "f32")
    np.testing.assert_array_equal(y2, 2 * y)
    inp3 = dict(inp); inp3["dy"] = (inp["dy"].float() * 2).to(torch.bfloat16)
    _, _, g3 = _run(inp3, k, "f32")
    for key in ("dx", "dWg", "dW1", "dW3", "dW2", "dg"):
        np.testing.assert_array_equal(g3[key], 2 * g[key], err_msg=key)
    perm = torch.randperm(cfg.T, generator=torch.Generator().manual_seed(0))
    inp4 = dict(inp); inp4["x"] = inp["x"][perm]
    y4, _ = cref.layer_fwd(inp4["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], k)
    np.testing.assert_array_equal(y4, y[perm.numpy()])


def test_threads_do_not_change_results(monkeypatch):
    """Every sum runs in one thread in a fixed order: the record is bitwise
    the same for any thread count (checked in a child process with 1 thread)."""
    import subprocess
    import sys
    code = (
        "import numpy as np, oracle.cref as c\n"
        "from tests.helpers import conditioned_inputs, small_config\n"
        "cfg = small_config(T=64, h=32, f=48, E=5, k=2, seed=9)\n"
        "inp = conditioned_inputs(cfg)\n"
        "y, ctx = c.layer_fwd(inp['x'], inp['Wg'], inp['b'], inp['W1'], inp['W3'], inp['W2'], 2)\n"
        "g = c.layer_bwd(inp['dy'], inp['x'], inp['Wg'], inp['W1'], inp['W3'], inp['W2'], ctx)\n"
        "import sys; sys.stdout.buffer.write(y.tobytes() + g['dW1'].tobytes() + g['dx'].tobytes()"
        " + g['dWg'].tobytes())\n")
    root = __import__("os").path.dirname(__import__("os").path.dirname(__file__))
    outs = []
    for n in ("1", "3"):
        env = dict(__import__("os").environ, OMP_NUM_THREADS=n, PYTHONPATH=root)
        outs.append(subprocess.run([sys.executable, "-c", code], capture_output=True, env=env,
                                   cwd=root, check=True).stdout)
    assert len(outs[0]) > 0 and outs[0] == outs[1]


# ------------------------------------------------- sampled / per-token forms ---

def test_token_and_column_forms_match_layer():
    k = 3
    cfg = small_config(T=24, h=16, f=32, E=5, k=k, seed=81)
    inp = conditioned_inputs(cfg)
    for prec in ("f64", "f32"):
        y, ctx, g = _run(inp, k, prec)
        W = lambda e: (inp["W1"][e], inp["W3"][e], inp["W2"][e])  # noqa: E731
        toks = [0, 5, 23]
        r = cref.tokens_fwd_bwd(inp["x"][toks], inp["dy"][toks], inp["Wg"], inp["b"], k, W,
                                prec=prec)
        np.testing.assert_array_equal(r["topk_idx"], ctx["topk_idx"][toks])
        tol = 1e-12 if prec == "f64" else 1e-6
        np.testing.assert_allclose(r["y"], y[toks], rtol=tol, atol=tol)
        np.testing.assert_allclose(r["dx"], g["dx"][toks], rtol=tol, atol=tol)
        np.testing.assert_allclose(r["dg"], g["dg"][toks], rtol=tol, atol=tol)
        for e in range(cfg.E):
            lo, hi = ctx["offsets"][e], ctx["offsets"][e + 1]
            a = ctx["perm_src"][lo:hi]
            dY_e = inp["dy"][torch.from_numpy(a // k)]
            g_e = ctx["gates"].ravel()[a]
            cols = [0, 7, 31]
            w = cref.expert_wgrad_columns(ctx["x_perm"][lo:hi], dY_e, g_e, *W(e), cols,
                                          prec=prec)
            np.testing.assert_allclose(w["dW1"], g["dW1"][e][:, cols], rtol=tol, atol=tol)
            np.testing.assert_allclose(w["dW3"], g["dW3"][e][:, cols], rtol=tol, atol=tol)
            np.testing.assert_allclose(w["dW2"], g["dW2"][e][cols, :], rtol=tol, atol=tol)
            # all of the expert's rows through expert_terms: its whole weight gradient
            t = cref.expert_terms(ctx["x_perm"][lo:hi], dY_e, g_e, *W(e), prec=prec, wgrads=True)
            for n in ("dW1", "dW3", "dW2"):
                np.testing.assert_allclose(t[n], g[n][e], rtol=tol, atol=tol, err_msg=n)
    # the whole batch's sampled tokens with drops: the slots the batch dropped add nothing
    cap = 10
    y, ctx, g = _run(inp, k, "f64", capacity=cap)
    keep = (ctx["perm_dst"] >= 0).reshape(cfg.T, k)
    assert not keep.all()
    seen = {}
    r = cref.tokens_fwd_bwd(inp["x"], inp["dy"], inp["Wg"], inp["b"], k, W, keep=keep,
                            prec="f64", on_expert_wgrads=lambda e, *w: seen.setdefault(e, w))
    for e, w in seen.items():
        for n, v in zip(("dW1", "dW3", "dW2"), w):
            np.testing.assert_allclose(v, g[n][e], rtol=1e-12, atol=1e-12, err_msg=n)
    np.testing.assert_allclose(r["y"], y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["dx"], g["dx"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["dWg"], g["dWg"], rtol=1e-12, atol=1e-12)


# ---------------------------------------------- the two oracles agree ---

@pytest.mark.parametrize("T,h,f,E,k,cap", [(48, 16, 32, 4, 2, None), (96, 32, 48, 8, 3, None),
                                           (64, 24, 40, 6, 2, 12), (50, 16, 16, 16, 1, None)])
def test_record_agrees_with_numpy_float64_oracle(T, h, f, E, k, cap):
    cfg = small_config(T=T, h=h, f=f, E=E, k=k, seed=T + E)
    inp = conditioned_inputs(cfg)
    y, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"],
                              k, capacity=cap)
    g = oracle.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    y2, ctx2, g2 = _run(inp, k, "f32", capacity=cap)
    for n in ("topk_idx", "counts", "offsets", "perm_src", "perm_dst"):
        np.testing.assert_array_equal(ctx2[n], ctx[n], err_msg=n)
    assert rel_l2(y2, y) <= TOL32
    for n in ("x_perm", "A", "B", "H", "O", "gates"):
        assert rel_l2(ctx2[n], ctx[n]) <= TOL32, n
    for n in ("dx", "dWg", "dW1", "dW3", "dW2", "dg", "dO", "dA", "dB", "dX_perm"):
        assert rel_l2(g2[n], g[n]) <= TOL32, n


# ------------------------------------------------------- number formats ---

def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-6, 6, 100000)).astype(np.float32)
    hi = rng.integers(0x30000000, 0x4F000000, 1000).astype(np.uint32) & np.uint32(0xFFFF0000)
    t = (hi | np.uint32(0x8000)).view(np.float32)                 # exact ties
    v = np.concatenate([v, t, -t])
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(cref.bf16_round(v), ref)


def test_e4m3_round_matches_torch_and_fixes_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = codes.float().double().numpy()
    vals = vals[np.isfinite(vals)]
    np.testing.assert_array_equal(cref.e4m3_round(vals), vals)
    rng = np.random.default_rng(1)
    mag = 2.0 ** rng.uniform(-12, np.log2(448.0), 100000)
    v = (np.where(rng.random(mag.size) < 0.5, -1.0, 1.0) * mag).astype(np.float32)
    c = np.unique(np.abs(vals))
    mids = ((c[1:] + c[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, (np.arange(1, 64) * 2.0 ** -11).astype(np.float32)])
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).float().double().numpy()
    np.testing.assert_array_equal(cref.e4m3_round(v), ref)
    np.testing.assert_array_equal(cref.e4m3_round(np.array([449.0, 1e6, -500.0])),
                                  [448, 448, -448])


def test_quantisers_exact_on_power_of_two_scaled_codes():
    rng = np.random.default_rng(3)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    c = codes.float().double().numpy()
    c = c[np.isfinite(c)]
    q = rng.choice(c, size=(12, 40))
    q[:, 0] = 448.0
    j = rng.integers(-20, 20, size=12)
    X = q * np.ldexp(1.0, j)[:, None]
    Xq, s = cref.quantize_rows_e4m3(X)
    np.testing.assert_array_equal(s, np.ldexp(1.0, j).astype(np.float32))
    np.testing.assert_array_equal(Xq, q)
    Wq, sw = cref.quantize_cols_e4m3(np.transpose(X.reshape(3, 4, 40), (0, 2, 1)))
    np.testing.assert_array_equal(sw, np.ldexp(1.0, j).astype(np.float32).reshape(3, 4))
    np.testing.assert_array_equal(Wq, np.transpose(q.reshape(3, 4, 40), (0, 2, 1)))
    X0 = rng.standard_normal((40, 24)) * np.exp(rng.uniform(-3, 3, (40, 1)))
    X1 = rng.standard_normal((40, 16)) * np.exp(rng.uniform(-3, 3, (40, 1)))
    X1[3] *= 100.0
    q0, q1, sj = cref.quantize_rows_joint_e4m3(X0, X1)
    qc, sc = cref.quantize_rows_e4m3(np.concatenate([X0, X1], axis=1))
    np.testing.assert_array_equal(sj, sc)
    np.testing.assert_array_equal(np.concatenate([q0, q1], axis=1), qc)
    Z = np.zeros((2, 8))
    Zq, zs = cref.quantize_rows_e4m3(Z)
    assert np.all(zs == 1.0) and np.all(Zq == 0.0)


def test_quantize_rows_error_bound():
    rng = np.random.default_rng(4)
    X = (rng.standard_normal((64, 300)) * np.exp(rng.uniform(-8, 8, (64, 1)))).astype(np.float32)
    Xq, s = cref.quantize_rows_e4m3(X)
    err = np.abs(Xq * s[:, None].astype(np.float64) - X)
    bound = np.maximum(2.0 ** -4 * np.abs(X), 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)
    assert np.all(np.max(np.abs(Xq), axis=1) == 448.0)
