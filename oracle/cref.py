"""The C++ oracle (moe_oracle.cpp) through ctypes: the oracle of record.

TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and the
benchmark's CPU legs may import this module.  It shares no code with the CUDA
library; the C++ source shares none either.

Every function here only marshals arrays into the C++ library and back: the
arithmetic (routing, dispatch, the expert matmuls, the combine, the backward,
the e4m3 and bf16 roundings) all runs in moe_oracle.cpp.  The functions follow
the float64 numpy oracle (moe_oracle.py) by name and by the layout of what
they return, so a test can run either.

Precision (`prec`):
  "f32"  the record.  bf16 tensors (x, W1, W3, W2, dy) go in as their 16-bit
         patterns (a tensor that is not bf16 is first rounded to bf16 by
         torch); Wg and b as fp32.  fp32 accumulation, fp32 intermediates.
  "f64"  the same C++ templates in double, on double inputs of any value (no
         rounding to bf16): the form finite differences need.
"""
from __future__ import annotations

import ctypes

import numpy as np

__all__ = [
    "lib", "num_threads", "route", "dispatch", "permute_rows", "unpermute_rows",
    "expert_ffn_fwd", "combine", "layer_fwd", "expert_ffn_bwd", "router_bwd", "layer_bwd",
    "expert_terms", "tokens_fwd_bwd", "expert_wgrad_columns", "token_grads",
    "E4M3_MAX", "e4m3_round", "bf16_round", "quantize_rows_e4m3", "quantize_cols_e4m3",
    "quantize_rows_joint_e4m3", "expert_ffn_fwd_fp8", "layer_fwd_fp8", "fc1_dgrad_fp8",
    "expert_ffn_bwd_fp8", "layer_bwd_fp8",
]

E4M3_MAX = 448.0
_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_longlong


def lib():
    """The loaded C++ oracle library (built from source if needed)."""
    global _LIB
    if _LIB is None:
        from oracle import cbuild
        L = ctypes.CDLL(cbuild.build())
        for name, (args, ret) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ret
        _LIB = L
    return _LIB


def _sig(*kinds, ret=None):
    m = {"p": _P, "i": _I, "l": _L}
    return [m[c] for c in kinds], ret


_SIGS = {
    "oracle_num_threads": _sig(ret=_I),
    "oracle_round_bf16": _sig("l", "p", "p"),
    "oracle_round_e4m3": _sig("l", "p", "p"),
    "oracle_dispatch": _sig("l", "i", "i", "p", "l", "i", "i", "p", "p", "p", "p", "p", ret=_L),
    "oracle_route_f32": _sig("l", "i", "i", "i", *"pppppp"),
    "oracle_route_f64": _sig("l", "i", "i", "i", *"pppppp"),
    "oracle_permute_rows_f32": _sig("l", "i", "i", "p", "p", "p"),
    "oracle_permute_rows_f64": _sig("l", "i", "i", "p", "p", "p"),
    "oracle_expert_ffn_fwd_f32": _sig("i", "i", "i", *"p" * 9),
    "oracle_expert_ffn_fwd_f64": _sig("i", "i", "i", *"p" * 9),
    "oracle_combine_f32": _sig("l", "i", "i", "p", "p", "p", "p"),
    "oracle_combine_f64": _sig("l", "i", "i", "p", "p", "p", "p"),
    "oracle_expert_ffn_bwd_f32": _sig("i", "i", "i", *"p" * 15),
    "oracle_expert_ffn_bwd_f64": _sig("i", "i", "i", *"p" * 15),
    "oracle_router_bwd_f32": _sig("l", "i", "p", "p", "p"),
    "oracle_router_bwd_f64": _sig("l", "i", "p", "p", "p"),
    "oracle_layer_fwd_f32": _sig("l", "i", "i", "i", "i", "l", *"p" * 19, ret=_L),
    "oracle_layer_fwd_f64": _sig("l", "i", "i", "i", "i", "l", *"p" * 19, ret=_L),
    "oracle_layer_bwd_f32": _sig("l", "i", "i", "i", "i", *"p" * 27),
    "oracle_layer_bwd_f64": _sig("l", "i", "i", "i", "i", *"p" * 27),
    "oracle_token_grads_f32": _sig("l", "i", "i", "i", *"p" * 10),
    "oracle_token_grads_f64": _sig("l", "i", "i", "i", *"p" * 10),
    "oracle_expert_terms_f32": _sig("l", "i", "i", *"p" * 12),
    "oracle_expert_terms_f64": _sig("l", "i", "i", *"p" * 12),
    "oracle_expert_wgrad_columns_f32": _sig("l", "i", *"p" * 6, "i", "p", "p", "p"),
    "oracle_expert_wgrad_columns_f64": _sig("l", "i", *"p" * 6, "i", "p", "p", "p"),
    "oracle_quantize_rows_e4m3": _sig("l", "l", "p", "p", "p"),
    "oracle_quantize_rows_joint_e4m3": _sig("l", "l", "l", *"p" * 5),
    "oracle_quantize_cols_e4m3": _sig("i", "l", "l", "p", "p", "p"),
    "oracle_expert_ffn_fwd_fp8": _sig("i", "i", "i", *"p" * 19),
    "oracle_fc1_dgrad_fp8": _sig("l", "i", "i", *"p" * 5),
    "oracle_expert_ffn_bwd_fp8": _sig("i", "i", "i", *"p" * 15),
    "oracle_layer_fwd_fp8": _sig("l", "i", "i", "i", "i", "l", *"p" * 29, ret=_L),
    "oracle_layer_bwd_fp8": _sig("l", "i", "i", "i", "i", *"p" * 27),
}


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(lib().oracle_num_threads())


# ------------------------------------------------------------- marshalling ---

def _is_torch(t):
    return hasattr(t, "detach") and hasattr(t, "dtype")


def _bits(t) -> np.ndarray:
    """bf16 patterns (uint16) of a tensor: bf16 as is, other values rounded to
    bf16 by torch."""
    import torch
    if not _is_torch(t):
        t = torch.from_numpy(np.ascontiguousarray(np.asarray(t, dtype=np.float32)))
    t = t.detach().to("cpu")
    if t.dtype != torch.bfloat16:
        t = t.float().to(torch.bfloat16)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f32(t) -> np.ndarray:
    if _is_torch(t):
        t = t.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.float32))


def _f64(t) -> np.ndarray:
    if _is_torch(t):
        t = t.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _i32(a) -> np.ndarray:
    if _is_torch(a):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return None if a is None else a.ctypes.data_as(_P)


def _check(prec):
    if prec not in ("f32", "f64"):
        raise ValueError("prec must be 'f32' or 'f64'")
    return np.float32 if prec == "f32" else np.float64


def _act(t, prec):
    """An activation-like input (bf16 tensor): bits for f32, doubles for f64."""
    return _bits(t) if prec == "f32" else _f64(t)


def _flt(t, prec):
    return _f32(t) if prec == "f32" else _f64(t)


# ------------------------------------------------------------------ router ---

def route(x, Wg, b, k, prec="f32"):
    """Softmax top-k gating.  Returns topk_idx [T,k] int32, gates [T,k] and
    the logits [T,E] (DisagMoE §2.1)."""
    dt = _check(prec)
    xa = _act(x, prec)
    T, h = xa.shape
    Wga = _flt(Wg, prec)
    E = Wga.shape[1]
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ba = None if b is None else _flt(b, prec)
    idx = np.empty((T, k), np.int32)
    gates = np.empty((T, k), dt)
    logits = np.empty((T, E), dt)
    getattr(lib(), f"oracle_route_{prec}")(T, h, E, k, _p(xa), _p(Wga), _p(ba), _p(idx),
                                           _p(gates), _p(logits))
    return idx, gates, logits


# ---------------------------------------------------------------- dispatch ---

def dispatch(topk_idx, E, capacity=None, experts=None, keep=None):
    """Counts, offsets and the stable expert-major permutation (see
    moe_oracle.dispatch).  keep[a] = False drops assignment a up front.
    Returns counts [EL], offsets [EL+1], perm_src [placed rows], perm_dst [T*k]
    (-1 for a dropped assignment)."""
    idx = _i32(topk_idx)
    if idx.ndim == 1:
        idx = idx.reshape(-1, 1)
    T, k = idx.shape
    e_lo, e_hi = (0, E) if experts is None else (int(experts[0]), int(experts[1]))
    EL = e_hi - e_lo
    counts = np.empty(EL, np.int32)
    offsets = np.empty(EL + 1, np.int32)
    perm_src = np.empty(max(T * k, 1), np.int32)
    perm_dst = np.empty(max(T * k, 1), np.int32)
    kp = None if keep is None else np.ascontiguousarray(np.asarray(keep, dtype=np.uint8).ravel())
    R = lib().oracle_dispatch(T, k, E, _p(idx), -1 if capacity is None else int(capacity),
                              e_lo, e_hi, _p(kp), _p(counts), _p(offsets), _p(perm_src),
                              _p(perm_dst))
    if R < 0:
        raise ValueError("expert id out of range")
    return counts, offsets, perm_src[:R].copy(), perm_dst[:T * k].copy()


def permute_rows(x, perm_src, k, prec="f32"):
    """x_perm[p] = x[perm_src[p] // k] (the values of the bf16 rows)."""
    dt = _check(prec)
    xa = _act(x, prec)
    h = xa.shape[1]
    ps = _i32(perm_src)
    out = np.empty((ps.size, h), dt)
    getattr(lib(), f"oracle_permute_rows_{prec}")(ps.size, h, k, _p(xa), _p(ps), _p(out))
    return out


def unpermute_rows(rows_perm, perm_dst):
    """rows_assign[a] = rows_perm[perm_dst[a]], a zero row where perm_dst[a] = -1
    (a gather: no arithmetic)."""
    rows_perm = np.asarray(rows_perm)
    dst = np.asarray(perm_dst, dtype=np.int64)
    out = np.zeros((dst.size,) + rows_perm.shape[1:], dtype=rows_perm.dtype)
    kept = dst >= 0
    out[kept] = rows_perm[dst[kept]]
    return out


# ----------------------------------------------------------------- experts ---

def _weights(W1, W3, W2, prec):
    if prec == "f32":
        return _bits(W1), _bits(W3), _bits(W2)
    return _f64(W1), _f64(W3), _f64(W2)


def expert_ffn_fwd(x_perm, offsets, W1, W3, W2, prec="f32"):
    """A = X W1, B = X W3, H = silu(A) * B, O = H W2 per expert (review §三
    核心公式).  Returns A, B, H, O."""
    dt = _check(prec)
    w1, w3, w2 = _weights(W1, W3, W2, prec)
    E, h, f = w1.shape
    X = _flt(x_perm, prec)
    off = _i32(offsets)
    R = int(off[E])
    A = np.zeros((R, f), dt); B = np.zeros((R, f), dt); H = np.zeros((R, f), dt)
    O = np.zeros((R, h), dt)
    getattr(lib(), f"oracle_expert_ffn_fwd_{prec}")(h, f, E, _p(X), _p(off), _p(w1), _p(w3),
                                                    _p(w2), _p(A), _p(B), _p(H), _p(O))
    return A, B, H, O


def combine(O, gates, perm_dst, T, k, prec="f32"):
    """y[t] = sum_j g[t,j] O[perm_dst[t*k+j]] in slot order; dropped slots add
    nothing (DisagMoE §2.1)."""
    dt = _check(prec)
    Oa = _flt(O, prec)
    h = Oa.shape[1]
    g = _flt(np.asarray(gates).reshape(T, k) if not _is_torch(gates) else gates, prec)
    pd = _i32(perm_dst)
    y = np.empty((T, h), dt)
    getattr(lib(), f"oracle_combine_{prec}")(T, k, h, _p(Oa), _p(g), _p(pd), _p(y))
    return y


def layer_fwd(x, Wg, b, W1, W3, W2, k, capacity=None, prec="f32"):
    """route -> dispatch -> permute -> expert FFN -> combine.  Returns y and a
    context dict with every intermediate (the placed rows only)."""
    dt = _check(prec)
    xa = _act(x, prec)
    T, h = xa.shape
    Wga = _flt(Wg, prec)
    E = Wga.shape[1]
    ba = None if b is None else _flt(b, prec)
    w1, w3, w2 = _weights(W1, W3, W2, prec)
    f = w1.shape[2]
    R = T * k
    y = np.empty((T, h), dt)
    idx = np.empty((T, k), np.int32)
    gates = np.empty((T, k), dt)
    logits = np.empty((T, E), dt)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm_src = np.empty(max(R, 1), np.int32)
    perm_dst = np.empty(max(R, 1), np.int32)
    x_perm = np.empty((R, h), dt)
    A = np.empty((R, f), dt); B = np.empty((R, f), dt); H = np.empty((R, f), dt)
    O = np.empty((R, h), dt)
    n = getattr(lib(), f"oracle_layer_fwd_{prec}")(
        T, h, f, E, k, -1 if capacity is None else int(capacity), _p(xa), _p(Wga), _p(ba),
        _p(w1), _p(w3), _p(w2), _p(y), _p(idx), _p(gates), _p(logits), _p(counts), _p(offsets),
        _p(perm_src), _p(perm_dst), _p(x_perm), _p(A), _p(B), _p(H), _p(O))
    ctx = dict(topk_idx=idx, gates=gates, logits=logits, counts=counts, offsets=offsets,
               perm_src=perm_src[:n].copy(), perm_dst=perm_dst[:R].copy(), x_perm=x_perm[:n],
               A=A[:n], B=B[:n], H=H[:n], O=O[:n], k=k, prec=prec)
    return y, ctx


# ---------------------------------------------------------------- backward ---

def expert_ffn_bwd(dO, x_perm, offsets, W1, W3, W2, A, B, H, prec="f32"):
    """Backward of the per-expert SwiGLU FFN given dO.  Returns dA, dB,
    dX_perm, dW1, dW3, dW2."""
    dt = _check(prec)
    w1, w3, w2 = _weights(W1, W3, W2, prec)
    E, h, f = w1.shape
    off = _i32(offsets)
    R = int(off[E])
    dOa, X = _flt(dO, prec), _flt(x_perm, prec)
    Aa, Ba, Ha = _flt(A, prec), _flt(B, prec), _flt(H, prec)
    dA = np.zeros((R, f), dt); dB = np.zeros((R, f), dt); dX = np.zeros((R, h), dt)
    dW1 = np.empty((E, h, f), dt); dW3 = np.empty((E, h, f), dt); dW2 = np.empty((E, f, h), dt)
    getattr(lib(), f"oracle_expert_ffn_bwd_{prec}")(
        h, f, E, _p(dOa), _p(X), _p(off), _p(w1), _p(w3), _p(w2), _p(Aa), _p(Ba), _p(Ha),
        _p(dA), _p(dB), _p(dX), _p(dW1), _p(dW3), _p(dW2))
    return dict(dA=dA, dB=dB, dX_perm=dX, dW1=dW1, dW3=dW3, dW2=dW2)


def router_bwd(gates, dg, prec="f32"):
    """dl_j = g_j sum_i g_i (dg_j - dg_i) for the selected logits."""
    dt = _check(prec)
    g = _flt(gates, prec)
    d = _flt(dg, prec)
    T, k = g.shape
    out = np.empty((T, k), dt)
    getattr(lib(), f"oracle_router_bwd_{prec}")(T, k, _p(g), _p(d), _p(out))
    return out


def layer_bwd(dy, x, Wg, W1, W3, W2, ctx, prec=None):
    """Gradients of L = <dy, y> with respect to x, Wg, W1, W3, W2, plus dg."""
    prec = prec or ctx.get("prec", "f32")
    dt = _check(prec)
    k = ctx["k"]
    xa, dya = _act(x, prec), _act(dy, prec)
    T, h = xa.shape
    Wga = _flt(Wg, prec)
    E = Wga.shape[1]
    w1, w3, w2 = _weights(W1, W3, W2, prec)
    f = w1.shape[2]
    R = int(ctx["offsets"][-1])
    c = {n: _flt(ctx[n], prec) for n in ("gates", "x_perm", "A", "B", "H", "O")}
    ii = {n: _i32(ctx[n]) for n in ("topk_idx", "offsets", "perm_src", "perm_dst")}
    dx = np.empty((T, h), dt); dWg = np.empty((h, E), dt)
    dW1 = np.empty((E, h, f), dt); dW3 = np.empty((E, h, f), dt); dW2 = np.empty((E, f, h), dt)
    dg = np.empty((T, k), dt); dl = np.empty((T, E), dt)
    dO = np.zeros((R, h), dt); dA = np.zeros((R, f), dt); dB = np.zeros((R, f), dt)
    dX = np.zeros((R, h), dt)
    getattr(lib(), f"oracle_layer_bwd_{prec}")(
        T, h, f, E, k, _p(xa), _p(dya), _p(Wga), _p(w1), _p(w3), _p(w2), _p(ii["topk_idx"]),
        _p(c["gates"]), _p(ii["offsets"]), _p(ii["perm_src"]), _p(ii["perm_dst"]),
        _p(c["x_perm"]), _p(c["A"]), _p(c["B"]), _p(c["H"]), _p(c["O"]), _p(dx), _p(dWg),
        _p(dW1), _p(dW3), _p(dW2), _p(dg), _p(dl), _p(dO), _p(dA), _p(dB), _p(dX))
    return dict(dx=dx, dWg=dWg, dg=dg, dl=dl, dO=dO, dA=dA, dB=dB, dX_perm=dX, dW1=dW1,
                dW3=dW3, dW2=dW2)


def token_grads(x, Wg, topk_idx, gates, perm_dst, dg, dX_perm, prec="f32"):
    """The token side of the backward: dl (router_bwd, scattered to [T,E]),
    dx = sum of the kept slots' dX_perm rows + sum_j dl_j Wg[:, e_j], and
    dWg = x^T dl.  Returns dict(dx, dWg, dl)."""
    dt = _check(prec)
    xa = _act(x, prec)
    T, h = xa.shape
    Wga = _flt(Wg, prec)
    E = Wga.shape[1]
    idx = _i32(topk_idx).reshape(T, -1)
    k = idx.shape[1]
    g = _flt(np.asarray(gates).reshape(T, k) if not _is_torch(gates) else gates, prec)
    pd, d = _i32(perm_dst), _flt(np.asarray(dg).reshape(T, k), prec)
    dX = _flt(dX_perm, prec)
    dx = np.empty((T, h), dt); dWg = np.empty((h, E), dt); dl = np.empty((T, E), dt)
    getattr(lib(), f"oracle_token_grads_{prec}")(T, h, E, k, _p(xa), _p(Wga), _p(idx), _p(g),
                                                 _p(pd), _p(d), _p(dX), _p(dx), _p(dWg),
                                                 _p(dl))
    return dict(dx=dx, dWg=dWg, dl=dl)


# ------------------------------------------------------- sampled forms ---

def expert_terms(X, dY, g, W1e, W3e, W2e, prec="f32", wgrads=False):
    """Rows X [n,h] through one expert with gates g [n] and loss rows dY:
    o = FFN_e(X), dg = <dY, o>, dx = the expert's part of the row gradient
    (rows backward of dO = g dY).  X and dY are values (bf16 rows as float).
    wgrads=True adds dW1, dW3 [h,f] and dW2 [f,h] from these rows alone."""
    dt = _check(prec)
    w1, w3, w2 = _weights(W1e, W3e, W2e, prec)
    h, f = w1.shape
    Xa = _flt(np.asarray(X).reshape(-1, h) if not _is_torch(X) else X.reshape(-1, h), prec)
    n = Xa.shape[0]
    dYa = _flt(np.asarray(dY).reshape(n, h) if not _is_torch(dY) else dY.reshape(n, h), prec)
    ga = _flt(np.asarray(g).reshape(n), prec)
    o = np.empty((n, h), dt); dg = np.empty(n, dt); dx = np.empty((n, h), dt)
    w = (np.empty((h, f), dt), np.empty((h, f), dt), np.empty((f, h), dt)) if wgrads else \
        (None, None, None)
    getattr(lib(), f"oracle_expert_terms_{prec}")(n, h, f, _p(Xa), _p(dYa), _p(ga), _p(w1),
                                                  _p(w3), _p(w2), _p(o), _p(dg), _p(dx),
                                                  _p(w[0]), _p(w[1]), _p(w[2]))
    out = dict(o=o, dg=dg, dx=dx)
    if wgrads:
        out.update(dW1=w[0], dW3=w[1], dW2=w[2])
    return out


def tokens_fwd_bwd(x_rows, dy_rows, Wg, b, k, expert_weights, keep=None, prec="f32",
                   on_expert_wgrads=None):
    """The layer for a sample of tokens, one expert at a time.

    x_rows, dy_rows: [n, h] bf16 rows of the sampled tokens.  expert_weights(e)
    returns (W1[e], W3[e], W2[e]).  keep [n, k] (optional) marks the slots the
    whole batch kept (capacity drops depend on the other tokens).  Each
    token's y and dx depend on that token alone, so they equal the whole
    layer's rows.  Returns dict(topk_idx, gates, y, dx, dg, dWg): dWg is the
    sample's share sum_{t in sample} x[t]^T dl[t].  on_expert_wgrads(e, dW1,
    dW3, dW2), when given, receives each expert's weight gradients from the
    sample's (kept) rows alone, one expert at a time.
    """
    dt = _check(prec)
    idx, gates, _ = route(x_rows, Wg, b, k, prec)
    n = idx.shape[0]
    xv = _flt(x_rows, prec)
    dyv = _flt(dy_rows, prec)
    h = xv.shape[1]
    kp = np.ones((n, k), bool) if keep is None else np.asarray(keep, bool).reshape(n, k)
    O = np.zeros((n * k, h), dt)
    dg = np.zeros(n * k, dt)
    dX = np.zeros((n * k, h), dt)
    flat = idx.ravel()
    for e in sorted(set(flat[kp.ravel()].tolist())):
        rows = np.nonzero((flat == e) & kp.ravel())[0]
        W1e, W3e, W2e = expert_weights(int(e))
        t = expert_terms(xv[rows // k], dyv[rows // k], gates.ravel()[rows], W1e, W3e, W2e, prec,
                         wgrads=on_expert_wgrads is not None)
        O[rows], dg[rows], dX[rows] = t["o"], t["dg"], t["dx"]
        if on_expert_wgrads is not None:
            on_expert_wgrads(int(e), t["dW1"], t["dW3"], t["dW2"])
            del t
    perm_dst = np.where(kp.ravel(), np.arange(n * k), -1).astype(np.int32)
    y = combine(O, gates, perm_dst, n, k, prec)
    tg = token_grads(x_rows, Wg, idx, gates, perm_dst, dg, dX, prec)
    return dict(topk_idx=idx, gates=gates, y=y, dx=tg["dx"], dg=dg.reshape(n, k),
                dWg=tg["dWg"], dl=tg["dl"])


def expert_wgrad_columns(X_e, dY_e, g_e, W1e, W3e, W2e, cols, prec="f32"):
    """Columns `cols` of dW1[e], dW3[e] and rows `cols` of dW2[e] from all of an
    expert's rows X_e [n,h], their loss rows dY_e [n,h] and gates g_e [n]
    (values).  Returns dW1 [h, nc], dW3 [h, nc], dW2 [nc, h]."""
    dt = _check(prec)
    cc = np.asarray(cols, dtype=np.int64).ravel()
    if _is_torch(W1e):
        ci = __import__("torch").from_numpy(cc)
        W1c, W3c, W2r = W1e[:, ci].t(), W3e[:, ci].t(), W2e[ci, :]
    else:
        W1c, W3c, W2r = np.asarray(W1e)[:, cc].T, np.asarray(W3e)[:, cc].T, np.asarray(W2e)[cc, :]
    w1, w3, w2 = _weights(W1c, W3c, W2r, prec)
    nc, h = w1.shape
    X = _flt(X_e, prec).reshape(-1, h)
    n = X.shape[0]
    dY = _flt(dY_e, prec).reshape(n, h)
    g = _flt(np.asarray(g_e).reshape(n) if not _is_torch(g_e) else g_e.reshape(n), prec)
    d1 = np.empty((nc, h), dt); d3 = np.empty((nc, h), dt); d2 = np.empty((nc, h), dt)
    getattr(lib(), f"oracle_expert_wgrad_columns_{prec}")(n, h, _p(X), _p(dY), _p(g), _p(w1),
                                                          _p(w3), _p(w2), nc, _p(d1), _p(d3),
                                                          _p(d2))
    return dict(dW1=d1.T.copy(), dW3=d3.T.copy(), dW2=d2)


# --------------------------------------------------------- number formats ---

def bf16_round(v) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); float32 out."""
    a = _f32(v)
    out = np.empty_like(a)
    lib().oracle_round_bf16(a.size, _p(a), _p(out))
    return out


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3 value (ties to even, saturating at 448), in float64."""
    a = _f64(v)
    out = np.empty_like(a)
    lib().oracle_round_e4m3(a.size, _p(a), _p(out))
    return out


# --------------------------------------------------------------------- FP8 ---

def quantize_rows_e4m3(X):
    """Per-row fp32 scales s = amax/448 (1 for a zero row) and e4m3 values of
    X / s (fp32 division)."""
    Xa = _f32(X)
    n, m = Xa.shape
    q = np.empty_like(Xa); s = np.empty(n, np.float32)
    lib().oracle_quantize_rows_e4m3(n, m, _p(Xa), _p(q), _p(s))
    return q, s


def quantize_rows_joint_e4m3(X0, X1):
    """Rows i of X0 and X1 quantised with one shared scale."""
    a0, a1 = _f32(X0), _f32(X1)
    n, m0 = a0.shape
    if a1.shape[0] != n:
        raise ValueError("X0 and X1 need the same number of rows")
    q0, q1 = np.empty_like(a0), np.empty_like(a1)
    s = np.empty(n, np.float32)
    lib().oracle_quantize_rows_joint_e4m3(n, m0, a1.shape[1], _p(a0), _p(a1), _p(q0), _p(q1),
                                          _p(s))
    return q0, q1, s


def quantize_cols_e4m3(W):
    """Per-(expert, output column) scales of W [E, K, N] (amax over K) and the
    e4m3 values: returns q [E, K, N], s [E, N]."""
    Wa = _f32(W)
    E, K, N = Wa.shape
    q = np.empty_like(Wa); s = np.empty((E, N), np.float32)
    lib().oracle_quantize_cols_e4m3(E, K, N, _p(Wa), _p(q), _p(s))
    return q, s


def expert_ffn_fwd_fp8(x_perm, offsets, W1, W3, W2):
    """The expert forward on e4m3 codes (row scales for x_perm and H, column
    scales for the weights); H is the stored bf16 copy its codes come from."""
    X = _f32(x_perm)
    w1, w3, w2 = _f32(W1), _f32(W3), _f32(W2)
    E, h, f = w1.shape
    off = _i32(offsets)
    R = int(off[E])
    z = lambda *s: np.zeros(s, np.float32)  # noqa: E731
    out = dict(A=z(R, f), B=z(R, f), H=z(R, f), O=z(R, h), Xq=z(R, h), sx=z(R), Hq=z(R, f),
               sh=z(R), W1q=z(E, h, f), s1=z(E, f), W3q=z(E, h, f), s3=z(E, f),
               W2q=z(E, f, h), s2=z(E, h))
    lib().oracle_expert_ffn_fwd_fp8(h, f, E, _p(X), _p(off), _p(w1), _p(w3), _p(w2),
                                    *[_p(out[n]) for n in ("A", "B", "H", "O", "Xq", "sx", "Hq",
                                                           "sh", "W1q", "s1", "W3q", "s3", "W2q",
                                                           "s2")])
    return out


def layer_fwd_fp8(x, Wg, b, W1, W3, W2, k, capacity=None):
    """layer_fwd with the expert matmuls on e4m3 codes.  The context feeds
    layer_bwd / layer_bwd_fp8."""
    xa = _bits(x)
    T, h = xa.shape
    Wga = _f32(Wg)
    E = Wga.shape[1]
    ba = None if b is None else _f32(b)
    w1, w3, w2 = _bits(W1), _bits(W3), _bits(W2)
    f = w1.shape[2]
    R = T * k
    z = lambda *s: np.zeros(s, np.float32)  # noqa: E731
    y = z(T, h)
    idx = np.empty((T, k), np.int32)
    gates, logits = z(T, k), z(T, E)
    counts, offsets = np.empty(E, np.int32), np.empty(E + 1, np.int32)
    perm_src, perm_dst = np.empty(max(R, 1), np.int32), np.empty(max(R, 1), np.int32)
    f8 = dict(x_perm=z(R, h), A=z(R, f), B=z(R, f), H=z(R, f), O=z(R, h), Xq=z(R, h), sx=z(R),
              Hq=z(R, f), sh=z(R), W1q=z(E, h, f), s1=z(E, f), W3q=z(E, h, f), s3=z(E, f),
              W2q=z(E, f, h), s2=z(E, h))
    n = lib().oracle_layer_fwd_fp8(
        T, h, f, E, k, -1 if capacity is None else int(capacity), _p(xa), _p(Wga), _p(ba),
        _p(w1), _p(w3), _p(w2), _p(y), _p(idx), _p(gates), _p(logits), _p(counts), _p(offsets),
        _p(perm_src), _p(perm_dst),
        *[_p(f8[m]) for m in ("x_perm", "A", "B", "H", "O", "Xq", "sx", "Hq", "sh", "W1q", "s1",
                              "W3q", "s3", "W2q", "s2")])
    for m in ("x_perm", "A", "B", "H", "O", "Xq", "sx", "Hq", "sh"):
        f8[m] = f8[m][:n]
    ctx = dict(topk_idx=idx, gates=gates, logits=logits, counts=counts, offsets=offsets,
               perm_src=perm_src[:n].copy(), perm_dst=perm_dst[:R].copy(), x_perm=f8["x_perm"],
               k=k, fp8=f8, A=f8["A"], B=f8["B"], H=f8["H"], O=f8["O"], prec="f32")
    return y, ctx


def fc1_dgrad_fp8(dA, dB, W1e, W3e):
    """dX = dA W1e^T + dB W3e^T on e4m3 codes (joint row scales)."""
    a, bb = _f32(dA), _f32(dB)
    w1, w3 = _f32(W1e), _f32(W3e)
    n, f = a.shape
    h = w1.shape[0]
    dX = np.empty((n, h), np.float32)
    lib().oracle_fc1_dgrad_fp8(n, h, f, _p(a), _p(bb), _p(w1), _p(w3), _p(dX))
    return dX


def expert_ffn_bwd_fp8(dO, x_perm, offsets, W1, W3, W2, A, B, H):
    """expert_ffn_bwd with the FC1 dgrad on e4m3 codes; A, B, H, dA and dB are
    taken as their bf16 copies (see moe_oracle.cpp)."""
    w1, w3, w2 = _f32(W1), _f32(W3), _f32(W2)
    E, h, f = w1.shape
    off = _i32(offsets)
    R = int(off[E])
    dOa, X = _f32(dO), _f32(x_perm)
    Aa, Ba, Ha = _f32(A), _f32(B), _f32(H)
    z = lambda *s: np.zeros(s, np.float32)  # noqa: E731
    out = dict(dA=z(R, f), dB=z(R, f), dX_perm=z(R, h), dW1=z(E, h, f), dW3=z(E, h, f),
               dW2=z(E, f, h))
    lib().oracle_expert_ffn_bwd_fp8(h, f, E, _p(dOa), _p(X), _p(off), _p(w1), _p(w3), _p(w2),
                                    _p(Aa), _p(Ba), _p(Ha),
                                    *[_p(out[m]) for m in ("dA", "dB", "dX_perm", "dW1", "dW3",
                                                           "dW2")])
    return out


def layer_bwd_fp8(dy, x, Wg, W1, W3, W2, ctx):
    """layer_bwd with the FP8 FC1 dgrad; dO = bf16(g dy) (product in fp32)."""
    k = ctx["k"]
    xa, dya = _bits(x), _bits(dy)
    T, h = xa.shape
    Wga = _f32(Wg)
    E = Wga.shape[1]
    w1, w3, w2 = _bits(W1), _bits(W3), _bits(W2)
    f = w1.shape[2]
    R = int(ctx["offsets"][-1])
    c = {n: _f32(ctx[n]) for n in ("gates", "x_perm", "A", "B", "H", "O")}
    ii = {n: _i32(ctx[n]) for n in ("topk_idx", "offsets", "perm_src", "perm_dst")}
    z = lambda *s: np.zeros(s, np.float32)  # noqa: E731
    out = dict(dx=z(T, h), dWg=z(h, E), dW1=z(E, h, f), dW3=z(E, h, f), dW2=z(E, f, h),
               dg=z(T, k), dl=z(T, E), dO=z(R, h), dA=z(R, f), dB=z(R, f), dX_perm=z(R, h))
    lib().oracle_layer_bwd_fp8(
        T, h, f, E, k, _p(xa), _p(dya), _p(Wga), _p(w1), _p(w3), _p(w2), _p(ii["topk_idx"]),
        _p(c["gates"]), _p(ii["offsets"]), _p(ii["perm_src"]), _p(ii["perm_dst"]),
        _p(c["x_perm"]), _p(c["A"]), _p(c["B"]), _p(c["H"]), _p(c["O"]),
        *[_p(out[m]) for m in ("dx", "dWg", "dW1", "dW3", "dW2", "dg", "dl", "dO", "dA", "dB",
                               "dX_perm")])
    return out

