"""CPU oracle for one top-k MoE FFN layer with SwiGLU experts (dropless by
default; optional per-expert capacity and local expert range in dispatch).

TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import or run this module.  The CUDA library
never calls it, and it shares no code, table or helper with the CUDA sources.

What it computes, with the passages it follows:

* Router and gating.  A trainable gate network scores every expert for each
  token and the k experts with the highest probability are chosen; their
  outputs are summed, weighted (DisagMoE, §2.1 "混合专家（MoE）结构"; the
  MegaScale-MoE review lists the gate network as a component, §三 模型组件).
  Probabilities are a softmax over all E router logits l = x Wg + b; the k
  selected probabilities are renormalised to sum to one.  Ties go to the lower
  expert id; the k slots are in descending logit order.
* Dispatch.  Token copies are sorted by expert, then by source (MegaScale-MoE
  digest §3.3 under Diagram C; the review's "extra scatter to keep memory
  contiguous", §四 自适应EP通信策略详解).  On one GPU the source order is the
  token order, so the permutation is a stable sort of assignments a = t*k + j
  by expert id: counts, their exclusive scan (offsets) and the maps
  perm_src[p] = a, perm_dst[a] = p.
* Experts.  Each expert is a SwiGLU FFN (review §三 核心公式: "SwiGLU structure
  with MoE", compute 3k*bsh*h_ffn multiply-adds at n = 1), run for all
  experts as one GroupedGEMM (digest glossary "GroupedGEMM"; review 训练流程,
  专家计算（GroupedGEMM）):  A = X W1,  B = X W3,  H = silu(A) * B,  O = H W2.
* Combine.  y[t] = sum_j g[t,j] * O[perm_dst[t*k+j]] (DisagMoE §2.1 weighted sum;
  review 训练流程 Token聚合).
* Backward.  The layer's backward written out as explicit operators (digest §3.3:
  forward and backward of the MoE layer are explicit operators, not autograd);
  FC2's gradients take fc2_in (= H) and the gradient of fc2_out (review
  选择性激活重计算).  Router gradient flows through the renormalised gates.

Precision.  Inputs are the exact values of the bf16 / fp32 bytes the layer
receives.  Every product and sum is float64, with no intermediate rounding.
The one integer decision that floating point takes, the choice of the top-k
experts, is taken on float32 logits (x Wg accumulated in float32, + b in
float32), the precision the CUDA router decides in; inputs are conditioned
(condition_router_margins) so that no float32 rounding order can flip it.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "as_f64", "router_logits", "route", "dispatch", "permute_rows",
    "unpermute_rows", "silu", "expert_ffn_fwd", "combine", "layer_fwd",
    "expert_ffn_bwd", "router_bwd", "layer_bwd", "token_fwd_bwd", "expert_terms",
    "assemble_token",
    "expert_wgrad_columns", "condition_router_margins", "router_margin",
    "gemm_macs_fwd", "dispatch_bytes_per_token", "activation_bytes",
    "E4M3_MAX", "e4m3_round", "bf16_round", "quantize_rows_e4m3", "quantize_cols_e4m3",
    "expert_ffn_fwd_fp8", "layer_fwd_fp8", "quantize_rows_joint_e4m3",
    "fc1_dgrad_fp8", "expert_ffn_bwd_fp8", "layer_bwd_fp8",
]


# ----------------------------------------------------------------- inputs ---

def as_f64(t) -> np.ndarray:
    """Exact float64 value of a bf16 / fp32 tensor (torch or numpy)."""
    if hasattr(t, "detach"):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def _as_f32(t) -> np.ndarray:
    if hasattr(t, "detach"):
        return t.detach().to("cpu").float().numpy()
    return np.asarray(t, dtype=np.float32)


# ----------------------------------------------------------------- router ---

def router_logits(x, Wg, b=None):
    """l[t,e] = sum_i x[t,i] Wg[i,e] + b[e]: float64 values and float32 values.

    The float32 copy (float32 products and sums, then + b in float32) is the
    one the top-k decision is taken on.  DisagMoE §2.1 (gate network scores).
    """
    x64, W64 = as_f64(x), as_f64(Wg)
    l64 = x64 @ W64
    l32 = _as_f32(x) @ _as_f32(Wg)
    if b is not None:
        l64 = l64 + as_f64(b)[None, :]
        l32 = (l32 + _as_f32(b)[None, :]).astype(np.float32)
    return l64, l32


def route(x, Wg, b, k):
    """Softmax top-k gating.

    Returns topk_idx [T,k] int32 (descending logit, ties -> lower id),
    gates [T,k] float64 = p[sel] / sum(p[sel]) with p = softmax over all E,
    and the float64 logits.  DisagMoE §2.1: the gate picks the k experts with
    the highest probability scores.
    """
    l64, l32 = router_logits(x, Wg, b)
    T, E = l64.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    # stable sort of -l: equal logits keep ascending expert id
    order = np.argsort(-l32, axis=1, kind="stable")
    topk_idx = order[:, :k].astype(np.int32)
    m = l64.max(axis=1, keepdims=True)
    ex = np.exp(l64 - m)
    p = ex / ex.sum(axis=1, keepdims=True)
    psel = np.take_along_axis(p, topk_idx.astype(np.int64), axis=1)
    gates = psel / psel.sum(axis=1, keepdims=True)
    return topk_idx, gates, l64


def router_margin(l64, k):
    """Smallest gap between consecutive values among each row's k+1 largest
    logits (k largest when k = E)."""
    s = -np.sort(-l64, axis=1)
    top = s[:, : min(k + 1, s.shape[1])]
    if top.shape[1] < 2:
        return np.full(l64.shape[0], np.inf)
    return (top[:, :-1] - top[:, 1:]).min(axis=1)


def condition_router_margins(x, Wg, b, k, fresh_rows, margin=1e-3, max_attempts=64):
    """Replace rows of x whose router decision is numerically ambiguous.

    A row is ambiguous when two of its k+1 largest float64 logits are closer
    than `margin`.  fresh_rows(row_ids, attempt) must return replacement bf16
    rows (torch, CPU).  Returns (new x as torch bf16, number of rows replaced).
    Input conditioning only: no value computed here is an expected output.
    """
    import torch
    xc = x.detach().to("cpu").clone()
    W64 = as_f64(Wg)
    b64 = np.zeros(W64.shape[1]) if b is None else as_f64(b)
    l64 = as_f64(xc) @ W64 + b64[None, :]
    bad = np.nonzero(router_margin(l64, k) < margin)[0]
    replaced = set()
    attempt = 0
    while bad.size:
        attempt += 1
        if attempt > max_attempts:
            raise RuntimeError("router margin conditioning did not converge")
        new = fresh_rows(bad, attempt)
        xc[torch.as_tensor(bad, dtype=torch.int64)] = new.to(xc.dtype)
        replaced.update(bad.tolist())
        lb = as_f64(xc[torch.as_tensor(bad, dtype=torch.int64)]) @ W64 + b64[None, :]
        bad = bad[router_margin(lb, k) < margin]
    return xc, len(replaced)


# --------------------------------------------------------------- dispatch ---

def dispatch(topk_idx, E, capacity=None, experts=None):
    """Counts, offsets and the stable expert-major permutation.

    Dropless (the defaults): counts[e] = #{a : topk_idx[a] = e};  offsets =
    exclusive scan, offsets[E] = T*k;  perm_src[p] = the assignment a placed at
    permuted row p, ordered by expert then by a (so by token);  perm_dst =
    inverse of perm_src.  MegaScale-MoE digest §3.3 (tokens sorted by expert,
    then by source).

    experts = (e_lo, e_hi): only assignments to experts e_lo <= e < e_hi are
    placed, the others are dropped -- the local "scatter & drop" that follows
    the all-gather of every token (digest §3.2, Diagram B; review §四
    自适应EP通信策略详解, step 2).  counts and offsets then cover the e_hi - e_lo
    local experts.

    capacity = C: each expert takes at most C assignments, the first C in
    assignment order a = t*k + j (earlier tokens first, then slot order); the
    rest are dropped -- the token dropping used for load balance (digest §3.2,
    the paragraph after Figure 7; the pages give no drop order, this one is the
    plainest deterministic choice).  Gates are not renormalised after a drop.

    Returns counts [EL], offsets [EL+1], perm_src [offsets[EL]] (placed rows
    only) and perm_dst [T*k] with -1 for every dropped assignment.
    """
    flat = np.asarray(topk_idx, dtype=np.int64).ravel()
    e_lo, e_hi = (0, E) if experts is None else (int(experts[0]), int(experts[1]))
    EL = e_hi - e_lo
    cap = flat.size if capacity is None else int(capacity)
    # stable sort by expert: within an expert, ascending a
    order = np.argsort(flat, kind="stable")
    full = np.bincount(flat, minlength=E)
    start = np.zeros(E + 1, dtype=np.int64)
    start[1:] = np.cumsum(full)
    counts = np.minimum(full[e_lo:e_hi], cap).astype(np.int32)
    offsets = np.zeros(EL + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm_src = np.concatenate(
        [order[start[e]:start[e] + counts[e - e_lo]] for e in range(e_lo, e_hi)]
        + [np.zeros(0, dtype=np.int64)]).astype(np.int32)
    perm_dst = np.full(flat.size, -1, dtype=np.int32)
    perm_dst[perm_src] = np.arange(perm_src.size, dtype=np.int32)
    return counts, offsets, perm_src, perm_dst


def permute_rows(x, perm_src, k):
    """x_perm[p] = x[perm_src[p] // k]: one copy of a token per assignment."""
    return np.asarray(x)[np.asarray(perm_src, dtype=np.int64) // k]


def unpermute_rows(rows_perm, perm_dst):
    """rows_assign[a] = rows_perm[perm_dst[a]] (assignment order a = t*k+j);
    a zero row where perm_dst[a] = -1 (a dropped assignment)."""
    rows_perm = np.asarray(rows_perm)
    dst = np.asarray(perm_dst, dtype=np.int64)
    out = np.zeros((dst.size,) + rows_perm.shape[1:], dtype=rows_perm.dtype)
    kept = dst >= 0
    out[kept] = rows_perm[dst[kept]]
    return out


# ---------------------------------------------------------------- experts ---

def silu(z):
    """silu(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def _sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


class MacCounter:
    """Counts multiply-adds of the expert matmuls as they are performed."""

    def __init__(self):
        self.macs = 0

    def matmul(self, a, b):
        self.macs += a.shape[0] * a.shape[1] * b.shape[1]
        return a @ b


def expert_ffn_fwd(x_perm, offsets, W1, W3, W2, counter=None):
    """Per-expert SwiGLU FFN over the expert-contiguous rows (GroupedGEMM).

    For each e, rows p in [offsets[e], offsets[e+1]):  A = X_e W1[e],
    B = X_e W3[e], H = silu(A) * B, O = H W2[e].  Returns A, B, H, O (float64).
    Review §三 核心公式 (SwiGLU MoE compute) and 训练流程 (GroupedGEMM).
    """
    c = counter if counter is not None else MacCounter()
    X = as_f64(x_perm)
    W1, W3, W2 = as_f64(W1), as_f64(W3), as_f64(W2)
    R = X.shape[0]
    f, h = W1.shape[2], W1.shape[1]
    A = np.zeros((R, f)); B = np.zeros((R, f)); O = np.zeros((R, h))
    for e in range(W1.shape[0]):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        Xe = X[lo:hi]
        A[lo:hi] = c.matmul(Xe, W1[e])
        B[lo:hi] = c.matmul(Xe, W3[e])
        O[lo:hi] = c.matmul(silu(A[lo:hi]) * B[lo:hi], W2[e])
    H = silu(A) * B
    return A, B, H, O


def combine(O, gates, perm_dst, T, k):
    """y[t] = sum_{j<k} g[t,j] * O[perm_dst[t*k+j]], summed in slot order; a
    dropped slot (perm_dst = -1) adds nothing.
    DisagMoE §2.1 (outputs reduced by a weighted sum)."""
    O = np.asarray(O)
    idx = np.asarray(perm_dst, dtype=np.int64).reshape(T, k)
    g = np.asarray(gates, dtype=np.float64).reshape(T, k)
    y = np.zeros((T, O.shape[1]))
    for j in range(k):
        kept = idx[:, j] >= 0
        y[kept] += g[kept, j:j + 1] * O[idx[kept, j]]
    return y


def layer_fwd(x, Wg, b, W1, W3, W2, k, counter=None, capacity=None):
    """route -> dispatch -> permute -> expert FFN -> combine.

    capacity: see dispatch (None = dropless).  Returns y (float64 [T,h]) and a
    context dict with every intermediate.
    """
    T = x.shape[0]
    E = Wg.shape[1]
    topk_idx, gates, l64 = route(x, Wg, b, k)
    counts, offsets, perm_src, perm_dst = dispatch(topk_idx, E, capacity)
    x64 = as_f64(x)
    x_perm = permute_rows(x64, perm_src, k)
    A, B, H, O = expert_ffn_fwd(x_perm, offsets, W1, W3, W2, counter)
    y = combine(O, gates, perm_dst, T, k)
    ctx = dict(topk_idx=topk_idx, gates=gates, logits=l64, counts=counts,
               offsets=offsets, perm_src=perm_src, perm_dst=perm_dst,
               x_perm=x_perm, A=A, B=B, H=H, O=O, k=k)
    return y, ctx


# --------------------------------------------------------------- backward ---

def expert_ffn_bwd(dO, x_perm, offsets, W1, W3, W2, A, B, H, counter=None):
    """Backward of the per-expert SwiGLU FFN given dO = dL/dO (float64).

    dH = dO W2[e]^T;  dA = dH * B * sigma(A) (1 + A (1 - sigma(A)));
    dB = dH * silu(A);  dW2[e] = H_e^T dO_e;  dW1[e] = X_e^T dA_e;
    dW3[e] = X_e^T dB_e;  dX_perm = dA W1[e]^T + dB W3[e]^T.
    FC2's weight gradient uses fc2_in (H) and d(fc2_out) (review 选择性激活重计算).
    """
    c = counter if counter is not None else MacCounter()
    W1, W3, W2 = as_f64(W1), as_f64(W3), as_f64(W2)
    E, h, f = W1.shape
    X = np.asarray(x_perm, dtype=np.float64)
    dW1 = np.zeros((E, h, f)); dW3 = np.zeros((E, h, f)); dW2 = np.zeros((E, f, h))
    dA = np.zeros_like(A); dB = np.zeros_like(B); dX = np.zeros_like(X)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        dH = c.matmul(dO[lo:hi], W2[e].T)
        a = A[lo:hi]
        s = _sigmoid(a)
        dA[lo:hi] = dH * B[lo:hi] * s * (1.0 + a * (1.0 - s))
        dB[lo:hi] = dH * silu(a)
        dW2[e] = c.matmul(H[lo:hi].T, dO[lo:hi])
        dW1[e] = c.matmul(X[lo:hi].T, dA[lo:hi])
        dW3[e] = c.matmul(X[lo:hi].T, dB[lo:hi])
        dX[lo:hi] = c.matmul(dA[lo:hi], W1[e].T) + c.matmul(dB[lo:hi], W3[e].T)
    return dict(dA=dA, dB=dB, dX_perm=dX, dW1=dW1, dW3=dW3, dW2=dW2)


def router_bwd(gates, dg):
    """dL/dl for the selected logits: dl_j = g_j (dg_j - sum_i g_i dg_i).

    The renormalised gates equal a softmax over the k selected logits (the
    full-softmax denominator cancels), whose Jacobian is g_j (delta_ij - g_i).
    With sum_i g_i = 1 the product is evaluated as g_j sum_i g_i (dg_j - dg_i),
    the same value without the cancellation of dg_j - sum_i g_i dg_i when one
    gate is close to 1.  Unselected logits get zero (selection is piecewise
    constant).
    """
    g = np.asarray(gates, dtype=np.float64)
    d = np.asarray(dg, dtype=np.float64)
    diff = d[:, :, None] - d[:, None, :]          # [T, j, i] = dg_j - dg_i
    return g * np.einsum("ti,tji->tj", g, diff)


def layer_bwd(dy, x, Wg, W1, W3, W2, ctx, counter=None):
    """Gradients of L = <dy, y> with respect to x, Wg, W1, W3, W2, plus dg.

    dO[p] = g[a] dy[t];  dg[a] = <dy[t], O[p]> (0 for a dropped a);  expert
    backward;  dx[t] = sum_j dX_perm[perm_dst[t*k+j]] (kept slots) +
    sum_j dl[t,j] Wg[:, e_j];
    dWg = x^T dl  (dl is zero outside each token's k selected experts).
    """
    k = ctx["k"]
    dy64 = as_f64(dy)
    T, h = dy64.shape
    Wg64 = as_f64(Wg)
    E = Wg64.shape[1]
    perm_src = np.asarray(ctx["perm_src"], dtype=np.int64)
    perm_dst = np.asarray(ctx["perm_dst"], dtype=np.int64)
    g_flat = np.asarray(ctx["gates"], dtype=np.float64).ravel()
    tok = perm_src // k
    dO = g_flat[perm_src][:, None] * dy64[tok]
    dg_perm = np.einsum("ph,ph->p", dy64[tok], ctx["O"])
    dg = np.zeros(T * k)          # a dropped slot has no output: dg = 0
    dg[perm_src] = dg_perm
    dg = dg.reshape(T, k)
    ex = expert_ffn_bwd(dO, ctx["x_perm"], ctx["offsets"], W1, W3, W2,
                        ctx["A"], ctx["B"], ctx["H"], counter)
    dl_sel = router_bwd(ctx["gates"], dg)
    idx = np.asarray(ctx["topk_idx"], dtype=np.int64)
    dl = np.zeros((T, E))
    np.put_along_axis(dl, idx, dl_sel, axis=1)
    dx = unpermute_rows(ex["dX_perm"], perm_dst).reshape(T, k, h).sum(axis=1)
    dx = dx + dl @ Wg64.T
    dWg = as_f64(x).T @ dl
    out = dict(dx=dx, dWg=dWg, dg=dg, dl=dl, dO=dO)
    out.update(ex)
    return out


# ---------------------------------------------- per-token / sampled forms ---

def expert_terms(X, dY, g, W1e, W3e, W2e):
    """Rows X [n,h] through one expert, with their gates g [n] and loss rows dY.

    Returns o = FFN_e(X) [n,h], dg = <dY, o> [n] and dx_e = g * J_e(X)^T dY
    [n,h], the expert's part of the token gradient (the SwiGLU chain rule:
    dH = g dY W2^T, dA = dH * B * s (1 + A (1 - s)), dB = dH * silu(A),
    dx = dA W1^T + dB W3^T).
    """
    X = np.asarray(X, dtype=np.float64).reshape(-1, W1e.shape[0])
    dY = np.asarray(dY, dtype=np.float64).reshape(X.shape[0], -1)
    g = np.asarray(g, dtype=np.float64).reshape(-1, 1)
    a = X @ W1e
    bb = X @ W3e
    o = (silu(a) * bb) @ W2e
    dg = np.einsum("nh,nh->n", dY, o)
    dh = g * (dY @ W2e.T)
    s = _sigmoid(a)
    da = dh * bb * s * (1.0 + a * (1.0 - s))
    db = dh * silu(a)
    return dict(o=o, dg=dg, dx=da @ W1e.T + db @ W3e.T)


def assemble_token(gates, idx, terms, Wg):
    """y, dg and dx of one token from its k per-expert terms (slot order).

    terms[j] = expert_terms(...) of slot j for this token (one row each).
    dx adds the router path: sum_j dl_j Wg[:, e_j], dl = router_bwd(g, dg).
    """
    g = np.asarray(gates, dtype=np.float64)
    y = sum(g[j] * terms[j]["o"][0] for j in range(len(idx)))
    dg = np.array([terms[j]["dg"][0] for j in range(len(idx))])
    dl = router_bwd(g[None, :], dg[None, :])[0]
    Wg64 = as_f64(Wg)
    dx = sum(terms[j]["dx"][0] for j in range(len(idx)))
    for j, e in enumerate(idx):
        dx = dx + dl[j] * Wg64[:, int(e)]
    return dict(y=y, dg=dg, dx=dx)


def token_fwd_bwd(x_t, dy_t, Wg, b, k, expert):
    """The layer for one token, straight from the definition (no dispatch).

    expert(e) -> (W1[e], W3[e], W2[e]) as float64 arrays.  Returns a dict with
    topk_idx, gates, y, dg, dx for this token: y = sum_j g_j FFN_{e_j}(x_t),
    dx = sum_j g_j J_{e_j}(x_t)^T dy + sum_j dl_j Wg[:, e_j].
    """
    x = as_f64(x_t).reshape(1, -1)
    dy = as_f64(dy_t).reshape(1, -1)
    idx, gates, _ = route(x_t.reshape(1, -1), Wg, b, k)
    idx, gates = idx[0], gates[0]
    terms = [expert_terms(x, dy, gates[j], *expert(int(e))) for j, e in enumerate(idx)]
    out = assemble_token(gates, idx, terms, Wg)
    out.update(topk_idx=idx, gates=gates)
    return out


def expert_wgrad_columns(X_e, dO_e, W1e, W3e, W2e, cols):
    """Columns `cols` of dW1[e] and dW3[e] and rows `cols` of dW2[e].

    X_e [n,h] are the expert's token rows in permuted order, dO_e [n,h] the
    matching g * dy rows.  Column c of the FFN width needs only A[:,c], B[:,c]
    and dH[:,c] = dO_e W2[e][c,:]^T.
    """
    X = np.asarray(X_e, dtype=np.float64)
    dO = np.asarray(dO_e, dtype=np.float64)
    cols = np.asarray(cols, dtype=np.int64)
    a = X @ W1e[:, cols]
    bb = X @ W3e[:, cols]
    dh = dO @ W2e[cols, :].T
    s = _sigmoid(a)
    da = dh * bb * s * (1.0 + a * (1.0 - s))
    db = dh * silu(a)
    hh = silu(a) * bb
    return dict(dW1=X.T @ da, dW3=X.T @ db, dW2=hh.T @ dO)


# ----------------------------------------------------- closed-form counts ---

def gemm_macs_fwd(T, h, f, k):
    """Forward expert multiply-adds, 3*k*T*h*f.

    Review §三 核心公式: comp_time = 3k * bsh * h_ffn / n / peak, at n = 1,
    with bs = T tokens (each MAC of the three h x h_ffn matmuls per copy).
    """
    return 3 * k * T * h * f


def dispatch_bytes_per_token(k, h, elem_bytes=2):
    """Bytes one token contributes to dispatch: k copies of its h-vector,
    k*h*2 in BF16 (digest §3.2 table: 3 x 4096 x 2 = 24,576 B)."""
    return k * h * elem_bytes


def activation_bytes(b, s, h, elem_bytes=2):
    """Bytes of a [b*s, h] activation, bsh*2 in BF16 (digest §3.2 table)."""
    return b * s * h * elem_bytes


# ------------------------------------------------------ FP8 (e4m3) forward ---
#
# FP8 training with per-token quantisation instead of per-tensor (review §三
# 创新点 "FP8训练优化": per-token scales address the wider value range after
# SwiGLU; digest §3.4: per-token scales on the FP8 path).  The pages give no
# further recipe; the plain reading used here:
#   * activations entering an expert matmul (x_perm, H) get one scale per row
#     (per token copy): s = amax(|row|) / 448 in float32 (s = 1 for a zero
#     row), q = e4m3(row / s) with the division in float32;
#   * weights get one scale per output column of each expert (amax over the
#     contraction dimension), quantised the same way;
#   * the matmul multiplies the e4m3 values exactly and sums them; the result
#     is scaled by s_row * s_col;
#   * H is stored in bf16 (as on the default path) and that bf16 H is what is
#     quantised for FC2; A, B and O are kept for the backward, which is the
#     default bf16 backward on these activations.

E4M3_MAX = 448.0


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, subnormals down to 2**-9, no infinities, largest finite 448), ties
    to the even mantissa; magnitudes above 448 saturate to 448.  Returns the
    exact values in float64."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))      # a = m 2**ex, m in [0.5, 1)
    e = np.clip(ex - 1, -6, 8)                      # binade; -6 and below: subnormal spacing
    step = np.ldexp(1.0, (e - 3).astype(np.int64))  # spacing of e4m3 values in that binade
    r = np.round(a / step) * step                   # np.round: half to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(v < 0, -r, r)


def bf16_round(v) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); float64 out."""
    f = np.asarray(v, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def quantize_rows_e4m3(X):
    """Per-row scales and e4m3 values: s[i] = amax_j |X[i,j]| / 448 (float32;
    1 for a zero row), q = e4m3(X / s) with a float32 division."""
    X32 = np.asarray(X, dtype=np.float32)
    amax = np.max(np.abs(X32), axis=1) if X32.shape[1] else np.zeros(X32.shape[0], np.float32)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = e4m3_round((X32 / s[:, None]).astype(np.float32))
    return q, s


def quantize_cols_e4m3(W):
    """Per-output-column scales of expert weights W [E, K, N] (amax over K)
    and their e4m3 values: returns q [E, K, N] and s [E, N]."""
    W32 = np.asarray(W, dtype=np.float32)
    amax = np.max(np.abs(W32), axis=1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = e4m3_round((W32 / s[:, None, :]).astype(np.float32))
    return q, s


def expert_ffn_fwd_fp8(x_perm, offsets, W1, W3, W2):
    """expert_ffn_fwd with both matmuls in e4m3 (recipe above).

    Returns A, B, H (bf16-rounded, as stored and quantised), O, and the
    quantised operands: Xq, sx, Hq, sh, (W1q, s1), (W3q, s3), (W2q, s2).
    """
    Xq, sx = quantize_rows_e4m3(as_f64(x_perm))
    W1q, s1 = quantize_cols_e4m3(as_f64(W1))
    W3q, s3 = quantize_cols_e4m3(as_f64(W3))
    W2q, s2 = quantize_cols_e4m3(as_f64(W2))
    R = Xq.shape[0]
    E, h, f = W1q.shape
    A = np.zeros((R, f)); B = np.zeros((R, f))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        sxe = sx[lo:hi, None].astype(np.float64)
        A[lo:hi] = (Xq[lo:hi] @ W1q[e]) * sxe * s1[e][None, :]
        B[lo:hi] = (Xq[lo:hi] @ W3q[e]) * sxe * s3[e][None, :]
    H = bf16_round(silu(A) * B)
    Hq, sh = quantize_rows_e4m3(H)
    O = np.zeros((R, h))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        O[lo:hi] = (Hq[lo:hi] @ W2q[e]) * sh[lo:hi, None] * s2[e][None, :]
    return dict(A=A, B=B, H=H, O=O, Xq=Xq, sx=sx, Hq=Hq, sh=sh, W1q=W1q, s1=s1, W3q=W3q,
                s3=s3, W2q=W2q, s2=s2)


def layer_fwd_fp8(x, Wg, b, W1, W3, W2, k, capacity=None):
    """layer_fwd with the expert matmuls of expert_ffn_fwd_fp8.  The context
    feeds layer_bwd unchanged (the backward runs on these activations)."""
    T = x.shape[0]
    E = Wg.shape[1]
    topk_idx, gates, l64 = route(x, Wg, b, k)
    counts, offsets, perm_src, perm_dst = dispatch(topk_idx, E, capacity)
    x_perm = permute_rows(as_f64(x), perm_src, k)
    f8 = expert_ffn_fwd_fp8(x_perm, offsets, W1, W3, W2)
    y = combine(f8["O"], gates, perm_dst, T, k)
    ctx = dict(topk_idx=topk_idx, gates=gates, logits=l64, counts=counts, offsets=offsets,
               perm_src=perm_src, perm_dst=perm_dst, x_perm=x_perm, k=k, fp8=f8,
               A=f8["A"], B=f8["B"], H=f8["H"], O=f8["O"])
    return y, ctx


# ------------------------------------------------------ FP8 (e4m3) dgrad ---
#
# The backward's FC1 data-gradient matmul on e4m3 codes, with the same
# per-token reading as the forward: the left operand's rows get one scale each
# and the weights' output rows one scale each (amax over the contraction
# dimension), so the scales again factor out of the sums.
#   FC1 dgrad  dX = dA W1^T + dB W3^T, one contraction over both halves: a row
#              of dA and the same row of dB share one scale (amax over both
#              bf16 rows), and row n of W1[e] and row n of W3[e] share one.
# FC2 dgrad (dH = dO W2^T with the SwiGLU backward) stays bf16: its time is
# the fused SwiGLU-backward epilogue, which e4m3 operands do not shorten.  The
# weight gradients stay bf16 matmuls on the bf16 dO, dA, dB; dO is the bf16
# value of g * dy (product in float32).

def quantize_rows_joint_e4m3(X0, X1):
    """Row i of X0 and row i of X1 quantised with one shared float32 scale
    amax(|X0[i]|, |X1[i]|) / 448 (1 if both rows are zero)."""
    X0_32 = np.asarray(X0, dtype=np.float32)
    X1_32 = np.asarray(X1, dtype=np.float32)
    amax = np.maximum(np.max(np.abs(X0_32), axis=1), np.max(np.abs(X1_32), axis=1))
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q0 = e4m3_round((X0_32 / s[:, None]).astype(np.float32))
    q1 = e4m3_round((X1_32 / s[:, None]).astype(np.float32))
    return q0, q1, s


def fc1_dgrad_fp8(dA, dB, W1e, W3e):
    """dX = dA W1e^T + dB W3e^T on e4m3 codes: rows of dA and dB [n, f] share a
    scale; rows n of W1e and W3e ([h, f]) share a scale."""
    aq, bq, sa = quantize_rows_joint_e4m3(dA, dB)
    w1q, w3q, sw = quantize_rows_joint_e4m3(W1e, W3e)
    return (aq @ w1q.T + bq @ w3q.T) * sa[:, None].astype(np.float64) * sw[None, :].astype(
        np.float64)


def expert_ffn_bwd_fp8(dO, x_perm, offsets, W1, W3, W2, A, B, H):
    """expert_ffn_bwd with the FC1 dgrad on e4m3 codes (recipe above).  dO must
    be the bf16 values of g * dy.  The activations are taken as stored, in
    bf16 (A, B, H are rounded here): the e4m3 codes of dA and dB are integer
    decisions, so they are made from the same values the layer keeps.  dA and
    dB are rounded to bf16 (as stored) before the FC1 dgrad, and the weight
    gradients use those bf16 copies."""
    W1, W3, W2 = as_f64(W1), as_f64(W3), as_f64(W2)
    E, h, f = W1.shape
    X = np.asarray(x_perm, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    A, B, H = bf16_round(A), bf16_round(B), bf16_round(H)
    dW1 = np.zeros((E, h, f)); dW3 = np.zeros((E, h, f)); dW2 = np.zeros((E, f, h))
    dA = np.zeros_like(A); dB = np.zeros_like(B); dX = np.zeros_like(X)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        dH = dO[lo:hi] @ W2[e].T
        a = A[lo:hi]
        sg = _sigmoid(a)
        dA[lo:hi] = bf16_round(dH * B[lo:hi] * sg * (1.0 + a * (1.0 - sg)))
        dB[lo:hi] = bf16_round(dH * silu(a))
        dW2[e] = H[lo:hi].T @ dO[lo:hi]
        dW1[e] = X[lo:hi].T @ dA[lo:hi]
        dW3[e] = X[lo:hi].T @ dB[lo:hi]
        dX[lo:hi] = fc1_dgrad_fp8(dA[lo:hi], dB[lo:hi], W1[e], W3[e])
    return dict(dA=dA, dB=dB, dX_perm=dX, dW1=dW1, dW3=dW3, dW2=dW2)


def layer_bwd_fp8(dy, x, Wg, W1, W3, W2, ctx):
    """layer_bwd with the expert dgrad of expert_ffn_bwd_fp8; dO = bf16(g dy)
    with the product in float32, dg = <dy, O> in float64."""
    k = ctx["k"]
    dy64 = as_f64(dy)
    T, h = dy64.shape
    Wg64 = as_f64(Wg)
    E = Wg64.shape[1]
    perm_src = np.asarray(ctx["perm_src"], dtype=np.int64)
    perm_dst = np.asarray(ctx["perm_dst"], dtype=np.int64)
    g32 = np.asarray(ctx["gates"], dtype=np.float32).ravel()
    tok = perm_src // k
    dO = bf16_round(g32[perm_src][:, None] * dy64[tok].astype(np.float32))
    dg_perm = np.einsum("ph,ph->p", dy64[tok], ctx["O"])
    dg = np.zeros(T * k)
    dg[perm_src] = dg_perm
    dg = dg.reshape(T, k)
    ex = expert_ffn_bwd_fp8(dO, ctx["x_perm"], ctx["offsets"], W1, W3, W2,
                            ctx["A"], ctx["B"], ctx["H"])
    dl_sel = router_bwd(ctx["gates"], dg)
    idx = np.asarray(ctx["topk_idx"], dtype=np.int64)
    dl = np.zeros((T, E))
    np.put_along_axis(dl, idx, dl_sel, axis=1)
    dx = unpermute_rows(ex["dX_perm"], perm_dst).reshape(T, k, h).sum(axis=1)
    dx = dx + dl @ Wg64.T
    dWg = as_f64(x).T @ dl
    out = dict(dx=dx, dWg=dWg, dg=dg, dl=dl, dO=dO)
    out.update(ex)
    return out

