"""Exact pins of the FP8 expert forward's FC2 half and of the FP8 backward
(no GPU), on constructed inputs, for both oracles (the C++ record and the
float64 numpy oracle).

The inputs are chosen so that every step has a closed form:
  * A >= 64, so sigmoid(A) = 1 and silu(A) = A exactly in fp32 and fp64
    (e^-64 is below half an ulp of 1 in both);
  * activation rows and weight columns (or rows) that are e4m3 codes times a
    power of two with 448 times that power in them, so their per-row or
    per-column scale is that power of two and the codes are the values;
  * one-hot rows where a single product decides a sum.
The expected values then come from plain float64 arithmetic on exact values
and from torch's own bf16 and float8_e4m3fn conversions: no formula of the
oracles is retyped.  Each case also shows that the plausible misreading it
guards against (codes from the unrounded H, another expert's scale, unrounded
A/B/H or dA/dB in the backward) gives a different result.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.cref as cref

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

IMPLS = {"numpy": oracle, "cpp": cref}
# the record sums and scales in fp32: products of a 4-bit code and a 24-bit
# scale round once or twice
RTOL = {"numpy": 0.0, "cpp": 4e-7}


def _codes(lo=0.0, hi=448.0):
    c = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    v = c.float().double().numpy()
    v = v[np.isfinite(v)]
    return v[(np.abs(v) >= lo) & (np.abs(v) <= hi)]


def _bf16(v):
    return torch.from_numpy(np.asarray(v, np.float64)).to(torch.bfloat16).double().numpy()


def _e4m3(v32):
    return torch.from_numpy(np.asarray(v32, np.float32)).to(torch.float8_e4m3fn).double().numpy()


def _row_deq(Hrow):
    """torch's e4m3 codes of one row under its amax/448 fp32 scale, and the scale."""
    s = np.float32(np.max(np.abs(Hrow))) / np.float32(448.0)
    q = _e4m3(np.asarray(Hrow, np.float32) / s)
    return q, np.float64(s)


def _close(got, want, rtol):
    got = np.asarray(got, np.float64)
    if rtol == 0.0:
        np.testing.assert_array_equal(got, want)
    else:
        np.testing.assert_allclose(got, want, rtol=rtol, atol=0)


# --------------------------------------------------- forward: the FC2 half ---

def _fc2_case(seed):
    rng = np.random.default_rng(seed)
    R, h, f, E = 8, 16, 16, 2
    u = rng.integers(0, 3, R)
    X = np.zeros((R, h))
    X[:, 0] = X[:, 1] = 56.0 * np.ldexp(1.0, -u)          # row scale 2^(-3-u), codes 448
    W1 = np.zeros((E, h, f)); W1[:, 0, :] = 448.0            # column scale 1, A = 25088 2^-u
    kE = np.array([0, 1])
    q = rng.choice(_codes(1.0, 448.0), (E, f))
    W3 = np.zeros((E, h, f))
    W3[:, 0, :] = 448.0 * np.ldexp(1.0, kE)[:, None]
    W3[:, 1, :] = q * np.ldexp(1.0, kE)[:, None]             # column scale 2^kE, codes [448, q]
    mE = np.array([0, 2])                                    # the two experts' W2 scales differ
    W2 = np.zeros((E, f, h))
    for e in range(E):
        W2[e][np.arange(f), np.arange(f)] = 448.0 * np.ldexp(1.0, -mE[e])
    offsets = np.array([0, 3, R])
    ex = np.repeat(np.arange(E), np.diff(offsets))
    A = 25088.0 * np.ldexp(1.0, -u)[:, None] * np.ones((1, f))
    B = 56.0 * (448.0 + q[ex]) * np.ldexp(1.0, kE[ex] - u)[:, None]
    H = A * B                                               # exact: <= 22 significant bits
    return X, W1, W3, W2, offsets, ex, mE, A, B, H


@pytest.mark.parametrize("impl", list(IMPLS))
def test_fp8_forward_fc2_half_exact_and_codes_from_the_bf16_H(impl):
    orc = IMPLS[impl]
    X, W1, W3, W2, offsets, ex, mE, A, B, H = _fc2_case(seed=17)
    f8 = orc.expert_ffn_fwd_fp8(X, offsets, W1, W3, W2)
    np.testing.assert_array_equal(np.asarray(f8["A"], np.float64), A)
    np.testing.assert_array_equal(np.asarray(f8["B"], np.float64), B)
    Hb = _bf16(H)
    assert np.any(Hb != H)
    np.testing.assert_array_equal(np.asarray(f8["H"], np.float64), Hb)
    want = np.zeros_like(H)
    alt = np.zeros_like(H)
    wrong_expert = np.zeros_like(H)
    codes_differ = False
    for r in range(H.shape[0]):
        qb, sb = _row_deq(Hb[r])
        qu, su = _row_deq(H[r])
        codes_differ |= bool(np.any(qb != qu))
        want[r] = qb * sb * 448.0 * np.ldexp(1.0, -mE[ex[r]])
        alt[r] = qu * su * 448.0 * np.ldexp(1.0, -mE[ex[r]])
        wrong_expert[r] = qb * sb * 448.0 * np.ldexp(1.0, -mE[1 - ex[r]])
    assert codes_differ, "the case must make H and bf16(H) quantise differently"
    _close(f8["O"], want, RTOL[impl])
    O = np.asarray(f8["O"], np.float64)
    for other in (alt, wrong_expert):
        assert np.linalg.norm(O - other) > 1e-4 * np.linalg.norm(other)


# ------------------------------------------------------------- backward ---

def _codes_scaled_rows(rng, n, m, lo, hi, cmax=16.0):
    q = rng.choice(_codes(1.0, cmax), (n, m))
    q[np.arange(n), rng.integers(0, m, n)] = 448.0
    return q * np.ldexp(1.0, rng.integers(lo, hi, n))[:, None]


@pytest.mark.parametrize("impl", list(IMPLS))
def test_fp8_backward_exact_on_jointly_quantisable_dA_dB(impl):
    """A >= 64 makes dA = dH * B and dB = dH * A exactly; rows of [dA | dB] are
    codes times 2^p with 448 * 2^p among them, and rows of [W1 | W3] are
    codes times a power of two: the e4m3 FC1 dgrad is then exact."""
    orc = IMPLS[impl]
    rng = np.random.default_rng(23)
    n, h, f = 6, 12, 16
    p = rng.integers(-6, 2, n)
    A = np.abs(rng.choice(_codes(64.0, 448.0), (n, f))); A[:, 0] = 448.0
    B = rng.choice(_codes(1.0, 448.0), (n, f)) * np.where(rng.random((n, f)) < 0.5, -1, 1)
    dO = np.zeros((n, h)); dO[:, 0] = np.ldexp(1.0, p)       # bf16 values of g * dy
    W2 = rng.standard_normal((1, f, h)); W2[0, :, 0] = 1.0      # dH[r, c] = 2^p_r
    W13 = _codes_scaled_rows(rng, h, 2 * f, -8, -3)
    W1, W3 = W13[None, :, :f], W13[None, :, f:]
    X = rng.choice(_codes(1.0, 8.0), (n, h)) * np.where(rng.random((n, h)) < 0.5, -1, 1)
    H = _bf16(A * B)
    out = orc.expert_ffn_bwd_fp8(dO, X, np.array([0, n]), W1, W3, W2, A, B, H)
    dA = np.ldexp(1.0, p)[:, None] * B
    dB = np.ldexp(1.0, p)[:, None] * A
    _close(out["dA"], dA, 0.0)
    _close(out["dB"], dB, 0.0)
    _close(out["dX_perm"], dA @ W1[0].T + dB @ W3[0].T, RTOL[impl])
    _close(out["dW1"][0], X.T @ dA, RTOL[impl])
    _close(out["dW3"][0], X.T @ dB, RTOL[impl])
    _close(out["dW2"][0], H.T @ dO, RTOL[impl])


@pytest.mark.parametrize("impl", list(IMPLS))
def test_fp8_backward_rounds_A_B_H_and_dA_dB_to_bf16(impl):
    """The backward works on the bf16 copies the layer keeps: A, B, H are
    rounded on entry, dA and dB are rounded before they feed the weight
    gradients and the FC1 dgrad codes."""
    orc = IMPLS[impl]
    rng = np.random.default_rng(29)
    n, h, f = 5, 8, 8
    A = np.full((n, f), 64.25)                 # bf16: 64
    B = np.full((n, f), 3.0)
    B[:, 1::2] = -255.0                        # bf16 exact
    H = np.full((n, f), 1.0 + 2.0 ** -9)       # bf16: 1
    p = rng.integers(-4, 1, n)
    dO = np.zeros((n, h)); dO[:, 0] = np.ldexp(1.0, p)
    W2 = rng.standard_normal((1, f, h)); W2[0, :, 0] = 255.0   # dH = 255 * 2^p
    W13 = _codes_scaled_rows(rng, h, 2 * f, -8, -3)
    W1, W3 = W13[None, :, :f], W13[None, :, f:]
    X = rng.choice(_codes(1.0, 8.0), (n, h))
    out = orc.expert_ffn_bwd_fp8(dO, X, np.array([0, n]), W1, W3, W2, A, B, H)
    dH = 255.0 * np.ldexp(1.0, p)[:, None]
    dA = _bf16(dH * _bf16(B))                  # 765 -> 764 where B = 3
    dB = _bf16(dH * _bf16(A))                  # 255 * 64, exact
    assert np.any(dA != dH * B) and np.any(_bf16(dH * A) != dB)
    _close(out["dA"], dA, 0.0)
    _close(out["dB"], dB, 0.0)
    _close(out["dW1"][0], X.T @ dA, RTOL[impl])
    _close(out["dW3"][0], X.T @ dB, RTOL[impl])
    _close(out["dW2"][0], _bf16(H).T @ dO, RTOL[impl])
    assert not np.allclose(np.asarray(out["dW2"][0], np.float64), H.T @ dO, rtol=1e-4, atol=0)
    # FC1 dgrad from the codes of the rounded dA, dB (torch's e4m3) and the
    # exact codes of W1, W3 (rows of codes times 2^j)
    want = np.zeros((n, h))
    for r in range(n):
        row = np.concatenate([dA[r], dB[r]])
        q, s = _row_deq(row)
        want[r] = (q[:f] @ (W1[0] / _row_scale(W13)[:, None]).T
                   + q[f:] @ (W3[0] / _row_scale(W13)[:, None]).T) * s * _row_scale(W13)
    _close(out["dX_perm"], want, RTOL[impl])


def _row_scale(W13):
    return np.max(np.abs(W13), axis=1) / 448.0
