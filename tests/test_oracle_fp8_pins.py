"""Pins of the oracle's FP8 (e4m3, per-token scale) forward (no GPU).

The e4m3 rounding is checked against torch's float8_e4m3fn conversion and the
format's own fixed points; bf16 rounding against torch; the per-row and
per-column quantisers against exact power-of-two cases and the format's error
bound; the FP8 expert forward against the exact forward on inputs that
quantise without error.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import conditioned_inputs, rel_l2, small_config

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).float().double().numpy()


def test_e4m3_fixed_points_are_every_finite_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = codes.float().double().numpy()
    vals = vals[np.isfinite(vals)]
    assert vals.size == 254 and np.max(vals) == 448.0 and np.min(vals[vals > 0]) == 2.0 ** -9
    np.testing.assert_array_equal(oracle.e4m3_round(vals), vals)


def test_e4m3_matches_torch_in_range_including_ties_and_subnormals():
    rng = np.random.default_rng(1)
    mag = 2.0 ** rng.uniform(-12, np.log2(448.0), 100000)
    sign = np.where(rng.random(mag.size) < 0.5, -1.0, 1.0)
    v = (sign * mag).astype(np.float32)
    # exact midpoints between neighbouring codes (ties) and subnormal values
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    c = np.unique(np.abs(codes.float().double().numpy()[np.isfinite(codes.float().numpy())]))
    mids = ((c[1:] + c[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, (np.arange(1, 64) * 2.0 ** -11).astype(np.float32)])
    v = v[np.abs(v) <= 448.0]
    np.testing.assert_array_equal(oracle.e4m3_round(v), _torch_e4m3(v))


def test_e4m3_saturates():
    v = np.array([448.0, 449.0, 463.99, 464.0, 1e6, -500.0], dtype=np.float32)
    np.testing.assert_array_equal(oracle.e4m3_round(v), [448, 448, 448, 448, 448, -448])


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-6, 6, 100000)).astype(np.float32)
    # exact ties: low 16 bits 0x8000
    hi = rng.integers(0x30000000, 0x4F000000, 1000).astype(np.uint32) & np.uint32(0xFFFF0000)
    t = (hi | np.uint32(0x8000)).view(np.float32)
    v = np.concatenate([v, t])
    ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.bf16_round(v), ref)


def test_quantize_rows_exact_on_power_of_two_scaled_codes():
    rng = np.random.default_rng(3)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    c = codes.float().double().numpy()
    c = c[np.isfinite(c)]
    q = rng.choice(c, size=(12, 40))
    q[:, 0] = 448.0                              # every row's amax is 448 * 2**j
    j = rng.integers(-20, 20, size=12)
    X = q * np.ldexp(1.0, j)[:, None]
    Xq, s = oracle.quantize_rows_e4m3(X)
    np.testing.assert_array_equal(s, np.ldexp(1.0, j).astype(np.float32))
    np.testing.assert_array_equal(Xq, q)
    Wq, sw = oracle.quantize_cols_e4m3(np.transpose(X.reshape(3, 4, 40), (0, 2, 1)))
    np.testing.assert_array_equal(sw, np.ldexp(1.0, j).astype(np.float32).reshape(3, 4))
    np.testing.assert_array_equal(Wq, np.transpose(q.reshape(3, 4, 40), (0, 2, 1)))


def test_quantize_rows_error_bound_and_zero_row():
    rng = np.random.default_rng(4)
    X = (rng.standard_normal((64, 300)) * np.exp(rng.uniform(-8, 8, (64, 1)))).astype(np.float32)
    X[5] = 0.0
    Xq, s = oracle.quantize_rows_e4m3(X)
    assert s[5] == 1.0 and np.all(Xq[5] == 0)
    err = np.abs(Xq * s[:, None].astype(np.float64) - X)
    # half a spacing: 2**-4 relative in the normal range, 2**-10 * s below it
    bound = np.maximum(2.0 ** -4 * np.abs(X), 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)
    assert np.all(np.abs(Xq) <= 448.0) and np.all(np.max(np.abs(Xq), axis=1)[s != 1] == 448.0)


def test_fp8_expert_forward_is_exact_on_quantisable_inputs():
    """x rows and weight columns that are e4m3 codes times powers of two
    quantise without error, so A and B equal the exact forward's."""
    rng = np.random.default_rng(5)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    c = codes.float().double().numpy()
    c = c[np.isfinite(c) & (np.abs(c) <= 8)]
    R, h, f, E = 24, 32, 48, 3
    X = rng.choice(c, (R, h)); X[:, 3] = 448.0
    X *= np.ldexp(1.0, rng.integers(-12, -6, R))[:, None]
    W1 = rng.choice(c, (E, h, f)); W1[:, 7, :] = 448.0
    W1 *= np.ldexp(1.0, rng.integers(-14, -8, (E, 1, f)))
    W3 = rng.choice(c, (E, h, f)); W3[:, 1, :] = -448.0
    W3 *= np.ldexp(1.0, rng.integers(-14, -8, (E, 1, f)))
    W2 = rng.standard_normal((E, f, h)) * 0.1
    offsets = np.array([0, 5, 5, R])
    f8 = oracle.expert_ffn_fwd_fp8(X, offsets, W1, W3, W2)
    A, B, H, O = oracle.expert_ffn_fwd(X, offsets, W1, W3, W2)
    np.testing.assert_allclose(f8["A"], A, rtol=1e-13, atol=0)
    np.testing.assert_allclose(f8["B"], B, rtol=1e-13, atol=0)
    np.testing.assert_array_equal(f8["H"], oracle.bf16_round(silu_np(A) * B))
    # O from the quantised H and W2: within the e4m3 error of the exact O
    assert rel_l2(f8["O"], O) < 0.08


def silu_np(z):
    return z / (1 + np.exp(-z))


@pytest.mark.parametrize("E,k", [(4, 2), (6, 3)])
def test_fp8_layer_close_to_exact_and_backward_runs(E, k):
    cfg = small_config(T=64, h=64, f=96, E=E, k=k, seed=600 + E)
    inp = conditioned_inputs(cfg)
    y, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], k)
    y8, ctx8 = oracle.layer_fwd_fp8(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                                    inp["W2"], k)
    np.testing.assert_array_equal(ctx8["perm_src"], ctx["perm_src"])
    e = rel_l2(y8, y)
    # e4m3 keeps 3 mantissa bits: about 2.5% rms error per operand, four operands
    assert 1e-2 < e < 0.1, e
    g = oracle.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    g8 = oracle.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx8)
    for key in ("dx", "dW1", "dW2", "dWg"):
        assert rel_l2(g8[key], g[key]) < 0.2, key


# ------------------------------------------------------------ FP8 dgrads ---

def _codes_scaled(rng, shape, lo, hi):
    """e4m3 codes times a power of two per row, with 448 in every row."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    c = codes.float().double().numpy()
    c = c[np.isfinite(c) & (np.abs(c) <= 16)]
    q = rng.choice(c, shape)
    q[:, int(rng.integers(0, shape[1]))] = 448.0
    j = rng.integers(lo, hi, shape[0])
    return q * np.ldexp(1.0, j)[:, None], q, np.ldexp(1.0, j)


def test_joint_row_quantiser_equals_quantiser_of_the_concatenation():
    rng = np.random.default_rng(7)
    X0 = rng.standard_normal((40, 24)) * np.exp(rng.uniform(-3, 3, (40, 1)))
    X1 = rng.standard_normal((40, 16)) * np.exp(rng.uniform(-3, 3, (40, 1)))
    X1[3] *= 100.0                                   # the amax sits in X1 for some rows
    q0, q1, s = oracle.quantize_rows_joint_e4m3(X0, X1)
    qc, sc = oracle.quantize_rows_e4m3(np.concatenate([X0, X1], axis=1))
    np.testing.assert_array_equal(s, sc)
    np.testing.assert_array_equal(np.concatenate([q0, q1], axis=1), qc)


def test_fc1_dgrad_fp8_exact_on_jointly_quantisable_rows():
    rng = np.random.default_rng(9)
    dAB, _, _ = _codes_scaled(rng, (10, 48), -14, -4)
    dA, dB = dAB[:, :24], dAB[:, 24:]
    W13, _, _ = _codes_scaled(rng, (16, 48), -12, -6)     # rows n of [W1 | W3]
    W1, W3 = W13[:, :24], W13[:, 24:]
    np.testing.assert_allclose(oracle.fc1_dgrad_fp8(dA, dB, W1, W3), dA @ W1.T + dB @ W3.T,
                               rtol=1e-13, atol=0)
    # a separate scale for each half (instead of one shared) is not exact here
    def deq(X, W):
        q, s = oracle.quantize_rows_e4m3(X)
        return q * s[:, None].astype(np.float64)
    sep = deq(dA, None) @ deq(W1, None).T + deq(dB, None) @ deq(W3, None).T
    assert not np.allclose(sep, dA @ W1.T + dB @ W3.T, rtol=1e-9, atol=0)


@pytest.mark.parametrize("E,k", [(4, 2), (6, 3)])
def test_fp8_backward_close_to_exact_and_dO_is_bf16_of_fp32_product(E, k):
    cfg = small_config(T=64, h=64, f=96, E=E, k=k, seed=700 + E)
    inp = conditioned_inputs(cfg)
    y, ctx = oracle.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], k)
    g = oracle.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    g8 = oracle.layer_bwd_fp8(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"],
                              ctx)
    # dO: the float32 product of gate and dy, rounded to bf16 (torch's conversion)
    a = torch.from_numpy(np.asarray(ctx["perm_src"], dtype=np.int64))
    gt = torch.from_numpy(np.asarray(ctx["gates"], dtype=np.float32)).reshape(-1)[a]
    ref = (gt[:, None] * inp["dy"].float()[a // k]).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(g8["dO"], ref)
    np.testing.assert_array_equal(g8["dg"], g["dg"])
    for key in ("dx", "dW1", "dW3", "dW2", "dWg"):
        e = rel_l2(g8[key], g[key])
        assert e < 0.12, (key, e)
    assert rel_l2(g8["dx"], g["dx"]) > 1e-3          # the quantisation is really there
