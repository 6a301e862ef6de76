"""Seeded synthetic inputs for one MoE FFN layer (random numbers only).

Every element is a pure function of (seed, tensor id, element index):

  mix   = splitmix64 output function (two xor-shift-multiply rounds)
  key   = mix(seed * 2**32 + tensor_id + GAMMA)
  z_j   = mix(key + (2*i + j) * GAMMA)                 j = 1, 2
  u1    = (z_1 >> 11 + 1) * 2**-53  in (0, 1]
  u2    = (z_2 >> 11)     * 2**-53  in [0, 1)
  n_i   = sqrt(-2 ln u1) * cos(2 pi u2)                (Box-Muller, float64)

splitmix64 is Vigna's published mixer (state += GAMMA; two xor-shift-multiply
rounds; final xor-shift).  The integer part is exact on CPU and GPU (torch
int64 arithmetic wraps modulo 2**64); the float64 transform may differ by an
ulp between devices, which the bf16/fp32 rounding of the result absorbs.

Value recipe (the workloads' "same init scheme"):
  x, dy   ~ N(0, 1)        -> bf16 (round-to-nearest-even via fp32)
  Wg      ~ N(0, 1/h)      -> fp32
  W1, W3  ~ N(0, 1/h)      -> bf16   (fan_in = h)
  W2      ~ N(0, 1/f)      -> bf16   (fan_in = f)
  b       = 0, or a fixed Zipf-shaping bias (see zipf_router_bias)

This module holds random-number generation and tensor formatting only.  It
computes nothing of the layer itself.
"""
from __future__ import annotations

import math

import numpy as np
import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB

# tensor ids of the streams
TID_X, TID_WG, TID_W1, TID_W3, TID_W2, TID_DY, TID_BIAS_FIT = 1, 2, 3, 4, 5, 6, 7
TID_X_RESAMPLE = 1000      # + attempt number: replacement rows for x

_CHUNK = 1 << 25           # elements generated per device pass


def _s64(v: int) -> int:
    """Python int in [0, 2**64) -> the int64 with the same bits."""
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def splitmix64_py(state: int) -> int:
    """Scalar splitmix64 output for an already-advanced state (pure Python)."""
    z = state & MASK64
    z = ((z ^ (z >> 30)) * _MIX1) & MASK64
    z = ((z ^ (z >> 27)) * _MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    return splitmix64_py((seed << 32) + tensor_id + GAMMA)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _s64(_MIX1)
    z = (z ^ _lsr(z, 27)) * _s64(_MIX2)
    return z ^ _lsr(z, 31)


def normal_from_index(seed: int, tensor_id: int, idx: torch.Tensor) -> torch.Tensor:
    """float64 N(0,1) draws for the int64 element indices `idx` (any device)."""
    key = _s64(stream_key(seed, tensor_id))
    g = _s64(GAMMA)
    base = idx * 2
    z1 = _mix((base + 1) * g + key)
    z2 = _mix((base + 2) * g + key)
    u1 = (_lsr(z1, 11) + 1).to(torch.float64) * (2.0 ** -53)
    u2 = _lsr(z2, 11).to(torch.float64) * (2.0 ** -53)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal(seed: int, tensor_id: int, shape, std: float, dtype: torch.dtype,
           device="cpu") -> torch.Tensor:
    """Tensor of N(0, std^2) draws rounded to `dtype` (fp32 first, then dtype)."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = torch.empty(n, dtype=dtype, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        idx = torch.arange(s, e, dtype=torch.int64, device=device)
        v = normal_from_index(seed, tensor_id, idx) * std
        out[s:e] = v.to(torch.float32).to(dtype)
    return out.view(shape)


def rows(seed: int, tensor_id: int, row_ids, ncols: int, std: float,
         dtype: torch.dtype, device="cpu") -> torch.Tensor:
    """Rows `row_ids` of the [*, ncols] matrix drawn from stream `tensor_id`."""
    r = torch.as_tensor(row_ids, dtype=torch.int64, device=device).view(-1, 1)
    idx = r * ncols + torch.arange(ncols, dtype=torch.int64, device=device).view(1, -1)
    v = normal_from_index(seed, tensor_id, idx) * std
    return v.to(torch.float32).to(dtype)


def zipf_router_bias(E: int, k: int, s: float, seed: int, n_zero: int = 1,
                     samples: int = 32768, iters: int = 200) -> np.ndarray:
    """Fixed fp32 router bias that skews expert load towards Zipf(s).

    Experts 0..E-n_zero-1 get target shares proportional to (e+1)^-s; the last
    `n_zero` experts get -1e4 so that no token ever selects them.  The bias is
    fitted to i.i.d. N(0,1) surrogate scores (one row of E draws per sample,
    drawn from this module's own stream), not to any layer input: it is a
    parameter of the workload, and only the shape of the resulting load is
    claimed.  Each iteration counts how often each expert lands among the k
    largest surrogate scores and moves its bias by half the log-ratio of target
    to observed share.
    """
    live = E - n_zero
    target = np.array([(r + 1.0) ** (-s) for r in range(live)])
    target /= target.sum()
    z = normal(seed, TID_BIAS_FIT, (samples, E), 1.0, torch.float64).numpy()
    b = np.zeros(E)
    b[live:] = -1.0e4
    floor = 0.5 / (samples * k)
    for _ in range(iters):
        top = np.argpartition(-(z + b), k - 1, axis=1)[:, :k]
        share = np.bincount(top.ravel(), minlength=E)[:live] / float(samples * k)
        b[:live] += 0.5 * (np.log(target) - np.log(np.maximum(share, floor)))
        b[:live] -= b[:live].max()
    return b.astype(np.float32)


def make_layer(cfg, device="cpu", with_dy: bool = True) -> dict:
    """All inputs of one layer config as tensors on `device`.

    Returns x, Wg, b, W1, W3, W2 (and dy).  Shapes: x, dy [T,h] bf16; Wg [h,E]
    fp32; b [E] fp32; W1, W3 [E,h,f] bf16; W2 [E,f,h] bf16.
    """
    T, h, f, E = cfg.T, cfg.h, cfg.f, cfg.E
    sd = cfg.seed
    out = {
        "x": normal(sd, TID_X, (T, h), 1.0, torch.bfloat16, device),
        "Wg": normal(sd, TID_WG, (h, E), 1.0 / math.sqrt(h), torch.float32, device),
        "W1": normal(sd, TID_W1, (E, h, f), 1.0 / math.sqrt(h), torch.bfloat16, device),
        "W3": normal(sd, TID_W3, (E, h, f), 1.0 / math.sqrt(h), torch.bfloat16, device),
        "W2": normal(sd, TID_W2, (E, f, h), 1.0 / math.sqrt(f), torch.bfloat16, device),
    }
    if cfg.zipf_s > 0:
        bias = zipf_router_bias(E, cfg.k, cfg.zipf_s, sd)
        out["b"] = torch.from_numpy(bias).to(device)
    else:
        out["b"] = torch.zeros(E, dtype=torch.float32, device=device)
    if with_dy:
        out["dy"] = normal(sd, TID_DY, (T, h), 1.0, torch.bfloat16, device)
    return out


def replacement_x_rows(cfg, row_ids, attempt: int, device="cpu") -> torch.Tensor:
    """Fresh N(0,1) bf16 rows for x, from the attempt-th replacement stream."""
    return rows(cfg.seed, TID_X_RESAMPLE + attempt, row_ids, cfg.h, 1.0,
                torch.bfloat16, device)
