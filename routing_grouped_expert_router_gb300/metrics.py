"""Throughput and roofline arithmetic used by the benchmark."""
from __future__ import annotations


def tokens_per_s(tokens: int, ms: float) -> float:
    """Tokens processed per second: tokens per step / seconds per step
    (the digest's throughput arithmetic, §5: sequences x length / step time)."""
    return tokens / (ms * 1e-3)


def tflops(flops: float, ms: float) -> float:
    return flops / (ms * 1e-3) / 1e12


def gbs(nbytes: float, ms: float) -> float:
    return nbytes / (ms * 1e-3) / 1e9


# Algorithmic work per kernel launch of the layer (FLOPs for the tensor-core
# GroupedGEMMs, minimum HBM bytes for the rest).  R = T*k permuted rows.
def kernel_work(T: int, h: int, f: int, E: int, k: int) -> dict:
    R = T * k
    gemm = {
        "gg_fc1_fwd_swiglu": 2 * 2 * R * h * f,
        "gg_fc2_fwd": 2 * R * f * h,
        "gg_fc2_dgrad_swiglu_bwd": 2 * R * h * f,
        "gg_fc2_dgrad_swiglu_bwd_sar": 2 * R * h * f,
        "gg_fc1_fwd_swiglu_fp8": 2 * 2 * R * h * f,
        "gg_fc2_fwd_fp8": 2 * R * f * h,
        "gg_fc1_dgrad_fp8": 2 * 2 * R * f * h,
        "gg_fc2_wgrad": 2 * R * f * h,
        "gg_fc1_dgrad": 2 * 2 * R * f * h,
        "gg_fc1_wgrad": 2 * 2 * R * h * f,
    }
    hbm = {
        "router_topk": T * h * 2 + h * E * 4 + R * 8,
        "dispatch_hist": R * 4 + (R // 1024 + 1) * E * 4,
        "dispatch_scan": 2 * (R // 1024 + 1) * E * 4 + (2 * E + 1) * 4,
        "dispatch_scatter": R * 4 + R * 8,
        "permute_rows": T * h * 2 + R * h * 2 + R * 4,
        "combine": R * h * 2 + T * h * 2 + R * 8,
        "bwd_prep": T * h * 2 + 2 * R * h * 2 + R * 12,
        "permute_dy": T * h * 2 + R * h * 2 + R * 12,
        "dg_reduce": R * ((f + 255) // 256) * 4 + R * 8,
        "quant_x_perm": T * h * 2 + R * h + R * 8,
        "permute_quant_x": T * h * 2 + R * h * 2 + R * h + R * 8,
        "quant_h": R * f * 2 + R * f + R * 4,
        "quant_w1": E * h * f * (2 + 1) + E * f * 4,
        "quant_w3": E * h * f * (2 + 1) + E * f * 4,
        "quant_w2": E * h * f * (2 + 1) + E * h * 4,
        "quant_w13_rows": 2 * E * h * f * (2 + 1) + E * h * 4,
        "quant_dAdB": 2 * R * f * 3 + R * 4,
        "transpose_wg": 2 * h * E * 4,
        "token_grad": R * h * 4 + T * h * 2 + E * h * 4 + R * 16 + T * E * 4,
        "router_wgrad": T * h * 2 + T * E * 4 + h * E * 4,
    }
    return {"flops": gemm, "bytes": hbm}
