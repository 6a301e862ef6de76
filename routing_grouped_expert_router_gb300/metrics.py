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
