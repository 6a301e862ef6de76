"""The five synthetic MoE-layer workloads.

Shapes follow the model table of the MegaScale-MoE paper review (xllm-io,
"五、实验结果 / 基准测试配置": hidden size h, expert width h_ffn, expert
count and top-k per model).  Tokens are flat: the layer sees b*s tokens as T
rows (the pages' "bsh" activation, MegaScale-MoE digest §3.2).

Every layer is a dropless top-k MoE with SwiGLU experts:
  W1, W3 : [E, h, f]   (fan_in h)      W2 : [E, f, h]   (fan_in f)
  Wg     : [h, E] fp32 router weight   b  : [E] fp32 fixed router bias
"""
from __future__ import annotations

from dataclasses import dataclass, asdict


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int          # tokens
    h: int          # hidden size
    f: int          # expert FFN width (h_ffn)
    E: int          # experts
    k: int          # experts per token
    seed: int
    zipf_s: float = 0.0   # >0: router bias skews expert load to Zipf(s)
    source: str = ""

    @property
    def rows(self) -> int:
        """Permuted rows = token-expert assignments (dropless: T*k)."""
        return self.T * self.k

    def gemm_macs_fwd(self) -> int:
        """Forward expert multiply-adds: 3*k*T*h*f (MegaScale-MoE review,
        核心公式, comp_time numerator at n = 1)."""
        return 3 * self.k * self.T * self.h * self.f

    def gemm_flops_fwd_bwd(self) -> int:
        """Useful GroupedGEMM FLOPs of forward + backward: 2 * 3 MACs-units
        (fwd 3, dgrad 3, wgrad 3 matmul passes per assignment) = 18*k*T*h*f."""
        return 2 * 3 * self.gemm_macs_fwd()

    def as_dict(self) -> dict:
        return asdict(self)


CONFIGS = {
    "tiny": LayerConfig("tiny", T=256, h=128, f=256, E=8, k=2, seed=0,
                        source="small case"),
    "deepseekmoe": LayerConfig("deepseekmoe", T=8192, h=2048, f=1408, E=64, k=6,
                               seed=1, source="DeepSeekMoE row of the model table"),
    "mixtral8x7b": LayerConfig("mixtral8x7b", T=16384, h=4096, f=14336, E=8, k=2,
                               seed=2, source="Mixtral-8x7B row of the model table"),
    "internal352b": LayerConfig("internal352b", T=16384, h=4096, f=14336, E=32, k=3,
                                seed=3, zipf_s=1.2,
                                source="Internal-352B row of the model table, skewed load"),
    "hunyuan": LayerConfig("hunyuan", T=32768, h=6400, f=18304, E=16, k=1, seed=4,
                           source="Hunyuan-Large row of the model table"),
}

# The layer whose throughput is the headline: the Mixtral-8x7B-shaped layer.
BENCH_CONFIG = "mixtral8x7b"


def get(name: str) -> LayerConfig:
    try:
        return CONFIGS[name]
    except KeyError:
        raise KeyError(f"unknown layer config {name!r}; known: {sorted(CONFIGS)}")
