"""Shared test helpers: conditioned synthetic inputs and comparison metrics."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from routing_grouped_expert_router_gb300 import synth
from routing_grouped_expert_router_gb300.configs import LayerConfig


def small_config(name="small", T=48, h=16, f=32, E=4, k=2, seed=11, zipf_s=0.0):
    return LayerConfig(name, T=T, h=h, f=f, E=E, k=k, seed=seed, zipf_s=zipf_s)


def scaled(cfg: LayerConfig, **kw) -> LayerConfig:
    return dataclasses.replace(cfg, **kw)


def conditioned_inputs(cfg: LayerConfig, device="cpu", margin=1e-3):
    """synth inputs with x rows resampled until every router margin >= margin.

    Conditioning runs on the CPU; tensors are then moved to `device`.
    """
    inp = synth.make_layer(cfg, "cpu")

    def fresh(row_ids, attempt):
        return synth.replacement_x_rows(cfg, row_ids, attempt)

    x, n = oracle.condition_router_margins(inp["x"], inp["Wg"], inp["b"], cfg.k,
                                           fresh, margin=margin)
    inp["x"] = x
    inp["n_resampled"] = n
    if device != "cpu":
        for key, v in list(inp.items()):
            if isinstance(v, torch.Tensor):
                inp[key] = v.to(device)
    return inp


def rel_l2(a, b) -> float:
    """||a - b||_2 / ||b||_2 in float64; inf if ||b|| = 0 and a != 0."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b.ravel())
    d = np.linalg.norm((a - b).ravel())
    if nb == 0.0:
        return 0.0 if d == 0.0 else float("inf")
    return float(d / nb)
