"""Runs the CUDA layer through the C ABI on torch-allocated device memory."""
from __future__ import annotations

import torch

from routing_grouped_expert_router_gb300 import binding as mb

SAVED_TENSORS = {
    # name: (dtype, shape(cfg))
    "topk_idx": (torch.int32, lambda d: (d.T, d.k)),
    "gates": (torch.float32, lambda d: (d.T, d.k)),
    "counts": (torch.int32, lambda d: (d.E,)),
    "offsets": (torch.int32, lambda d: (d.E + 1,)),
    "perm_src": (torch.int32, lambda d: (d.T * d.k,)),
    "perm_dst": (torch.int32, lambda d: (d.T * d.k,)),
    "x_perm": (torch.bfloat16, lambda d: (d.T * d.k, d.h)),
    "A": (torch.bfloat16, lambda d: (d.T * d.k, d.f)),
    "B": (torch.bfloat16, lambda d: (d.T * d.k, d.f)),
    "H": (torch.bfloat16, lambda d: (d.T * d.k, d.f)),
    "O": (torch.bfloat16, lambda d: (d.T * d.k, d.h)),
}


# activations a sar context does not keep
SAR_DROPPED = ("x_perm", "H", "O")


def saved_tensor(d, saved: torch.Tensor, name: str) -> torch.Tensor:
    dtype, shp = SAVED_TENSORS[name]
    shape = shp(d)
    off = mb.moe_saved_view(d, saved, name) - saved.data_ptr()
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    return saved[off:off + nbytes].view(dtype).view(shape)


def workspace(d, op, device="cuda") -> torch.Tensor:
    return torch.zeros(max(mb.moe_workspace_bytes(d, op), 256), dtype=torch.uint8, device=device)


class LayerRun:
    """Buffers and calls for one layer shape on one device."""

    def __init__(self, d, device="cuda"):
        self.d = d
        self.device = device
        T, h, f, E = d.T, d.h, d.f, d.E
        self.saved = torch.zeros(max(mb.moe_saved_bytes(d), 256), dtype=torch.uint8, device=device)
        self.ws_f = workspace(d, mb.OP_LAYER_FWD, device)
        self.ws_b = workspace(d, mb.OP_LAYER_BWD, device)
        self.y = torch.empty(T, h, dtype=torch.bfloat16, device=device)
        self.dx = torch.empty(T, h, dtype=torch.bfloat16, device=device)
        self.dWg = torch.empty(h, E, dtype=torch.float32, device=device)
        self.dW1 = torch.empty(E, h, f, dtype=torch.float32, device=device)
        self.dW3 = torch.empty(E, h, f, dtype=torch.float32, device=device)
        self.dW2 = torch.empty(E, f, h, dtype=torch.float32, device=device)

    def fwd(self, inp, stream=None):
        mb.moe_layer_fwd(self.d, inp["x"], inp["Wg"], inp["b"] if self.d.has_bias else None,
                         inp["W1"], inp["W3"], inp["W2"], self.y, self.saved, self.ws_f,
                         stream=stream)

    def bwd(self, inp, stream=None):
        mb.moe_layer_bwd(self.d, inp["x"], inp["dy"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"],
                         self.saved, self.dx, self.dWg, self.dW1, self.dW3, self.dW2, self.ws_b,
                         stream=stream)

    def status(self) -> int:
        return max(mb.moe_read_device_status(self.ws_f), mb.moe_read_device_status(self.ws_b))

    def saved_view(self, name):
        return saved_tensor(self.d, self.saved, name)

    def outputs(self) -> dict:
        kept = [n for n in SAVED_TENSORS if not (self.d.sar and n in SAR_DROPPED)]
        out = {n: self.saved_view(n).detach().cpu().clone() for n in kept}
        for n in ("y", "dx", "dWg", "dW1", "dW3", "dW2"):
            out[n] = getattr(self, n).detach().cpu().clone()
        return out
