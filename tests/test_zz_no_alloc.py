"""moe_permute_noalloc: dispatch for callers that cannot allocate device
memory (for example inside a runtime that owns a fixed memory budget).  Its
scratch is a fixed array in the library, so the test checks that two calls in
a row -- the second one reusing whatever the first left in that array -- give
exactly the outputs of the regular entry point, which takes a caller
workspace.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import pytest
import torch

from routing_grouped_expert_router_gb300 import binding as mb
from routing_grouped_expert_router_gb300 import build as mbuild
from routing_grouped_expert_router_gb300 import synth
from tests.helpers import small_config

pytestmark = pytest.mark.gpu


def _routing(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    return idx


def _outputs(fn, d, idx, x):
    T, h, E, k = d.T, d.h, d.E, d.k
    R = T * k
    out = dict(counts=torch.full((E,), -1, dtype=torch.int32, device="cuda"),
               offsets=torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
               psrc=torch.full((R,), -1, dtype=torch.int32, device="cuda"),
               pdst=torch.full((R,), -1, dtype=torch.int32, device="cuda"),
               xp=torch.zeros(R, h, dtype=torch.bfloat16, device="cuda"))
    fn(idx, x, out)
    torch.cuda.synchronize()
    return {key: v.cpu() for key, v in out.items()}


@pytest.mark.parametrize("shape", [(1000, 128, 8, 2), (3000, 64, 64, 6)])
def test_noalloc_matches_workspace_entry_point(shape):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    mb.load()
    T, h, E, k = shape
    d = mb.dims(T, h, 128, E, k)
    ws = torch.zeros(mb.moe_workspace_bytes(d, mb.OP_PERMUTE), dtype=torch.uint8, device="cuda")

    def with_ws(idx, x, o):
        mb.moe_permute(d, idx, x, o["counts"], o["offsets"], o["psrc"], o["pdst"], o["xp"], ws)

    def no_alloc(idx, x, o):
        mb.moe_permute_noalloc(d, idx, x, o["counts"], o["offsets"], o["psrc"], o["pdst"],
                               o["xp"])

    cfg = small_config(T=T, h=h, f=128, E=E, k=k, seed=T + E)
    for call in range(2):   # the second call reuses the scratch the first one left
        idx = _routing(T, E, k, seed=17 * call + E).cuda()
        x = synth.normal(cfg.seed + call, 1, (T, h), 1.0, torch.bfloat16, "cuda")
        ref = _outputs(with_ws, d, idx, x)
        got = _outputs(no_alloc, d, idx, x)
        for key in ref:
            assert torch.equal(got[key].view(torch.uint8) if got[key].dtype == torch.bfloat16
                               else got[key],
                               ref[key].view(torch.uint8) if ref[key].dtype == torch.bfloat16
                               else ref[key]), (call, key)
        assert int(got["offsets"][-1]) == T * k


def test_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    lib = mb.load()
    # ceil(T*k/1024) * E = 2049 * 64 > 131072.  Real buffers of the declared
    # sizes (about 8 MB each): were the size check ever to pass, the call
    # would compute on them instead of touching memory it does not own.
    T, E, k = (1 << 18) + 128, 64, 8
    d = mb.dims(T, 64, 64, E, k)
    R = T * k
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.zeros(R, **i32)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    psrc, pdst = torch.empty(R, **i32), torch.empty(R, **i32)
    st = lib.moe_permute_noalloc(ctypes.byref(d), idx.data_ptr(), None, counts.data_ptr(),
                                 offsets.data_ptr(), psrc.data_ptr(), pdst.data_ptr(), None, None)
    torch.cuda.synchronize()
    assert st == mb.MOE_ERR_UNSUPPORTED
