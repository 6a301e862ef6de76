"""Device-side index checks: an expert id, permutation entry or expert offset
that is out of range, written into an input from the host, is reported as
MOE_ERR_DEVICE_INDEX through the status word and the element is skipped; the
rest of the output is what the oracle gives for the valid elements alone.

The corrupted values only make the kernels take their error branch: every
kernel that reads such an index checks it before any access that depends on
it, so nothing here reads or writes out of bounds."""
import numpy as np
import pytest
import torch

import oracle.cref as ref
from routing_grouped_expert_router_gb300 import binding as mb
from routing_grouped_expert_router_gb300 import build as mbuild
from routing_grouped_expert_router_gb300 import synth
from tests.gpu_runner import LayerRun, workspace
from tests.helpers import conditioned_inputs, rel_l2, small_config

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    return mb.load()


def _routing(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)


def test_permute_reports_bad_expert_ids(lib):
    T, h, E, k = 3000, 128, 16, 2
    d = mb.dims(T, h, 128, E, k)
    idx = _routing(T, E, k, 5)
    bad = torch.tensor([7, 1500, 2999 * k + 1])
    flat = idx.view(-1).clone()
    flat[bad] = torch.tensor([E, -1, E + 1000], dtype=torch.int32)
    idx_bad = flat.view(T, k)
    x = synth.normal(3, 1, (T, h), 1.0, torch.bfloat16)
    i32 = dict(dtype=torch.int32, device="cuda")
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    psrc, pdst = torch.empty(T * k, **i32), torch.empty(T * k, **i32)
    xp = torch.zeros(T * k, h, dtype=torch.bfloat16, device="cuda")
    ws = workspace(d, mb.OP_PERMUTE)
    mb.moe_permute(d, idx_bad.cuda(), x.cuda(), counts, offsets, psrc, pdst, xp, ws)
    assert mb.moe_read_device_status(ws) == mb.MOE_ERR_DEVICE_INDEX
    assert mb.moe_read_device_status(ws) == mb.MOE_OK          # reading clears it
    keep = np.ones(T * k, bool)
    keep[bad.numpy()] = False
    fixed = flat.clone()
    fixed[bad] = 0
    c, o, s, p = ref.dispatch(fixed.view(T, k), E, keep=keep.reshape(T, k))
    n = int(o[-1])
    assert n == T * k - len(bad)
    np.testing.assert_array_equal(counts.cpu().numpy(), c)
    np.testing.assert_array_equal(offsets.cpu().numpy(), o)
    np.testing.assert_array_equal(psrc.cpu().numpy()[:n], s)
    np.testing.assert_array_equal(pdst.cpu().numpy(), p)
    np.testing.assert_array_equal(xp[:n].cpu().float().numpy(), ref.permute_rows(x, s, k))
    # the same call on clean ids leaves the status at OK
    mb.moe_permute(d, idx.cuda(), x.cuda(), counts, offsets, psrc, pdst, xp, ws)
    assert mb.moe_read_device_status(ws) == mb.MOE_OK


def test_combine_and_unpermute_report_rows_past_the_end(lib):
    T, h, k = 500, 256, 3
    R = T * k
    d = mb.dims(T, h, 128, 8, k)
    O = synth.normal(9, 1, (R, h), 1.0, torch.bfloat16)
    gates = torch.rand(T, k, generator=torch.Generator().manual_seed(2))
    pdst = torch.randperm(R, generator=torch.Generator().manual_seed(3)).to(torch.int32)
    pdst[[4, 700]] = torch.tensor([R, R + 12345], dtype=torch.int32)
    mb.moe_clear_device_status(None)
    y = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    mb.moe_combine(d, O.cuda(), gates.cuda(), pdst.cuda(), y)
    assert mb.moe_read_device_status(None) == mb.MOE_ERR_DEVICE_INDEX
    keep = (pdst >= 0) & (pdst < R)
    p_ok = torch.where(keep, pdst, torch.full_like(pdst, -1))
    y_ref = ref.combine(O, gates.numpy(), p_ok.numpy(), T, k)
    assert rel_l2(y.cpu().double().numpy(), y_ref) <= 3e-3
    back = torch.full((R, h), 7.0, dtype=torch.bfloat16, device="cuda")
    mb.moe_unpermute(d, pdst.cuda(), O.cuda(), back)
    assert mb.moe_read_device_status(None) == mb.MOE_ERR_DEVICE_INDEX
    want = ref.unpermute_rows(O.float().numpy(), p_ok.numpy())
    np.testing.assert_array_equal(back.cpu().float().numpy(), want)
    assert mb.moe_read_device_status(None) == mb.MOE_OK


def test_expert_ffn_reports_bad_offsets(lib):
    cfg = small_config(name="off", T=256, h=128, f=256, E=4, k=2, seed=3)
    inp = conditioned_inputs(cfg)
    _, ctx = ref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], cfg.k)
    d = mb.dims_of(cfg, has_bias=False)
    R = cfg.T * cfg.k
    dev = {n: v.cuda() for n, v in inp.items() if isinstance(v, torch.Tensor)}
    psrc = torch.from_numpy(ctx["perm_src"]).cuda()
    A = torch.empty(R, cfg.f, dtype=torch.bfloat16, device="cuda")
    B, H = torch.empty_like(A), torch.empty_like(A)
    O = torch.empty(R, cfg.h, dtype=torch.bfloat16, device="cuda")
    for off in ([0, 300, 200, 400, R], [0, 100, 200, 300, R + 1], [5, 100, 200, 300, R]):
        ws = workspace(d, mb.OP_EXPERT_FFN_FWD)
        offs = torch.tensor(off, dtype=torch.int32, device="cuda")
        mb.moe_expert_ffn_fwd(d, dev["x"], psrc, offs, dev["W1"], dev["W3"], dev["W2"], A, B, H,
                              O, ws)
        assert mb.moe_read_device_status(ws) == mb.MOE_ERR_DEVICE_INDEX, off
    ws = workspace(d, mb.OP_EXPERT_FFN_FWD)
    mb.moe_expert_ffn_fwd(d, dev["x"], psrc, torch.from_numpy(ctx["offsets"]).cuda(), dev["W1"],
                          dev["W3"], dev["W2"], A, B, H, O, ws)
    assert mb.moe_read_device_status(ws) == mb.MOE_OK
    assert rel_l2(O.cpu().double().numpy(), ctx["O"]) <= 5e-3


def test_router_bwd_reports_bad_expert_ids(lib):
    cfg = small_config(name="rb", T=300, h=128, f=128, E=6, k=2, seed=4)
    inp = conditioned_inputs(cfg)
    _, ctx = ref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"], inp["W2"], cfg.k)
    g = ref.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    d = mb.dims_of(cfg, has_bias=False)
    T, h, E, k = cfg.T, cfg.h, cfg.E, cfg.k
    idx = torch.from_numpy(ctx["topk_idx"].copy())
    idx[11, 1] = E + 3
    dx = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dWg = torch.empty(h, E, dtype=torch.float32, device="cuda")
    ws = workspace(d, mb.OP_ROUTER_BWD)
    mb.moe_router_bwd(d, inp["x"].cuda(), inp["Wg"].cuda(), idx.cuda(),
                      torch.from_numpy(ctx["gates"]).cuda(),
                      torch.from_numpy(g["dg"].ravel()).float().cuda(),
                      torch.from_numpy(g["dX_perm"]).float().cuda(),
                      torch.from_numpy(ctx["perm_src"]).cuda(),
                      torch.from_numpy(ctx["perm_dst"]).cuda(),
                      torch.from_numpy(ctx["offsets"]).cuda(), dx, dWg, ws)
    assert mb.moe_read_device_status(ws) == mb.MOE_ERR_DEVICE_INDEX
    # every other token's gradient is untouched by the bad entry
    others = np.ones(T, bool)
    others[11] = False
    assert rel_l2(dx.cpu().double().numpy()[others], g["dx"][others]) <= 5e-3


def test_clean_layer_leaves_status_ok(lib):
    cfg = small_config(name="clean", T=512, h=256, f=256, E=8, k=2, seed=6)
    inp = {n: v.cuda() for n, v in conditioned_inputs(cfg).items() if isinstance(v, torch.Tensor)}
    run = LayerRun(mb.dims_of(cfg, has_bias=False))
    run.fwd(inp)
    run.bwd(inp)
    assert run.status() == mb.MOE_OK
    assert mb.moe_read_device_status(None) == mb.MOE_OK
