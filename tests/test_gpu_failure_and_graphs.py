"""Device failure reporting and graph capture (GPU).

* The bounded-wait path: moe_selftest_wait_timeout makes one mbarrier wait
  that nothing can complete run out (a 20 ms limit); the kernel records
  MOE_ERR_DEVICE_TIMEOUT in the workspace status word and returns.  The host
  reads the status, and the same context then runs a layer correctly.  Nothing
  faults, traps or hangs.
* A launch failure injected on the host (moe_test_fail_launch_after) makes the
  entry point that hit it return MOE_ERR_CUDA at that launch, wherever it falls
  in the forward or the backward; the next layer on the same context runs
  clean and matches the oracle.
* The layer is a fixed sequence of launches with no host synchronisation or
  allocation, so moe_layer_fwd + moe_layer_bwd capture into a CUDA graph; the
  replay gives bitwise the eager results.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import oracle.cref as ref
from routing_grouped_expert_router_gb300 import binding as mb
from routing_grouped_expert_router_gb300 import build as mbuild
from tests.gpu_runner import LayerRun, workspace
from tests.helpers import conditioned_inputs, rel_l2, small_config

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    return mb.load()


def _inputs():
    cfg = small_config(name="g", T=512, h=256, f=384, E=8, k=2, seed=31)
    inp = conditioned_inputs(cfg)
    return cfg, inp, {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def test_bounded_wait_reports_timeout_and_context_survives(lib):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    mb.moe_selftest_wait_timeout(ws, 20000)
    assert mb.moe_read_device_status(ws) == mb.MOE_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert mb.moe_read_device_status(ws) == mb.MOE_OK        # reading cleared it
    # the context is intact: a layer runs and matches the oracle
    cfg, inp, dev = _inputs()
    y_ref, ctx = ref.layer_fwd(inp["x"], inp["Wg"], inp["b"], inp["W1"], inp["W3"],
                                  inp["W2"], cfg.k)
    run = LayerRun(mb.dims_of(cfg, has_bias=False))
    run.fwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    assert rel_l2(run.y.double().cpu().numpy(), y_ref) <= 5e-3


def test_layer_captures_into_a_cuda_graph(lib):
    cfg, inp, dev = _inputs()
    d = mb.dims_of(cfg, has_bias=False)
    eager = LayerRun(d)
    eager.fwd(dev)
    eager.bwd(dev)
    torch.cuda.synchronize()
    ref = eager.outputs()

    run = LayerRun(d)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):          # warm-up on the capture stream
        run.fwd(dev)
        run.bwd(dev)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for t in (run.y, run.dx, run.dW1, run.dWg):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    k0 = mb.moe_kernel_launches()
    with torch.cuda.graph(g):
        run.fwd(dev)
        run.bwd(dev)
    captured = mb.moe_kernel_launches() - k0
    assert captured >= 15
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    out = run.outputs()
    for key in ref:
        a, b = out[key], ref[key]
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b), key


@pytest.mark.parametrize("n", [1, 4, 8, 12, 17])
def test_injected_launch_failure_is_reported_and_the_context_recovers(lib, n):
    cfg, inp, dev = _inputs()
    d = mb.dims_of(cfg, has_bias=False)
    run = LayerRun(d)
    before = mb.moe_kernel_launches()
    mb.moe_test_fail_launch_after(n)
    with pytest.raises(mb.MoeError) as err:
        run.fwd(dev)
        run.bwd(dev)
    assert err.value.status == mb.MOE_ERR_CUDA
    assert mb.moe_kernel_launches() - before == n  # nothing launched after the failure
    torch.cuda.synchronize()
    run.fwd(dev)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
    y, ctx = ref.layer_fwd(inp["x"], inp["Wg"], None, inp["W1"], inp["W3"], inp["W2"], cfg.k)
    g = ref.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
    out = run.outputs()
    assert rel_l2(out["y"].double().numpy(), y) <= 5e-3
    assert rel_l2(out["dx"].double().numpy(), g["dx"]) <= 5e-3
    assert rel_l2(out["dW1"].numpy(), g["dW1"]) <= 1e-2


def test_cleared_injection_does_not_fire(lib):
    cfg, inp, dev = _inputs()
    run = LayerRun(mb.dims_of(cfg, has_bias=False))
    mb.moe_test_fail_launch_after(3)
    mb.moe_test_fail_launch_after(0)
    run.fwd(dev)
    run.bwd(dev)
    torch.cuda.synchronize()
    assert run.status() == mb.MOE_OK
