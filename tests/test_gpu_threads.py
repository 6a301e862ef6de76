"""Two host threads drive two layers at once, each on its own CUDA stream, and
both match the oracle.  The library's per-launch settings (shared-memory
attributes, the co-resident cluster count of the persistent CTA-pair grid, the
SM count) are kept per kernel and device behind a lock, so concurrent first
calls from several threads set them once and correctly."""
import threading

import numpy as np
import pytest
import torch

import oracle.cref as ref
from routing_grouped_expert_router_gb300 import binding as mb
from routing_grouped_expert_router_gb300 import build as mbuild
from tests.gpu_runner import LayerRun
from tests.helpers import conditioned_inputs, rel_l2, small_config

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


def test_two_layers_from_two_threads_on_two_streams():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mbuild.build()
    mb.load()
    cases = [small_config(name="t0", T=1024, h=256, f=512, E=8, k=2, seed=31),
             small_config(name="t1", T=700, h=192, f=320, E=32, k=3, seed=32)]
    inputs = [conditioned_inputs(c) for c in cases]
    runs = [LayerRun(mb.dims_of(c, has_bias=False)) for c in cases]
    devs = [{n: v.cuda() for n, v in i.items() if isinstance(v, torch.Tensor)} for i in inputs]
    torch.cuda.synchronize()
    start = threading.Barrier(2)
    errors = []

    def work(i):
        try:
            stream = torch.cuda.Stream()
            start.wait()
            for _ in range(3):
                runs[i].fwd(devs[i], stream=stream.cuda_stream)
                runs[i].bwd(devs[i], stream=stream.cuda_stream)
            stream.synchronize()
        except Exception as exc:  # reported on the main thread
            errors.append(exc)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for c, inp, run in zip(cases, inputs, runs):
        assert run.status() == mb.MOE_OK
        y, ctx = ref.layer_fwd(inp["x"], inp["Wg"], None, inp["W1"], inp["W3"], inp["W2"], c.k)
        g = ref.layer_bwd(inp["dy"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ctx)
        out = run.outputs()
        np.testing.assert_array_equal(out["topk_idx"].numpy(), ctx["topk_idx"])
        assert rel_l2(out["y"].double().numpy(), y) <= 5e-3
        assert rel_l2(out["dx"].double().numpy(), g["dx"]) <= 5e-3
        for key in ("dW1", "dW3", "dW2", "dWg"):
            assert rel_l2(out[key].numpy(), g[key]) <= 1e-2, key
