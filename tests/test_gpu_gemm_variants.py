"""Both GroupedGEMM kernels (one CTA per tile, and the CTA pair with
tcgen05 cta_group::2), and both tile orders, against the oracle for all six
expert matmuls.

The library picks one kernel and one tile order per matmul; MOE_GEMM_CTAS
forces one kind of kernel for every matmul, and MOE_GEMM_RASTER one order and
group size (small groups, so that every expert's tile grid splits into several
groups with a ragged last one).  The choice is read once per process, so each
setting runs the layer parity cases in a fresh interpreter."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ctas,raster", [("1", ""), ("2", ""), ("1", "m3"), ("1", "n3"),
                                          ("2", "n2"), ("2", "m1")])
def test_layer_parity_with_each_gemm_kernel(ctas, raster):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MOE_GEMM_CTAS=ctas)
    if raster:
        env["MOE_GEMM_RASTER"] = raster
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "-q", "-x", "-p",
         "no:cacheprovider", "-k", "layer_matches_oracle or stage_entry or one_expert"],
        env=env, cwd=ROOT, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
