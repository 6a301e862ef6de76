"""The benchmark's roofline bookkeeping on CPU: the DRAM traffic it reports
per GroupedGEMM comes from the committed one-pass ncu summary
(profiles/dram_traffic_gemms.json), only for the workload and the GEMM sources
that summary was captured from; each figure is the captured launch's bytes
times the summary's stated scale, and at least about the matmul's algorithmic
bytes (every operand read once and every output written once)."""
import json

import pytest

import bench
from routing_grouped_expert_router_gb300.configs import CONFIGS

GEMMS = ("gg_fc1_fwd_swiglu", "gg_fc2_fwd", "gg_fc2_dgrad_swiglu_bwd", "gg_fc2_wgrad",
         "gg_fc1_dgrad", "gg_fc1_wgrad")


def _recorded():
    with open(bench.TRAFFIC_PROFILE) as f:
        return json.load(f)


def _algorithmic_bytes(cfg):
    """Operands read once and outputs written once, per launch (bf16 = 2 bytes,
    the fp32 data and weight gradients 4)."""
    R, h, f, E = cfg.T * cfg.k, cfg.h, cfg.f, cfg.E
    x, hf, w = R * h * 2, R * f * 2, E * h * f * 2
    return {
        "gg_fc1_fwd_swiglu": x + 2 * w + 3 * hf,          # x_perm, W1|W3 -> A, B, H
        "gg_fc2_fwd": hf + w + x,                          # H, W2 -> O
        "gg_fc2_dgrad_swiglu_bwd": x + w + 2 * hf + 2 * hf,  # dO, W2, A, B -> dA, dB
        "gg_fc2_wgrad": hf + x + 2 * w,                    # H, dO -> dW2 (fp32)
        "gg_fc1_dgrad": 2 * hf + 2 * w + 2 * x,            # dA|dB, W1|W3 -> dX_perm (fp32)
        "gg_fc1_wgrad": x + 2 * hf + 4 * w,                # x_perm, dA|dB -> dW1|dW3 (fp32)
    }


def test_summary_is_for_the_bench_workload():
    rec = _recorded()
    assert rec["workload"] == bench.workload_desc(CONFIGS["mixtral8x7b"])
    assert set(GEMMS) <= set(rec["kernels"])


def test_traffic_is_the_capture_scaled(monkeypatch):
    rec = _recorded()
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: rec["source_sha256"])
    cfg = CONFIGS["mixtral8x7b"]
    alg = _algorithmic_bytes(cfg)
    for name in GEMMS:
        ent = rec["kernels"][name]
        t = bench.measured_traffic(name, bench.workload_desc(cfg))
        assert t == pytest.approx(rec["scale"] * (ent["captured_read_bytes"]
                                                  + ent["captured_write_bytes"]))
        # part of a kernel's output can still sit in L2 when it ends
        assert 0.95 * alg[name] <= t <= 5.0 * alg[name], name


def test_traffic_withheld_for_changed_sources_or_other_workloads(monkeypatch):
    rec = _recorded()
    cfg = CONFIGS["mixtral8x7b"]
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 64)
    assert bench.measured_traffic("gg_fc1_wgrad", bench.workload_desc(cfg)) is None
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: rec["source_sha256"])
    assert bench.measured_traffic("gg_fc1_wgrad", bench.workload_desc(CONFIGS["hunyuan"])) is None
    assert bench.measured_traffic("no_such_kernel", bench.workload_desc(cfg)) is None


def test_source_hash_covers_the_gemm_sources(tmp_path, monkeypatch):
    """Any edit to a GEMM source changes the hash (and so withholds the traffic)."""
    h0 = bench.gemm_source_hash()
    import shutil
    src = tmp_path / "routing_grouped_expert_router_gb300" / "csrc"
    src.mkdir(parents=True)
    for name in bench.GEMM_SOURCES:
        shutil.copy(f"{bench.ROOT}/routing_grouped_expert_router_gb300/csrc/{name}", src / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.gemm_source_hash() == h0
    with open(src / bench.GEMM_SOURCES[0], "a") as f:
        f.write("\n// edited\n")
    assert bench.gemm_source_hash() != h0


@pytest.mark.parametrize("tokens,ranks,steps,ms", [(16384, 1, 30, 672.0), (16384, 8, 5, 120.0)])
def test_job_throughput_counts_every_rank(tokens, ranks, steps, ms):
    assert bench.job_tokens_per_s(tokens, ranks, steps, ms) == pytest.approx(
        tokens * ranks * steps / (ms / 1e3))


def test_oracle_leg_times_a_calibrated_sample():
    """The CPU legs time the C++ oracle on a sample sized by a calibration run."""
    import dataclasses
    cfg = dataclasses.replace(CONFIGS["tiny"], T=64)
    tps, n, dt, threads = bench.time_oracle(cfg, 0.05, 2, 1)
    assert 8 <= n <= 64 and dt > 0 and threads >= 1
    assert tps == pytest.approx(n * 2 / dt)
