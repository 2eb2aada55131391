"""Host-side arithmetic of bench.py that feeds its JSON line, on CPU.

The roofline's traffic figure is read from the committed ncu summary only
while that summary was taken on the current kernel sources; the theoretical
peak is SMs x SM clock x 8192 FLOP per clock and SM (the dense fp16 / bf16
tensor rate); the CPU baseline is the oracle on a bounded sample.  None of
these touch a GPU.
"""
import importlib.util
import json
import os
import types

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_host_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_kernel_sha_depends_on_every_profiled_source(tmp_path, monkeypatch):
    bench = _bench()
    csrc = tmp_path / "attention_forward_fwd_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        (csrc / name).write_text("// " + name + "\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench._kernel_sha()
    assert len(base) == 16 and int(base, 16) >= 0
    for name in bench.KERNEL_SOURCES:
        p = csrc / name
        old = p.read_text()
        p.write_text(old + "// changed\n")
        assert bench._kernel_sha() != base, name
        p.write_text(old)
        assert bench._kernel_sha() == base


def test_traffic_is_reported_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    bench = _bench()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({
        "w": {"kernel_sha": "aaaa", "dram_bytes_per_launch": 123.0},
    }))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "_kernel_sha", lambda: "aaaa")
    assert bench._traffic("w") == 123.0
    assert bench._traffic("other") is None
    monkeypatch.setattr(bench, "_kernel_sha", lambda: "bbbb")
    assert bench._traffic("w") is None


def test_traffic_without_a_summary_is_none(tmp_path, monkeypatch):
    bench = _bench()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("s4096") is None


def test_committed_traffic_entries_name_existing_summaries():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    assert d
    for name, entry in d.items():
        assert entry["dram_bytes_per_launch"] > 0, name
        assert len(entry["kernel_sha"]) == 16, name
        assert os.path.exists(os.path.join(ROOT, entry["source"])), (name, entry["source"])


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    bench = _bench()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    burst, sustained, kind = bench._peaks()
    assert (burst, sustained, kind) == (1900.0, 1700.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1750.5,
                                                               "bf16_tflops_sustained": 1600.25}))
    assert bench._peaks() == (1750.5, 1600.25, "measured")


def test_theoretical_peak_arithmetic(monkeypatch):
    bench = _bench()
    import torch
    monkeypatch.setattr(torch.cuda, "get_device_properties",
                        lambda dev: types.SimpleNamespace(multi_processor_count=152))
    out = bench._theoretical(1000.0, {"sm_max_mhz": 2000, "sm_mhz": 1000}, 0)
    # 152 SMs x 2.0e9 clk/s x 8192 FLOP/clk = 2490.368 TFLOP/s
    assert out["sms"] == 152 and out["flop_per_clk_per_sm"] == 8192
    assert out["at_max_clock"]["tflops"] == pytest.approx(2490.368)
    assert out["at_max_clock"]["pct"] == pytest.approx(100.0 * 1000.0 / 2490.368)
    assert out["at_sampled_clock"]["tflops"] == pytest.approx(1245.184)
    assert bench._theoretical(1.0, {"sm_max_mhz": None, "sm_mhz": 0}, 0)["at_max_clock"] is None


def test_cpu_baseline_takes_at_least_one_row_block():
    bench = _bench()
    w = bench.fa_inputs.WORKLOADS["s256"]
    out = bench.cpu_baseline(w, budget_s=0.0)
    assert out["kind"] == "oracle" and out["unit"] == "TFLOP/s"
    assert out["value"] > 0 and out["cores"] >= 1
    assert out["sample"].startswith("1 row blocks of s256")


@pytest.mark.parametrize("S", [1, 7, 256, 1999, 8192])
@pytest.mark.parametrize("causal", [False, True])
def test_cpu_baseline_row_blocks_cover_each_row_once_and_sum_to_the_convention(S, causal):
    """The row blocks of a head partition its rows, and their counted FLOPs
    add up to the convention for the whole head (4 S^2 D, half causal)."""
    bench = _bench()
    blocks, _ = bench._row_blocks(S)
    rows = np.sort(np.concatenate(blocks))
    assert np.array_equal(rows, np.arange(S))
    total = sum(bench._row_flops(r, S, 64, causal) for r in blocks)
    assert total == pytest.approx(bench.fa_inputs.attention_flops(1, 1, S, 64, causal), rel=1e-12)


def test_one_thread_oracle_sample_and_cpu_model():
    bench = _bench()
    assert bench._cpu_model()
    out = bench.cpu_baseline_one_thread("s256", budget_s=0.05)
    assert "error" not in out, out
    assert out["cores"] == 1 and out["kind"] == "oracle" and out["value"] > 0
    assert "BLAS threads = 1" in out["sample"]
