"""Host-side benchmark logic on CPU: the one-GPU refusal, the JSON-facing
helpers and the compact summary that closes the bench line."""
import json

import pytest

import bench
import workloads


def test_more_than_one_gpu_is_refused():
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "2"])
    assert e.value.code != 0


def test_multi_process_launch_is_refused(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit) as e:
        bench.main(["--impl", "reference"])
    assert e.value.code != 0


def test_rate_units():
    assert bench._rate(2e12, 1000.0, "TFLOP/s") == pytest.approx(2.0)
    assert bench._rate(5e9, 1.0, "GB/s") == pytest.approx(5000.0)


def test_visible_pair_counts():
    assert workloads.visible_pairs(4, 4, False) == 16
    assert workloads.visible_pairs(4, 4, True) == 10
    assert workloads.visible_pairs(2, 5, True) == 4 + 5  # bottom-right alignment
    assert workloads.visible_pairs(5, 2, True) == 0 + 0 + 0 + 1 + 2
    assert workloads.C2_CAUSAL.flops() == pytest.approx(4 * 4 * 32 * 128 * 4096 * 4097 / 2)


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["0, 1800, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 1900, 2070, 950.1, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_mhz"] == 1850 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def _fake_result(unit, bound):
    roof = {"bound": bound, "frac": 0.5, "achieved": 1.0, "peak": 2.0}
    if bound == "tensor":
        roof["tensor_pipe_active"] = 0.6
    return {"value": 1234.56789, "unit": unit, "ms_per_step": 0.3391, "roofline": roof,
            "e2e": {"value": 99.99}, "clocks": {"sm_mhz": 2070.0, "reasons": []}}


def test_summary_lists_the_five_configs_last_and_stays_short():
    results = {}
    for name, label in bench.SUMMARY_ORDER:
        unit, bound = ("GB/s", "hbm") if name.startswith("decode") else ("TFLOP/s", "tensor")
        results[name] = (_fake_result(unit, bound), {"value": 0.0612345, "cores": 16})
    summary = {label: bench._summary_entry(*results[name]) for name, label in bench.SUMMARY_ORDER}
    assert list(summary)[-4:] == ["C2", "C3", "C4", "C5"]
    assert summary["C3"]["tensor_pipe_active"] == 0.6
    assert "tensor_pipe_active" not in summary["C4"]
    assert summary["C5"]["cpu_baseline"] == {"value": 0.06123, "cores": 16}
    # The three configurations that close the line fit well inside 1500 bytes.
    tail = json.dumps({k: summary[k] for k in ("C3", "C4", "C5")})
    assert len(tail) < 900


def test_ncu_record_is_dropped_when_the_kernel_source_changed(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    csrc = tmp_path / "attention_flash_attn_fwd_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"w": {"kernel": "k", "bytes_per_launch": 10, "tensor_pipe_active": 0.5,
                 "source_hash": bench._source_hash("k.cu")}}
    (prof / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench._ncu_record("w", "k", ["k.cu"])["tensor_pipe_active"] == 0.5
    assert bench._ncu_record("w", "other", ["k.cu"]) == {}
    (csrc / "k.cu").write_text("kernel v2")
    assert bench._ncu_record("w", "k", ["k.cu"]) == {}
