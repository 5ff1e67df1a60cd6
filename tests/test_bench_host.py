"""Host-side logic of bench.py, checked without a GPU: the FLOP count, the
workload names, the peak table, the summary of the clock samples (throttle
reasons) and the rule that a stored DRAM-traffic figure is reported only
while the kernel source it was measured on is unchanged."""
import hashlib
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_flop_count_is_two_products_per_head(bench):
    """Forward FLOPs: S = Q K^T and O = P V, each S*S*d multiply-adds per
    (batch, head); causal counts half the score matrix.  Counted here by
    walking a tiny problem's multiply-adds."""
    w = bench.Workload("tiny", 2, 3, 5, 4, "bf16", (True,), 1.0, 0)
    madds = 0
    for _ in range(w.B * w.H):
        for _i in range(w.S):
            for _j in range(w.S):
                madds += w.d          # one score
                madds += w.d          # its row of P times V
    assert bench.flops_fwd(w, causal=False) == 2 * madds
    assert bench.flops_fwd(w, causal=True) == madds


def test_workload_config_names_the_mask(bench):
    w = bench.workload("c3")
    assert bench.workload_config(w, True)["workload"].endswith(" causal bf16")
    assert bench.workload_config(w, False)["workload"].endswith(" non-causal bf16")
    assert bench.workload_config(w, False)["causal"] is False


def test_workload_names(bench):
    w = bench.workload("sweep:8192:128")
    assert (w.B, w.H, w.S, w.d, w.dtype) == (1, 16, 8192, 128, "bf16")
    assert bench.workload("sweep:1024:32:fp32").dtype == "fp32"
    c2 = bench.workload("c2")
    assert (c2.B, c2.H, c2.S, c2.d) == (4, 12, 1024, 64)
    with pytest.raises(SystemExit):
        bench.workload("no-such-workload")


def test_peaks_fall_back_without_the_measured_table(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.load_peaks()
    assert pk["source"] == "fallback" and pk["hbm_gbs"] == 6800.0 and pk["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 1950.0}))
    pk = bench.load_peaks()
    assert pk["source"] == "measured" and pk["bf16_tflops_sustained"] == 1950.0


def _row(sm, mx, hw="Not Active", thermal="Not Active", sw_thermal="Not Active", power="Not Active"):
    return ["2026/01/01 00:00:00.000", "0", str(sm), str(mx), "850.0", "0x0", hw, thermal, sw_thermal, power]


def test_clock_summary_median_and_reasons(bench):
    cs = bench.ClockSampler(0)
    cs.rows = [(10.0, _row(1900, 2070)), (10.1, _row(2000, 2070, power="Active")),
               (10.2, _row(2070, 2070)), (50.0, _row(300, 2070, hw="Active"))]   # last one outside the window
    s = cs.summary(10.0, 10.2)
    assert s["sm_mhz"] == 2000.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3
    s = cs.summary(49.9, 50.1)
    assert s["reasons"] == ["hw_slowdown"] and s["sm_mhz"] == 300.0


def test_clock_summary_without_samples(bench):
    cs = bench.ClockSampler(0)
    s = cs.summary(0.0, 1.0)
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["no samples"]
    cs.rows = [(5.0, _row("[N/A]", "[N/A]"))]        # unreadable fields are skipped, not parsed
    s = cs.summary(100.0, 101.0)                     # no row in the window: all rows are used
    assert s["samples"] == 1 and s["sm_mhz"] is None and s["sm_max_mhz"] is None


def test_traffic_used_only_while_the_source_is_unchanged(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("k", "c2") is None                          # no record at all
    src = tmp_path / "kern.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    rec = {"k": {"c2": {"source": "kern.cu", "source_sha256_16": sha, "dram_bytes_per_launch": 1234}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic("k", "c2") == 1234
    assert bench.load_traffic("k", "c3") is None                          # other workload
    assert bench.load_traffic("other", "c2") is None                      # other kernel
    src.write_bytes(b"__global__ void k() { /* changed */ }\n")
    assert bench.load_traffic("k", "c2") is None                          # stale figure dropped


def test_traffic_record_covers_the_included_headers(bench, tmp_path, monkeypatch):
    """A figure is dropped when a header the kernel includes changes, not only its .cu file."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_bytes(b"#include \"h.cuh\"\n")
    (tmp_path / "h.cuh").write_bytes(b"// v1\n")
    (tmp_path / "profiles").mkdir()
    rec = {"k": {"c4": {"sources": ["k.cu", "h.cuh"], "source_sha256_16": bench.sources_sha16(["k.cu", "h.cuh"]),
                        "dram_bytes_per_launch": 99}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic("k", "c4") == 99
    (tmp_path / "h.cuh").write_bytes(b"// v2\n")
    assert bench.load_traffic("k", "c4") is None


def test_committed_traffic_record_is_well_formed():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert rec, "empty traffic record"
    for kern, by_workload in rec.items():
        for wl, ent in by_workload.items():
            for src in ent.get("sources", [ent.get("source")]):
                assert src and os.path.exists(os.path.join(ROOT, src)), (kern, wl)
            assert os.path.exists(os.path.join(ROOT, ent["from"])), (kern, wl)
            assert len(ent["source_sha256_16"]) == 16
            assert isinstance(ent["dram_bytes_per_launch"], int) and ent["dram_bytes_per_launch"] > 0


def test_reference_arm_line(bench, capsys):
    """The reference arm (the oracle on the host cores) prints one line with
    the workload keys both arms share, cpu_baseline = its own value and an
    e2e object with no host-device traffic."""
    import types
    args = types.SimpleNamespace(workload="c1", steps=2, warmup=1, gpus=1)
    assert bench.run_reference(args, 1, 0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = bench.workload("c1")
    for key, val in bench.workload_config(w, True).items():
        assert line["config"][key] == val
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1 and line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert bench.run_reference(args, 2, 1) == 0                      # other ranks: no work, no line
    assert capsys.readouterr().out == ""


def test_backward_rates_name_the_kernel_and_the_whole_backward(bench):
    """The backward's TFLOP/s come from the backward's own event times: one
    figure for the main backward kernel alone, one for the whole backward
    (D preprocess + main kernel + dQ conversion); never from a step time."""
    f_fwd = 1e12
    prof = {"fwd": (4.0, 4), "bwd_preprocess": (0.4, 4), "bwd_main": (8.0, 4), "dq_convert": (0.8, 4),
            "dq_pass": (0.0, 0)}
    r = bench.bwd_rates(f_fwd, prof)
    assert r["bwd_kernel_tflops"] == pytest.approx(2.5 * f_fwd / 2e-3 / 1e12)
    assert r["bwd_step_ms"] == pytest.approx(0.1 + 2.0 + 0.2)
    assert r["bwd_step_tflops"] == pytest.approx(2.5 * f_fwd / 2.3e-3 / 1e12)
    assert r["bwd_step_tflops"] < r["bwd_kernel_tflops"]
    # The deterministic backward has no conversion launch: the step is preprocess + main.
    r = bench.bwd_rates(f_fwd, {"bwd_preprocess": (0.4, 4), "bwd_main": (8.0, 4), "dq_convert": (0.0, 0)})
    assert r["bwd_step_ms"] == pytest.approx(2.1)
    assert bench.bwd_rates(f_fwd, {"bwd_main": (0.0, 0)})["bwd_kernel_tflops"] is None


def test_default_workload_is_the_largest_single_gpu_config(bench, monkeypatch):
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    args = bench.parse()
    w = bench.workload(args.workload)
    assert (w.B, w.H, w.S, w.d, w.qkv_scale) == (4, 32, 4096, 80, 2.0)
    assert [(S, d) for S, d in bench.TARGET_SHAPES] == [(4096, 64), (4096, 128), (8192, 64), (8192, 128)]
