"""Host-side logic of bench.py that needs no GPU: workload specs, the names the
traffic figures are keyed by, launch counts, and the CPU-oracle baseline legs
on tiny layers."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _spec(monkeypatch, *argv):
    monkeypatch.setattr(sys, "argv", ["bench.py", *argv])
    args = bench.parse_args()
    if args.workload == "prefill" and args.m == 1:
        args.m = 2048                                   # as main() does
    return args, bench.workload_spec(args)


def test_default_line_is_the_dense_mlp_with_its_traffic_figure(monkeypatch):
    args, spec = _spec(monkeypatch)
    assert spec["kind"] == "mlp" and args.m == 1 and args.gpus == 1
    assert bench.GEMV_TRAFFIC_BYTES.get(spec["name"]) is not None


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill_traffic_figures_are_keyed_by_the_workload_names(monkeypatch, fp8):
    _, spec = _spec(monkeypatch, "--workload", "prefill", *(["--fp8"] if fp8 else []))
    assert spec["fp8"] is fp8
    assert spec["rounding"] == ("e4m3" if fp8 else "fp16")
    assert spec["name"] in bench.PREFILL_TRAFFIC_BYTES


def test_fp8_only_changes_the_prefill(monkeypatch):
    _, spec = _spec(monkeypatch, "--fp8")
    assert spec["kind"] == "mlp" and spec["fp8"] is False and spec["rounding"] == "fp16"


def test_prefill_call_is_two_kernels():
    for m, k, n in [(2048, 5120, 17408), (64, 17408, 256), (1, 128, 128)]:
        for fp8 in (False, True):
            assert bench.prefill_launches(m, k, n, 152, fp8) == 2


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill_cpu_baseline_leg_on_a_tiny_layer(fp8):
    spec = dict(kind="prefill", layers=[(256, 256, 2)], seed=1234, fp8=fp8,
                rounding="e4m3" if fp8 else "fp16", name="tiny")
    tflops, cores, sample = bench.prefill_oracle_rate(spec, 8, 0.05)
    assert tflops > 0 and cores > 0 and "8 tokens" in sample


def test_every_workload_parses(monkeypatch):
    for wl in ("mlp", "linear512", "sweep", "prefill", "moe", "encode"):
        _, spec = _spec(monkeypatch, "--workload", wl)
        assert spec["name"] and spec["layers"]


def test_timed_region_repeats():
    assert bench.repeats_for(1.4) == 179          # 20 steps of 70 us: about 0.25 s in all
    assert bench.repeats_for(0.01) == bench.MAX_REPEATS
    assert bench.repeats_for(1000.0) == bench.MIN_REPEATS
    assert bench.repeats_for(10.0) == 25
    assert bench.repeats_for(5.0, asked=3) == 3


def test_issue_roofline_is_the_tighter_of_issue_and_alu(monkeypatch):
    _, spec = _spec(monkeypatch)
    r = bench.issue_roofline(spec["name"], 4.0e12, 152, {"sm_mhz": 2000.0})
    mix = bench.GEMV_ISSUE_MIX[spec["name"]]
    f = 152 * 4 * 2000e6
    assert abs(r["peak"] * 1e12 - min(f * 32 / mix["issue"], f * 16 / mix["alu"])) < 1e3
    assert abs(r["frac"] - 4.0e12 / (r["peak"] * 1e12)) < 1e-12
    assert bench.issue_roofline(None, 1.0, 152, None) is None
    assert bench.issue_roofline("no capture of this workload", 1.0, 152, None) is None


def test_default_line_prefill_half_is_the_2048_token_gemm(monkeypatch):
    args, spec = _spec(monkeypatch)
    p = bench.prefill_spec(args)
    assert p["kind"] == "prefill" and p["layers"] == [(5120, 17408, 3)]
    assert not p["fp8"] and p["rounding"] == "fp16" and "M=2048" in p["name"]
    assert bench.PREFILL_TRAFFIC_BYTES.get(p["name"]) is not None
    assert args.workload == "mlp" and args.m == 1          # the decode half is unchanged


def test_both_arms_print_one_metric_string_per_kind():
    src = open(os.path.join(ROOT, "bench.py")).read()
    # every "metric" key of either arm takes one of the three shared strings
    import re
    vals = re.findall(r'"metric": ([A-Za-z_"][^,]*),', src)
    assert vals and set(vals) <= {"METRIC_DECODE", "METRIC_PREFILL", "METRIC_ENCODE"}


def test_prefill_peak_is_sustained_for_long_regions():
    """A region of half a second or more is compared with the sustained tensor
    peak, a shorter one with the burst peak; E4M3 doubles either."""
    import bench
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    assert bench.tensor_peak(peaks, "measured", 1.2, 4000, False)[0] == 1700.0
    assert bench.tensor_peak(peaks, "measured", 0.006, 20, False)[0] == 1900.0
    assert bench.tensor_peak(peaks, "measured", 1.2, 4000, True)[0] == 3400.0
    peak, note = bench.tensor_peak(peaks, "measured", 0.006, 20, True)
    assert peak == 3800.0 and "bf16_tflops x 2" in note
