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
    assert bench.PREFILL_TRAFFIC_BYTES.get(spec["name"]) is not None


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
