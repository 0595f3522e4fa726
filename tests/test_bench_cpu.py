"""Host logic of bench.py that needs no GPU: the step's call schedule (including
the wgrad calls spread over several streams), the guard on the recorded DRAM
traffic, the choice of the tensor peak and the gate targets."""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeStream:
    def __init__(self, handle, log):
        self.cuda_stream = handle
        self.log = log

    def wait_stream(self, other):
        self.log.append(("wait", self.cuda_stream, other.cuda_stream))


def _record_calls(monkeypatch):
    calls = []

    def fake(kind):
        def f(wl, i, sh, side=-1):
            calls.append((kind, i, sh, side))
            return 2 if kind == "wgrad" else 1
        return f

    monkeypatch.setattr(bench, "_fwd", fake("fwd"))
    monkeypatch.setattr(bench, "_dgrad", fake("dgrad"))
    monkeypatch.setattr(bench, "_wgrad", fake("wgrad"))
    return calls


@pytest.mark.parametrize("nstreams", [1, 2, 3])
def test_step_schedule(monkeypatch, nstreams):
    calls = _record_calls(monkeypatch)
    log = []
    wl = types.SimpleNamespace(layers=list(range(7)))
    streams = None
    if nstreams > 1:
        streams = tuple(_FakeStream(100 + k, log) for k in range(nstreams))
    marks = []
    n = bench.run_step(wl, 100, mark=marks.append, streams=streams)
    assert n == 7 + 7 + 2 * 7
    assert marks == ["start", "fwd", "dgrad", "wgrad"]
    # forward in network order and dgrad in reverse, all on the launching stream
    assert [(k, i, sh) for k, i, sh, _ in calls if k == "fwd"] == [("fwd", i, 100) for i in range(7)]
    assert [(k, i, sh) for k, i, sh, _ in calls if k == "dgrad"] == [
        ("dgrad", i, 100) for i in reversed(range(7))]
    # every wgrad exactly once, in reverse order, round-robin over the streams,
    # each extra stream with its own workspace index
    w = [(i, sh, side) for k, i, sh, side in calls if k == "wgrad"]
    assert [i for i, _, _ in w] == list(reversed(range(7)))
    for j, (_, sh, side) in enumerate(w):
        k = j % nstreams
        assert sh == 100 + k
        assert side == (k - 1 if k else -1)
    if nstreams > 1:
        # fork: every side stream waits for the launching stream; join: the
        # launching stream waits for every side stream
        forks = [e for e in log if e[2] == 100]
        joins = [e for e in log if e[1] == 100]
        assert sorted(e[1] for e in forks) == [100 + k for k in range(1, nstreams)]
        assert sorted(e[2] for e in joins) == [100 + k for k in range(1, nstreams)]
        assert log.index(forks[-1]) < log.index(joins[0])


def test_interleaved_schedule(monkeypatch):
    calls = _record_calls(monkeypatch)
    wl = types.SimpleNamespace(layers=list(range(4)))
    bench.run_step(wl, 5, interleave=True)
    back = [(k, i) for k, i, _, _ in calls if k != "fwd"]
    assert back == [(k, i) for i in reversed(range(4)) for k in ("dgrad", "wgrad")]


def test_recorded_traffic_guard(monkeypatch):
    monkeypatch.setattr(bench, "RECORDED_TRAFFIC", {("l1", "fwd"): 1.5e8})
    monkeypatch.setattr(bench, "TRAFFIC_SHA256", bench.sources_sha256())
    assert bench.sources_sha256() is not None
    assert bench.recorded_traffic("l1", "fwd") == 1.5e8
    # no capture for this config or pass
    assert bench.recorded_traffic("l2", "fwd") is None
    assert bench.recorded_traffic("l1", "wgrad") is None
    # kernel sources changed since the capture: no figure
    monkeypatch.setattr(bench, "TRAFFIC_SHA256", "0" * 64)
    assert bench.recorded_traffic("l1", "fwd") is None


def test_recorded_pass_traffic_by_workload(monkeypatch):
    monkeypatch.setattr(bench, "RECORDED_TRAFFIC", {("l1", "fwd"): 1.5e8})
    monkeypatch.setattr(bench, "RECORDED_STEP_TRAFFIC", {"fwd": 1.5e9})
    monkeypatch.setattr(bench, "TRAFFIC_SHA256", bench.sources_sha256())
    assert bench.recorded_pass_traffic("unet", "fwd") == 1.5e9
    assert bench.recorded_pass_traffic("l1", "fwd") == 1.5e8
    # the step's figure never stands for another workload, nor the plain kernels' for variants
    assert bench.recorded_pass_traffic("l2", "fwd") is None
    assert bench.recorded_pass_traffic("stack", "fwd") is None
    assert bench.recorded_pass_traffic("unet", "fwd", fused_act=True) is None
    assert bench.recorded_pass_traffic("unet", "fwd", concat_free=True) is None
    assert bench.recorded_pass_traffic("l1", "fwd", path="simt") is None
    monkeypatch.setattr(bench, "TRAFFIC_SHA256", "0" * 64)
    assert bench.recorded_pass_traffic("unet", "fwd") is None


def test_peak_choice():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0}
    assert bench.pick_peak(peaks, full, 0.3) == ("bf16_tflops", 1900.0)
    # a long timed region, a clock well below its maximum, or no clock record:
    # the sustained figure
    assert bench.pick_peak(peaks, full, 3.0) == ("bf16_tflops_sustained", 1700.0)
    assert bench.pick_peak(peaks, {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0}, 0.3)[0] == \
        "bf16_tflops_sustained"
    assert bench.pick_peak(peaks, None, 0.3)[0] == "bf16_tflops_sustained"


def test_gate_targets():
    # the small-channel stem is held to the HBM roofline, the others to the tensor peak
    g = {name: (bound, target) for name, bound, target in bench.GATES}
    assert g == {"stem": ("hbm", 0.70), "l1": ("tensor", 0.60), "l2": ("tensor", 0.60),
                 "l3": ("tensor", 0.60)}


def test_wgrad_streams_validated():
    with pytest.raises(SystemExit):
        bench.main(["--wgrad-streams", "0"])
