"""Host-side logic of bench.py, on CPU: the work counts its figures divide by, the traffic table's guard, and the
clock sampler's parsing.  No GPU and no nvidia-smi are needed."""
import os
import subprocess
import sys
import tempfile

import pytest

from causal_sliding_window_fwd_b300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    sys.path.insert(0, ROOT)
    import bench as b
    return b


@pytest.mark.parametrize("T", [1, 2, 7, 128, 300])
@pytest.mark.parametrize("window", [0, 1, 2, 5, 128, 299, 300, 1000])
def test_pairs_in_window_counts_visible_pairs(T, window):
    W = T if (window <= 0 or window >= T) else window
    brute = sum(1 for i in range(T) for j in range(T) if j <= i and i - j < W)
    assert workloads.pairs_in_window(T, window) == brute


def test_flop_counts(bench):
    call = workloads.D20_PAIR.calls[0]
    pairs = call.B * call.H * workloads.pairs_in_window(call.T, call.window)
    # forward: QK^T and PV, 2 D flops each per pair; training step adds the backward's 10 D
    assert bench.fwd_flops(call) == 4.0 * call.D * pairs
    assert bench.useful_flops(call) == 14.0 * call.D * pairs


def test_min_bytes(bench):
    call = workloads.D20_PAIR.calls[0]
    t = call.B * call.T * call.H * call.D * 2
    lse = call.B * call.H * call.T * 4
    assert bench.min_bytes(call, "fwd") == 4 * t + lse        # q, k, v in; o, lse out
    assert bench.min_bytes(call, "bwd") == 8 * t + lse        # q, k, v, o, dO, lse in; dq, dk, dv out


def test_traffic_table_guard(bench):
    """A recorded DRAM figure is returned only for the kernel source it was captured from, and it can never be
    below the algorithmic minimum of the call."""
    for name in bench.TRAFFIC:
        for W, call in ((1024, workloads.D20_PAIR.calls[0]), (2048, workloads.D20_PAIR.calls[1])):
            got = bench.traffic_per_call(name, W)
            if got is None:
                continue  # the kernel changed since the capture: the bench reports null
            which = "fwd" if name.endswith("fwd") else "bwd"
            assert got >= bench.min_bytes(call, which)


def test_traffic_table_rejects_a_changed_source(bench, monkeypatch):
    t = dict(bench.TRAFFIC["nc_attn_fwd"])
    t["sha256"] = "0" * 64
    monkeypatch.setitem(bench.TRAFFIC, "nc_attn_fwd", t)
    assert bench.traffic_per_call("nc_attn_fwd", 1024) is None


def test_clock_sampler_parsing(bench):
    """Median over the samples under load (power at least half the highest), every throttle reason seen, and
    rows with unreadable fields tolerated."""
    c = bench.ClockSampler(0)
    fd, c.path = tempfile.mkstemp(suffix=".csv")
    os.close(fd)
    with open(c.path, "w") as f:
        f.write("0, 2032, 2032, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")   # idle lead-in
        f.write("0, 1900, 2032, 1000.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 1950, 2032, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1960, 2032, [N/A], 0x0, Not Active, Active, Not Active, Not Active\n")
        f.write("garbage line\n")
    c.proc = subprocess.Popen([sys.executable, "-c", "import time; time.sleep(30)"])
    r = c.stop()
    assert r["samples"] == 4
    assert r["samples_under_load"] == 2
    assert r["sm_mhz"] == pytest.approx(1925.0)
    assert r["sm_max_mhz"] == 2032.0
    assert r["power_w_max"] == 1000.0
    assert r["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert not os.path.exists(c.path)


def test_clock_sampler_without_nvidia_smi(bench):
    c = bench.ClockSampler(0)
    r = c.stop()  # never started: no process
    assert r["sm_mhz"] is None and "nvidia-smi unavailable" in r["reasons"]
