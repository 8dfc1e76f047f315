"""Host-side legs of bench.py that need no GPU: the oracle's CPU-baseline
timing (backward and forward) on a bounded sample, the workload description,
the flop counts and the traffic lookup."""
import os

import pytest
import torch

import bench
import synth
from tests import _support as S


@pytest.fixture(scope="module")
def tiny():
    w = synth.WORKLOADS[0]
    x = S.workload_inputs(w, "cpu")
    return w, x


@pytest.mark.parametrize("forward", [False, True])
def test_oracle_baseline_times_a_bounded_sample(tiny, forward):
    w, x = tiny
    tflops, dt, n = bench.time_oracle(w, x, 0.2, forward=forward)
    assert tflops > 0 and dt > 0 and 1 <= n <= w.t1


def test_workload_config_names_the_workload():
    w = synth.WORKLOADS[2]
    c = bench.workload_config(w, False)
    assert c["workload"] == "long_context" and c["mode"] == "default"
    assert c["seq_len_q"] == [32768] and c["n1"] == 64 and c["n2"] == 4
    assert "no flush" in c["l2"]                         # inputs larger than L2
    assert "flushed" in bench.workload_config(synth.WORKLOADS[0], True)["l2"]
    assert bench.workload_config(w, True)["mode"] == "deterministic"


def test_flop_counts():
    w = synth.WORKLOADS[2]
    L = w.block_size * w.block_count
    assert w.flops() == 2.0 * L * (3 * w.d_qk + 2 * w.d_v) * w.t1 * w.n1
    assert bench.fwd_flops(w, w.t1 * w.n1) == 2.0 * L * (w.d_qk + w.d_v) * w.t1 * w.n1


def test_traffic_lookup_misses_unknown_keys():
    assert bench.profiled_traffic("no_such_workload", False) is None
    assert bench.profiled_traffic("long_context", False, "no_such_mode") is None


def test_traffic_lookup_follows_the_dq_path():
    """The long-context entries cover the main kernel storing dS and the
    fixed-order dQ pass after it: no figure for the in-kernel reductions."""
    import json
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")) as f:
        e = json.load(f)["long_context:default"]
    assert e["kernels"] == "main_dq_pass"
    assert bench.profiled_traffic("long_context", False, dq_path=0) is None
    got = bench.profiled_traffic("long_context", False, dq_path=1)
    assert got is None or got == e["dram_bytes_per_launch"]
