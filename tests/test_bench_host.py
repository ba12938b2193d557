"""Host-side arithmetic of bench.py (no GPU): the roofline's algorithmic
bytes and FLOPs, the traffic record's source check, the launch count, and
the capacity sweep."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from bit_mla_kv_qmla_gb300 import workloads as W  # noqa: E402

PK = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "source": "test"}


def test_token_bytes_follow_the_layout():
    # the roofline's bytes per token are the oracle's block bytes / 64 slots
    for name, code in W.FORMATS.items():
        assert bench.TOKEN_BYTES[name] * 64 == oracle.block_bytes(code), name


def test_roofline_hbm_bound_16_heads():
    lens = [8192] * 32
    t = 50e-6
    r = bench.roofline_for("C4R4", 16, lens, t, PK, None)
    nbytes = 32 * 8192 * 324 + 32 * 16 * (576 * 2 + 512 * 2 + 4)
    assert r["bound"] == "hbm" and r["algorithmic_bytes"] == nbytes
    assert r["achieved"] == round(nbytes / t / 1e9, 1)
    assert r["frac"] == round(nbytes / t / 1e9 / PK["hbm_gbs"], 4)


def test_roofline_tensor_bound_128_heads():
    lens = [131072] * 4
    t = 380e-6
    r = bench.roofline_for("C4R4", 128, lens, t, PK, None)
    flops = 4 * 131072 * 128 * 2 * (576 + 512)
    assert r["bound"] == "tensor" and r["algorithmic_flops"] == flops
    assert r["frac"] == round(flops / t / 1e12 / PK["bf16_tflops"], 4)


def test_recorded_traffic_only_for_the_current_sources(monkeypatch):
    d = json.load(open(os.path.join(ROOT, "profiles", "decode_traffic.json")))
    name = "c4r4_b32_h16_l8192_append1"
    if d[name]["kernel_hash"] == bench.decode_kernel_hash():
        assert bench.recorded_traffic(name) == d[name]["traffic_bytes_per_launch"]
    assert bench.recorded_traffic("no_such_workload") is None
    monkeypatch.setattr(bench, "decode_kernel_hash", lambda: "0" * 16)
    assert bench.recorded_traffic(name) is None


@pytest.mark.parametrize("heads,batch,tc,n_app,want", [
    (16, 32, True, 1, 3),    # append (advances the lengths) + decode + merge
    (16, 150, True, 1, 4),   # above 64 sequences the planner kernel runs too
    (128, 4, True, 0, 3),    # planner + decode + merge
    (32, 8, False, 0, 2),    # CUDA-core kernel plans for itself
    (16, 32, True, 3, 4),    # several tokens: append + length update
])
def test_step_launches(heads, batch, tc, n_app, want):
    w = W.Workload("x", "C4R4", batch, heads, 1024)
    assert bench.step_launches(w, n_app, tc) == want


def test_capacity_sweep_shows_the_pressure_gap():
    r = bench.capacity_sweep({"C4R4": 4e9, "BF16": 2e9, "C2R4": None})
    at8 = r["by_budget"]["8GB"]
    assert at8["BF16"]["preemptions"] > 0 and at8["C4R4"]["preemptions"] == 0
    assert at8["BF16"]["steps"] > at8["C4R4"]["steps"]
    assert "decode_s_at_measured_rate" in at8["C4R4"]
    assert "decode_s_at_measured_rate" not in at8["C2R4"]


def test_oracle_multicore_covers_disjoint_units():
    # two processes, each its own (sequences, heads) unit of the workload
    v, t, desc, procs = bench.oracle_multicore(1, "C4R4", 2, steps=1, warmup=0)
    assert v > 0 and t > 0 and procs == 2 and "2 processes" in desc
    # each sequence's appended tokens come from its own stream: splitting the
    # sequences or the heads over runners appends the same bytes and counts
    # the same work (head subsets as their fraction of the decode)
    one = bench.OracleRunner(1, "C4R4", 4, 1)
    two = [bench.OracleRunner(1, "C4R4", 2, 1, first=f) for f in (0, 2)]
    halves = [bench.OracleRunner(1, "C4R4", 4, 1, h0=h, n_heads=8) for h in (0, 8)]
    a = one.step()
    assert a == sum(r.step() for r in two) == sum(r.step() for r in halves)
    assert (one.qc[2:] == two[1].qc).all()
    assert (one.qc[:, 8:] == halves[1].qc).all()
    bb = oracle.block_bytes(one.f)
    for b, (r, rb) in enumerate([(two[0], 0), (two[0], 1), (two[1], 0), (two[1], 1)]):
        for j in range(one.table.shape[1]):
            x, y = one.table[b, j], r.table[rb, j]
            if x < 0:
                break
            assert (one.pool[x * bb:(x + 1) * bb] == r.pool[y * bb:(y + 1) * bb]).all()


def test_host_cpu_names_the_cores():
    c = bench.host_cpu()
    assert c["logical_cores"] == os.cpu_count() and c["arch"]
