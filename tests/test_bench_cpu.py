"""Host-side pieces of the benchmark: the group counts and the algorithmic-byte formulas the roofline
lines divide by (no GPU needed)."""

import numpy as np

import bench
from synth import WORKLOADS, make_inputs, scaled


def _brute_groups(idx):
    return sum(len({int(s) for s in row.ravel() if s >= 0}) for row in idx)


def test_group_counts_match_a_brute_force_count():
    w = scaled(WORKLOADS["wide_ragged"], P=2, T=300, S=512)   # ragged: ids -1 in the last step
    x = make_inputs(w)
    assert bench.count_groups(x, w) == _brute_groups(x["k_idx"])
    assert bench.count_read_groups(x) == _brute_groups(x["q_idx"])


def test_algorithmic_bytes_of_the_large_workload():
    """The per-pass byte counts quoted for the large workload: forward 714.1 + 2210.4 MB with 4,186,081
    write groups; Phase A 6.67 GB (f32 grad rows), GDS 5.57 GB with 4,185,964 read groups, GWR 2.40 GB."""
    w = WORKLOADS["large"]
    x = {"k_idx": np.zeros((w.N, w.C, w.W), np.int32)}
    ab = bench.algorithmic_bytes(w, x, 4186081)
    assert round(ab["phase1"] / 1e6, 1) == 714.1 and round(ab["dw"] / 1e6, 1) == 2210.4
    assert round(bench.pa_algorithmic_bytes(w, 4186081, 4) / 1e9, 2) == 6.67
    assert round(bench.gds_algorithmic_bytes(w, 4185964, 4) / 1e9, 2) == 5.57
    assert round(bench.gwr_algorithmic_bytes(w, 4) / 1e9, 2) == 2.40
    # bf16 grad rows move half the grad bytes
    assert bench.pa_algorithmic_bytes(w, 4186081, 2) < bench.pa_algorithmic_bytes(w, 4186081, 4)


def test_traffic_keys_name_known_kernels():
    for key in bench.NCU_TRAFFIC:
        workload, dom, h = key.split(":")
        assert workload in WORKLOADS and len(h) == 12
        assert dom.split("_")[0] in ("dw", "phase1", "pa", "gds", "gwr", "read")


def test_reference_arm_every_mode(capsys):
    """`bench.py --impl reference` prints one JSON line per mode with the GPU arm's metric names (tiny
    workload, a fraction of a second of oracle time each)."""
    import argparse
    import json

    for mode, metric in (("", bench.METRIC_FWD), ("pa", bench.METRIC_PA), ("gds", bench.METRIC_GDS),
                         ("gwr", bench.METRIC_GWR), ("read", bench.METRIC_READ)):
        args = argparse.Namespace(workload="tiny", steps=1, warmup=0, cpu_seconds=0.2, pa=mode == "pa",
                                  gds=mode == "gds", gwr=mode == "gwr", read=mode == "read", pa_grad="f32")
        bench.run_reference(args)
        d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        assert d["impl"] == "reference" and d["metric"] == metric and d["value"] > 0
        assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
