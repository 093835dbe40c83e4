"""bench.py's reference arm on CPU (the oracle on a bounded sample of the
tiny workload): its one JSON line carries the keys the benchmark contract
names, with the e2e and cpu_baseline objects describing this run."""

import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line_has_the_contract_keys():
    sys.path.insert(0, ROOT)
    import bench
    args = type("A", (), dict(steps=2, warmup=1, workload="tiny"))()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1
    assert (d["steps"], d["warmup"]) == (2, 1)
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny"
    # the GPU arm prints the same config object for the same workload
    assert d["config"] == bench.bench_config(bench.W.WORKLOADS["tiny"])
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert (e2e["value"], e2e["unit"]) == (d["value"], d["unit"])
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_cpu_baseline_reports_cores_model_and_one_thread_run():
    sys.path.insert(0, ROOT)
    import bench
    from invariant_mmdit_joint_gb300 import workloads as W
    w = W.WORKLOADS["tiny"]
    cb = bench.cpu_baseline(w, W.make_batch(w, seed=0), budget_s=0.0)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] == os.cpu_count()
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    one = cb["one_thread"]
    assert one["cores"] == 1 and one["value"] > 0 and one["unit"] == "TFLOP/s", one


def test_cpu_baseline_extrapolates_a_head_subset_at_the_larger_shapes():
    """Away from the 1024^2 CFG pair the oracle runs heads 0 and H-1 of every
    sample and scales the time per head to all heads, labelled as such."""
    sys.path.insert(0, ROOT)
    import bench
    from invariant_mmdit_joint_gb300 import workloads as W
    w = W.Workload("small4", B=2, H=4, T_txt=16, grid_h=6, grid_w=6, valid_len=(5, 16))
    cb = bench.cpu_baseline(w, W.make_batch(w, seed=0), budget_s=0.0)
    assert cb["extrapolated"] is True and cb["value"] > 0
    assert abs(cb["extrapolated_step_seconds"] - cb["seconds_per_head"] * 4) < 0.02
    assert "heads [0, 3]" in cb["sample"]
