"""The reference arm of bench.py (the fp64 oracle timed on the host cores) prints the JSON line
the bench contract requires.  Run on the tiny workload, where one oracle step takes well
under a second; the bench itself times the metric's 27B workload."""
import json
import types

import bdsynth
import bench


def test_reference_arm_line_carries_the_contract_keys():
    args = types.SimpleNamespace(steps=2, warmup=1, seed=0, gpus=1)
    line = bench.reference_line(bdsynth.TINY, args)
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert abs(line["ms_per_step"] * line["value"] - 1000.0) < 1e-6 * 1000.0
    assert line["steps"] == 2 and line["warmup"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == bdsynth.TINY.name
    json.loads(json.dumps(line))
