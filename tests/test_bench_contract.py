"""bench.py on the host alone: the reference arm (the fp64 oracle on the host
cores) prints one JSON line with the keys the benchmark contract names, and
our arm refuses to run without a GPU (it has no CPU path)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ENV = {**os.environ, "CUDA_VISIBLE_DEVICES": ""}


def _bench(*args, timeout=900):
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, env=ENV, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_prints_the_contract_line():
    out = _bench("--impl", "reference", "--shape", "small", "--steps", "1", "--warmup", "0")
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0
    assert "workload" in line["config"] and "model" not in line["config"]


def test_our_arm_refuses_to_run_without_a_gpu():
    out = _bench("--steps", "1", "--warmup", "0", "--no-cpu-baseline", timeout=600)
    assert out.returncode != 0
    assert not out.stdout.strip().startswith("{")


def test_both_arms_describe_the_workload_with_the_same_config():
    """The reference arm's config is the one our arm prints for the same
    flags: workload_config depends on the layer shape, weight type and batch
    sizes alone (timing details live outside config)."""
    out = _bench("--impl", "reference", "--shape", "small", "--steps", "1", "--warmup", "0")
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    import dataclasses
    shape = dataclasses.replace(wl.MIXTRAL, name="profile-small", p=3584)
    assert line["config"] == bench.workload_config(shape, "bf16", wl.DECODE_TOKENS)
    assert set(line["config"]) == {"workload", "m", "p", "E", "k", "expert", "tokens_per_step",
                                   "parallelism", "l2"}
