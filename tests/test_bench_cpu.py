"""The benchmark's JSON contract, checked on the CPU through its reference arm.

``bench.py --impl reference`` times the fp64 oracle on the host, so it runs
without a GPU; its line must carry the keys the contract names, for the
forward, for the backward (``--only bwd``) and for the gated delta rule
(``--only gdn``)."""

from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e", "gpu_launches"}


def _run(*extra):
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "small", "--steps", "1", "--warmup", "0",
                          "--ref-seconds", "0.5", *extra],
                         capture_output=True, text=True, env=env, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("only", ["both", "bwd", "gdn"])
def test_reference_line_keeps_the_contract(only):
    line = _run("--only", only)
    assert KEYS <= set(line), sorted(KEYS - set(line))
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("B1-H2-T256-dk64-dv64")
    assert ("chunk-bwd" in line["metric"]) == (only == "bwd")
    assert ("Gated DeltaNet" in line["metric"]) == (only == "gdn")
    assert line["ms_per_step"] > 0
