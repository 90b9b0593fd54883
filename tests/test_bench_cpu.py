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


def test_roofline_binds_on_the_slower_roof():
    """The roofline's bound is whichever of bytes / HBM peak and flops / tensor peak
    takes longer, and its fraction is that roof's time over the measured time."""
    sys.path.insert(0, ROOT)
    import bench
    pk = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}
    # 1 GB at 1000 GB/s = 1 ms; 50 GFLOP at 100 TF/s = 0.5 ms: HBM binds
    r = bench.roofline(10**9, 5 * 10**10, 2e-3, pk, "test")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - 0.5) < 1e-12 and abs(r["achieved"] - 500.0) < 1e-9
    assert abs(r["tensor_frac"] - 0.25) < 1e-12
    # 200 GFLOP = 2 ms against 1 ms of bytes: the tensor roof binds
    r = bench.roofline(10**9, 2 * 10**11, 4e-3, pk, "test")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - 0.5) < 1e-12 and abs(r["hbm_frac"] - 0.25) < 1e-12
    assert list(r)[:5] == ["bound", "achieved", "peak", "unit", "frac"]


def test_chunk_flops_use_the_kernel_chunk():
    sys.path.insert(0, ROOT)
    import bench
    from synth import CHUNK_CONFIGS
    cfg = CHUNK_CONFIGS["long"]
    per_token = (bench.KERNEL_CHUNK + 1) * (cfg.dk + cfg.dv) + 4 * cfg.dk * cfg.dv
    assert bench.KERNEL_CHUNK == 128
    assert bench.chunk_flops(cfg) == cfg.tokens * per_token
