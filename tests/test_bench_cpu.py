"""The benchmark's reference arm times the fp64 oracle on the host cores; it needs no GPU, so its
JSON line is checked here: the same metric and config as the kernels' arm, the oracle named as
the baseline, and no host-device bytes.  Under a multi-rank launch only rank 0 prints."""
import json
import os
import subprocess
import sys

from conftest import ROOT


def _run(extra_env=None, *args):
    env = dict(os.environ, **(extra_env or {}))
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny_fp32", "--steps", "1", "--warmup", "1", *args]
    return subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)


def test_reference_line_matches_the_kernel_arm_contract():
    import bench
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    p = _run()
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s"
    assert line["higher_is_better"] is True
    assert line["config"] == bench.layer_config(S.WORKLOADS["tiny_fp32"], False, 1)
    assert line["value"] > 0 and line["steps"] == 1 and line["warmup"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_prints_nothing_on_other_ranks():
    p = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr
    assert not [l for l in p.stdout.splitlines() if l.startswith("{")]
