"""The parts of the benchmark that need no GPU.

The reference arm times the fp64 oracle on the host cores: its JSON line carries the same metric
and config as the kernels' arm, names the oracle as the baseline and moves no host-device bytes;
under a multi-rank launch only rank 0 prints.  The roofline's algorithmic FLOPs and bytes are
checked against their closed forms."""
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


def test_algorithmic_flops_match_the_closed_forms():
    """Per token, the K2 layer is 2dE (router) + (k + 1) * 6dI (eight routed experts and the
    shared one) = 798,228,480 FLOPs; the K3 latent layer adds the down- and up-projections (4dL)
    and runs the routed experts at width L: 2dE + 4dL + k * 6LI + 6dI = 548,667,392."""
    import bench
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    d, E, k, I, L = 7168, 384, 8, 2048, 3584
    assert 2 * d * E + (k + 1) * 6 * d * I == 798_228_480
    assert 2 * d * E + 4 * d * L + k * 6 * L * I + 6 * d * I == 548_667_392
    assert bench.flops(S.WORKLOADS["k2_decode_bf16"], 1)["layer"] == 798_228_480
    assert bench.flops(S.WORKLOADS["k2_prefill_bf16"], 3)["layer"] == 3 * 798_228_480
    assert bench.flops(S.WORKLOADS["k3_latent_bf16"], 1)["layer"] == 548_667_392
    f = bench.flops(S.WORKLOADS["k2_decode_bf16"], 1)
    assert f["router"] + f["gemm13"] + f["gemm2"] == 798_228_480


def test_algorithmic_bytes_count_each_touched_expert_once():
    """A bf16 K2 expert is 3 * I * d * 2 = 88,080,384 bytes and an e4m3 one 44,040,192 bytes plus
    2,688 fp32 block scales; the layer's bytes are the touched experts, the shared expert, the fp32
    router weight, x in and the output out -- whatever the number of tokens that share an
    expert."""
    import numpy as np
    import bench
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    d, E, I = 7168, 384, 2048
    w = S.WORKLOADS["k2_decode_bf16"]
    T = 128
    idx = np.tile(np.arange(8, dtype=np.int32), (T, 1))  # every token on experts 0..7
    by = bench.touched_bytes(w, idx)
    assert by["touched_experts"] == 8
    assert by["layer"] == (8 + 1) * 88_080_384 + E * d * 4 + 2 * T * d * 2
    idx_all = (np.arange(T * 8, dtype=np.int32) % E).reshape(T, 8)
    by_all = bench.touched_bytes(w, idx_all)
    assert by_all["touched_experts"] == E
    assert by_all["layer"] == (E + 1) * 88_080_384 + E * d * 4 + 2 * T * d * 2
    wq = S.WORKLOADS["k2_fp8"]
    byq = bench.touched_bytes(wq, idx)
    assert 3 * I * d * 4.0 / (128 * 128) == 2688 * 4
    assert byq["layer"] == (8 + 1) * (44_040_192 + 2688 * 4) + E * d * 4 + 2 * T * d * 2
    # expert outputs: bf16 by default for e4m3 experts, fp32 on request (or for bf16 experts)
    P = T * 8
    assert (bench.touched_bytes(wq, idx, y_bytes=4)["gemm2"] - byq["gemm2"]
            == (P * d + T * d) * 2)
    assert (by["gemm2"] - bench.touched_bytes(w, idx, y_bytes=2)["gemm2"] == (P * d + T * d) * 2)


def test_traffic_ratio_is_refused_once_its_sources_change(tmp_path, monkeypatch):
    """A traffic ratio belongs to the kernel source it was measured on: with the current digests
    it is used, with any other digest it is dropped (traffic null)."""
    import bench
    srcs = ["csrc/gemm_tc.cu", "csrc/common.cuh"]
    good = bench.source_digest(srcs)
    stale = dict(good, **{"csrc/common.cuh": "0" * 64})
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"entries": [
        {"kernel": "gemm13_swiglu_rows", "ratio": 1.05, "capture": "a test case", "sources": good},
        {"kernel": "gemm2_rows", "ratio": 0.98, "capture": "a test case", "sources": stale}]}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.traffic_ratio("gemm13_swiglu_rows", False)[0] == 1.05
    assert bench.traffic_ratio("gemm13_swiglu_rows", True)[0] is None  # no latent capture
    r, note = bench.traffic_ratio("gemm2_rows", False)
    assert r is None and "changed" in note
    assert bench.traffic_ratio("gemm13_swiglu_swap", False)[0] is None


def test_default_run_is_the_prefill_layer_with_the_other_configurations(monkeypatch):
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    assert a.workload == "k2_prefill_bf16" and a.others
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "k2_decode_bf16"])
    a = bench.parse_args()
    assert a.workload == "k2_decode_bf16" and not a.others
    names = [n for n, _, _ in bench.OTHER_WORKLOADS]
    assert set(names) == {"k2_decode_bf16", "k3_latent_bf16", "k2_fp8", "k2_int4_decode"}


def test_oracle_check_reports_plain_and_beyond_rounding_errors():
    """On a tiny bf16 layer (CPU), an 'output' that is the oracle's own result rounded to bf16 has
    a plain error of up to half a bf16 ulp and nothing beyond its rounding."""
    from dataclasses import replace
    import numpy as np
    import torch
    import bench
    from oracle import torch_bridge as OB
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    w = replace(S.WORKLOADS["tiny_fp32"], name="tiny_bf16", act="bf16", T=40)
    layer = S.make_layer(w, seed=3, device="cpu")
    ref = OB.forward(layer)
    out = torch.tensor(ref["out"], dtype=torch.float32).to(torch.bfloat16)
    rows = torch.arange(0, 40, 3)
    chk = bench.oracle_check(layer, out, rows, 2)
    assert chk["tokens"] == len(rows) and chk["compared"] + chk["near_tie_tokens"] == len(rows)
    assert chk["max_err_rms_beyond_rounding"] <= 1e-9
    assert 0 < chk["max_err_rms"] <= 2.0 ** -8 * np.abs(ref["out"]).max() / np.sqrt(
        np.mean(ref["out"][rows.numpy()] ** 2))


def test_fused_decode_work_is_both_expert_gemms_without_h():
    """The persistent decode launch is credited with both expert GEMMs' FLOPs and with their
    bytes less h, which never leaves the launch: gemm13 + gemm2 - 2 (T k + T) I * 2 bytes."""
    import numpy as np
    import bench
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    w = S.WORKLOADS["k2_decode_bf16"]
    T, I = 128, 2048
    idx = (np.arange(T * 8, dtype=np.int32) % 300).reshape(T, 8)
    by = bench.touched_bytes(w, idx)
    assert by["experts_fused"] == by["gemm13"] + by["gemm2"] - 2 * (T * 8 + T) * I * 2
    f = bench.flops(w, T)
    assert f["experts_fused"] == f["gemm13"] + f["gemm2"]
