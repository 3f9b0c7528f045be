#!/usr/bin/env python
"""Benchmark of the GB300 MoE FFN layer: tokens/s and the roofline fraction.

One step = one pass of the whole layer (router -> permute -> experts -> combine) over one batch of
synthetic tokens, through the C ABI (moe_forward).  Default workload: the Kimi K2 layer in the
prefill regime (16384 tokens = 4 x 4096, d=7168, 384 experts top-8, expert intermediate 2048, one
shared expert, bf16 with fp32 router logits, tokens drawn from 16 Gaussian clusters), the largest
single-GPU configuration.  The default run also measures, in the same process and after the
headline, the decode batch (128 tokens), the K3 latent layer (8192 tokens), fp8 experts (8192
tokens) and INT4 experts at decode, each with its own roofline and an oracle check on a sample,
under "other_workloads".  Other workloads as the headline: --workload k2_decode_bf16 |
k3_latent_bf16 | k2_fp8 | k2_int4_decode | tiny_fp32, and the dense block-0 MLP (moe_dense_mlp,
d=7168, I=18432) as k2_dense_decode_bf16 | k2_dense_prefill_bf16 | tiny_dense_fp32.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs an independent replica of the layer on its
own batch (the layer has no exchange step); value = tokens of all ranks / max-over-ranks time.
`--impl reference` times the fp64 CPU oracle (the only reference there is) on the host cores.
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (d=7168, 384 experts top-8) and % of roofline (HBM or TC)"
DEFAULT_WORKLOAD = "k2_prefill_bf16"
# measured in the default run after the headline: (workload, timed steps, oracle sample tokens)
OTHER_WORKLOADS = (("k2_decode_bf16", 100, 128), ("k3_latent_bf16", 20, 128),
                   ("k2_fp8", 20, 128), ("k2_int4_decode", 50, 128))
# DRAM traffic / algorithmic bytes of the dominant kernels, from ncu captures of small cases, with
# the digests of the sources the captured kernel was built from (a ratio is used only while the
# sources are unchanged)
TRAFFIC_FILE = os.path.join(ROOT, "mixture_experts_ffn_gemm_gb300", "measured_traffic.json")
DENSE_METRIC = "Dense block-0 MLP tokens/s (d=7168, I=18432) and % of roofline (HBM or TC)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of the ranks' values, returned on every rank (collective; the value itself
    for one rank).  Replicas finish when the slowest one does."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput of `world` replicas: the units every rank processed over the time of
    the slowest rank (weak scaling: the work per rank is fixed)."""
    return world * units_per_rank / max_seconds


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None,
                    help=f"layer or dense workload (default {DEFAULT_WORKLOAD}, with the other "
                         f"layer configurations measured after it)")
    ap.add_argument("--no-others", dest="others", action="store_false",
                    help="measure the headline workload only")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=0,
                    help="tokens in the oracle's timed sample (0 = automatic)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the routed expert count (small profiling cases)")
    ap.add_argument("--tokens", type=int, default=0, help="override the token count")
    ap.add_argument("--block", action="store_true",
                    help="time the block's FFN half (moe_forward_block: RMSNorm, layer, residual)")
    ap.add_argument("--flags", type=lambda v: int(v, 0), default=0,
                    help="moe_config_t.flags tuning overrides (MOE_FLAG_*)")
    args = ap.parse_args()
    if args.workload is None:
        args.workload = DEFAULT_WORKLOAD
    else:
        args.others = False  # a named workload is measured alone
    if args.experts or args.tokens or args.block or args.flags:
        args.others = False
    return args


# ----------------------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS if k in p}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [ln.split(", ") for ln in self.tmp.read().strip().splitlines() if ln.strip()]
        os.unlink(self.tmp.name)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def touched_bytes(w, idx: np.ndarray, y_bytes=None) -> dict:
    """Algorithmic bytes of one layer pass: the expert weights the routing touches (each once),
    the shared expert, the router weight, the input read and the output write; per kernel also the
    activations it reads and writes (h in the activation type, or e4m3 + scales for fp8 experts;
    expert outputs in fp32, or bf16 (y_bytes = 2): the library's default for e4m3 experts)."""
    yb = y_bytes if y_bytes is not None else (2 if w.fp8 else 4)
    touched = np.unique(idx)
    ab = 4 if w.act == "f32" else 2
    int4 = getattr(w, "int4", False)
    wb = 1 if w.fp8 else (0.5 if int4 else ab)   # bytes per expert weight
    sb = 4.0 / (128 * 128) if w.fp8 else (2.0 / 32 if int4 else 0.0)  # scale bytes per weight
    hb = 1 + 4.0 / 128 if w.fp8 else ab           # bytes per activation entering a GEMM
    de = w.d_expert
    T, P = idx.shape[0], idx.size
    w13 = 2 * w.I * de * (wb + sb)
    w2 = de * w.I * (wb + sb)
    sh13 = 2 * w.I_shared * w.d * (wb + sb) if w.n_shared else 0
    sh2 = w.d * w.I_shared * (wb + sb) if w.n_shared else 0
    lat = 2 * w.d_latent * w.d * ab if w.d_latent else 0
    rows_sh = T * w.n_shared  # the shared expert rides in both expert launches, at width d
    return {
        "touched_experts": int(touched.size),
        # gemm13: W1|W3 of the touched experts and of the shared expert, activations in, h out
        "gemm13": len(touched) * w13 + sh13 + P * de * hb + rows_sh * w.d * hb
        + (P + rows_sh) * w.I * hb,
        # gemm2: W2 of the touched experts and of the shared expert, h in, expert outputs out
        "gemm2": len(touched) * w2 + sh2 + (P + rows_sh) * w.I * hb + P * de * yb
        + rows_sh * w.d * yb,
        "layer": len(touched) * (w13 + w2) + sh13 + sh2 + lat + w.E * w.d * 4
        + 2 * T * w.d * ab,
        # both expert GEMMs in one launch: h stays inside it (written and read back on chip or
        # through L2), so only the weights, the activations in and the expert outputs count
        "experts_fused": len(touched) * (w13 + w2) + sh13 + sh2 + P * de * hb
        + rows_sh * w.d * hb + P * de * yb + rows_sh * w.d * yb,
    }


def flops(w, T: int) -> dict:
    """Algorithmic FLOPs: the router, the k selected experts and the shared expert per token."""
    de = w.d_expert
    P = T * w.k
    rows13 = P + (0 if w.d_latent else T * w.n_shared)
    f = {
        "gemm13": 2 * rows13 * de * 2 * w.I,
        "gemm2": 2 * rows13 * w.I * de,
        "router": 2 * T * w.d * w.E,
    }
    f["layer"] = (2 * T * w.d * w.E + P * 6 * de * w.I + T * w.n_shared * 6 * w.d * w.I_shared
                  + (4 * T * w.d * w.d_latent if w.d_latent else 0))
    f["experts_fused"] = f["gemm13"] + f["gemm2"]
    return f


def prepare_oracle(layer, rows):
    """Host inputs of the fp64 oracle for `rows` of the layer: the rows, the router and the
    weights of the experts those rows select (copied once, outside any timed part)."""
    import oracle
    from oracle import torch_bridge as OB
    x, W_r, b = OB.route_inputs(layer, rows)
    cfg = OB.config(layer, x.data.shape[0])
    experts = np.unique(oracle.route(cfg, x, W_r, b)["idx"])
    W13, W2 = OB.expert_mats(layer, experts)
    sh = (OB.mat(layer.Ws13, layer.Ws13_scale), OB.mat(layer.Ws2, layer.Ws2_scale),
          OB.mat(layer.W_down), OB.mat(layer.W_up))
    return cfg, (x, W_r, b, W13, W2, *sh)


def time_oracle(prep, nthreads: int) -> float:
    """Seconds of one oracle pass (as it stands) over the prepared rows."""
    import oracle
    cfg, args = prep
    t0 = time.perf_counter()
    oracle.forward(cfg, *args, nthreads=nthreads)
    return time.perf_counter() - t0


def layer_config(w, block: bool, world: int) -> dict:
    """The JSON line's `config` for a layer workload, the same on both arms."""
    return {"workload": w.name + ("_block" if block else ""), "tokens": w.T, "d": w.d,
            "experts": w.E, "top_k": w.k, "block_ffn_half": bool(block),
            "expert_intermediate": w.I, "shared_intermediate": w.I_shared,
            "d_latent": w.d_latent, "router": "fp32 logits",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (expert weights stream from HBM every step; no flush)"}


def dense_config(w, world: int) -> dict:
    """The JSON line's `config` for a dense-MLP workload, the same on both arms."""
    return {"workload": w.name, "tokens": w.T, "d": w.d, "intermediate": w.I,
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (0.8 GB of weights stream from HBM every step; "
                  "no flush)"}


# ----------------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ----------------------------------------------------------------------------------------------
def run_reference(args, w, rank: int, world: int):
    if rank != 0:
        return
    import torch
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    cores = os.cpu_count() or 1
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    layer = S.make_layer(w, seed=0, device=dev)
    # a step is a bounded sample of the batch, sized so that the whole run stays within minutes
    core_s_per_token = time_oracle(prepare_oracle(layer, S.subset_rows(w.T, 1, seed=2)), 1)
    budget_s = 150.0 / max(1, args.steps + args.warmup)
    n = args.cpu_sample or int(max(1, min(w.T, budget_s * cores / max(core_s_per_token, 1e-9))))
    prep = prepare_oracle(layer, S.subset_rows(w.T, n, seed=1))
    for _ in range(args.warmup):
        time_oracle(prep, cores)
    secs = [time_oracle(prep, cores) for _ in range(args.steps)]
    tps = n / statistics.mean(secs)
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * statistics.mean(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": layer_config(w, False, world),
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} of {w.T} tokens (seed 1) per step, fp64 C oracle, "
                                   f"{cores} threads"},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------------
def source_digest(paths) -> dict:
    """sha256 of each listed source file (paths relative to the package)."""
    import hashlib
    base = os.path.join(ROOT, "mixture_experts_ffn_gemm_gb300")
    out = {}
    for rel in paths:
        with open(os.path.join(base, rel), "rb") as f:
            out[rel] = hashlib.sha256(f.read()).hexdigest()
    return out


def traffic_ratio(kernel: str, latent: bool):
    """(ratio, note) for a kernel label from the traffic file; ratio None when there is no
    capture, or when a source listed for it changed since the capture."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no traffic file"
    with open(TRAFFIC_FILE) as f:
        entries = json.load(f)["entries"]
    for e in entries:
        if e["kernel"] == kernel and bool(e.get("latent", False)) == bool(latent):
            if source_digest(e["sources"]) != e["sources"]:
                return None, f"{kernel}: sources changed since its ncu capture ({e['capture']})"
            return e["ratio"], (f"ncu DRAM bytes / algorithmic bytes = {e['ratio']} on "
                                f"{e['capture']}, scaled to this launch")
    return None, f"{kernel}: no ncu capture of this kernel"


def time_steps(step, steps: int, stream, dev, world: int):
    """Device time of `steps` back-to-back steps (CUDA events on the launching stream, barrier and
    synchronise on both sides), the launches counted, the per-kernel profile and the clocks."""
    import torch
    import torch.distributed as dist
    from mixture_experts_ffn_gemm_gb300 import binding as B
    gpu_id = str(getattr(torch.cuda.get_device_properties(dev), "uuid", dev.index or 0))
    if not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    B.moe_profile_enable(True)
    B.moe_profile_read()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = B.moe_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    launches = B.moe_launch_count() - launches0
    ms_total = ev0.elapsed_time(ev1)
    prof = B.moe_profile_read()
    B.moe_profile_enable(False)
    clocks = sampler.stop()
    return ms_total, launches, prof, clocks


def rooflines(w, idx_np, prof, ms_step, y_bytes=None) -> tuple:
    """(dominant-kernel roofline, layer roofline, per-kernel times).  Peaks: the measured burst
    figures (the timed loop runs well under a second of tensor work), the sustained one beside."""
    peaks, peak_src = load_peaks()
    by = touched_bytes(w, idx_np, y_bytes)
    fl = flops(w, w.T)
    kernels = {k: {"ms_per_launch": v[0] / max(v[1], 1), "launches": v[1]} for k, v in prof.items()}
    ratio_fp8 = 2.0 if w.fp8 else 1.0  # an fp8 contraction: nominal dense fp8 / bf16 = 4.5 / 2.25
    tc_peak = ratio_fp8 * peaks["bf16_tflops"]
    tc_sus = ratio_fp8 * peaks["bf16_tflops_sustained"]
    tc_src = (f"{peak_src} bf16_tflops (burst)" + (" x 2 (nominal dense fp8 / bf16 ratio 4.5 / "
                                                    "2.25)" if w.fp8 else ""))
    dom = max(prof.items(), key=lambda kv: kv[1][0])[0] if prof else None
    roof = None
    if dom is not None:
        ms_launch = kernels[dom]["ms_per_launch"]
        unit_key = ("gemm2" if dom.startswith("gemm2") else
                    "experts_fused" if dom.startswith("experts_fused") else "gemm13")
        # the kernel's bound: the larger of its algorithmic time at tensor peak and at HBM peak
        t_tc_k = fl.get(unit_key, 0) / (tc_peak * 1e12)
        t_hbm_k = by[unit_key] / (peaks["hbm_gbs"] * 1e9)
        if t_tc_k > t_hbm_k:
            achieved = fl.get(unit_key, 0) / (ms_launch / 1000.0) / 1e12
            roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tc_peak,
                    "unit": "TFLOP/s", "frac": achieved / tc_peak,
                    "frac_of_sustained_peak": achieved / tc_sus, "peak_source": tc_src,
                    "work_per_launch": fl.get(unit_key, 0)}
        else:
            achieved = by[unit_key] / (ms_launch / 1000.0) / 1e9
            roof = {"kernel": dom, "bound": "hbm", "achieved": achieved,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "peak_source": f"{peak_src} hbm_gbs", "work_per_launch": by[unit_key]}
        ratio, note = traffic_ratio(dom, bool(w.d_latent))
        roof["traffic"] = ratio * by[unit_key] if ratio else None
        roof["traffic_source"] = note
    t_tc = fl["layer"] / (tc_peak * 1e12)
    t_hbm = by["layer"] / (peaks["hbm_gbs"] * 1e9)
    t_roof = max(t_tc, t_hbm)
    layer_roof = {"t_roof_ms": 1000 * t_roof, "bound": "tensor" if t_tc > t_hbm else "hbm",
                  "frac": 1000 * t_roof / ms_step,
                  "frac_of_sustained_peak": 1000 * max(fl["layer"] / (tc_sus * 1e12), t_hbm)
                  / ms_step, "tensor_peak_tflops": tc_peak, "hbm_peak_gbs": peaks["hbm_gbs"],
                  "algorithmic_bytes": by["layer"], "algorithmic_flops": fl["layer"],
                  "touched_experts": by["touched_experts"],
                  "kernel_algorithmic_bytes": {k: by[k] for k in ("gemm13", "gemm2",
                                                                  "experts_fused")}}
    return roof, layer_roof, kernels


def oracle_check(layer, out, rows, nthreads: int) -> dict:
    """The fp64 oracle on `rows` (timed), and the GPU output on those rows against it: the plain
    max |GPU - oracle| / rms, the same beyond the output's own bf16 rounding (2^-8 |oracle| per
    element), the rms error, near ties (k-th / (k+1)-th key margin < 1e-5, left out)."""
    prep = prepare_oracle(layer, rows)
    import oracle
    cfg, oargs = prep
    t0 = time.perf_counter()
    ref = oracle.forward(cfg, *oargs, nthreads=nthreads)
    sec = time.perf_counter() - t0
    keep = ref["margin"] >= 1e-5
    got = out[rows.to(out.device)].float().cpu().numpy()[keep]
    r = ref["out"][keep]
    res = {"seconds": sec, "tokens": int(len(rows)), "compared": int(keep.sum()),
           "near_tie_tokens": int((~keep).sum())}
    if keep.any():
        rms = float(np.sqrt(np.mean(r * r)))
        dlt = np.abs(got - r)
        res["max_err_rms"] = float(dlt.max()) / rms
        res["max_err_rms_beyond_rounding"] = (float(np.max(dlt - 2.0 ** -8 * np.abs(r))) / rms
                                              if layer.w.act != "f32" else res["max_err_rms"])
        res["rms_err"] = float(np.sqrt(np.mean(dlt * dlt))) / rms
    return res


def near_ties_all(layer, cfg_c, ws) -> int:
    """Tokens of the whole batch whose k-th / (k+1)-th key margin is below 1e-5, from the GPU's
    own fp32 logits and the oracle's selection rule."""
    import torch
    import oracle
    from oracle import torch_bridge as OB
    from mixture_experts_ffn_gemm_gb300 import binding as B
    w = layer.w
    dev = layer.x.device
    z = torch.empty(w.T, w.E, dtype=torch.float32, device=dev)
    idx = torch.empty(w.T, w.k, dtype=torch.int32, device=dev)
    wgt = torch.empty(w.T, w.k, dtype=torch.float32, device=dev)
    B.moe_router(cfg_c, layer.x, layer.W_r, layer.b, z, idx, wgt, ws)
    _, _, margin = oracle.route_from_logits(OB.config(layer), z.cpu().numpy(),
                                            layer.b.cpu().numpy())
    return int((margin < 1e-5).sum())


def measure_workload(args, w, rank: int, world: int, dev, steps: int, warmup: int,
                     sample: int, with_e2e: bool, with_cpu: bool) -> dict:
    """One layer workload: warm-up, `steps` timed steps, rooflines; optionally the end-to-end leg
    through host buffers and the oracle on a sample of `sample` tokens."""
    import torch
    from mixture_experts_ffn_gemm_gb300 import binding as B
    from mixture_experts_ffn_gemm_gb300 import synthetic as S

    layer = S.make_layer(w, seed=rank, device=dev)  # each replica its own batch
    cfg = B.config_for(w, flags=args.flags)
    ws = B.alloc_workspace(cfg, dev)
    out = torch.empty(w.T, w.d, dtype=layer.x.dtype, device=dev)
    weights = B.layer_weights(layer)
    stream = torch.cuda.current_stream(dev)

    # the routing of this batch (deterministic; the same as inside every timed step)
    idx = torch.empty(w.T, w.k, dtype=torch.int32, device=dev)
    wgt = torch.empty(w.T, w.k, dtype=torch.float32, device=dev)
    B.moe_router(cfg, layer.x, layer.W_r, layer.b, None, idx, wgt, ws)
    idx_np = idx.cpu().numpy()

    norm_w = S.make_block_norm(w, seed=0, device=dev) if args.block else None

    def step(x=layer.x):
        if args.block:
            B.moe_forward_block(cfg, x, norm_w, *weights, out, ws, stream=stream)
        else:
            B.moe_forward(cfg, x, *weights, out, ws, stream=stream)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    status = B.moe_device_status(ws)
    if status != B.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {B.status_string(status)}")
    ms_total, launches, prof, clocks = time_steps(step, steps, stream, dev, world)
    status = B.moe_device_status(ws)
    if status != B.MOE_OK:
        raise RuntimeError(f"device status after the timed steps: {B.status_string(status)}")
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / steps
    res = {"ms_per_step": ms_step, "value": replica_throughput(w.T, world, ms_step / 1000.0),
           "launches": int(launches), "clocks": clocks}

    # ------------------------------------------------------------- end to end (host buffers)
    if with_e2e:
        io_bytes = w.T * w.d * layer.x.element_size()
        x_host = layer.x.cpu().pin_memory()
        out_host = torch.empty(w.T, w.d, dtype=layer.x.dtype).pin_memory()
        x_dev = torch.empty_like(layer.x)

        def e2e_step():
            if args.block:  # host x'_n -> device, the block, device x_{n+1} -> host
                x_dev.copy_(x_host, non_blocking=True)
                step(x=x_dev)
                out_host.copy_(out, non_blocking=True)
                torch.cuda.synchronize(dev)
            else:
                B.moe_forward_host_io(cfg, x_host, *weights, out_host, ws, stream=stream)

        for _ in range(3):
            e2e_step()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
        res["e2e"] = {
            "value": replica_throughput(w.T * args.e2e_steps, world, e2e_s), "unit": "tokens/s",
            "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
            "path": ("pinned host x'_n -> moe_forward_block -> pinned host x_{n+1}, "
                     "synchronised per step") if args.block else
                    "moe_forward_host_io (pinned host x / out, synchronised per step)"}
    if rank != 0:
        return res

    # bytes per expert output: bf16 on request, and by default for e4m3 experts
    y_bytes = 2 if (cfg.flags & B.MOE_FLAG_EXPERT_OUT_BF16 or
                    (w.fp8 and not cfg.flags & B.MOE_FLAG_EXPERT_OUT_F32)) else 4
    res["roofline"], res["layer_roofline"], res["kernels"] = rooflines(w, idx_np, prof, ms_step,
                                                                      y_bytes)

    # ------------------------------------------------------------- the oracle on a sample
    if with_cpu:
        step()  # `out` holds this batch's result (every step computes the same)
        torch.cuda.synchronize(dev)
        cores = os.cpu_count() or 1
        n = min(w.T, sample)
        chk = oracle_check(layer, out, S.subset_rows(w.T, n, seed=1), cores)
        res["cpu_baseline"] = {"value": n / chk["seconds"], "unit": "tokens/s", "cores": cores,
                               "kind": "oracle",
                               "sample": f"{n} of {w.T} tokens (seed 1), fp64 C oracle, one "
                                         f"pass, {chk['seconds']:.1f} s"}
        acc = {k: v for k, v in chk.items() if k != "seconds"}
        if not args.block:
            acc["near_tie_tokens_all"] = near_ties_all(layer, cfg, ws)
            acc["tokens_all"] = int(w.T)
        acc["rule"] = ("max|GPU-oracle|/rms(oracle) on the sample, plain and beyond the bf16 "
                       "output's own rounding (2^-8|oracle|); bounds 1e-4 fp32, 2e-2 bf16, 6e-2 "
                       "fp8 experts on the latter")
        res["accuracy"] = acc
    return res


def run_ours(args, w, rank: int, world: int, local_rank: int):
    import torch
    from mixture_experts_ffn_gemm_gb300 import binding as B
    from mixture_experts_ffn_gemm_gb300 import build as BLD
    from mixture_experts_ffn_gemm_gb300 import synthetic as S

    if rank == 0:
        BLD.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    B.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    sample = args.cpu_sample or (512 if w.d >= 4096 else w.T)
    r = measure_workload(args, w, rank, world, dev, args.steps, args.warmup, sample,
                         with_e2e=not args.no_e2e, with_cpu=not args.no_cpu_baseline)
    others = {}
    if args.others and world == 1:
        torch.cuda.empty_cache()
        for name, steps, n in OTHER_WORKLOADS:
            try:
                o = measure_workload(args, S.WORKLOADS[name], rank, world, dev, steps,
                                     min(args.warmup, 5), n, with_e2e=False,
                                     with_cpu=not args.no_cpu_baseline)
                others[name] = {
                    "tokens": S.WORKLOADS[name].T, "value": o["value"], "unit": "tokens/s",
                    "ms_per_step": o["ms_per_step"], "steps": steps,
                    "layer_roofline": o.get("layer_roofline"), "roofline": o.get("roofline"),
                    "kernels": o.get("kernels"), "accuracy": o.get("accuracy"),
                    "gpu_launches": o["launches"], "clocks": o["clocks"]}
            except Exception as exc:  # reported, not fatal for the headline line
                others[name] = {"error": f"{type(exc).__name__}: {exc}"}
            torch.cuda.empty_cache()
    if rank != 0:
        return
    acc = r.get("accuracy") or {}
    line = {
        "metric": METRIC, "value": r["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.act == "f32" else ("e4m3" if w.fp8 else
                                               "int4 weights, bf16" if getattr(w, "int4", False)
                                               else "bf16"),
        "data": "synthetic",
        "config": layer_config(w, args.block, world),
        "roofline": r["roofline"],
        "layer_roofline": r["layer_roofline"],
        "cpu_baseline": r.get("cpu_baseline"),
        "e2e": r.get("e2e"),
        "near_tie_tokens": acc.get("near_tie_tokens_all", acc.get("near_tie_tokens")),
        "max_err_rms": acc.get("max_err_rms"),
        "accuracy": acc or None,
        "gpu_launches": r["launches"],
        "kernels": r["kernels"],
        "clocks": r["clocks"],
    }
    if others:
        line["other_workloads"] = others
    print(json.dumps(line), flush=True)

# ----------------------------------------------------------------------------------------------
# the dense block MLP (moe_dense_mlp): a second workload on the same GEMM kernels
# ----------------------------------------------------------------------------------------------
def dense_work(w) -> dict:
    """Algorithmic bytes and FLOPs of the dense MLP per kernel and for the whole MLP: weights once,
    x in and y out (and h between the two GEMMs, for the kernels)."""
    T, d, I = w.T, w.d, w.I
    ab = 4 if w.act == "f32" else 2
    return {"gemm13": (2 * I * d * ab + T * d * ab + T * I * ab, 2 * T * d * 2 * I),
            "gemm2": (d * I * ab + T * I * ab + T * d * ab, 2 * T * I * d),
            "layer": (3 * d * I * ab + 2 * T * d * ab, 6 * T * d * I)}


def time_dense_oracle(layer, rows, nthreads: int) -> float:
    from oracle import torch_bridge as OB
    t0 = time.perf_counter()
    OB.dense_mlp(layer, rows=rows, nthreads=nthreads)
    return time.perf_counter() - t0


def run_dense(args, w, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist
    from mixture_experts_ffn_gemm_gb300 import binding as B
    from mixture_experts_ffn_gemm_gb300 import build as BLD
    from mixture_experts_ffn_gemm_gb300 import synthetic as S

    cores = os.cpu_count() or 1
    if args.impl == "reference":
        if rank != 0:
            return
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        layer = S.make_dense(w, seed=0, device=dev)
        per_token = time_dense_oracle(layer, S.subset_rows(w.T, 1, seed=2), 1)
        budget_s = 150.0 / max(1, args.steps + args.warmup)
        n = args.cpu_sample or int(max(1, min(w.T, budget_s * cores / max(per_token, 1e-9))))
        rows = S.subset_rows(w.T, n, seed=1)
        for _ in range(args.warmup):
            time_dense_oracle(layer, rows, cores)
        secs = [time_dense_oracle(layer, rows, cores) for _ in range(args.steps)]
        tps = n / statistics.mean(secs)
        print(json.dumps({
            "impl": "reference", "metric": DENSE_METRIC, "value": tps, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * statistics.mean(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dense_config(w, world),
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} of {w.T} tokens (seed 1) per step, fp64 C oracle"},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return

    if rank == 0:
        BLD.build()
    if world > 1:
        dist.barrier()
    B.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    layer = S.make_dense(w, seed=rank, device=dev)  # each replica its own batch
    ws = torch.zeros(B.moe_dense_mlp_workspace_size(w.T, w.d, w.I, layer.x.dtype),
                     dtype=torch.uint8, device=dev)
    out = torch.empty(w.T, w.d, dtype=layer.x.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(x=layer.x, y=out):
        B.moe_dense_mlp(x, layer.W13, layer.W2, y, ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if B.moe_device_status(ws) != B.MOE_OK:
        raise RuntimeError("device status after warm-up")
    gpu_id = str(getattr(torch.cuda.get_device_properties(dev), "uuid", local_rank))
    if not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    B.moe_profile_enable(True)
    B.moe_profile_read()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = B.moe_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    launches = B.moe_launch_count() - launches0
    prof = B.moe_profile_read()
    B.moe_profile_enable(False)
    clocks = sampler.stop()
    if B.moe_device_status(ws) != B.MOE_OK:
        raise RuntimeError("device status after the timed steps")
    ms_step = max_over_ranks(ev0.elapsed_time(ev1), world, dev) / args.steps
    value = replica_throughput(w.T, world, ms_step / 1000.0)

    e2e = None
    if not args.no_e2e:  # host x -> device, the MLP, device y -> host, every step
        io_bytes = w.T * w.d * layer.x.element_size()
        x_host = layer.x.cpu().pin_memory()
        y_host = torch.empty(w.T, w.d, dtype=layer.x.dtype).pin_memory()
        x_dev = torch.empty_like(layer.x)

        def e2e_step():
            x_dev.copy_(x_host, non_blocking=True)
            step(x=x_dev)
            y_host.copy_(out, non_blocking=True)
            torch.cuda.synchronize(dev)

        for _ in range(3):
            e2e_step()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": replica_throughput(w.T * args.e2e_steps, world, e2e_s), "unit": "tokens/s",
               "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
               "path": "pinned host x -> moe_dense_mlp -> pinned host y, synchronised per step"}
    if rank != 0:
        return

    peaks, peak_src = load_peaks()
    work = dense_work(w)
    tc_peak = peaks["bf16_tflops"]  # burst: the timed loop runs well under a second
    kernels = {k: {"ms_per_launch": v[0] / max(v[1], 1), "launches": v[1]} for k, v in prof.items()}
    dom = max(prof.items(), key=lambda kv: kv[1][0])[0] if prof else None
    roof = None
    if dom is not None:
        by, fl = work["gemm2" if "gemm2" in dom else "gemm13"]
        sec = kernels[dom]["ms_per_launch"] / 1000.0
        if fl / (tc_peak * 1e12) > by / (peaks["hbm_gbs"] * 1e9):
            roof = {"kernel": dom, "bound": "tensor", "achieved": fl / sec / 1e12, "peak": tc_peak,
                    "unit": "TFLOP/s", "frac": fl / sec / 1e12 / tc_peak,
                    "peak_source": f"{peak_src} bf16_tflops (burst)", "work_per_launch": fl,
                    "frac_of_sustained_peak": fl / sec / 1e12 / peaks["bf16_tflops_sustained"]}
        else:
            roof = {"kernel": dom, "bound": "hbm", "achieved": by / sec / 1e9,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": by / sec / 1e9 / peaks["hbm_gbs"],
                    "peak_source": f"{peak_src} hbm_gbs", "work_per_launch": by}
        roof["traffic"] = None
    lb, lf = work["layer"]
    t_roof = max(lf / (tc_peak * 1e12), lb / (peaks["hbm_gbs"] * 1e9))
    cpu = None
    if not args.no_cpu_baseline:
        n = args.cpu_sample or min(w.T, 64)
        sec = time_dense_oracle(layer, S.subset_rows(w.T, n, seed=1), cores)
        cpu = {"value": n / sec, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} of {w.T} tokens (seed 1), fp64 C oracle, one pass, {sec:.1f} s"}
    print(json.dumps({
        "metric": DENSE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.act == "f32" else "bf16", "data": "synthetic",
        "config": dense_config(w, world),
        "roofline": roof,
        "layer_roofline": {"t_roof_ms": 1000 * t_roof, "frac": 1000 * t_roof / ms_step,
                           "bound": "tensor" if lf / (tc_peak * 1e12) > lb / (peaks["hbm_gbs"] * 1e9)
                           else "hbm", "algorithmic_bytes": lb, "algorithmic_flops": lf},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches), "kernels": kernels,
        "clocks": clocks}), flush=True)


def main():
    args = parse_args()
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload in S.DENSE_WORKLOADS:
        w = S.DENSE_WORKLOADS[args.workload]
        if args.tokens:
            w = w.with_tokens(args.tokens)
        if world > 1 and args.impl != "reference":
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        try:
            run_dense(args, w, rank, world, local_rank)
        finally:
            if world > 1 and args.impl != "reference":
                import torch.distributed as dist
                dist.destroy_process_group()
        return
    w = S.WORKLOADS[args.workload]
    if args.experts or args.tokens:
        from dataclasses import replace
        w = replace(w, name=f"{w.name}_E{args.experts or w.E}_T{args.tokens or w.T}",
                    E=args.experts or w.E, T=args.tokens or w.T)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
