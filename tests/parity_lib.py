"""Helpers for the GPU parity tests: run the layer through the C ABI (stage by stage and as one
moe_forward), and compare with the fp64 oracle on the same seeded inputs.

The rule, the same for every workload and every test:
  * routing: the oracle's selection rule fed the GPU's own fp32 logits must give bit-identical
    expert indices, except tokens whose k-th / (k+1)-th key margin is below 1e-5 (near ties,
    counted and reported, not compared);
  * fp32 values (the fp32 layer's outputs, the fp32 expert rows of y_perm, the shared expert's
    rows): max |GPU - oracle| <= tol * rms(oracle);
  * values rounded to bf16 as the layer's result (bf16 and fp8-expert outputs, and the expert
    rows of y_perm when they are bf16 on request): the same bound on
    the error beyond the result's own rounding, max(|GPU - oracle| - 2^-8 |oracle|) <= tol *
    rms(oracle).  2^-8 |v| bounds half a bf16 ulp of v, the representation error of the output
    type itself, which no bf16 result can avoid; an output near 5 rms already carries up to
    1.95e-2 rms of it.  The plain max |GPU - oracle| / rms is reported next to it every time;
  * in addition the rms of the error must stay below 1e-5 (fp32) / 5e-3 (bf16) / 2e-2 (fp8) of
    rms(oracle), which catches a systematic error the max bound could hide.
tol is 1e-4 for the fp32 layer, 2e-2 for the bf16 layer and 6e-2 for fp8 experts, against the
unrounded fp64 oracle.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import numpy as np
import torch

import oracle
from oracle import torch_bridge as OB
from mixture_experts_ffn_gemm_gb300 import binding as B

TOL = {"f32": 1e-4, "bf16": 2e-2, "fp8": 6e-2}
RMS_TOL = {"f32": 1e-5, "bf16": 5e-3, "fp8": 2e-2}


def kind(w) -> str:
    """Tolerance class of a workload: fp32, bf16, or fp8 experts."""
    return "fp8" if w.fp8 else w.act
NEAR_TIE = 1e-5
NTHREADS = os.cpu_count() or 4


@dataclass
class GpuResult:
    logits: torch.Tensor
    idx: torch.Tensor
    weight: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    perm_src: torch.Tensor
    perm_dst: torch.Tensor
    y_perm: torch.Tensor
    out: torch.Tensor       # stage by stage
    out_fwd: torch.Tensor   # moe_forward
    status: int
    status_fwd: int


def run_gpu(layer, flags: int = 0) -> GpuResult:
    w = layer.w
    cfg = B.config_for(w, T=layer.x.shape[0], flags=flags)
    T, E, k, d, de = layer.x.shape[0], w.E, w.k, w.d, w.d_expert
    dev = layer.x.device
    act = layer.x.dtype
    ws = B.alloc_workspace(cfg, dev)
    logits = torch.full((T, E), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    wgt = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
    B.moe_router(cfg, layer.x, layer.W_r, layer.b, logits, idx, wgt, ws)
    counts = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 2,), -7, dtype=torch.int32, device=dev)
    perm_src = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    perm_dst = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    B.moe_permute(cfg, idx, counts, offsets, perm_src, perm_dst, ws)
    # bf16 expert outputs on request, and by default for e4m3 experts
    y_bf16 = flags & B.MOE_FLAG_EXPERT_OUT_BF16 or (w.fp8 and not flags & B.MOE_FLAG_EXPERT_OUT_F32)
    y_dtype = torch.bfloat16 if y_bf16 else torch.float32
    y_perm = torch.full((T * k * de + T * w.n_shared * d,), float("nan"), dtype=y_dtype,
                        device=dev)
    B.moe_experts(cfg, layer.x, offsets, perm_src, layer.W13, layer.W2, layer.W13_scale,
                  layer.W2_scale, layer.Ws13, layer.Ws2, layer.Ws13_scale, layer.Ws2_scale,
                  layer.W_down, y_perm, ws)
    out = torch.full((T, d), float("nan"), dtype=act, device=dev)
    B.moe_combine(cfg, y_perm, perm_dst, wgt, layer.W_up, out, ws)
    status = B.moe_device_status(ws)
    out_fwd = torch.full((T, d), float("nan"), dtype=act, device=dev)
    B.moe_forward(cfg, layer.x, *B.layer_weights(layer), out_fwd, ws)
    status_fwd = B.moe_device_status(ws)
    return GpuResult(logits, idx, wgt, counts, offsets, perm_src, perm_dst, y_perm, out, out_fwd,
                  status, status_fwd)


def check_routing(layer, g: GpuResult) -> dict:
    """Bit-exact indices (near ties excepted) and gates against the oracle's rule on the GPU's
    logits.  The selected set is compared exactly; the slot order too, except between selected
    experts whose keys are less than the near-tie margin apart (their order is decided by the
    last bits of two sigmoid evaluations, as a near tie at the selection boundary is).  Returns
    counts for reporting."""
    cfg = OB.config(layer, layer.x.shape[0])
    z = g.logits.cpu().numpy()
    assert np.isfinite(z).all(), "router logits not written"
    idx_o, gates_o, margin, keys = oracle.route_from_logits(cfg, z, layer.b.cpu().numpy(),
                                                            with_keys=True)
    near = margin < NEAR_TIE
    idx_g = g.idx.cpu().numpy()
    # slots whose order is unique: separated from both neighbours by at least the margin
    gap = np.abs(np.diff(keys.astype(np.float64), axis=1)) >= NEAR_TIE
    fixed = np.ones_like(idx_o, dtype=bool)
    fixed[:, 1:] &= gap
    fixed[:, :-1] &= gap
    set_mism = (np.sort(idx_g, 1) != np.sort(idx_o, 1)).any(1)
    order_mism = ((idx_g != idx_o) & fixed).any(1)
    mism = set_mism | order_mism
    assert not (mism & ~near).any(), \
        f"{int((mism & ~near).sum())} tokens routed differently away from a near tie"
    wg = g.weight.cpu().numpy().astype(np.float64)
    ok = ~near
    # gates matched by expert (the slot order may differ where keys are within the margin)
    og, oo = np.argsort(idx_g, 1), np.argsort(idx_o, 1)
    wg_e = np.take_along_axis(wg, og, 1)
    wo_e = np.take_along_axis(gates_o, oo, 1)
    assert np.allclose(wg_e[ok], wo_e[ok], rtol=2e-6, atol=2e-6)
    assert np.allclose(wg.sum(1), layer.w.gate_scale, rtol=0, atol=2e-5)
    return {"near_ties": int(near.sum()), "tokens": int(len(near))}


def check_permutation(layer, g: GpuResult):
    """counts / offsets / permutation bit-exact against a stable sort of the expert ids."""
    T, E, k = layer.x.shape[0], layer.w.E, layer.w.k
    idx = g.idx.cpu().numpy().reshape(-1)
    counts = g.counts.cpu().numpy()
    offsets = g.offsets.cpu().numpy()
    assert np.array_equal(counts[:E], np.bincount(idx, minlength=E))
    assert counts[E] == T * layer.w.n_shared
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    perm_src = g.perm_src.cpu().numpy()
    perm_dst = g.perm_dst.cpu().numpy()
    assert np.array_equal(perm_src, np.argsort(idx, kind="stable"))
    assert np.array_equal(perm_dst[perm_src], np.arange(T * k))


def rel_err(a: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(a - ref))) / max(rms, 1e-30)


def rms_err(a: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.sqrt(np.mean((a - ref) ** 2))) / max(rms, 1e-30)


BF16_HALF_ULP = 2.0 ** -8  # half a bf16 ulp of v is at most 2^-8 |v| (8 significant bits)


def beyond_rounding_err(a: np.ndarray, ref: np.ndarray) -> float:
    """max(|a - ref| - 2^-8 |ref|) / rms(ref): the error beyond a bf16 result's own rounding."""
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(a - ref) - BF16_HALF_ULP * np.abs(ref))) / max(rms, 1e-30)


def compare(got: np.ndarray, ref: np.ndarray, act: str, tol=None, rounded: bool = False) -> dict:
    """The parity rule of this module on one set of values.  ``rounded``: the values are the
    layer's bf16 result (the bound applies beyond their own rounding); else they are fp32 values
    (the plain bound).  Returns the bounded figure ("err"), the plain one and the rms one."""
    tol = tol if tol is not None else TOL[act]
    e_plain = rel_err(got, ref)
    e_max = beyond_rounding_err(got, ref) if rounded and act in ("bf16", "fp8") else e_plain
    e_rms = rms_err(got, ref)
    assert e_max <= tol, f"max err / rms = {e_max:.3e} > {tol} (plain {e_plain:.3e})"
    assert e_rms <= RMS_TOL[act], f"rms err = {e_rms:.3e} > {RMS_TOL[act]}"
    return {"err": e_max, "err_plain": e_plain, "rms_err": e_rms}


class HostExperts:
    """Host copies of a layer's expert weights for the oracle, each expert copied once and only
    when a compared token or row needs it (a full K2 layer is 34 GB)."""

    def __init__(self, layer):
        self.layer = layer
        self.W13 = [None] * layer.w.E
        self.W2 = [None] * layer.w.E
        self._shared = None

    def need(self, experts):
        missing = [int(e) for e in np.unique(np.asarray(experts, dtype=np.int64))
                   if self.W13[int(e)] is None]
        if missing:
            W13, W2 = OB.expert_mats(self.layer, missing)
            for e in missing:
                self.W13[e], self.W2[e] = W13[e], W2[e]
        return self

    def shared(self):
        if self._shared is None:
            L = self.layer
            self._shared = (OB.mat(L.Ws13, L.Ws13_scale), OB.mat(L.Ws2, L.Ws2_scale),
                            OB.mat(L.W_down), OB.mat(L.W_up))
        return self._shared


def oracle_forward(layer, rows, host: HostExperts, nthreads: int = NTHREADS) -> dict:
    """The oracle on ``rows`` of the layer's tokens (its own routing), with the expert weights
    from ``host``."""
    x, W_r, b = OB.route_inputs(layer, torch.as_tensor(rows))
    cfg = OB.config(layer, x.data.shape[0])
    host.need(oracle.route(cfg, x, W_r, b)["idx"])
    return oracle.forward(cfg, x, W_r, b, host.W13, host.W2, *host.shared(), nthreads=nthreads)


def check_outputs(layer, g: GpuResult, rows=None, tol=None, host: HostExperts = None) -> dict:
    """Layer outputs (and the shared expert rows of y_perm) against the oracle on `rows`
    (all rows by default), near-tie tokens excluded and counted."""
    T = layer.x.shape[0]
    rows_np = np.arange(T) if rows is None else np.asarray(rows)
    host = host or HostExperts(layer)
    ref = oracle_forward(layer, rows_np, host)
    keep = ref["margin"] >= NEAR_TIE
    out = g.out.float().cpu().numpy()[rows_np]
    out_fwd = g.out_fwd.float().cpu().numpy()[rows_np]
    assert np.isfinite(out).all() and np.isfinite(out_fwd).all()
    assert np.array_equal(out, out_fwd), "moe_forward differs from the stage-by-stage path"
    res = {"compared": int(keep.sum()), "sample_near_ties": int((~keep).sum())}
    act = kind(layer.w)
    if keep.any():
        res.update(compare(out[keep], ref["out"][keep], act, tol, rounded=act != "f32"))
    w = layer.w
    if w.n_shared:
        P, de, d = T * w.k, w.d_expert, w.d
        ysh = g.y_perm[P * de:].view(T, d).float().cpu().numpy()[rows_np]
        res["shared_err"] = compare(ysh, ref["shared"], act, tol,
                                    rounded=g.y_perm.dtype == torch.bfloat16)["err"]
    return res


def expert_rows_to_check(g: GpuResult, E: int, nrows: int, seed: int) -> np.ndarray:
    """Permuted rows of y_perm to compare: ``nrows`` seeded random ones, plus the last row of
    every non-empty expert (its ragged tail tile) and the very last row."""
    offsets = g.offsets.cpu().numpy().astype(np.int64)
    P = int(offsets[E])
    if P == 0:
        return np.zeros(0, np.int64)
    rng = np.random.default_rng(seed)
    ends = offsets[1:E + 1]
    tails = ends[ends > offsets[:E]] - 1
    pick = rng.choice(P, size=min(nrows, P), replace=False)
    return np.unique(np.concatenate([pick, tails, [P - 1]]))


def check_expert_rows(layer, g: GpuResult, nrows: int = 64, seed: int = 0, tol=None,
                      host: HostExperts = None) -> dict:
    """Permuted rows of y_perm against one oracle SwiGLU of that row's token and expert (K2
    path): isolates the grouped GEMMs from the combine.  Compares ``nrows`` seeded rows and the
    last row of every expert, so that every expert's last (ragged) row tile is checked."""
    w = layer.w
    if w.d_latent:
        return {}
    T, k, d = layer.x.shape[0], w.k, w.d
    P = T * k
    rows = expert_rows_to_check(g, w.E, nrows, seed)
    if rows.size == 0:
        return {"expert_rows": 0}
    perm_src = g.perm_src.cpu().numpy()
    idx = g.idx.cpu().numpy().reshape(-1)
    src = perm_src[rows].astype(np.int64)
    toks, exps = src // k, idx[src]
    host = host or HostExperts(layer)
    host.need(exps)
    y = g.y_perm[: P * d].view(P, d)
    got = y[torch.as_tensor(rows, device=y.device)].float().cpu().numpy()
    xs = layer.x[torch.as_tensor(toks, device=layer.x.device)].double().cpu().numpy()
    quant = w.fp8

    def one(i):
        e = int(exps[i])
        return oracle.swiglu_row(xs[i], host.W13[e], host.W2[e], I=w.I, qb=w.quant_block,
                                 quant_act=quant)

    from concurrent.futures import ThreadPoolExecutor  # the oracle's C call releases the GIL
    with ThreadPoolExecutor(max_workers=NTHREADS) as ex:
        ref = np.stack(list(ex.map(one, range(rows.size))))
    worst = {"err": 0.0, "err_plain": 0.0, "rms_err": 0.0}
    rounded = g.y_perm.dtype == torch.bfloat16  # bf16 expert outputs on request
    for i in range(rows.size):
        r = compare(got[i], ref[i], kind(w), tol, rounded=rounded)
        worst = {kk: max(worst[kk], r[kk]) for kk in worst}
    return {"expert_rows": int(rows.size), "expert_rows_err": worst["err"]}
