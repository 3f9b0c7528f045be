"""What an ideal bf16 implementation of the layer reaches against the fp64 oracle (TEST HELPER).

A bf16 implementation has to round some values to bf16 because they are bf16 GEMM operands or the
result: h (the W2 operand), the layer's output, and on the K3 latent path also x_lat (the latent
experts' operand) and u_hat (the up-projection's operand).  This model computes the layer exactly
(fp64, numpy matmuls) with the oracle's own routing and gates, and rounds exactly those values to
bf16 (nearest, ties to even) -- nothing else.  With every rounding switched off it is the oracle's
definition itself, which the CPU tests check against oracle.forward to 1e-12; with the roundings on,
its distance to the oracle is the error floor of any bf16 pipeline with these operands.

Sources: "Kimi K2 · Transformer blocks > MoE transformer block", "Mixture of experts" steps (g, u,
a, h, E_i, the gate-weighted sum and the shared expert); "Kimi K3 · Latent up-projection", its
equation (latent down-projection, RMSNorm, up-projection, shared expert on the full-width x).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import torch_bridge as OB


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rn(v: np.ndarray, on: bool) -> np.ndarray:
    return OB.round_bf16(v) if on else v


def _silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def _mlp(x: np.ndarray, W13: np.ndarray, W2: np.ndarray, I: int, round_h: bool) -> np.ndarray:
    """SwiGLU rows: h = SiLU(x W1^T) * (x W3^T), then h W2^T (W13 holds W1 rows, then W3 rows)."""
    g = x @ W13[:I].T
    u = x @ W13[I:].T
    return _rn(_silu(g) * u, round_h) @ W2.T


def ideal_forward(layer, rows=None, round_h=True, round_out=True, round_xlat=True,
                  round_uhat=True, round_y=False) -> dict:
    """The layer on ``rows`` (all by default) with only the listed bf16 roundings; returns the
    output and the oracle's routing it used.  ``round_y`` also rounds every expert's output
    E_i(x) (and the shared expert's) to bf16 before the gate-weighted sum, as a pipeline that
    keeps its expert outputs in bf16 does."""
    w = layer.w
    T = layer.x.shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    xr = layer.x[torch.as_tensor(rows, device=layer.x.device)]
    xm, W_r, b = OB.route_inputs(layer, torch.as_tensor(rows))
    cfg = OB.config(layer, len(rows))
    rt = oracle.route(cfg, xm, W_r, b)
    x = _f64(xr)
    if w.d_latent:
        x_e = _rn(x @ _f64(layer.W_down).T, round_xlat)
    else:
        x_e = x
    y = np.zeros((len(rows), w.d_expert), np.float64)
    for e in np.unique(rt["idx"]):
        t, j = np.nonzero(rt["idx"] == e)
        ye = _rn(_mlp(x_e[t], _f64(layer.W13[e]), _f64(layer.W2[e]), w.I, round_h), round_y)
        y[t] += rt["gates"][t, j][:, None] * ye
    shared = (_rn(_mlp(x, _f64(layer.Ws13), _f64(layer.Ws2), w.I_shared, round_h), round_y)
              if w.n_shared else np.zeros((len(rows), w.d)))
    if w.d_latent:
        if w.latent_norm:
            y = y / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + w.rms_eps)
        y = _rn(y, round_uhat) @ _f64(layer.W_up).T
    out = _rn(y + shared, round_out)
    return {"out": out, "margin": rt["margin"], "idx": rt["idx"]}


def pages_combine_forward(layer, rows=None) -> dict:
    """The K2 layer with the rounding sequence of the pages' own code ("Kimi K3 · Latent
    up-projection", `moe_infer` back half, and the block's `forward`): h rounded to bf16 (the W2
    operand), each expert's output rounded to bf16 (the module's output type), cast to the gate
    type (fp32) and multiplied by its gate, summed over the slots, cast back to bf16; the shared
    expert's output in bf16; the two added in bf16.  Everything else exact, as in
    ideal_forward."""
    w = layer.w
    assert not w.d_latent, "the K2 path"
    T = layer.x.shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    xr = layer.x[torch.as_tensor(rows, device=layer.x.device)]
    xm, W_r, b = OB.route_inputs(layer, torch.as_tensor(rows))
    cfg = OB.config(layer, len(rows))
    rt = oracle.route(cfg, xm, W_r, b)
    x = _f64(xr)
    y = np.zeros((len(rows), w.d), np.float64)
    for e in np.unique(rt["idx"]):
        t, j = np.nonzero(rt["idx"] == e)
        ye = OB.round_bf16(_mlp(x[t], _f64(layer.W13[e]), _f64(layer.W2[e]), w.I, True))
        gates = rt["gates"][t, j].astype(np.float32).astype(np.float64)  # the gate type
        y[t] += gates[:, None] * ye
    routed = OB.round_bf16(y)
    shared = (OB.round_bf16(_mlp(x, _f64(layer.Ws13), _f64(layer.Ws2), w.I_shared, True))
              if w.n_shared else np.zeros_like(routed))
    return {"out": OB.round_bf16(routed + shared), "margin": rt["margin"], "idx": rt["idx"]}


def errors(got: np.ndarray, ref: np.ndarray) -> dict:
    """Plain max error, max error beyond the result's own bf16 rounding, rms error; each over
    rms(ref)."""
    rms = float(np.sqrt(np.mean(ref * ref)))
    d = np.abs(got - ref)
    return {"plain": float(d.max()) / rms,
            "beyond_rounding": float(np.max(d - 2.0 ** -8 * np.abs(ref))) / rms,
            "rms": float(np.sqrt(np.mean(d * d))) / rms}
