"""Turn a synthetic layer's torch tensors into the oracle's numpy inputs (TEST INFRASTRUCTURE).

Only host copies are made; nothing here computes any part of the layer.  Experts are copied one by
one and only when asked for, so that a sample of tokens at full size needs only the experts those
tokens select.
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np
import torch

from . import Config, Mat
from . import dense_mlp as _dense_mlp


def _np_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def mat(t: Optional[torch.Tensor], scale: Optional[torch.Tensor] = None) -> Optional[Mat]:
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return Mat(_np_bits(t), "bf16")
    if t.dtype == torch.float8_e4m3fn:
        return Mat(_np_bits(t), "e4m3", _np_bits(scale.float()))
    if t.dtype == torch.uint8:  # 4-bit integer groups: packed codes, bf16 scales [K/32][rows]
        return Mat(_np_bits(t), "int4", _np_bits(scale.float()))
    if t.dtype == torch.float32:
        return Mat(_np_bits(t), "f32")
    if t.dtype == torch.float64:
        return Mat(_np_bits(t), "f64")
    raise TypeError(f"unsupported dtype {t.dtype}")


def config(layer, T: Optional[int] = None) -> Config:
    w = layer.w
    return Config(T=w.T if T is None else T, d=w.d, E=w.E, k=w.k, I=w.I, I_shared=w.I_shared,
                  n_shared=w.n_shared, d_latent=w.d_latent, latent_norm=w.latent_norm,
                  fp8=int(w.fp8), quant_block=w.quant_block, gate_scale=w.gate_scale,
                  rms_eps=w.rms_eps)


def expert_mats(layer, experts: Iterable[int]):
    """Per-expert W13 / W2 lists with host copies of ``experts`` only (None elsewhere)."""
    E = layer.w.E
    W13 = [None] * E
    W2 = [None] * E
    for e in sorted(set(int(v) for v in experts)):
        s13 = layer.W13_scale[e] if layer.W13_scale is not None else None
        s2 = layer.W2_scale[e] if layer.W2_scale is not None else None
        W13[e] = mat(layer.W13[e], s13)
        W2[e] = mat(layer.W2[e], s2)
    return W13, W2


def route_inputs(layer, rows: Optional[torch.Tensor] = None):
    """(x Mat, W_r, b) for the given token rows (all rows by default)."""
    x = layer.x if rows is None else layer.x[rows.to(layer.x.device)]
    return mat(x), _np_bits(layer.W_r.float()), _np_bits(layer.b.float())


def forward(layer, rows: Optional[torch.Tensor] = None, experts: Optional[Iterable[int]] = None,
            nthreads: int = 1) -> dict:
    """Oracle forward on ``rows`` of the layer's tokens.  ``experts`` limits the expert weights
    copied to the host; by default the oracle's own routing of these rows (which reads no expert
    weight) picks them, and only those experts are copied."""
    from . import forward as orc_forward, route as orc_route
    x, W_r, b = route_inputs(layer, rows)
    cfg = config(layer, x.data.shape[0])
    if experts is None:
        experts = np.unique(orc_route(cfg, x, W_r, b)["idx"])
    W13, W2 = expert_mats(layer, experts)
    return orc_forward(cfg, x, W_r, b, W13, W2, mat(layer.Ws13, layer.Ws13_scale),
                       mat(layer.Ws2, layer.Ws2_scale), mat(layer.W_down), mat(layer.W_up),
                       nthreads=nthreads)


def dense_mlp(layer, rows: Optional[torch.Tensor] = None, nthreads: int = 1) -> np.ndarray:
    """The oracle's dense block MLP on a synthetic DenseLayer (optionally a subset of its rows):
    fp64 [rows][d]."""
    x = layer.x if rows is None else layer.x[rows.to(layer.x.device)]
    return _dense_mlp(mat(x.cpu()), mat(layer.W13.cpu()), mat(layer.W2.cpu()),
                            nthreads=nthreads)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (8 significant bits, ties to even), in fp64.
    Normal-range values only (the block's normalised activations are O(1))."""
    m, e = np.frexp(np.asarray(v, dtype=np.float64))  # v = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def block_forward(layer, norm_w: torch.Tensor, rows: Optional[torch.Tensor] = None,
                  nthreads: int = 1) -> dict:
    """The FFN half of a transformer block around the layer ("Kimi K2 · Transformer blocks > MoE
    transformer block": x_ffn = RMSNorm(x'_n), the mixture of experts, x_{n+1} = x'_n + D_ffn),
    in fp64 on ``rows`` of the layer's x, which plays x'_n.  The RMSNorm is the oracle's unit
    RMSNorm times the weight; x_ffn is then rounded once to the activation type, as the layer's
    GEMM operand.  Returns the layer forward's dict with "delta" (D_ffn), "x_ffn" and
    "out" = x'_n + D_ffn."""
    from . import forward as orc_forward, route as orc_route, rmsnorm_unit
    xr = layer.x if rows is None else layer.x[rows.to(layer.x.device)]
    x64 = _np_bits(xr.float()).astype(np.float64)
    g64 = _np_bits(norm_w.float()).astype(np.float64)
    eps = float(layer.w.rms_eps)
    xn = np.stack([rmsnorm_unit(r, eps) for r in x64]) * g64[None, :] if len(x64) else x64
    # x_ffn is the router's and the experts' GEMM operand: rounded once to the activation type
    if layer.w.act == "bf16":
        xn = round_bf16(xn)
    elif layer.w.act == "f32":
        xn = xn.astype(np.float32).astype(np.float64)
    x = Mat(np.ascontiguousarray(xn), "f64")
    W_r, b = _np_bits(layer.W_r.float()), _np_bits(layer.b.float())
    cfg = config(layer, xn.shape[0])
    experts = np.unique(orc_route(cfg, x, W_r, b)["idx"])
    W13, W2 = expert_mats(layer, experts)
    res = orc_forward(cfg, x, W_r, b, W13, W2, mat(layer.Ws13, layer.Ws13_scale),
                      mat(layer.Ws2, layer.Ws2_scale), mat(layer.W_down), mat(layer.W_up),
                      nthreads=nthreads)
    res["delta"] = res["out"]
    res["x_ffn"] = xn
    res["out"] = x64 + res["out"]
    return res
