"""Seeded synthetic inputs for the MoE FFN layer: activations and random-init weights.

This module holds none of the layer's arithmetic (no routing, no GEMM, no activation quantisation):
it only draws tensors.  It is the one module that both the CUDA path and the fp64 oracle's tests
consume, so that both see exactly the same stored values.

Workloads (shapes from the nnterp "kimi_k2" Config table: hidden_size 7168, n_routed_experts 384,
num_experts_per_tok 8, moe_intermediate_size 2048, n_shared_experts 1, routed_scaling_factor 2.827;
the latent width 3584 from "Kimi K3 · Latent up-projection"):

=================  ======  =====  ===  ==  ====  ======  =====================================
name               T       d      E    k   I     latent  values
=================  ======  =====  ===  ==  ====  ======  =====================================
tiny_fp32          64      256    16   4   128   -       fp32; x~N(0,1); W~N(0,1/fan_in);
                                                          b~U(-0.1,0.1)
k2_decode_bf16     128     7168   384  8   2048  -       bf16; x~N(0,1); W~N(0,0.02^2);
                                                          b~U(-0.05,0.05)
k2_prefill_bf16    16384   7168   384  8   2048  -       bf16; x = one of 16 N(0,1) centres +
                                                          0.5 N(0,1) noise; W, b as decode
k3_latent_bf16     8192    7168   384  8   2048  3584    bf16; x~N(0,1); W~N(0,1/fan_in);
                                                          b~U(-0.05,0.05); RMSNorm on
k2_fp8             8192    7168   384  8   2048  -       as prefill; expert weights e4m3 with one
                                                          fp32 scale (amax/448) per 128x128 block
=================  ======  =====  ===  ==  ====  ======  =====================================

Dense block MLP workloads (the first block's DeepseekV3MLP, nnterp "kimi_k2" "Printout":
gate_proj / up_proj 7168 -> 18432, down_proj 18432 -> 7168):

============================  ======  =====  =====  ==========================================
name                          T       d      I      values
============================  ======  =====  =====  ==========================================
tiny_dense_fp32               48      64     96     fp32; x~N(0,1); W~N(0,1/fan_in)
k2_dense_decode_bf16          128     7168   18432  bf16; x~N(0,1); W~N(0,0.02^2)
k2_dense_prefill_bf16         16384   7168   18432  bf16; x as k2_prefill_bf16; W~N(0,0.02^2)
============================  ======  =====  =====  ==========================================

Draw order for a dense workload: x, W13 (W1 rows, then W3 rows), W2.

Readings: "N(0, 1/fan_in)" is a variance (std = fan_in**-0.5); "N(0, 0.02)" is a standard deviation
(the usual initializer range); the 16 cluster centres are picked uniformly per token.

Draw order (fixed): x, W_r, b, routed W13 (expert by expert), routed W2 (expert by expert), shared
W13, shared W2, W_down, W_up.  Every draw uses one ``torch.Generator`` on the target device seeded
with ``seed``; the same seed gives the same values on the same device type.

Layouts (the pages' Linear weights are stored [out, in]):
  x [T, d];  W_r [E, d] fp32;  b [E] fp32;
  W13 [E, 2I, d_e] (rows 0..I-1 = W1 = gate_proj, rows I..2I-1 = W3 = up_proj);  W2 [E, d_e, I];
  Ws13 [2 I_s, d];  Ws2 [d, I_s];  W_down [L, d];  W_up [d, L];  (d_e = L on the latent path)
  fp8: W13 / W2 / Ws13 / Ws2 as float8_e4m3fn bytes plus fp32 block scales
       [E, 2I/128, d/128], [E, d/128, I/128], [2I_s/128, d/128], [d/128, I_s/128].
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, Optional

import torch

GATE_SCALE = 2.827
RMS_EPS = 1e-6


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    I_shared: int
    n_shared: int = 1
    d_latent: int = 0
    latent_norm: int = 0
    act: str = "bf16"        # activation / weight storage: "f32" | "bf16"
    fp8: bool = False        # expert weights e4m3 + block scales, activations quantised
    int4: bool = False       # expert weights 4-bit integer groups of 32 (bf16 scales)
    x_dist: str = "normal"   # "normal" | "clusters16"
    w_init: str = "std0.02"  # "std0.02" | "fan_in"
    bias_range: float = 0.05
    gate_scale: float = GATE_SCALE
    rms_eps: float = RMS_EPS
    quant_block: int = 128

    @property
    def d_expert(self) -> int:
        return self.d_latent if self.d_latent > 0 else self.d

    def with_tokens(self, T: int) -> "Workload":
        return replace(self, T=T)


WORKLOADS: Dict[str, Workload] = {
    "tiny_fp32": Workload("tiny_fp32", T=64, d=256, E=16, k=4, I=128, I_shared=128, act="f32",
                          w_init="fan_in", bias_range=0.1),
    "k2_decode_bf16": Workload("k2_decode_bf16", T=128, d=7168, E=384, k=8, I=2048,
                               I_shared=2048),
    "k2_prefill_bf16": Workload("k2_prefill_bf16", T=16384, d=7168, E=384, k=8, I=2048,
                                I_shared=2048, x_dist="clusters16"),
    "k3_latent_bf16": Workload("k3_latent_bf16", T=8192, d=7168, E=384, k=8, I=2048,
                               I_shared=2048, d_latent=3584, latent_norm=1, w_init="fan_in"),
    "k2_fp8": Workload("k2_fp8", T=8192, d=7168, E=384, k=8, I=2048, I_shared=2048,
                       x_dist="clusters16", fp8=True),
    "k2_int4_decode": Workload("k2_int4_decode", T=128, d=7168, E=384, k=8, I=2048,
                               I_shared=2048, int4=True, quant_block=32),
}


@dataclass(frozen=True)
class DenseWorkload:
    name: str
    T: int
    d: int
    I: int
    act: str = "bf16"
    x_dist: str = "normal"
    w_init: str = "std0.02"

    def with_tokens(self, T: int) -> "DenseWorkload":
        return replace(self, T=T)


DENSE_WORKLOADS: Dict[str, DenseWorkload] = {
    "tiny_dense_fp32": DenseWorkload("tiny_dense_fp32", T=48, d=64, I=96, act="f32",
                                     w_init="fan_in"),
    "k2_dense_decode_bf16": DenseWorkload("k2_dense_decode_bf16", T=128, d=7168, I=18432),
    "k2_dense_prefill_bf16": DenseWorkload("k2_dense_prefill_bf16", T=16384, d=7168, I=18432,
                                           x_dist="clusters16"),
}


@dataclass
class DenseLayer:
    """The dense block MLP's input and weights, resident on one device."""
    w: DenseWorkload
    x: torch.Tensor
    W13: torch.Tensor
    W2: torch.Tensor


@dataclass
class Layer:
    """One layer's inputs and weights, resident on one device."""
    w: Workload
    x: torch.Tensor
    W_r: torch.Tensor
    b: torch.Tensor
    W13: torch.Tensor
    W2: torch.Tensor
    Ws13: Optional[torch.Tensor] = None
    Ws2: Optional[torch.Tensor] = None
    W_down: Optional[torch.Tensor] = None
    W_up: Optional[torch.Tensor] = None
    W13_scale: Optional[torch.Tensor] = None
    W2_scale: Optional[torch.Tensor] = None
    Ws13_scale: Optional[torch.Tensor] = None
    Ws2_scale: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)


def _std(w: Workload, fan_in: int) -> float:
    return fan_in ** -0.5 if w.w_init == "fan_in" else 0.02


def _act_dtype(w: Workload) -> torch.dtype:
    return torch.float32 if w.act == "f32" else torch.bfloat16


def _block_quantize(m: torch.Tensor, qb: int):
    """Store a weight matrix as e4m3 codes with one fp32 scale (amax/448, 1 for an all-zero
    block) per qb x qb block.  Input preparation for the fp8 workload (the checkpoint format)."""
    R, C = m.shape
    assert R % qb == 0 and C % qb == 0
    blk = m.reshape(R // qb, qb, C // qb, qb).float()
    amax = blk.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blk / scale[:, None, :, None]).clamp(-448.0, 448.0).reshape(R, C)
    return q.to(torch.float8_e4m3fn), scale.contiguous()


# nibble n of a packed 32-bit word holds code _W4_CODE_OF_NIBBLE[n] of its 8 channels
_W4_CODE_OF_NIBBLE = (0, 2, 4, 6, 1, 3, 5, 7)


def _int4_quantize(m: torch.Tensor, group: int = 32):
    """Store a weight matrix [R][C] as 4-bit integer groups (the MOE_INT4 format): per row and 32
    input channels a bf16 scale (amax / 7, rounded to bf16; 1 for an all-zero group) and codes
    round(w / scale) clamped to -8..7, stored as nibbles u = code + 8, packed eight to a
    little-endian 32-bit word with code i in nibble (i / 2) + 4 (i % 2).  Returns (packed uint8
    [R][C/2], scales bf16 [C/32][R]).  Input preparation for the int4 workload."""
    R, C = m.shape
    assert C % group == 0 and C % 8 == 0
    g = m.float().reshape(R, C // group, group)
    scale = (g.abs().amax(dim=2) / 7.0).to(torch.bfloat16)
    scale = torch.where(scale == 0, torch.ones_like(scale), scale)
    codes = torch.round(g / scale.float()[:, :, None]).clamp(-8, 7).to(torch.int32) + 8
    words = codes.reshape(R, C // 8, 8)
    nib = words[:, :, list(_W4_CODE_OF_NIBBLE)]  # nibble n's code
    packed = (nib[:, :, 0::2] | (nib[:, :, 1::2] << 4)).to(torch.uint8)  # byte b: nibbles 2b, 2b+1
    return packed.reshape(R, C // 2).contiguous(), scale.t().contiguous()


def make_layer(w: Workload, seed: int = 0, device="cuda") -> Layer:
    """Draw one layer's inputs and weights on ``device`` from ``seed``."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    adt = _act_dtype(w)
    T, d, E, I, Is, L = w.T, w.d, w.E, w.I, w.I_shared, w.d_latent
    de = w.d_expert

    def randn(*shape, std=1.0):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std

    # x
    if w.x_dist == "clusters16":
        centres = randn(16, d)
        member = torch.randint(0, 16, (T,), generator=g, device=device)
        x = centres[member] + 0.5 * randn(T, d)
    else:
        x = randn(T, d)
    x = x.to(adt).contiguous()
    # router
    W_r = randn(E, d, std=_std(w, d)).contiguous()
    b = ((torch.rand(E, generator=g, device=device, dtype=torch.float32) * 2 - 1)
         * w.bias_range).contiguous()

    qb = w.quant_block
    W13_scale = W2_scale = None
    if w.int4:  # packed codes [rows][K/2] and bf16 scales [K/32][rows] per expert
        W13 = torch.empty(E, 2 * I, de // 2, device=device, dtype=torch.uint8)
        W2 = torch.empty(E, de, I // 2, device=device, dtype=torch.uint8)
        W13_scale = torch.empty(E, de // 32, 2 * I, device=device, dtype=torch.bfloat16)
        W2_scale = torch.empty(E, I // 32, de, device=device, dtype=torch.bfloat16)
    else:
        wdt = torch.float8_e4m3fn if w.fp8 else adt
        W13 = torch.empty(E, 2 * I, de, device=device, dtype=wdt)
        W2 = torch.empty(E, de, I, device=device, dtype=wdt)
    if w.fp8:
        W13_scale = torch.empty(E, 2 * I // qb, de // qb, device=device, dtype=torch.float32)
        W2_scale = torch.empty(E, de // qb, I // qb, device=device, dtype=torch.float32)
    for e in range(E):
        m = randn(2 * I, de, std=_std(w, de))
        if w.fp8:
            W13[e], W13_scale[e] = _block_quantize(m, qb)
        elif w.int4:
            W13[e], W13_scale[e] = _int4_quantize(m)
        else:
            W13[e] = m.to(W13.dtype)
    for e in range(E):
        m = randn(de, I, std=_std(w, I))
        if w.fp8:
            W2[e], W2_scale[e] = _block_quantize(m, qb)
        elif w.int4:
            W2[e], W2_scale[e] = _int4_quantize(m)
        else:
            W2[e] = m.to(W2.dtype)
    Ws13 = Ws2 = Ws13_scale = Ws2_scale = None
    if w.n_shared:
        m13 = randn(2 * Is, d, std=_std(w, d))
        m2 = randn(d, Is, std=_std(w, Is))
        if w.fp8:
            Ws13, Ws13_scale = _block_quantize(m13, qb)
            Ws2, Ws2_scale = _block_quantize(m2, qb)
        elif w.int4:
            Ws13, Ws13_scale = _int4_quantize(m13)
            Ws2, Ws2_scale = _int4_quantize(m2)
        else:
            Ws13, Ws2 = m13.to(adt).contiguous(), m2.to(adt).contiguous()
    W_down = W_up = None
    if L > 0:
        W_down = randn(L, d, std=_std(w, d)).to(adt).contiguous()
        W_up = randn(d, L, std=_std(w, L)).to(adt).contiguous()
    return Layer(w, x, W_r, b, W13, W2, Ws13, Ws2, W_down, W_up, W13_scale, W2_scale,
                 Ws13_scale, Ws2_scale)


def make_block_norm(w, seed: int = 0, device="cuda") -> torch.Tensor:
    """The post-attention RMSNorm weight of a block around the layer: [d] in the activation
    type, drawn U(0.8, 1.2) from its own generator (seed + 7919) so that the layer's draws are
    unchanged.  The layer's x then plays the residual stream x'_n."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed + 7919)
    adt = torch.float32 if w.act == "f32" else torch.bfloat16
    u = torch.rand(w.d, generator=g, device=device, dtype=torch.float32)
    return (0.8 + 0.4 * u).to(adt).contiguous()


def make_dense(w: DenseWorkload, seed: int = 0, device="cuda") -> DenseLayer:
    """Draw the dense MLP's input and weights on ``device`` from ``seed`` (order: x, W13, W2)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    adt = torch.float32 if w.act == "f32" else torch.bfloat16
    std = (lambda fan_in: fan_in ** -0.5) if w.w_init == "fan_in" else (lambda fan_in: 0.02)

    def randn(*shape, s=1.0):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * s

    if w.x_dist == "clusters16":
        centres = randn(16, w.d)
        member = torch.randint(0, 16, (w.T,), generator=g, device=device)
        x = centres[member] + 0.5 * randn(w.T, w.d)
    else:
        x = randn(w.T, w.d)
    x = x.to(adt).contiguous()
    W13 = randn(2 * w.I, w.d, s=std(w.d)).to(adt).contiguous()
    W2 = randn(w.d, w.I, s=std(w.I)).to(adt).contiguous()
    return DenseLayer(w, x, W13, W2)


def subset_rows(n: int, count: int, seed: int = 1) -> torch.Tensor:
    """A seeded sample of ``count`` distinct row ids in [0, n), sorted (CPU tensor)."""
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randperm(n, generator=g)[: min(count, n)].sort().values
