"""GPU parity of the FFN half of a block (moe_forward_block) with the fp64 oracle.

"Kimi K2 · Transformer blocks > MoE transformer block": x_ffn = RMSNorm(x'_n), the mixture of
experts on x_ffn, x_{n+1} = x'_n + D_ffn.  Both sides round x_ffn once to the activation type (it is
the router's and the experts' GEMM operand; the oracle rounds its fp64 value to nearest, ties to
even), so the routing agrees except within the usual near-tie margin (1e-5), whose tokens are
counted and left out.  The parity rule of the layer (parity_lib) applies to the block's output
x'_n + D_ffn.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from mixture_experts_ffn_gemm_gb300 import binding as B
from mixture_experts_ffn_gemm_gb300 import synthetic as S
from oracle import torch_bridge as OB
from parity_lib import NEAR_TIE, NTHREADS, compare, kind

pytestmark = pytest.mark.gpu


def _check(w, seed=0, flags=0, rows=None):
    layer = S.make_layer(w, seed=seed, device="cuda")
    g = S.make_block_norm(w, seed=seed, device="cuda")
    cfg = B.config_for(w, flags=flags)
    ws = B.alloc_workspace(cfg)
    out = torch.full((w.T, w.d), float("nan"), dtype=layer.x.dtype, device="cuda")
    B.moe_forward_block(cfg, layer.x, g, *B.layer_weights(layer), out, ws)
    torch.cuda.synchronize()
    assert B.moe_device_status(ws) == B.MOE_OK
    got = out.float().cpu().numpy()
    rows_t = torch.arange(w.T) if rows is None else torch.as_tensor(rows)
    ref = OB.block_forward(layer, g, rows=rows_t, nthreads=NTHREADS)
    got = got[rows_t.numpy()]
    assert np.isfinite(got).all()
    keep = ref["margin"] >= NEAR_TIE
    res = compare(got[keep], ref["out"][keep], kind(w), rounded=w.act != "f32")
    res["skipped_near_ties"] = int((~keep).sum())
    return res


SMALL_BF16 = replace(S.WORKLOADS["tiny_fp32"], name="small_bf16", act="bf16", T=300)


def test_block_fp32(cuda_device):
    _check(S.WORKLOADS["tiny_fp32"], seed=1)


@pytest.mark.parametrize("flags", [B.MOE_FLAG_GEMM_ROWS_MAJOR, B.MOE_FLAG_GEMM_SWAP_AB],
                         ids=["rows", "swap"])
def test_block_bf16_small(cuda_device, flags):
    _check(SMALL_BF16, seed=2, flags=flags)


def test_block_latent_small(cuda_device):
    w = replace(SMALL_BF16, name="latent_small", d=512, d_latent=256, latent_norm=1, T=300,
                w_init="fan_in")
    _check(w, seed=3)


def test_block_fp8_small(cuda_device):
    w = replace(S.WORKLOADS["tiny_fp32"], name="small_fp8", act="bf16", fp8=True, T=200,
                x_dist="clusters16", w_init="std0.02", bias_range=0.05)
    _check(w, seed=4)


def test_block_int4_small(cuda_device):
    w = replace(S.WORKLOADS["tiny_fp32"], name="small_int4", act="bf16", int4=True, quant_block=32,
                T=200, w_init="std0.02", bias_range=0.05)
    _check(w, seed=5)


def test_block_k2_decode_widths(cuda_device):
    """The K2 decode workload's shapes (128 tokens, d = 7168, 384 experts), every token."""
    _check(S.WORKLOADS["k2_decode_bf16"], seed=0)


def test_block_zero_tokens_is_a_no_op(cuda_device):
    w = SMALL_BF16.with_tokens(0)
    cfg = B.config_for(w)
    ws = B.alloc_workspace(cfg)
    layer = S.make_layer(SMALL_BF16.with_tokens(4), device="cuda")
    g = S.make_block_norm(w, device="cuda")
    out = torch.empty(0, w.d, dtype=torch.bfloat16, device="cuda")
    B.moe_forward_block(cfg, layer.x[:0], g, *B.layer_weights(layer), out, ws)
    torch.cuda.synchronize()
