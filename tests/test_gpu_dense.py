"""GPU parity of the dense block MLP (moe_dense_mlp) with the fp64 oracle.

The dense MLP of the first block is y = (SiLU(x W1) * (x W3)) W2 per token (nnterp "kimi_k2",
"Printout": layer 0's DeepseekV3MLP).  The library runs it as one dense group through the expert
GEMMs: token-rows tensor-core tiles for bf16, CUDA cores for fp32.  When the W2 GEMM has fewer
output tiles than one wave of CTAs holds (few tokens, or a narrow d), each tile is computed as
fp32 partial sums over up to 8 ranges of I that one more kernel adds in range order.
The parity rule of the layer (parity_lib): tol 1e-4 (fp32) / 2e-2 (bf16) of rms(oracle), for bf16
beyond the output's own rounding, the plain figure reported beside it."""
from dataclasses import replace

import numpy as np
import pytest
import torch

from mixture_experts_ffn_gemm_gb300 import binding as B
from mixture_experts_ffn_gemm_gb300 import synthetic as S
from oracle import torch_bridge as OB
from parity_lib import NTHREADS, compare

pytestmark = pytest.mark.gpu


def _run(L) -> torch.Tensor:
    T, d = L.x.shape
    I = L.W2.shape[1]
    out = torch.full((T, d), float("nan"), dtype=L.x.dtype, device="cuda")
    ws = torch.zeros(B.moe_dense_mlp_workspace_size(T, d, I, L.x.dtype), dtype=torch.uint8,
                     device="cuda")
    B.moe_dense_mlp(L.x, L.W13, L.W2, out, ws)
    torch.cuda.synchronize()
    assert B.moe_device_status(ws) == B.MOE_OK
    return out


def _dense(name, T=None, seed=0, **over):
    w = S.DENSE_WORKLOADS[name]
    if T is not None:
        w = w.with_tokens(T)
    if over:
        w = replace(w, **over)
    return S.make_dense(w, seed=seed, device="cuda")


def _check(L, rows=None, act=None):
    out = _run(L)
    assert torch.isfinite(out.float()).all()
    rows_t = None if rows is None else torch.as_tensor(rows)
    ref = OB.dense_mlp(L, rows=rows_t, nthreads=NTHREADS)
    got = out.float().cpu().numpy()
    if rows_t is not None:
        got = got[rows_t.numpy()]
    act = act or ("f32" if L.x.dtype == torch.float32 else "bf16")
    return compare(got, ref, act, rounded=act != "f32")


@pytest.mark.parametrize("T", [1, 48, 131])
def test_dense_fp32_cuda_cores(cuda_device, T):
    _check(_dense("tiny_dense_fp32", T=T))


@pytest.mark.parametrize("T", [1, 33, 200, 256])
def test_dense_bf16_few_tokens(cuda_device, T):
    """T <= 256: one or two 128-row token tiles, ragged tails; W2 split over 6 ranges of I."""
    _check(_dense("k2_dense_decode_bf16", T=T, d=512, I=384))


@pytest.mark.parametrize("T", [257, 700, 1300, 5000])
def test_dense_bf16_many_tokens(cuda_device, T):
    """T > 256: token-rows tiles (128 rows x 256 weight rows), several tiles and a ragged tail.
    With d = 512 the W2 GEMM has 2 output tiles per row tile: split over 6 ranges of I up to 1300
    tokens, unsplit at 5000 (80 tiles)."""
    _check(_dense("k2_dense_prefill_bf16", T=T, d=512, I=384))


def test_dense_zero_tokens_is_a_no_op(cuda_device):
    L = _dense("k2_dense_decode_bf16", T=4, d=256, I=128)
    ws = torch.zeros(B.moe_dense_mlp_workspace_size(0, 256, 128, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    empty = L.x[:0]
    out = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    B.moe_dense_mlp(empty, L.W13, L.W2, out, ws)
    torch.cuda.synchronize()


def test_dense_k2_block0_decode_full_size(cuda_device):
    """The K2 block-0 widths (d = 7168, I = 18432) at the decode batch (128 tokens), compared on
    every token."""
    _check(_dense("k2_dense_decode_bf16"))


def test_dense_k2_block0_two_row_tiles_split_in_two(cuda_device):
    """K2 block-0 widths at 200 tokens: 56 W2 output tiles, so two ranges of I; compared on 40
    tokens, 20 of them in the ragged second row tile."""
    L = _dense("k2_dense_decode_bf16", T=200, seed=4)
    rows = np.concatenate([S.subset_rows(128, 20, seed=5), 128 + S.subset_rows(72, 20, seed=6)])
    _check(L, rows=rows)


def test_dense_k2_block0_prefill_sampled(cuda_device):
    """The K2 block-0 widths at 2048 tokens (token-rows tiles), compared on 24 sampled tokens."""
    L = _dense("k2_dense_prefill_bf16", T=2048)
    _check(L, rows=S.subset_rows(2048, 24, seed=3))
