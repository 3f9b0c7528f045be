"""The C ABI without a GPU: the library loads, exports every entry point that include/moe.h
declares, and rejects bad arguments on the host (nothing is launched, no CUDA call is made)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from mixture_experts_ffn_gemm_gb300 import binding as B


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_entry_point_is_exported(moelib):
    names = _declared()
    assert "moe_forward" in names and len(names) >= 12
    for n in names:
        assert hasattr(moelib, n), n
    assert set(names) == set(B.EXPORTED)


def test_config_struct_matches_header_size(moelib):
    # int64 + 12 x int32 + 2 x float + int32 = 8 + 48 + 8 + 4 -> 72 with 8-byte alignment
    assert ctypes.sizeof(B.moe_config_t) == 72


def _cfg(**kw):
    base = dict(T=128, d=7168, E=384, k=8, I=2048, act_dtype=B.torch.bfloat16)
    base.update(kw)
    return B.make_config(**base)


def test_workspace_size_of_the_workloads(moelib):
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    for name, w in S.WORKLOADS.items():
        assert B.moe_workspace_size(B.config_for(w)) > 0, name
    # the prefill workspace holds the permuted activations, h and the expert outputs
    n = B.moe_workspace_size(B.config_for(S.WORKLOADS["k2_prefill_bf16"]))
    P = 16384 * 8
    assert n >= (P * 7168 + (P + 16384) * 2048 + (P + 16384) * 7168) * 2


@pytest.mark.parametrize("bad", [dict(k=0), dict(k=385), dict(E=0), dict(d=0), dict(T=-1),
                                 dict(n_shared=2), dict(I=0)])
def test_invalid_configs_have_no_workspace(moelib, bad):
    assert B.moe_workspace_size(_cfg(**bad)) == 0


@pytest.mark.parametrize("bad", [dict(d=7000), dict(I=2000), dict(k=33, E=64),
                                 dict(I_shared=4096)])
def test_unsupported_shapes_are_refused(moelib, bad):
    cfg = _cfg(**bad)
    assert B.moe_workspace_size(cfg) == 0
    st = moelib.moe_forward(ctypes.byref(cfg), *([0x1000] * 14), 0x1000, 1 << 40, None)
    assert st in (B.MOE_ERR_UNSUPPORTED, B.MOE_ERR_INVALID_ARG)


def test_host_validation_codes(moelib):
    cfg = _cfg()
    need = B.moe_workspace_size(cfg)
    p = 0x10000  # an aligned stand-in address: validation fails before anything dereferences it

    def fwd(c, ws=p, nbytes=need, **override):
        # x, W_r, b, W13, W2, W13_s, W2_s, Ws13, Ws2, Ws13_s, Ws2_s, W_down, W_up, out
        names = ["x", "W_r", "b", "W13", "W2", "W13_s", "W2_s", "Ws13", "Ws2", "Ws13_s",
                 "Ws2_s", "W_down", "W_up", "out"]
        ptrs = [override.get(n, p) for n in names]
        return moelib.moe_forward(c, *ptrs, ws, nbytes, None)

    c = ctypes.byref(cfg)
    assert fwd(c, nbytes=need - 1) == B.MOE_ERR_WORKSPACE
    assert fwd(c, ws=None) == B.MOE_ERR_WORKSPACE
    assert fwd(c, x=None) == B.MOE_ERR_INVALID_ARG
    assert fwd(c, out=None) == B.MOE_ERR_INVALID_ARG
    assert fwd(c, Ws13=None) == B.MOE_ERR_INVALID_ARG       # n_shared = 1 needs the shared expert
    assert fwd(c, W13=p + 2) == B.MOE_ERR_INVALID_ARG       # misaligned weight
    assert fwd(c, ws=p + 8) == B.MOE_ERR_INVALID_ARG        # misaligned workspace
    cfg.reserved_ = 1
    assert fwd(c) == B.MOE_ERR_INVALID_ARG
    assert fwd(None) == B.MOE_ERR_INVALID_ARG


def test_stage_entry_points_validate(moelib):
    cfg = _cfg()
    need = B.moe_workspace_size(cfg)
    p = 0x10000
    assert moelib.moe_router(ctypes.byref(cfg), p, p, p, None, None, p, p, need, None) == \
        B.MOE_ERR_INVALID_ARG
    assert moelib.moe_permute(ctypes.byref(cfg), p, p, p, None, p, p, need, None) == \
        B.MOE_ERR_INVALID_ARG
    assert moelib.moe_experts(ctypes.byref(cfg), p, p, p, p, None, *([None] * 7), p, p, need,
                              None) == B.MOE_ERR_INVALID_ARG
    assert moelib.moe_combine(ctypes.byref(cfg), p, p, p, None, None, p, need, None) == \
        B.MOE_ERR_INVALID_ARG
    lat = _cfg(d_latent=3584, latent_norm=1)
    need_l = B.moe_workspace_size(lat)
    assert moelib.moe_combine(ctypes.byref(lat), p, p, p, None, p, p, need_l, None) == \
        B.MOE_ERR_INVALID_ARG  # the latent path needs W_up
    assert moelib.moe_device_status(None, 0, None) == B.MOE_ERR_WORKSPACE
    assert moelib.moe_reset_device_status(None, 0, None) == B.MOE_ERR_WORKSPACE


def test_int4_host_validation(moelib):
    """4-bit group experts (MOE_INT4): bf16 activations, groups of 32, the K2 path, d % 256 and
    I % 128; anything else is refused before a launch, and the scales are required."""
    int4 = dict(w_dtype=B.torch.uint8, quant_block=32)
    assert B.moe_workspace_size(_cfg(**int4)) > 0
    for bad in (dict(quant_block=128), dict(act_dtype=B.torch.float32),
                dict(d_latent=3584, latent_norm=1), dict(d=7040), dict(I=2000)):
        assert B.moe_workspace_size(_cfg(**{**int4, **bad})) == 0, bad
    cfg = _cfg(**int4)
    need = B.moe_workspace_size(cfg)
    p = 0x10000  # aligned stand-in address: validation fails before anything dereferences it
    names = ["x", "W_r", "b", "W13", "W2", "W13_s", "W2_s", "Ws13", "Ws2", "Ws13_s", "Ws2_s",
             "W_down", "W_up", "out"]
    for missing in ("W13_s", "W2_s", "Ws13_s", "Ws2_s"):
        ptrs = [None if n == missing or n in ("W_down", "W_up") else p for n in names]
        assert moelib.moe_forward(ctypes.byref(cfg), *ptrs, p, need, None) == \
            B.MOE_ERR_INVALID_ARG, missing


def test_dense_mlp_host_validation(moelib):
    p = 0x10000  # aligned stand-in address: every call below fails (or returns) before using it
    bf, f32 = B.MOE_BF16, B.MOE_F32
    T, d, I = 16, 7168, 18432
    need = moelib.moe_dense_mlp_workspace_size(T, d, I, bf)
    a256 = lambda n: (n + 255) // 256 * 256
    # 16 tokens: the W2 GEMM's 28 output tiles are split over 5 ranges of I (fp32 partials), as
    # many as one wave of 152 CTAs holds; 16384 tokens fill the GPU without a split; no split in fp32
    assert need == 256 + a256(T * I * 2) + a256(5 * T * d * 4)
    assert moelib.moe_dense_mlp_workspace_size(16384, d, I, bf) == 256 + a256(16384 * I * 2)
    assert moelib.moe_dense_mlp_workspace_size(T, d, I, f32) == 256 + a256(T * I * 4)
    # few output tiles: at most 8 ranges, and never more ranges than 64-wide K-blocks
    assert moelib.moe_dense_mlp_workspace_size(T, 256, 1024, bf) == 256 + a256(T * 1024 * 2) + \
        a256(8 * T * 256 * 4)
    assert moelib.moe_dense_mlp_workspace_size(T, 256, 128, bf) == 256 + a256(T * 128 * 2) + \
        a256(2 * T * 256 * 4)
    assert moelib.moe_dense_mlp_workspace_size(-1, d, I, bf) == 0
    assert moelib.moe_dense_mlp_workspace_size(T, d, I, B.MOE_FP8_E4M3) == 0
    f = moelib.moe_dense_mlp

    def call(T=T, d=d, I=I, dt=bf, x=p, W13=p, W2=p, out=p, ws=p, nbytes=need):
        return f(T, d, I, dt, x, W13, W2, out, ws, nbytes, None)

    assert call(T=-1) == B.MOE_ERR_INVALID_ARG
    assert call(I=0) == B.MOE_ERR_INVALID_ARG
    assert call(dt=B.MOE_FP8_E4M3) == B.MOE_ERR_UNSUPPORTED
    assert call(d=7000) == B.MOE_ERR_UNSUPPORTED                    # bf16 tiles need d % 256
    assert call(d=64, I=40, dt=f32, nbytes=1 << 20) == B.MOE_ERR_UNSUPPORTED  # fp32: I % 16
    assert call(nbytes=need - 1) == B.MOE_ERR_WORKSPACE
    assert call(ws=None) == B.MOE_ERR_INVALID_ARG
    assert call(ws=p + 8) == B.MOE_ERR_INVALID_ARG
    assert call(x=None) == B.MOE_ERR_INVALID_ARG
    assert call(W2=p + 4) == B.MOE_ERR_INVALID_ARG
    # T = 0 is a no-op once the widths and the workspace are valid; empty tensors may be NULL
    need0 = moelib.moe_dense_mlp_workspace_size(0, d, I, bf)
    assert call(T=0, x=None, W13=None, W2=None, out=None, nbytes=need0) == B.MOE_OK


def test_block_host_validation(moelib):
    cfg = _cfg()
    need = B.moe_workspace_size(cfg)
    p = 0x10000

    def blk(c, ws=p, nbytes=need, **override):
        names = ["x", "norm_w", "W_r", "b", "W13", "W2", "W13_s", "W2_s", "Ws13", "Ws2",
                 "Ws13_s", "Ws2_s", "W_down", "W_up", "out"]
        ptrs = [override.get(n, p) for n in names]
        return moelib.moe_forward_block(c, *ptrs, ws, nbytes, None)

    c = ctypes.byref(cfg)
    assert blk(c, nbytes=need - 1) == B.MOE_ERR_WORKSPACE
    assert blk(c, norm_w=None) == B.MOE_ERR_INVALID_ARG
    assert blk(c, x=None) == B.MOE_ERR_INVALID_ARG
    assert blk(c, norm_w=p + 4) == B.MOE_ERR_INVALID_ARG
    lat = _cfg(d_latent=3584, latent_norm=1, n_shared=0)
    assert blk(ctypes.byref(lat), nbytes=B.moe_workspace_size(lat)) == B.MOE_ERR_UNSUPPORTED
    empty = _cfg(T=0)
    assert blk(ctypes.byref(empty), nbytes=B.moe_workspace_size(empty), x=None, norm_w=None,
               out=None) == B.MOE_OK


def test_status_strings(moelib):
    for code in range(7):
        assert B.status_string(code).startswith("MOE_")
    assert B.status_string(99) == "MOE_ERR_UNKNOWN"


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        B.load_library()
