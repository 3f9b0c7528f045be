"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by element.

Small shapes compare every token; the full workloads (K2 decode and INT4 decode 128 tokens,
K2 prefill 16384, K3 latent 8192, fp8 experts 8192) compare every routing decision, every token of
the decode batches and a seeded sample of 512 tokens of the others, and, on the K2 path, 64 seeded
rows of the fp32 expert outputs plus the last row of every expert (each expert's ragged last
tile), in the launch configuration the benchmark times.  Ragged token counts, empty experts, one
expert taking every token, k == E and T == 0 are covered.  The comparison rule (parity_lib) is the
same for every case.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from mixture_experts_ffn_gemm_gb300 import binding as B
from mixture_experts_ffn_gemm_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

ROWS = B.MOE_FLAG_GEMM_ROWS_MAJOR
SWAP = B.MOE_FLAG_GEMM_SWAP_AB
WIDE = B.MOE_FLAG_GEMM_SWAP_WIDE  # 256-token swap-AB tiles with a run-time MMA N
ROWS2 = B.MOE_FLAG_GEMM_ROWS_MAJOR | B.MOE_FLAG_GEMM_M2  # 256-row tiles of two M halves
FUSED = SWAP | B.MOE_FLAG_DECODE_FUSED  # decode expert GEMMs in one persistent launch
PAIR = B.MOE_FLAG_GEMM_ROWS_MAJOR | B.MOE_FLAG_GEMM_PAIR  # 256-row tiles on a pair of SMs
VARIANTS = [ROWS, ROWS2, PAIR, SWAP, FUSED, WIDE]
VARIANT_IDS = ["rows", "rows_m2", "rows_pair", "swap", "swap_fused", "wide"]


def _lib():
    import parity_lib as L
    return L


def _layer(w, seed=0):
    return S.make_layer(w, seed=seed, device="cuda")


def _full_check(layer, flags=0, rows=None, expert_rows=64):
    L = _lib()
    g = L.run_gpu(layer, flags)
    assert g.status == B.MOE_OK and g.status_fwd == B.MOE_OK
    L.check_permutation(layer, g)
    r = L.check_routing(layer, g)
    host = L.HostExperts(layer)
    e = L.check_expert_rows(layer, g, nrows=expert_rows, host=host)
    o = L.check_outputs(layer, g, rows=rows, host=host)
    return {**r, **e, **o}


# ---------------------------------------------------------------------------------------------
# fp32 tiny layer (CUDA-core GEMMs)
# ---------------------------------------------------------------------------------------------

def test_tiny_fp32_all_tokens(cuda_device):
    res = _full_check(_layer(S.WORKLOADS["tiny_fp32"]))
    assert res["err"] <= 1e-4


@pytest.mark.parametrize("T", [1, 3, 17, 200])
def test_tiny_fp32_ragged_tokens(cuda_device, T):
    _full_check(_layer(S.WORKLOADS["tiny_fp32"].with_tokens(T), seed=T))


def test_zero_tokens_is_a_no_op(cuda_device):
    w = S.WORKLOADS["tiny_fp32"].with_tokens(0)
    layer = _layer(w)
    cfg = B.config_for(w)
    ws = B.alloc_workspace(cfg)
    out = torch.empty(0, w.d, device="cuda")
    B.moe_forward(cfg, layer.x, *B.layer_weights(layer), out, ws)
    assert B.moe_device_status(ws) == B.MOE_OK


# ---------------------------------------------------------------------------------------------
# bf16, tensor-core GEMMs, small widths (many tiles, ragged groups)
# ---------------------------------------------------------------------------------------------

SMALL_BF16 = replace(S.WORKLOADS["tiny_fp32"], name="small_bf16", act="bf16", T=300)


@pytest.mark.parametrize("flags", VARIANTS, ids=VARIANT_IDS)
def test_bf16_small_all_tokens(cuda_device, flags):
    _full_check(_layer(SMALL_BF16, seed=1), flags)


@pytest.mark.parametrize("flags", VARIANTS, ids=VARIANT_IDS)
def test_bf16_one_expert_takes_every_token(cuda_device, flags):
    """k = 1 and a bias that forces expert 5: one group of T rows, every other group empty.

    Every output is 2.827 x one expert's output plus the shared expert, with no averaging over
    the k slots, so the bf16 roundings of h and of the output enter unaveraged (the CPU test
    test_bf16_rounding_bound measures what an ideal bf16 pipeline reaches on such a layer)."""
    w = replace(SMALL_BF16, k=1, T=333)
    layer = _layer(w, seed=2)
    layer.b.zero_()
    layer.b[5] = 10.0
    g = _lib().run_gpu(layer, flags)
    assert (g.idx.cpu() == 5).all()
    assert int(g.counts[5]) == 333 and int(g.counts[:5].sum() + g.counts[6:16].sum()) == 0
    print(_full_check(layer, flags, expert_rows=64))


@pytest.mark.parametrize("flags", VARIANTS, ids=VARIANT_IDS)
def test_bf16_every_expert_selected(cuda_device, flags):
    """k == E: every token visits every expert."""
    w = replace(SMALL_BF16, E=4, k=4, T=130)
    _full_check(_layer(w, seed=3), flags)


@pytest.mark.parametrize("flags", [SWAP, FUSED], ids=["two_launches", "fused"])
def test_bf16_decode_without_shared_expert(cuda_device, flags):
    """n_shared = 0: the decode expert launches with no trailing dense group."""
    w = replace(SMALL_BF16, name="small_bf16_noshared", n_shared=0, T=90)
    _full_check(_layer(w, seed=13), flags)


def test_fused_and_unfused_decode_agree_bit_for_bit(cuda_device):
    """The persistent decode launch computes every tile as the two launches do (same MMAs, same
    epilogues), so the layer outputs agree bit for bit."""
    w = replace(S.WORKLOADS["k2_decode_bf16"], name="k2_e48", E=48, T=100)
    layer = _layer(w, seed=14)
    a, _, _ = B.forward_layer(layer, flags=FUSED)
    b, _, _ = B.forward_layer(layer, flags=SWAP)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_bf16_tensor_core_router_top3(cuda_device):
    """The tensor-core router with k = 3 < 8 and a ragged last 128-token tile."""
    w = replace(SMALL_BF16, E=128, k=3, T=1100)
    res = _full_check(_layer(w, seed=15), ROWS | B.MOE_FLAG_ROUTER_TC,
                      rows=np.arange(0, 1100, 11))
    assert res["compared"] > 80


def test_bf16_tensor_core_router(cuda_device):
    """E = 128 with more than 1024 tokens takes the 3 x bf16 split router on the tensor cores."""
    w = replace(SMALL_BF16, E=128, k=8, T=1100)
    res = _full_check(_layer(w, seed=4), ROWS | B.MOE_FLAG_ROUTER_TC,
                      rows=np.arange(0, 1100, 7))
    assert res["compared"] > 100


def test_bf16_router_paths_agree(cuda_device):
    """The CUDA-core split-K router, the tensor-core split router and the split-K tensor-core
    router (the default below 1024 tokens) give the same selections (away from near ties) and
    logits within fp32 accumulation error."""
    w = replace(SMALL_BF16, E=128, k=8, T=257, d=512)
    layer = _layer(w, seed=5)
    L = _lib()
    a = L.run_gpu(layer, B.MOE_FLAG_ROUTER_SIMT)
    b = L.run_gpu(layer, B.MOE_FLAG_ROUTER_TC)
    c = L.run_gpu(layer, 0)
    za, zb, zc = (r.logits.cpu().double() for r in (a, b, c))
    assert float((za - zb).abs().max()) <= 1e-5 * float(za.abs().max())
    assert float((za - zc).abs().max()) <= 1e-5 * float(za.abs().max())
    for r in (a, b, c):
        L.check_routing(layer, r)


@pytest.mark.parametrize("T,E,d", [(1, 64, 256), (37, 128, 512), (128, 384, 1024),
                                   (300, 192, 7168), (1000, 64, 512)])
def test_splitk_tensor_core_router(cuda_device, T, E, d):
    """The split-K tensor-core router at one token, ragged token tiles, several 64-expert
    blocks and K slices (the slice count depends on T and E): logits against the fp64 oracle's
    within fp32 accumulation error, selections and gates by the oracle's rule."""
    import oracle
    from oracle import torch_bridge as OB
    w = replace(SMALL_BF16, E=E, k=min(8, E), T=T, d=d, I=128, I_shared=128)
    layer = _layer(w, seed=T + E)
    L = _lib()
    g = L.run_gpu(layer, 0)
    xm, W_r, b = OB.route_inputs(layer, torch.arange(T))
    z_ref = oracle.route(OB.config(layer, T), xm, W_r, b)["logits"]
    z = g.logits.cpu().double().numpy()
    # fp32 accumulation of d products: bound by the sum of |x| |w| per logit
    bound = (layer.x.double().abs() @ layer.W_r.double().abs().T).cpu().numpy()
    assert (np.abs(z - z_ref) <= 2e-6 * bound + 1e-30).all()
    L.check_routing(layer, g)


def test_latent_small_all_tokens(cuda_device):
    w = replace(SMALL_BF16, name="latent_small", d=512, d_latent=256, latent_norm=1, T=300,
                w_init="fan_in")
    _full_check(_layer(w, seed=6), ROWS)


def test_latent_small_wide_swap_tiles(cuda_device):
    """The latent path in 256-token swap-AB tiles (MOE_FLAG_GEMM_SWAP_WIDE): routed groups at
    width L and the full-width shared expert (its own K) in the same launches."""
    w = replace(SMALL_BF16, name="latent_small", d=512, d_latent=256, latent_norm=1, T=700,
                w_init="fan_in")
    _full_check(_layer(w, seed=9), WIDE)


def test_latent_small_two_m_halves(cuda_device):
    """The latent path with 256-row SwiGLU tiles: routed groups at width L (ragged, many end in
    their first M half) and the full-width shared expert in the same launch."""
    w = replace(SMALL_BF16, name="latent_small", d=512, d_latent=256, latent_norm=1, T=700,
                w_init="fan_in")
    _full_check(_layer(w, seed=12), ROWS2)


def test_latent_small_sm_pairs(cuda_device):
    """The latent path with 256-row tiles on SM pairs: routed groups at width L, many ending in
    the first SM's 128 rows, and the full-width shared expert in the same launches."""
    w = replace(SMALL_BF16, name="latent_small", d=512, d_latent=256, latent_norm=1, T=700,
                w_init="fan_in")
    _full_check(_layer(w, seed=12), PAIR)


def test_latent_small_without_norm(cuda_device):
    w = replace(SMALL_BF16, name="latent_small", d=512, d_latent=256, latent_norm=0, T=70,
                w_init="fan_in")
    _full_check(_layer(w, seed=7), SWAP)


@pytest.mark.parametrize("case", ["k1_forced", "k3_latent_norm", "k2_top4"])
def test_error_is_the_ideal_bf16_pipelines(cuda_device, case):
    """On the GPU-drawn inputs of the cases above, the kernels' plain and rms errors against the
    oracle are those of an ideal bf16 pipeline (rounding_model: exact arithmetic, the oracle's
    routing, only h, x_lat, u_hat and the output rounded to bf16), so any excess over the plain
    2e-2 bound is the rounding the data types force, not the kernels' own."""
    import rounding_model as R
    L = _lib()
    if case == "k1_forced":
        layer, flags = _layer(replace(SMALL_BF16, k=1, T=333), seed=2), ROWS
        layer.b.zero_()
        layer.b[5] = 10.0
    elif case == "k3_latent_norm":
        layer, flags = _layer(replace(SMALL_BF16, name="latent_small", d=512, d_latent=256,
                                      latent_norm=1, T=700, w_init="fan_in"), seed=9), 0
    else:
        layer, flags = _layer(SMALL_BF16, seed=1), 0
    g = L.run_gpu(layer, flags)
    ref = L.oracle_forward(layer, np.arange(layer.x.shape[0]), L.HostExperts(layer))
    keep = ref["margin"] >= L.NEAR_TIE
    ideal = R.errors(R.ideal_forward(layer)["out"][keep], ref["out"][keep])
    gpu = R.errors(g.out.float().cpu().numpy()[keep], ref["out"][keep])
    print(case, "gpu", {k: f"{v:.3e}" for k, v in gpu.items()},
          "ideal", {k: f"{v:.3e}" for k, v in ideal.items()})
    assert gpu["plain"] <= ideal["plain"] + 4e-3
    assert gpu["rms"] <= 1.25 * ideal["rms"]
    assert gpu["beyond_rounding"] <= 2e-2


@pytest.mark.parametrize("case", ["k2_top4", "k2_widths"])
def test_outputs_within_the_rule_of_the_pages_rounding_sequence(cuda_device, case):
    """The kernels' outputs against an emulation of the pages' own combine rounding (bf16 expert
    outputs cast to the gate type, multiplied, summed, cast back, plus the bf16 shared output;
    rounding_model.pages_combine_forward) on the same GPU-drawn inputs: within the bf16 rule, so
    the one-rounding fp32 sum the library uses agrees with the pages' arithmetic to the same
    tolerance it keeps against the fp64 oracle."""
    import rounding_model as R
    L = _lib()
    if case == "k2_top4":
        layer = _layer(SMALL_BF16, seed=1)
    else:
        layer = _layer(replace(S.WORKLOADS["k2_prefill_bf16"], name="k2_e32", E=32, T=256), seed=3)
    g = L.run_gpu(layer)
    pages = R.pages_combine_forward(layer)
    keep = pages["margin"] >= L.NEAR_TIE
    e = R.errors(g.out.float().cpu().numpy()[keep], pages["out"][keep])
    print(case, "gpu vs pages' sequence", {k: f"{v:.3e}" for k, v in e.items()})
    assert e["beyond_rounding"] <= 2e-2
    assert e["rms"] <= 5e-3


# ---------------------------------------------------------------------------------------------
# fp8 experts: e4m3 weights with 128 x 128 block scales, activations per token per 128 channels
# ---------------------------------------------------------------------------------------------

SMALL_FP8 = replace(S.WORKLOADS["tiny_fp32"], name="small_fp8", act="bf16", fp8=True, T=300,
                    x_dist="clusters16", w_init="std0.02", bias_range=0.05)


def test_fp8_small_all_tokens(cuda_device):
    _full_check(_layer(SMALL_FP8, seed=21))


@pytest.mark.parametrize("T", [1, 17, 129])
def test_fp8_ragged_tokens(cuda_device, T):
    _full_check(_layer(SMALL_FP8.with_tokens(T), seed=22 + T))


def test_fp8_k2_widths_32_experts(cuda_device):
    w = replace(S.WORKLOADS["k2_fp8"], name="k2_fp8_e32", E=32, T=72)
    _full_check(_layer(w, seed=23))


def test_fp8_zero_activation_group_gets_unit_scale(cuda_device):
    """An all-zero 128-channel group of x quantises with scale 1 (no 0/0) and contributes 0."""
    layer = _layer(replace(SMALL_FP8, T=64), seed=24)
    layer.x[:, :128] = 0.0
    _full_check(layer)


# ---------------------------------------------------------------------------------------------
# K2 widths (d = 7168, I = 2048) with fewer experts: every token checked
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("flags", VARIANTS, ids=VARIANT_IDS)
def test_k2_widths_32_experts(cuda_device, flags):
    w = replace(S.WORKLOADS["k2_decode_bf16"], name="k2_e32", E=32, T=72)
    _full_check(_layer(w, seed=8), flags)


# ---------------------------------------------------------------------------------------------
# 4-bit integer group experts (bf16 activations): the weights both sides use are the decoded
# RN_bf16((u - 8) * scale) values, so the bf16 bounds apply
# ---------------------------------------------------------------------------------------------

SMALL_INT4 = replace(S.WORKLOADS["tiny_fp32"], name="small_int4", act="bf16", int4=True,
                     quant_block=32, T=300, w_init="std0.02", bias_range=0.05)


def test_int4_small_all_tokens(cuda_device):
    _full_check(_layer(SMALL_INT4, seed=31))


@pytest.mark.parametrize("T", [1, 17, 129])
def test_int4_ragged_tokens(cuda_device, T):
    _full_check(_layer(SMALL_INT4.with_tokens(T), seed=32 + T))


def test_int4_zero_tokens_is_a_no_op(cuda_device):
    w = SMALL_INT4.with_tokens(0)
    layer = _layer(w)
    cfg = B.config_for(w)
    ws = B.alloc_workspace(cfg)
    out = torch.empty(0, w.d, dtype=torch.bfloat16, device="cuda")
    B.moe_forward(cfg, layer.x, *B.layer_weights(layer), out, ws)
    torch.cuda.synchronize()
    assert B.moe_device_status(ws) == B.MOE_OK


def test_int4_every_expert_skewed(cuda_device):
    """Clustered tokens: a few experts get several token tiles (their weights are expanded once
    per tile), most get one or none."""
    w = replace(SMALL_INT4, name="int4_clusters", T=600, x_dist="clusters16")
    _full_check(_layer(w, seed=34))


def test_int4_k2_widths_32_experts(cuda_device):
    w = replace(S.WORKLOADS["k2_int4_decode"], name="k2_int4_e32", E=32, T=72)
    _full_check(_layer(w, seed=33))


# ---------------------------------------------------------------------------------------------
# Full workloads, in the launch configuration of the benchmark (automatic flags)
# ---------------------------------------------------------------------------------------------

def _sample(T, n=512, seed=1):
    return S.subset_rows(T, n, seed=seed).numpy()


def _full_workload(name, flags=0):
    """One benchmark workload in the bench's launch configuration (or the given GEMM flags):
    routing and permutation on every token; 64 seeded rows of the fp32 expert outputs plus the
    last row of every expert; the outputs of every token for decode-sized batches (128 tokens),
    else of 512 seeded tokens."""
    w = S.WORKLOADS[name]
    layer = _layer(w)
    res = _full_check(layer, flags, rows=None if w.T <= 128 else _sample(w.T))
    del layer
    torch.cuda.empty_cache()
    assert res["compared"] + res["sample_near_ties"] == min(w.T, 512)
    return res


def test_full_k2_decode(cuda_device):
    res = _full_workload("k2_decode_bf16")
    print("k2_decode", res)


def test_full_k2_prefill(cuda_device):
    res = _full_workload("k2_prefill_bf16")
    print("k2_prefill", res)


def test_full_k2_prefill_sm_pairs(cuda_device):
    res = _full_workload("k2_prefill_bf16", PAIR)
    print("k2_prefill_pairs", res)


YBF16 = B.MOE_FLAG_EXPERT_OUT_BF16  # bf16 expert outputs (one more rounding, half the bytes)


@pytest.mark.parametrize("flags", [ROWS | YBF16, SWAP | YBF16, PAIR | YBF16, WIDE | YBF16,
                                   ROWS | B.MOE_FLAG_GEMM_N128 | YBF16,
                                   SWAP | B.MOE_FLAG_DECODE_FUSED | YBF16],
                         ids=["rows", "swap", "rows_pair", "wide", "rows_n128", "swap_fused_off"])
def test_bf16_expert_outputs_small(cuda_device, flags):
    """Expert outputs in bf16 on request: within the same parity rule (the error beyond the output
    rounding, 2e-2 rms), with one more bf16 rounding of every expert output before the sum; the
    sampled expert rows are compared as bf16 results under the same rule."""
    res = _full_check(_layer(SMALL_BF16, seed=1), flags)
    print("bf16 expert outputs", res)


def test_full_k2_prefill_bf16_expert_outputs(cuda_device):
    res = _full_workload("k2_prefill_bf16", YBF16)
    print("k2_prefill_bf16_expert_outputs", res)


@pytest.mark.parametrize("flags", [0, B.MOE_FLAG_EXPERT_OUT_F32], ids=["bf16_out", "f32_out"])
def test_fp8_experts_outputs_k2_widths(cuda_device, flags):
    """e4m3 experts: bf16 expert outputs (the default) and fp32 ones on request, 32 experts at
    the K2 widths, within the fp8 rule."""
    w = replace(S.WORKLOADS["k2_fp8"], E=32, T=300)
    res = _full_check(_layer(w, seed=23), flags)
    print("fp8 expert outputs", flags, res)


def test_bf16_expert_outputs_unsupported_elsewhere(cuda_device):
    for wl in ("k3_latent_bf16", "k2_int4_decode", "tiny_fp32"):
        cfg = B.config_for(S.WORKLOADS[wl].with_tokens(16), flags=YBF16)
        assert B.moe_workspace_size(cfg) == 0


def test_k2_prefill_65536_tokens_offsets_past_2_31(cuda_device):
    """65536 tokens at the K2 widths: the permuted activations (524288 rows x 7168) and the fp32
    expert outputs hold more than 2^31 elements, so every row * width product must be 64-bit.
    About 62 GB on the device; 64 sampled tokens and the last row of every expert against the
    oracle."""
    w = S.WORKLOADS["k2_prefill_bf16"].with_tokens(65536)
    layer = _layer(w, seed=11)
    res = _full_check(layer, 0, rows=_sample(w.T, n=64, seed=5), expert_rows=16)
    del layer
    torch.cuda.empty_cache()
    print("k2_prefill_65536", res)


def test_full_k3_latent(cuda_device):
    res = _full_workload("k3_latent_bf16")
    print("k3_latent", res)


def test_full_k2_int4_decode(cuda_device):
    res = _full_workload("k2_int4_decode")
    print("k2_int4_decode", res)


def test_full_k2_fp8(cuda_device):
    res = _full_workload("k2_fp8")
    print("k2_fp8", res)


# ---------------------------------------------------------------------------------------------
# Boundary behaviour on the GPU
# ---------------------------------------------------------------------------------------------

def test_host_io_entry_point_matches_device_path(cuda_device):
    w = SMALL_BF16
    layer = _layer(w, seed=9)
    cfg = B.config_for(w)
    ws = B.alloc_workspace(cfg)
    out_dev = torch.empty(w.T, w.d, dtype=torch.bfloat16, device="cuda")
    B.moe_forward(cfg, layer.x, *B.layer_weights(layer), out_dev, ws)
    x_host = layer.x.cpu().pin_memory()
    out_host = torch.empty(w.T, w.d, dtype=torch.bfloat16).pin_memory()
    B.moe_forward_host_io(cfg, x_host, *B.layer_weights(layer), out_host, ws)
    assert torch.equal(out_host, out_dev.cpu())


@pytest.mark.parametrize("latent,flags", [(False, 0), (True, 0), (False, B.MOE_FLAG_EXPERT_OUT_BF16),
                                          (False, B.MOE_FLAG_GEMM_N128)],
                         ids=["k2", "k3_latent", "k2_bf16_outputs", "k2_two_pieces"])
def test_host_io_overlapped_copies_match_device_path(cuda_device, latent, flags):
    """Inputs of 32 MB and more take the overlapped host-I/O path: the input in token chunks of
    2048 on two copy streams, each chunk's shared-expert rows computed in launches of their own
    while the next chunk arrives, then the routed experts without the shared expert, and the
    combine (K3: latent combine and up-projection) in eight token chunks, each copied out behind
    its part.  The output must equal moe_forward's (shared expert inside the routed launches) bit
    for bit, with ragged last chunks (3001 tokens); also with bf16 expert outputs, and with the
    128-column W2 tiles, under which x arrives in two pieces instead (no shared-expert chunks)."""
    base = S.WORKLOADS["k3_latent_bf16" if latent else "k2_prefill_bf16"]
    w = replace(base, name="host_io_large", E=32, T=3001)
    layer = _layer(w, seed=21)
    cfg = B.config_for(w, flags=flags)
    ws = B.alloc_workspace(cfg)
    assert w.T * w.d * 2 >= 32 << 20
    out_dev = torch.empty(w.T, w.d, dtype=torch.bfloat16, device="cuda")
    B.moe_forward(cfg, layer.x, *B.layer_weights(layer), out_dev, ws)
    x_host = layer.x.cpu().pin_memory()
    for _ in range(2):  # the copy streams and events are reused by a second call
        out_host = torch.full((w.T, w.d), float("nan"), dtype=torch.bfloat16).pin_memory()
        B.moe_forward_host_io(cfg, x_host, *B.layer_weights(layer), out_host, ws)
        assert torch.equal(out_host, out_dev.cpu())
    del layer, ws
    torch.cuda.empty_cache()


def test_forward_replays_from_a_cuda_graph(cuda_device):
    """moe_forward allocates nothing and never synchronises, so it can be captured into a CUDA
    graph; every replay must give the eager result bit for bit (decode shapes, 32 experts)."""
    w = replace(S.WORKLOADS["k2_decode_bf16"], name="k2_e32", E=32)
    layer = _layer(w, seed=21)
    out, ws, cfg = B.forward_layer(layer)
    torch.cuda.synchronize()
    ref = out.clone()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        B.forward_layer(layer, out=out, ws=ws, stream=st)  # warm-up on the capture stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        B.forward_layer(layer, out=out, ws=ws, stream=st)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert B.moe_device_status(ws) == B.MOE_OK


def test_out_of_range_expert_index_is_flagged(cuda_device):
    """An index outside [0, E) handed to moe_permute is skipped and reported, not followed."""
    w = SMALL_BF16
    cfg = B.config_for(w)
    ws = B.alloc_workspace(cfg)
    B.moe_reset_device_status(ws)
    idx = torch.randint(0, w.E, (w.T, w.k), dtype=torch.int32, device="cuda")
    idx[7, 1] = w.E + 3
    counts = torch.empty(w.E + 1, dtype=torch.int32, device="cuda")
    offsets = torch.empty(w.E + 2, dtype=torch.int32, device="cuda")
    ps = torch.empty(w.T * w.k, dtype=torch.int32, device="cuda")
    pd = torch.empty(w.T * w.k, dtype=torch.int32, device="cuda")
    B.moe_permute(cfg, idx, counts, offsets, ps, pd, ws)
    assert B.moe_device_status(ws) == B.MOE_ERR_DEVICE_CHECK
    assert int(counts[: w.E].sum()) == w.T * w.k - 1
    assert int(pd[7 * w.k + 1]) == -1


def test_expired_wait_is_reported_and_the_context_survives(cuda_device):
    """The failure path without a GPU fault: the test flag withholds the expert GEMM's copies, its
    bounded wait (50 ms) expires, the kernel returns with MOE_ERR_TIMEOUT in the device status;
    the next normal call on the same context gives correct results."""
    w = SMALL_BF16
    layer = _layer(w, seed=11)
    cfg = B.config_for(w, flags=ROWS | B.MOE_FLAG_TEST_STALL_EXPERTS)
    ws = B.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d, dtype=torch.bfloat16, device="cuda")
    B.moe_forward(cfg, layer.x, *B.layer_weights(layer), out, ws)
    assert B.moe_device_status(ws) == B.MOE_ERR_TIMEOUT
    _full_check(layer, ROWS)


def test_launch_counter_counts_kernels(cuda_device):
    w = SMALL_BF16
    layer = _layer(w, seed=10)
    B.moe_reset_launch_count()
    B.forward_layer(layer)
    torch.cuda.synchronize()
    n = B.moe_launch_count()
    # router GEMM + top-k, the permute (one kernel up to 1024 pairs, else count + scan + scatter),
    # gather, two grouped GEMMs, combine
    assert n >= 7
