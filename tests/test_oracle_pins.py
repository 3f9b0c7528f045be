"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics (no GPU).

Each test ties one part of the oracle to something other than itself: a number the pages print, a
hand-computed case, a closed form, a brute-force enumeration, an independent library routine
(numpy matmul, torch's float8 conversion) or an identity of the equations.  A plausible slip in the
oracle (a dropped term, a swapped W1/W3, a wrong sign, a transposed operand, a broken tie rule)
fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from conftest import read_golden

K2 = dict(d=7168, E=384, k=8, I=2048, I_shared=2048)


def silu(v):
    return v / (1.0 + np.exp(-v))


def dense_swiglu(x, W13, W2):
    """Textbook SwiGLU with numpy matmuls (a library routine independent of the oracle's loops):
    x [T, din], W13 [2I, din] (W1 rows then W3 rows), W2 [dout, I]."""
    I = W13.shape[0] // 2
    g = x @ W13[:I].T
    u = x @ W13[I:].T
    return (silu(g) * u) @ W2.T


def f64(m):
    return m.data.astype(np.float64) if m.dtype in ("f32", "f64") else None


# --------------------------------------------------------------------------------------------
# Parameter accounting printed on the pages
# --------------------------------------------------------------------------------------------

def test_param_count_k2_matches_page(orc):
    golden = {r[0]: int(r[1]) for r in read_golden("param_counts.txt")}
    cfg = orc.Config(T=1, **K2)
    assert orc.param_count(cfg) == golden["k2_mixture_of_experts"] == 16_958_226_816


def test_param_count_k3_latent_projections_match_page(orc):
    golden = {r[0]: int(r[1]) for r in read_golden("param_counts.txt")}
    cfg = orc.Config(T=1, d_latent=3584, latent_norm=1, **K2)
    br = orc.param_breakdown(cfg)
    assert br["up"] == golden["k3_latent_up_projection"] == 25_690_112
    assert br["down"] == br["up"]
    # the routed experts shrink to the latent width; router and shared expert stay full width
    assert br["routed"] == 384 * 3 * 3584 * 2048
    assert br["shared"] == 3 * 7168 * 2048 and br["router"] == 384 * 7168


def test_param_count_changes_with_every_shape(orc):
    base = orc.Config(T=1, d=256, E=16, k=4, I=128, I_shared=128)
    n0 = orc.param_count(base)
    for field in ("d", "E", "I", "I_shared"):
        c = orc.Config(**{**base.__dict__, field: getattr(base, field) * 2})
        assert orc.param_count(c) != n0, field


# --------------------------------------------------------------------------------------------
# e4m3 format (OCP FP8 E4M3, "fn": no infinities, max 448)
# --------------------------------------------------------------------------------------------

def test_e4m3_decode_definition(orc):
    assert orc.e4m3_decode(0x00) == 0.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9          # smallest subnormal
    assert orc.e4m3_decode(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert orc.e4m3_decode(0x08) == 2.0 ** -6          # smallest normal
    assert orc.e4m3_decode(0x38) == 1.0
    assert orc.e4m3_decode(0x39) == 1.125
    assert orc.e4m3_decode(0x7E) == 448.0
    assert math.isnan(orc.e4m3_decode(0x7F)) and math.isnan(orc.e4m3_decode(0xFF))
    assert orc.e4m3_decode(0xB8) == -1.0 and orc.e4m3_decode(0xFE) == -448.0
    assert math.copysign(1.0, orc.e4m3_decode(0x80)) == -1.0


def test_e4m3_decode_matches_torch_for_all_codes(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([orc.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])


def test_e4m3_encode_ties_to_even_and_saturates(orc):
    assert orc.e4m3_encode(1.0625) == 0x38      # halfway 1 .. 1.125 -> even mantissa
    assert orc.e4m3_encode(1.1875) == 0x3A      # halfway 1.125 .. 1.25 -> even mantissa
    assert orc.e4m3_encode(2.0 ** -10) == 0x00  # halfway 0 .. 2^-9 -> 0
    assert orc.e4m3_encode(3 * 2.0 ** -10) == 0x02
    assert orc.e4m3_encode(464.0) == 0x7E and orc.e4m3_encode(1e9) == 0x7E
    assert orc.e4m3_encode(-1e9) == 0xFE
    assert orc.e4m3_encode(float("nan")) == 0x7F


def test_e4m3_encode_matches_torch(orc):
    rng = np.random.default_rng(0)
    mag = np.exp2(rng.uniform(-12, np.log2(448.0), 4000))
    v = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([orc.e4m3_encode(float(a)) for a in v], np.uint8)
    assert np.array_equal(ref, ours)


def test_quantize_group_scales_and_codes(orc):
    rng = np.random.default_rng(1)
    v = rng.standard_normal(300).astype(np.float32)
    v[128:256] = 0.0                                   # an all-zero group
    q, s = orc.quantize_group_e4m3(v, 128)
    assert s.shape == (3,)
    assert s[1] == 1.0 and np.all(q[128:256] == 0)
    for g, (lo, hi) in enumerate([(0, 128), (256, 300)]):
        grp = v[lo:hi]
        gi = 0 if lo == 0 else 2
        assert s[gi] == np.float32(np.abs(grp).max()) / np.float32(448.0)
        amax_at = lo + int(np.argmax(np.abs(grp)))
        assert q[amax_at] & 0x7F == 0x7E               # the group maximum maps to +-448
        ref = torch.from_numpy(grp / s[gi]).clamp(-448, 448).to(torch.float8_e4m3fn)
        assert np.array_equal(ref.view(torch.uint8).numpy(), q[lo:hi])


# --------------------------------------------------------------------------------------------
# Routing: top_8(s + b), ties to the lower index, gates renormalised x 2.827
# --------------------------------------------------------------------------------------------

def _keys32(z, b):
    s32 = (1.0 / (1.0 + np.exp(-z.astype(np.float64)))).astype(np.float32)
    return s32 + b.astype(np.float32)


def _before(ki, i, kj, j):
    """Expert i is ordered before expert j: larger key, or an equal key and a lower index."""
    return ki > kj or (ki == kj and i < j)


@pytest.mark.parametrize("ties", [False, True])
def test_topk_matches_brute_force_enumeration(orc, ties):
    rng = np.random.default_rng(2 + ties)
    T, E, k = 300, 6, 3
    if ties:
        z = rng.integers(-1, 2, (T, E)).astype(np.float32)    # many exactly equal keys
        b = np.zeros(E, np.float32)
    else:
        z = rng.standard_normal((T, E)).astype(np.float32)
        b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    cfg = orc.Config(T=T, d=1, E=E, k=k, I=1)
    idx, gates, margin = orc.route_from_logits(cfg, z, b)
    key = _keys32(z, b)
    for t in range(T):
        winners = [S for S in itertools.combinations(range(E), k)
                   if all(_before(key[t, i], i, key[t, j], j)
                          for i in S for j in range(E) if j not in S)]
        assert len(winners) == 1
        assert sorted(idx[t]) == list(winners[0])
        # slots in order: each slot ordered before the next
        for a, c in zip(idx[t][:-1], idx[t][1:]):
            assert _before(key[t, a], a, key[t, c], c)
    # the selected keys it reports are those experts' keys, in slot order, and the margin is the
    # last selected key minus the best key left out
    _, _, margin2, sel = orc.route_from_logits(cfg, z, b, with_keys=True)
    np.testing.assert_array_equal(sel, np.take_along_axis(key, idx.astype(np.int64), 1))
    for t in range(T):
        rest = np.delete(key[t], idx[t])
        assert margin2[t] == np.float64(sel[t, -1]) - np.float64(rest.max())


def test_all_equal_scores_pick_lowest_indices(orc):
    T, E, k = 5, 16, 4
    cfg = orc.Config(T=T, d=1, E=E, k=k, I=1)
    idx, gates, margin = orc.route_from_logits(cfg, np.zeros((T, E), np.float32),
                                               np.zeros(E, np.float32))
    assert np.array_equal(idx, np.tile(np.arange(k), (T, 1)))
    assert np.allclose(gates, 2.827 / k, rtol=0, atol=1e-15)
    assert np.all(margin == 0.0)


def test_bias_selects_but_does_not_weight(orc):
    rng = np.random.default_rng(4)
    T, E, k = 50, 16, 2
    z = rng.standard_normal((T, E)).astype(np.float32)
    b = np.zeros(E, np.float32)
    b[[3, 11]] = 5.0                       # forces experts 3 and 11 for every token
    cfg = orc.Config(T=T, d=1, E=E, k=k, I=1)
    idx, gates, _ = orc.route_from_logits(cfg, z, b)
    assert all(sorted(r) == [3, 11] for r in idx)
    s = 1.0 / (1.0 + np.exp(-z.astype(np.float64)))
    expect = 2.827 * s[np.arange(T)[:, None], idx] / (s[:, 3] + s[:, 11])[:, None]
    assert np.allclose(gates, expect, rtol=1e-14, atol=0)
    b2 = b.copy()
    b2[[3, 11]] = 9.0                      # a different bias, the same selection
    _, gates2, _ = orc.route_from_logits(cfg, z, b2)
    assert np.array_equal(gates, gates2)


def test_gates_closed_form_from_rational_sigmoids(orc):
    """Logits ln 3, 0, -ln 3, -ln 9 have sigmoids 3/4, 1/2, 1/4, 1/10 exactly, so the gates have
    closed forms: with no bias the top two are experts 0 and 1 with 2.827 * (3/5, 2/5); a bias of
    0.6 on expert 2 lifts its key to 0.85 above expert 0's 0.75, and the gates, taken from the
    unbiased sigmoids, are 2.827 * (1/4, 3/4) in key order.  A sign slip in the sigmoid, a gate
    taken from the biased key, or a missing renormalisation fails one of these."""
    ln3 = math.log(3.0)
    z = np.array([[ln3, 0.0, -ln3, -math.log(9.0)]], np.float32)
    cfg = orc.Config(T=1, d=1, E=4, k=2, I=1)
    idx, gates, _ = orc.route_from_logits(cfg, z, np.zeros(4, np.float32))
    assert list(idx[0]) == [0, 1]
    np.testing.assert_allclose(gates[0], [2.827 * 0.6, 2.827 * 0.4], rtol=1e-6)
    idx, gates, _ = orc.route_from_logits(cfg, z, np.array([0, 0, 0.6, 0], np.float32))
    assert list(idx[0]) == [2, 0]
    np.testing.assert_allclose(gates[0], [2.827 * 0.25, 2.827 * 0.75], rtol=1e-6)


def _tiny_layer(T=64, seed=0, **over):
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    w = S.WORKLOADS["tiny_fp32"].with_tokens(T)
    if over:
        from dataclasses import replace
        w = replace(w, **over)
    return S.make_layer(w, seed=seed, device="cpu")


def test_gates_sum_to_scale_and_route_matches_forward(orc):
    from oracle import torch_bridge as B
    layer = _tiny_layer()
    res = B.forward(layer)
    assert np.allclose(res["gates"].sum(1), 2.827, rtol=0, atol=1e-12)
    assert np.all(res["gates"] > 0)
    x, W_r, b = B.route_inputs(layer)
    r = orc.route(B.config(layer), x, W_r, b)
    assert np.array_equal(r["idx"], res["idx"]) and np.array_equal(r["gates"], res["gates"])
    # logits are x W_r^T: compare with a numpy matmul
    ref = layer.x.double().numpy() @ layer.W_r.double().numpy().T
    assert np.allclose(r["logits"], ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------------------------
# Experts
# --------------------------------------------------------------------------------------------

def test_swiglu_hand_computed(orc):
    rows = {r[0]: np.array([float(v) for v in r[1:]]) for r in read_golden("swiglu_hand.txt")}
    W13 = np.concatenate([rows["W1"].reshape(2, 3), rows["W3"].reshape(2, 3)])
    W2 = rows["W2"].reshape(3, 2)
    y = orc.swiglu_row(rows["x"], orc.Mat(W13, "f64"), orc.Mat(W2, "f64"), I=2)
    assert np.allclose(y, rows["E"], rtol=0, atol=1e-15)


# --------------------------------------------------------------------------------------------
# 4-bit integer groups
# --------------------------------------------------------------------------------------------

def test_int4_hand_decoded(orc):
    """Two rows decoded by hand from the format definition (tests/golden/int4_hand.txt): the
    nibble order inside a word, the excess-8 codes, the per-32 scale and the bf16 rounding of the
    product (values that round up, round down and round away in magnitude)."""
    rows = {r[0]: r[1:] for r in read_golden("int4_hand.txt")}
    row_bytes = np.array([int(b, 16) for b in rows["bytes"]], np.uint8)
    packed = np.stack([row_bytes, row_bytes])                      # [2][16]
    scales = np.array([[float(v) for v in rows["scales"]]], np.float32)  # [K/32 = 1][rows = 2]
    W = orc.Mat(packed, "int4", scales)
    r0 = orc.dequant_row(W, 0, 32)
    assert np.array_equal(r0, np.array([float(v) for v in rows["row0"]]))
    r1 = orc.dequant_row(W, 1, 32)
    for pick in rows["row1_picks"]:
        ch, val = pick.split(":")
        assert r1[int(ch)] == float(val), pick


def test_int4_decode_against_torch(orc):
    """The oracle's int4 decode of synthetic weights against an independent decode in torch
    (nibbles by the format, excess-8, times the scale, torch's bf16 rounding)."""
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    g = torch.Generator().manual_seed(11)
    m = torch.randn(16, 256, generator=g) * 0.02
    packed, scale = S._int4_quantize(m)
    W = orc.Mat(packed.numpy(), "int4", scale.float().numpy())
    b = packed.to(torch.int32)                                        # [16][128] bytes
    nib = torch.stack([b & 15, b >> 4], dim=-1).reshape(16, 32, 8)    # per word: nibbles 0..7
    code = nib[:, :, [0, 4, 1, 5, 2, 6, 3, 7]].reshape(16, 256) - 8   # channel 8w + i
    ref = (code.double() * scale.t().double().repeat_interleave(32, dim=1)).float().bfloat16()
    for r in range(16):
        assert np.array_equal(orc.dequant_row(W, r, 256), ref[r].double().numpy())


def test_int4_layer_equals_the_bf16_layer_of_its_values(orc):
    """A layer with int4 experts gives exactly the output of the same layer with bf16 experts
    holding the decoded values (routing reads no expert weight; the GEMMs see equal fp64 values)."""
    from dataclasses import replace
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    from oracle import torch_bridge as TB
    w = replace(S.WORKLOADS["tiny_fp32"], name="tiny_int4", act="bf16", int4=True,
                quant_block=32, T=24)
    L4 = S.make_layer(w, seed=5, device="cpu")
    r4 = TB.forward(L4, nthreads=2)

    def decode(packed, scale):
        M = orc.Mat(packed.numpy(), "int4", scale.float().numpy())
        cols = packed.shape[1] * 2
        return torch.from_numpy(np.stack([orc.dequant_row(M, r, cols)
                                          for r in range(packed.shape[0])])).bfloat16()

    Lb = S.make_layer(replace(w, int4=False), seed=5, device="cpu")
    for e in range(w.E):
        Lb.W13[e] = decode(L4.W13[e], L4.W13_scale[e])
        Lb.W2[e] = decode(L4.W2[e], L4.W2_scale[e])
    Lb.Ws13 = decode(L4.Ws13, L4.Ws13_scale)
    Lb.Ws2 = decode(L4.Ws2, L4.Ws2_scale)
    rb = TB.forward(Lb, nthreads=2)
    assert np.array_equal(r4["idx"], rb["idx"])
    assert np.array_equal(r4["out"], rb["out"])


# --------------------------------------------------------------------------------------------
# The block around the layer: x_ffn = RMSNorm(x'_n), layer, x_{n+1} = x'_n + D_ffn
# --------------------------------------------------------------------------------------------

def test_bf16_rounding_matches_the_format(orc):
    """round_bf16 (8 significant bits, ties to even) against torch's fp32 -> bf16 conversion on
    values exact in fp32, including exact ties, and its own idempotence."""
    from oracle import torch_bridge as TB
    g = torch.Generator().manual_seed(3)
    v = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-20, 20, (20000,), generator=g).float())
    ties = (torch.randint(128, 256, (2000,), generator=g).double() * 2 + 1) / 512.0  # m + half ulp
    vals = torch.cat([v.double(), ties, -ties])
    ours = TB.round_bf16(vals.numpy())
    ref = vals.float().bfloat16().double().numpy()
    assert np.array_equal(ours, ref)
    assert np.array_equal(TB.round_bf16(ours), ours)


def test_block_with_zero_norm_weight_passes_the_residual(orc):
    """A zero RMSNorm weight makes x_ffn = 0: every expert and the shared expert see a zero input,
    SiLU(0) * 0 = 0, so D_ffn = 0 and the block returns x'_n unchanged, bit for bit."""
    from oracle import torch_bridge as TB
    layer = _tiny_layer(T=20)
    res = TB.block_forward(layer, torch.zeros(layer.w.d), nthreads=2)
    assert np.all(res["delta"] == 0.0)
    assert np.array_equal(res["out"], layer.x.double().numpy())


def test_block_norm_closed_form_and_scale_invariance(orc):
    """With unit weight every normalised row has mean square m / (m + eps) (m the row's mean
    square, up to the rounding of x_ffn to the activation type), and the FFN half is invariant to scaling x'_n (up to eps): block(4x) - 4x equals
    block(x) - x."""
    from oracle import torch_bridge as TB
    layer = _tiny_layer(T=16)
    x = layer.x.double().numpy()
    res = TB.block_forward(layer, torch.ones(layer.w.d), nthreads=2)
    m = np.mean(x * x, axis=1)
    # x_ffn is rounded once to the fp32 activation type: 2^-24 per element, 2^-23 per square
    assert np.allclose(np.mean(res["x_ffn"] ** 2, axis=1), m / (m + layer.w.rms_eps), rtol=3e-7)
    g = torch.rand(layer.w.d, generator=torch.Generator().manual_seed(5)) + 0.5
    r1 = TB.block_forward(layer, g, nthreads=2)
    layer.x = layer.x * 4.0
    r4 = TB.block_forward(layer, g, nthreads=2)
    assert np.allclose(r4["out"] - 4.0 * x, r1["out"] - x, rtol=1e-5, atol=1e-6)


def test_dense_mlp_hand_computed(orc):
    """The dense block MLP on the hand-computed SwiGLU case, with a zero token beside it:
    SiLU(0) * 0 = 0, so the second row must be exactly zero."""
    rows = {r[0]: np.array([float(v) for v in r[1:]]) for r in read_golden("swiglu_hand.txt")}
    W13 = np.concatenate([rows["W1"].reshape(2, 3), rows["W3"].reshape(2, 3)])
    W2 = rows["W2"].reshape(3, 2)
    x = np.stack([rows["x"], np.zeros(3)])
    y = orc.dense_mlp(orc.Mat(x, "f64"), orc.Mat(W13, "f64"), orc.Mat(W2, "f64"), nthreads=2)
    assert np.allclose(y[0], rows["E"], rtol=0, atol=1e-15)
    assert np.all(y[1] == 0.0)


def test_dense_mlp_is_one_always_selected_expert(orc):
    """A MoE layer with one expert, top-1 and no shared expert routes every token to expert 0 with
    gate 2.827 * s / s = 2.827: its output is 2.827 times the dense MLP with the same weights."""
    from oracle import torch_bridge as TB
    layer = _tiny_layer(T=24, E=1, k=1, n_shared=0)
    res = TB.forward(layer)
    x = orc.Mat(layer.x.numpy(), "f32")
    y = orc.dense_mlp(x, orc.Mat(layer.W13[0].numpy(), "f32"), orc.Mat(layer.W2[0].numpy(), "f32"),
                      nthreads=3)
    assert np.allclose(res["out"], 2.827 * y, rtol=1e-13, atol=1e-13)
    ref = dense_swiglu(layer.x.double().numpy(), layer.W13[0].double().numpy(),
                       layer.W2[0].double().numpy())
    assert np.allclose(y, ref, rtol=1e-11, atol=1e-12)


def test_dense_mlp_threads_do_not_change_the_result(orc):
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    L = S.make_dense(S.DENSE_WORKLOADS["tiny_dense_fp32"], device="cpu")
    args = (orc.Mat(L.x.numpy(), "f32"), orc.Mat(L.W13.numpy(), "f32"), orc.Mat(L.W2.numpy(), "f32"))
    assert np.array_equal(orc.dense_mlp(*args, nthreads=1), orc.dense_mlp(*args, nthreads=7))


def test_dense_reduction_one_forced_expert(orc):
    """top_k = 1 with a bias that forces expert 5: every gate is 2.827 and the layer is
    2.827 * MLP_5(x) + MLP_shared(x), a pair of dense SwiGLU MLPs."""
    from oracle import torch_bridge as B
    layer = _tiny_layer(T=32, k=1)
    layer.b.zero_()
    layer.b[5] = 10.0
    res = B.forward(layer)
    assert np.all(res["idx"] == 5) and np.allclose(res["gates"], 2.827, atol=1e-15)
    x = layer.x.double().numpy()
    ref = 2.827 * dense_swiglu(x, layer.W13[5].double().numpy(), layer.W2[5].double().numpy())
    ref += dense_swiglu(x, layer.Ws13.double().numpy(), layer.Ws2.double().numpy())
    assert np.allclose(res["out"], ref, rtol=1e-11, atol=1e-12)
    assert np.allclose(res["shared"] + res["routed"], res["out"], rtol=0, atol=1e-15)


def test_concatenation_identity(orc):
    """With every expert selected and equal gates 2.827/E, the routed sum is one dense SwiGLU of
    width E*I whose W1 / W3 rows and W2 columns are the experts' concatenated."""
    from oracle import torch_bridge as B
    E = 4
    layer = _tiny_layer(T=16, E=E, k=E)
    layer.W_r.zero_()                                  # s = 1/2 for all -> equal gates
    res = B.forward(layer)
    I = layer.w.I
    W1 = np.concatenate([layer.W13[e, :I].double().numpy() for e in range(E)])
    W3 = np.concatenate([layer.W13[e, I:].double().numpy() for e in range(E)])
    W2 = np.concatenate([layer.W2[e].double().numpy() for e in range(E)], axis=1)
    ref = (2.827 / E) * dense_swiglu(layer.x.double().numpy(), np.concatenate([W1, W3]), W2)
    assert np.allclose(res["routed"], ref, rtol=1e-11, atol=1e-12)


def test_rows_are_independent(orc):
    from oracle import torch_bridge as B
    layer = _tiny_layer()
    full = B.forward(layer)
    rows = torch.tensor([40, 3, 17, 63, 0])
    sub = B.forward(layer, rows=rows, experts=range(layer.w.E))
    assert np.array_equal(sub["out"], full["out"][rows.numpy()])
    assert np.array_equal(sub["idx"], full["idx"][rows.numpy()])


def test_threads_do_not_change_results(orc):
    from oracle import torch_bridge as B
    layer = _tiny_layer()
    assert np.array_equal(B.forward(layer, nthreads=1)["out"], B.forward(layer, nthreads=5)["out"])


# --------------------------------------------------------------------------------------------
# K3 latent path
# --------------------------------------------------------------------------------------------

def test_rmsnorm_closed_form(orc):
    eps = 1e-6
    assert np.allclose(orc.rmsnorm_unit(np.array([3.0, 4.0]), eps),
                       np.array([3.0, 4.0]) / math.sqrt(12.5 + eps), rtol=1e-15)
    c = -2.5
    assert np.allclose(orc.rmsnorm_unit(np.full(7, c), eps), c / math.sqrt(c * c + eps),
                       rtol=1e-15)


def test_latent_path_with_selection_projections_reduces_to_k2(orc):
    """W_down = [I_L | 0], W_up = its transpose, no norm: the latent layer's routed output is the
    full-width layer's routed output on the first L channels, padded with zeros."""
    from oracle import torch_bridge as B
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    from dataclasses import replace
    d, L = 256, 128
    wl = replace(S.WORKLOADS["tiny_fp32"], T=24, d_latent=L, latent_norm=0)
    lat = S.make_layer(wl, seed=3, device="cpu")
    lat.W_down.zero_()
    lat.W_down[:, :L] = torch.eye(L)
    lat.W_up.zero_()
    lat.W_up[:L, :] = torch.eye(L)
    lat.W_r[:, L:] = 0.0                               # the router sees only the first L channels
    res = B.forward(lat)
    wk = replace(S.WORKLOADS["tiny_fp32"], T=24, d=L)
    k2 = S.make_layer(wk, seed=3, device="cpu")
    k2.x = lat.x[:, :L].contiguous()
    k2.W_r = lat.W_r[:, :L].contiguous()
    k2.b = lat.b
    k2.W13, k2.W2 = lat.W13, lat.W2
    ref = B.forward(k2)
    assert np.array_equal(res["idx"], ref["idx"])
    assert np.allclose(res["routed"][:, :L], ref["routed"], rtol=1e-12, atol=1e-13)
    assert np.all(res["routed"][:, L:] == 0.0)


def test_latent_norm_applies_before_up_projection(orc):
    """With W_up = [I_L ; 0] the routed output is exactly RMSNorm(y_lat): unit RMS over L."""
    from oracle import torch_bridge as B
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    from dataclasses import replace
    L = 128
    wl = replace(S.WORKLOADS["tiny_fp32"], T=16, d_latent=L, latent_norm=1)
    lat = S.make_layer(wl, seed=5, device="cpu")
    lat.W_up.zero_()
    lat.W_up[:L, :] = torch.eye(L)
    res = B.forward(lat)
    y = res["routed"][:, :L]
    rms = np.sqrt((y * y).mean(1))
    ms = (y * y).mean(1)
    # y = v / sqrt(mean(v^2)+eps) => mean(y^2) = m / (m + eps) with m = mean(v^2) > 0
    assert np.all(rms < 1.0) and np.all(rms > 1.0 - 1e-3)
    assert np.all(ms <= 1.0)


# --------------------------------------------------------------------------------------------
# fp8 experts
# --------------------------------------------------------------------------------------------

def test_fp8_forward_matches_library_composition(orc):
    """The fp8 layer recomposed from torch's float8 conversion (an independent library routine):
    weights = e4m3 x block scale, x and h quantised per token per 128 channels with scale
    amax/448 (decided in fp32), everything else in fp64."""
    from oracle import torch_bridge as B
    from mixture_experts_ffn_gemm_gb300 import synthetic as S
    from dataclasses import replace
    w = replace(S.WORKLOADS["tiny_fp32"], T=12, E=4, k=2, fp8=True, act="bf16")
    layer = S.make_layer(w, seed=6, device="cpu")
    res = B.forward(layer)

    def deq_w(q, s):
        v = q.to(torch.float64)
        return (v * s.double().repeat_interleave(128, 0).repeat_interleave(128, 1)).numpy()

    def qact(v64):
        v = torch.from_numpy(v64.astype(np.float32))
        out = torch.empty_like(v, dtype=torch.float64)
        for g0 in range(0, v.numel(), 128):
            grp = v[g0:g0 + 128]
            amax = grp.abs().max()
            s = amax / torch.tensor(448.0) if amax > 0 else torch.tensor(1.0)
            q = (grp / s).clamp(-448, 448).to(torch.float8_e4m3fn)
            out[g0:g0 + 128] = q.to(torch.float64) * s.double()
        return out.numpy()

    def mlp(x, W13, W2, I):
        xq = qact(x)
        g = W13[:I] @ xq
        u = W13[I:] @ xq
        h = qact(silu(g) * u)
        return W2 @ h

    x = layer.x.double().numpy()
    I = w.I
    for t in range(w.T):
        ref = mlp(x[t], deq_w(layer.Ws13, layer.Ws13_scale), deq_w(layer.Ws2, layer.Ws2_scale), I)
        for j in range(w.k):
            e = res["idx"][t, j]
            ref = ref + res["gates"][t, j] * mlp(x[t], deq_w(layer.W13[e], layer.W13_scale[e]),
                                                  deq_w(layer.W2[e], layer.W2_scale[e]), I)
        assert np.allclose(res["out"][t], ref, rtol=1e-9, atol=1e-9)
