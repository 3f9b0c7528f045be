"""Why the bf16 outputs are bounded beyond their own rounding (CPU, no GPU).

The parity rule (parity_lib) holds a bf16 result to max(|GPU - oracle| - 2^-8 |oracle|) <= 2e-2
rms(oracle) and reports the plain max |GPU - oracle| / rms beside it.  These tests measure, with
the committed rounding model (rounding_model.py: exact fp64 arithmetic with the oracle's own
routing, plus only the bf16 roundings a bf16 pipeline cannot avoid -- h, x_lat, u_hat and the
output), that:
  * the model with no rounding is the oracle itself (1e-12), so the model computes the layer the
    pages define;
  * the ideal bf16 pipeline's plain error already exceeds 2e-2 rms on the K3 latent path and on a
    k = 1 layer (outputs that are one gate-amplified expert), so no bf16 implementation can meet
    the plain bound there; the K2 top-4 layer stays below it;
  * the output's own rounding is exactly what the 2^-8 |ref| term removes (beyond it, an output
    rounded from the exact value has no error left), and the ideal pipeline's error beyond its
    rounding stays well inside 2e-2.
Inputs are the GPU parity tests' small cases, drawn by the CPU generator with the same seeds.
"""
from dataclasses import replace

import numpy as np
import pytest

from oracle import torch_bridge as OB
from mixture_experts_ffn_gemm_gb300 import synthetic as S

import rounding_model as R

SMALL_BF16 = replace(S.WORKLOADS["tiny_fp32"], name="small_bf16", act="bf16", T=300)
LATENT = replace(SMALL_BF16, name="latent_small", d=512, d_latent=256, latent_norm=1, T=700,
                 w_init="fan_in")
CASES = {
    # name: (workload, seed, forced expert or None)
    "k2_top4": (SMALL_BF16, 1, None),
    "k1_forced": (replace(SMALL_BF16, k=1, T=333), 2, 5),
    "k3_latent_norm": (LATENT, 9, None),
    "k3_latent_no_norm": (replace(LATENT, latent_norm=0, T=300), 7, None),
}
# the ideal pipeline's plain error is above the plain 2e-2 bound on these cases
ABOVE_PLAIN_BOUND = {"k1_forced", "k3_latent_norm", "k3_latent_no_norm"}


def _case(name):
    w, seed, force = CASES[name]
    layer = S.make_layer(w, seed=seed, device="cpu")
    if force is not None:
        layer.b.zero_()
        layer.b[force] = 10.0
    ref = OB.forward(layer, nthreads=4)
    keep = ref["margin"] >= 1e-5
    return layer, ref, keep


@pytest.fixture(scope="module")
def cases():
    return {name: _case(name) for name in CASES}


@pytest.mark.parametrize("name", list(CASES))
def test_model_without_rounding_is_the_oracle(cases, name):
    layer, ref, _ = cases[name]
    exact = R.ideal_forward(layer, round_h=False, round_out=False, round_xlat=False,
                            round_uhat=False)
    rms = np.sqrt(np.mean(ref["out"] ** 2))
    assert np.array_equal(exact["idx"], ref["idx"])
    assert np.abs(exact["out"] - ref["out"]).max() <= 1e-12 * rms


@pytest.mark.parametrize("name", list(CASES))
def test_output_rounding_is_what_the_rule_removes(cases, name):
    """Rounding the exact output to bf16 and nothing else: the plain error is the rounding
    itself (up to 2^-8 of the largest output), and nothing is left beyond 2^-8 |ref|."""
    layer, ref, keep = cases[name]
    only_out = R.ideal_forward(layer, round_h=False, round_xlat=False, round_uhat=False)
    e = R.errors(only_out["out"][keep], ref["out"][keep])
    assert e["beyond_rounding"] <= 1e-9
    assert 0.25 * 2.0 ** -8 * np.abs(ref["out"][keep]).max() / np.sqrt(
        np.mean(ref["out"][keep] ** 2)) <= e["plain"]


@pytest.mark.parametrize("name", list(CASES))
def test_ideal_bf16_pipeline_against_the_bounds(cases, name):
    layer, ref, keep = cases[name]
    ideal = R.ideal_forward(layer)
    e = R.errors(ideal["out"][keep], ref["out"][keep])
    print(name, {k: f"{v:.3e}" for k, v in e.items()})
    if name in ABOVE_PLAIN_BOUND:
        assert e["plain"] > 2e-2  # the plain bound is out of reach of any bf16 pipeline here
    else:
        assert e["plain"] <= 2e-2
    assert e["beyond_rounding"] <= 1.5e-2  # inside the bound the parity tests apply
    assert e["rms"] <= 5e-3


@pytest.mark.parametrize("name", ["k2_top4", "k1_forced"])
def test_pages_rounding_sequence_against_the_one_rounding_sum(cases, name):
    """The pages' `moe_infer` rounds each expert's output to bf16, casts it to the gate type,
    multiplies, sums over the slots and casts back, then adds the bf16 shared output in bf16.  The
    library sums the fp32 expert outputs with the shared one and rounds once.  Against the fp64
    oracle: the pages' sequence is itself inside the parity rule (so the rule does not reject the
    pages' own arithmetic), and the one-rounding sum is the more accurate of the two, in the rms
    and in the error beyond the output's rounding."""
    layer, ref, keep = cases[name]
    pages = R.errors(R.pages_combine_forward(layer)["out"][keep], ref["out"][keep])
    ours = R.errors(R.ideal_forward(layer)["out"][keep], ref["out"][keep])
    print(name, "pages", {k: f"{v:.3e}" for k, v in pages.items()},
          "one rounding", {k: f"{v:.3e}" for k, v in ours.items()})
    assert pages["beyond_rounding"] <= 2e-2 and pages["rms"] <= 5e-3
    assert ours["rms"] < pages["rms"]
    assert ours["beyond_rounding"] < pages["beyond_rounding"]
