"""moe_permute_noalloc, the dispatch bookkeeping for callers that cannot allocate device memory
(for example a serving process that handed the GPU's free memory to its own pool at start-up, or
a latency-critical loop where cudaMalloc may synchronise the device).

The entry point keeps its scratch in a fixed array inside the library instead of a caller
workspace.  Checked through the C ABI against moe_permute (which uses a workspace), bit for bit,
on two calls in a row with different routings: the second call must not see the first call's
leftovers in the shared array.  This file is collected last so that a failure here comes after
every other GPU test has run.
"""
import pytest
import torch

from mixture_experts_ffn_gemm_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _routing(T, E, k, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    scores = torch.rand(T, E, generator=g, device="cuda")
    return scores.topk(k, dim=1).indices.to(torch.int32).contiguous()  # k distinct experts/token


def _outputs(T, E, k):
    z = lambda n: torch.full((n,), -9, dtype=torch.int32, device="cuda")  # noqa: E731
    return z(E + 1), z(E + 2), z(T * k), z(T * k)


@pytest.mark.parametrize("T,E,k", [(128, 384, 8), (16384, 384, 8), (37, 16, 4)])
def test_noalloc_permute_matches_workspace_permute(cuda_device, T, E, k):
    cfg = B.make_config(T=T, d=7168, E=E, k=k, I=2048)
    ws = B.alloc_workspace(cfg)
    for call, seed in enumerate((11, 12)):
        idx = _routing(T, E, k, seed + T)
        ref = _outputs(T, E, k)
        got = _outputs(T, E, k)
        B.moe_permute(cfg, idx, *ref, ws)
        B.moe_permute_noalloc(cfg, idx, *got)
        torch.cuda.synchronize()
        for name, a, b in zip(("counts", "offsets", "perm_src", "perm_dst"), ref, got):
            assert torch.equal(a, b), f"call {call + 1}: {name} differs"
        assert int(got[0][:E].sum()) == T * k


def _compare(cfg, ws, idx, T, E, k, what):
    ref = _outputs(T, E, k)
    got = _outputs(T, E, k)
    B.moe_permute(cfg, idx, *ref, ws)
    B.moe_permute_noalloc(cfg, idx, *got)
    torch.cuda.synchronize()
    for name, a, b in zip(("counts", "offsets", "perm_src", "perm_dst"), ref, got):
        assert torch.equal(a, b), f"{what}: {name} differs"
    return got


def test_noalloc_permute_after_a_larger_expert_count(cuda_device):
    """The shared array holds [chunks][E] counts, so its row stride follows E.  A call with many
    chunks and E = 1000 leaves counts at that stride; the next call, with fewer experts (E = 40,
    another stride) and a ragged last chunk, must not read any of them."""
    for T, E, k, seed in ((24000, 1000, 8, 31), (5000, 40, 6, 32), (1500, 7, 3, 33)):
        cfg = B.make_config(T=T, d=256, E=E, k=k, I=128)  # small widths: a small workspace
        ws = B.alloc_workspace(cfg)
        got = _compare(cfg, ws, _routing(T, E, k, seed), T, E, k, f"T={T} E={E}")
        assert int(got[0][:E].sum()) == T * k


@pytest.mark.parametrize("T", [100, 3000])
def test_noalloc_permute_skips_out_of_range_ids(cuda_device, T):
    """Expert ids outside [0, E) are not counted and their perm_dst entries are -1, exactly as
    moe_permute leaves them (one CTA up to 1024 pairs, the chunked kernels above)."""
    E, k = 64, 4
    cfg = B.make_config(T=T, d=256, E=E, k=k, I=128)
    ws = B.alloc_workspace(cfg)
    idx = _routing(T, E, k, 40 + T)
    bad = [(3, 1, E), (T // 2, 0, -1), (T - 1, 3, E + 77)]
    for t, j, v in bad:
        idx[t, j] = v
    got = _compare(cfg, ws, idx, T, E, k, f"T={T} with out-of-range ids")
    assert int(got[0][:E].sum()) == T * k - len(bad)
    for t, j, _ in bad:
        assert int(got[3][t * k + j]) == -1


def test_noalloc_permute_refuses_sizes_beyond_its_scratch(cuda_device):
    too_many_pairs = B.make_config(T=262144 // 8 + 1, d=7168, E=384, k=8, I=2048)
    out = _outputs(1, 384, 8)
    idx = torch.zeros(1, 8, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoEError) as ei:
        B.moe_permute_noalloc(too_many_pairs, idx, *out)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
    too_many_experts = B.make_config(T=4, d=7168, E=1024, k=8, I=2048)
    with pytest.raises(B.MoEError) as ei:
        B.moe_permute_noalloc(too_many_experts, idx, *out)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
