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
