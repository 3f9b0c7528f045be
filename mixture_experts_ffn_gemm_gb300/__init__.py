"""GB300 (sm_103a) mixture-of-experts FFN layer: Kimi K2 / DeepSeek-V3 routing and SwiGLU experts,
and the Kimi K3 latent variant, as a C-ABI CUDA library (``include/moe.h``) with a thin ctypes
binding.  Import the binding lazily so that ``synthetic`` stays usable without a built library."""

__all__ = ["binding", "synthetic", "build"]
