"""ctypes binding of the C ABI in ``include/moe.h`` (argument marshalling only).

Every function has the name of its C entry point and takes torch tensors (device memory) or
``None`` for a NULL pointer; the stream defaults to torch's current CUDA stream.  All compute runs
in the CUDA library ``_build/libmoe_gb300.so``; if that library is missing the first call raises:
there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_DEVICE_CHECK, MOE_ERR_TIMEOUT = 4, 5, 6
MOE_F32, MOE_BF16, MOE_FP8_E4M3, MOE_INT4 = 0, 1, 2, 3
MOE_FLAG_GEMM_ROWS_MAJOR, MOE_FLAG_GEMM_SWAP_AB = 0x1, 0x2
MOE_FLAG_ROUTER_SIMT, MOE_FLAG_ROUTER_TC = 0x4, 0x8
MOE_FLAG_TEST_STALL_EXPERTS = 0x100
MOE_FLAG_GEMM_N128 = 0x10
MOE_FLAG_GEMM_SWAP_WIDE = 0x20
MOE_FLAG_GEMM_M1, MOE_FLAG_GEMM_M2 = 0x40, 0x80
MOE_FLAG_DECODE_FUSED = 0x200
MOE_FLAG_GEMM_PAIR = 0x400
MOE_FLAG_EXPERT_OUT_BF16 = 0x800
MOE_FLAG_EXPERT_OUT_F32 = 0x1000

EXPORTED = ("moe_workspace_size", "moe_router", "moe_permute", "moe_experts", "moe_combine",
            "moe_forward", "moe_forward_host_io", "moe_reset_device_status", "moe_device_status",
            "moe_status_string", "moe_launch_count", "moe_reset_launch_count",
            "moe_profile_enable", "moe_profile_read", "moe_permute_noalloc",
            "moe_last_error_string", "moe_dense_mlp_workspace_size", "moe_dense_mlp",
            "moe_forward_block")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == MOE_ERR_CUDA:
            detail = " [" + load_library().moe_last_error_string().decode() + "]"
        super().__init__(f"{where}: {status_string(status)} ({status}){detail}")


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("I_shared", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("d_latent", ctypes.c_int32),
                ("latent_norm", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("w_dtype", ctypes.c_int32), ("quant_block", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("gate_scale", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("reserved_", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"the MoE CUDA library is not built ({LIB_PATH}); run "
                                   "`python -m mixture_experts_ffn_gemm_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            P, C = ctypes.c_void_p, ctypes.POINTER(moe_config_t)
            S = ctypes.c_int
            lib.moe_workspace_size.restype = ctypes.c_size_t
            lib.moe_workspace_size.argtypes = [C]
            lib.moe_router.restype = S
            lib.moe_router.argtypes = [C, P, P, P, P, P, P, P, ctypes.c_size_t, P]
            lib.moe_permute.restype = S
            lib.moe_permute.argtypes = [C, P, P, P, P, P, P, ctypes.c_size_t, P]
            lib.moe_experts.restype = S
            lib.moe_experts.argtypes = [C, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                        ctypes.c_size_t, P]
            lib.moe_combine.restype = S
            lib.moe_combine.argtypes = [C, P, P, P, P, P, P, ctypes.c_size_t, P]
            lib.moe_forward.restype = S
            lib.moe_forward.argtypes = [C, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                        ctypes.c_size_t, P]
            lib.moe_forward_block.restype = S
            lib.moe_forward_block.argtypes = [C, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                              ctypes.c_size_t, P]
            lib.moe_forward_host_io.restype = S
            lib.moe_forward_host_io.argtypes = lib.moe_forward.argtypes
            lib.moe_reset_device_status.restype = S
            lib.moe_reset_device_status.argtypes = [P, ctypes.c_size_t, P]
            lib.moe_device_status.restype = S
            lib.moe_device_status.argtypes = [P, ctypes.c_size_t, P]
            lib.moe_status_string.restype = ctypes.c_char_p
            lib.moe_status_string.argtypes = [S]
            lib.moe_launch_count.restype = ctypes.c_uint64
            lib.moe_launch_count.argtypes = []
            lib.moe_reset_launch_count.restype = None
            lib.moe_reset_launch_count.argtypes = []
            lib.moe_last_error_string.restype = ctypes.c_char_p
            lib.moe_last_error_string.argtypes = []
            lib.moe_permute_noalloc.restype = S
            lib.moe_permute_noalloc.argtypes = [C, P, P, P, P, P, P]
            lib.moe_dense_mlp_workspace_size.restype = ctypes.c_size_t
            lib.moe_dense_mlp_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int32,
                                                         ctypes.c_int32, S]
            lib.moe_dense_mlp.restype = S
            lib.moe_dense_mlp.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, S, P, P,
                                          P, P, P, ctypes.c_size_t, P]
            lib.moe_profile_enable.restype = S
            lib.moe_profile_enable.argtypes = [S]
            lib.moe_profile_read.restype = S
            lib.moe_profile_read.argtypes = [S, P, ctypes.c_size_t, P, P]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().moe_status_string(int(status)).decode()


def _dt(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return MOE_F32
    if dtype == torch.bfloat16:
        return MOE_BF16
    if dtype == torch.float8_e4m3fn:
        return MOE_FP8_E4M3
    if dtype == torch.uint8:  # packed 4-bit integer groups
        return MOE_INT4
    raise TypeError(f"unsupported dtype {dtype}")


def make_config(T: int, d: int, E: int, k: int, I: int, I_shared: Optional[int] = None,
                n_shared: int = 1, d_latent: int = 0, latent_norm: int = 0,
                act_dtype: torch.dtype = torch.bfloat16, w_dtype: Optional[torch.dtype] = None,
                quant_block: int = 128, flags: int = 0, gate_scale: float = 2.827,
                rms_eps: float = 1e-6) -> moe_config_t:
    return moe_config_t(int(T), int(d), int(E), int(k), int(I),
                        int(I if I_shared is None else I_shared), int(n_shared), int(d_latent),
                        int(latent_norm), _dt(act_dtype), _dt(w_dtype or act_dtype),
                        int(quant_block), int(flags), float(gate_scale), float(rms_eps), 0)


def config_for(w, T: Optional[int] = None, flags: int = 0) -> moe_config_t:
    """The C configuration of a synthetic ``Workload`` (optionally with another token count)."""
    act = torch.float32 if w.act == "f32" else torch.bfloat16
    return make_config(T=w.T if T is None else T, d=w.d, E=w.E, k=w.k, I=w.I,
                       I_shared=w.I_shared, n_shared=w.n_shared, d_latent=w.d_latent,
                       latent_norm=w.latent_norm, act_dtype=act,
                       w_dtype=(torch.float8_e4m3fn if w.fp8 else
                                torch.uint8 if getattr(w, "int4", False) else act),
                       quant_block=w.quant_block, flags=flags, gate_scale=w.gate_scale,
                       rms_eps=w.rms_eps)


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def _dev(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return _p(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


def moe_workspace_size(cfg: moe_config_t) -> int:
    return int(load_library().moe_workspace_size(ctypes.byref(cfg)))


def alloc_workspace(cfg: moe_config_t, device="cuda") -> torch.Tensor:
    n = moe_workspace_size(cfg)
    if n == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_router(cfg, x, W_r, b, logits, topk_idx, topk_weight, ws, stream=None):
    _check(load_library().moe_router(ctypes.byref(cfg), _dev(x), _dev(W_r), _dev(b), _dev(logits),
                                     _dev(topk_idx), _dev(topk_weight), _dev(ws), ws.numel(),
                                     _stream(stream)), "moe_router")


def moe_permute(cfg, topk_idx, counts, offsets, perm_src, perm_dst, ws, stream=None):
    _check(load_library().moe_permute(ctypes.byref(cfg), _dev(topk_idx), _dev(counts),
                                      _dev(offsets), _dev(perm_src), _dev(perm_dst), _dev(ws),
                                      ws.numel(), _stream(stream)), "moe_permute")


def moe_permute_noalloc(cfg, topk_idx, counts, offsets, perm_src, perm_dst, stream=None):
    """moe_permute for callers that cannot allocate: no workspace, fixed in-library scratch."""
    _check(load_library().moe_permute_noalloc(ctypes.byref(cfg), _dev(topk_idx), _dev(counts),
                                              _dev(offsets), _dev(perm_src), _dev(perm_dst),
                                              _stream(stream)), "moe_permute_noalloc")


def moe_experts(cfg, x, offsets, perm_src, W13, W2, W13_scale, W2_scale, Ws13, Ws2, Ws13_scale,
                Ws2_scale, W_down, y_perm, ws, stream=None):
    _check(load_library().moe_experts(ctypes.byref(cfg), _dev(x), _dev(offsets), _dev(perm_src),
                                      _dev(W13), _dev(W2), _dev(W13_scale), _dev(W2_scale),
                                      _dev(Ws13), _dev(Ws2), _dev(Ws13_scale), _dev(Ws2_scale),
                                      _dev(W_down), _dev(y_perm), _dev(ws), ws.numel(),
                                      _stream(stream)), "moe_experts")


def moe_combine(cfg, y_perm, perm_dst, topk_weight, W_up, out, ws, stream=None):
    _check(load_library().moe_combine(ctypes.byref(cfg), _dev(y_perm), _dev(perm_dst),
                                      _dev(topk_weight), _dev(W_up), _dev(out), _dev(ws),
                                      ws.numel(), _stream(stream)), "moe_combine")


def moe_forward(cfg, x, W_r, b, W13, W2, W13_scale, W2_scale, Ws13, Ws2, Ws13_scale, Ws2_scale,
                W_down, W_up, out, ws, stream=None):
    _check(load_library().moe_forward(ctypes.byref(cfg), _dev(x), _dev(W_r), _dev(b), _dev(W13),
                                      _dev(W2), _dev(W13_scale), _dev(W2_scale), _dev(Ws13),
                                      _dev(Ws2), _dev(Ws13_scale), _dev(Ws2_scale), _dev(W_down),
                                      _dev(W_up), _dev(out), _dev(ws), ws.numel(),
                                      _stream(stream)), "moe_forward")


def moe_forward_block(cfg, x_resid, norm_w, W_r, b, W13, W2, W13_scale, W2_scale, Ws13, Ws2,
                      Ws13_scale, Ws2_scale, W_down, W_up, out, ws, stream=None):
    """The FFN half of a block: out = x_resid + layer(RMSNorm(x_resid) * norm_w)."""
    _check(load_library().moe_forward_block(
        ctypes.byref(cfg), _dev(x_resid), _dev(norm_w), _dev(W_r), _dev(b), _dev(W13), _dev(W2),
        _dev(W13_scale), _dev(W2_scale), _dev(Ws13), _dev(Ws2), _dev(Ws13_scale), _dev(Ws2_scale),
        _dev(W_down), _dev(W_up), _dev(out), _dev(ws), ws.numel(), _stream(stream)),
        "moe_forward_block")


def moe_forward_host_io(cfg, x_host, W_r, b, W13, W2, W13_scale, W2_scale, Ws13, Ws2,
                        Ws13_scale, Ws2_scale, W_down, W_up, out_host, ws, stream=None):
    """x_host / out_host are CPU tensors (pinned for full copy bandwidth)."""
    if x_host.is_cuda or out_host.is_cuda:
        raise ValueError("moe_forward_host_io takes host tensors for x and out")
    _check(load_library().moe_forward_host_io(
        ctypes.byref(cfg), _p(x_host), _dev(W_r), _dev(b), _dev(W13), _dev(W2), _dev(W13_scale),
        _dev(W2_scale), _dev(Ws13), _dev(Ws2), _dev(Ws13_scale), _dev(Ws2_scale), _dev(W_down),
        _dev(W_up), _p(out_host), _dev(ws), ws.numel(), _stream(stream)), "moe_forward_host_io")


def moe_dense_mlp_workspace_size(T: int, d: int, I: int, act_dtype: torch.dtype) -> int:
    return int(load_library().moe_dense_mlp_workspace_size(int(T), int(d), int(I),
                                                           _dt(act_dtype)))


def moe_dense_mlp(x, W13, W2, out, ws, stream=None):
    """Dense SwiGLU MLP: x [T][d], W13 [2I][d] (W1 rows then W3 rows), W2 [d][I], out [T][d]."""
    T, d = x.shape
    I = W2.shape[1]
    _check(load_library().moe_dense_mlp(int(T), int(d), int(I), _dt(x.dtype), _dev(x), _dev(W13),
                                        _dev(W2), _dev(out), _dev(ws), ws.numel(),
                                        _stream(stream)), "moe_dense_mlp")


def moe_reset_device_status(ws, stream=None):
    _check(load_library().moe_reset_device_status(_dev(ws), ws.numel(), _stream(stream)),
           "moe_reset_device_status")


def moe_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns the translated device status code."""
    return int(load_library().moe_device_status(_dev(ws), ws.numel(), _stream(stream)))


def moe_launch_count() -> int:
    return int(load_library().moe_launch_count())


def moe_reset_launch_count():
    load_library().moe_reset_launch_count()


def moe_profile_enable(on: bool = True):
    _check(load_library().moe_profile_enable(1 if on else 0), "moe_profile_enable")


def moe_profile_read(max_entries: int = 64) -> dict:
    """{kernel name: (total ms, launches)} since the last read (synchronises on the events)."""
    name_len = 48
    names = ctypes.create_string_buffer(max_entries * name_len)
    ms = (ctypes.c_double * max_entries)()
    n_l = (ctypes.c_uint64 * max_entries)()
    n = load_library().moe_profile_read(max_entries, ctypes.cast(names, ctypes.c_void_p),
                                        name_len, ctypes.cast(ms, ctypes.c_void_p),
                                        ctypes.cast(n_l, ctypes.c_void_p))
    out = {}
    for i in range(n):
        nm = names.raw[i * name_len:(i + 1) * name_len].split(b"\0", 1)[0].decode()
        out[nm] = (float(ms[i]), int(n_l[i]))
    return out


# ----------------------------------------------------------------------------------------------
# Convenience: run a synthetic layer (mixture_experts_ffn_gemm_gb300.synthetic.Layer)
# ----------------------------------------------------------------------------------------------
def layer_weights(layer):
    """The weight arguments of moe_forward for a synthetic layer, in ABI order."""
    return (layer.W_r, layer.b, layer.W13, layer.W2, layer.W13_scale, layer.W2_scale, layer.Ws13,
            layer.Ws2, layer.Ws13_scale, layer.Ws2_scale, layer.W_down, layer.W_up)


def forward_layer(layer, out=None, ws=None, flags: int = 0, stream=None, x=None):
    """moe_forward on a synthetic layer; allocates out / ws when not given (outside the call)."""
    cfg = config_for(layer.w, T=(x if x is not None else layer.x).shape[0], flags=flags)
    x = layer.x if x is None else x
    if out is None:
        out = torch.empty(x.shape[0], layer.w.d, dtype=x.dtype, device=x.device)
    if ws is None:
        ws = alloc_workspace(cfg, x.device)
    moe_forward(cfg, x, *layer_weights(layer), out, ws, stream=stream)
    return out, ws, cfg
