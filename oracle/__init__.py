"""fp64 CPU oracle of the mixture-of-experts FFN layer (Kimi K2 / DeepSeek-V3, Kimi K3 latent).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / reference leg may import this package.  It shares no code with the CUDA library
and imports nothing from it; both sides only receive the same seeded input arrays.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64); this module compiles it with gcc and
marshals numpy arrays through ctypes.  Sources, by page title and section:

* "Kimi K2 · Transformer blocks > MoE transformer block", "Mixture of experts" steps (router,
  selection, gates, SwiGLU experts, routed sum, shared expert, D_ffn);
* nnterp encyclopedia "kimi_k2", note "The mixture of experts" (bias only selects; gates are the
  renormalised unbiased sigmoids times 2.827 and sum to 2.827) and its "Config" table;
* "Kimi K3 · Latent up-projection", its equation and parameter table and the ``forward`` /
  ``moe_infer`` code excerpts (latent down-projection, optional RMSNorm, up-projection, shared
  expert on the full-width input).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmoe_oracle.so")

F32, BF16, E4M3, F64, INT4 = 0, 1, 2, 3, 4
_DTYPES = {"f32": F32, "bf16": BF16, "e4m3": E4M3, "f64": F64, "int4": INT4}
_NP = {F32: np.float32, BF16: np.uint16, E4M3: np.uint8, F64: np.float64, INT4: np.uint8}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmoe_oracle.so`` (gcc, -O2, no fast-math,
    no FMA contraction so fp32 decisions round exactly as written)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest_src:
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class _Cfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("I_shared", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("d_latent", ctypes.c_int32),
                ("latent_norm", ctypes.c_int32), ("fp8", ctypes.c_int32),
                ("quant_block", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("gate_scale", ctypes.c_double), ("rms_eps", ctypes.c_double)]


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("scale", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.orc_forward.restype = ctypes.c_int
            lib.orc_forward.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int, _Tensor, P, P,
                                        ctypes.POINTER(_Tensor), ctypes.POINTER(_Tensor),
                                        _Tensor, _Tensor, _Tensor, _Tensor,
                                        P, P, P, P, P, P, P]
            lib.orc_route.restype = ctypes.c_int
            lib.orc_route.argtypes = [ctypes.POINTER(_Cfg), _Tensor, P, P, P, P, P, P]
            lib.orc_route_from_logits.restype = ctypes.c_int
            lib.orc_route_from_logits.argtypes = [ctypes.POINTER(_Cfg), P, P, P, P, P, P]
            lib.orc_param_count.restype = ctypes.c_int64
            lib.orc_param_count.argtypes = [ctypes.POINTER(_Cfg)]
            lib.orc_param_breakdown.restype = None
            lib.orc_param_breakdown.argtypes = [ctypes.POINTER(_Cfg), P]
            lib.orc_e4m3_decode.restype = ctypes.c_double
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_quantize_group_e4m3.restype = None
            lib.orc_quantize_group_e4m3.argtypes = [P, ctypes.c_int64, ctypes.c_int, P, P]
            lib.orc_swiglu_row.restype = ctypes.c_int
            lib.orc_swiglu_row.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _Tensor,
                                           _Tensor, ctypes.c_int, ctypes.c_int, P]
            lib.orc_rmsnorm_unit.restype = None
            lib.orc_rmsnorm_unit.argtypes = [P, ctypes.c_int, ctypes.c_double, P]
            lib.orc_dequant_row.restype = ctypes.c_int
            lib.orc_dequant_row.argtypes = [_Tensor, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                            P]
            lib.orc_dense_mlp.restype = ctypes.c_int
            lib.orc_dense_mlp.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          _Tensor, _Tensor, _Tensor, P]
            _lib = lib
    return _lib


@dataclass
class Config:
    """Layer shapes and constants (names follow the nnterp "Config" table)."""
    T: int
    d: int
    E: int
    k: int
    I: int
    I_shared: int = 0
    n_shared: int = 1
    d_latent: int = 0
    latent_norm: int = 0
    fp8: int = 0
    quant_block: int = 128
    gate_scale: float = 2.827
    rms_eps: float = 1e-6

    def _c(self) -> _Cfg:
        return _Cfg(self.T, self.d, self.E, self.k, self.I, self.I_shared or self.I,
                    self.n_shared, self.d_latent, self.latent_norm, self.fp8,
                    self.quant_block, 0, self.gate_scale, self.rms_eps)


@dataclass
class Mat:
    """A row-major matrix: ``data`` holds f32 / f64 values, bf16 bit patterns (uint16), e4m3
    codes (uint8, with ``scale`` one fp32 per quant_block x quant_block block) or int4 packed
    bytes (uint8 [rows][cols/2], with ``scale`` [cols/32][rows], the format of moe_oracle.h)."""
    data: np.ndarray
    dtype: str
    scale: Optional[np.ndarray] = None

    def __post_init__(self):
        code = _DTYPES[self.dtype]
        self.data = np.ascontiguousarray(self.data, dtype=_NP[code])
        if self.scale is not None:
            self.scale = np.ascontiguousarray(self.scale, dtype=np.float32)
        if code in (E4M3, INT4) and self.scale is None:
            raise ValueError("an e4m3 or int4 matrix needs its scales")

    def _c(self) -> _Tensor:
        rows = self.data.shape[0] if _DTYPES[self.dtype] == INT4 else 0
        return _Tensor(self.data.ctypes.data, _DTYPES[self.dtype], rows,
                       self.scale.ctypes.data if self.scale is not None else None)


_NULL = _Tensor(None, 0, 0, None)


def _ptr(a):
    return None if a is None else a.ctypes.data


def forward(cfg: Config, x: Mat, W_r: np.ndarray, b: np.ndarray,
            W13: Sequence[Optional[Mat]], W2: Sequence[Optional[Mat]],
            Ws13: Optional[Mat] = None, Ws2: Optional[Mat] = None,
            W_down: Optional[Mat] = None, W_up: Optional[Mat] = None,
            nthreads: int = 1) -> dict:
    """The layer in fp64 with the oracle's own routing.  ``W13`` / ``W2`` are per-expert lists;
    ``None`` marks an expert not supplied.  Returns out, routed, shared, idx, gates, margin,
    logits."""
    lib = _load()
    T, d, E, k = cfg.T, cfg.d, cfg.E, cfg.k
    W_r = np.ascontiguousarray(W_r, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    assert W_r.shape == (E, d) and b.shape == (E,) and len(W13) == E and len(W2) == E
    t13 = (_Tensor * E)(*[m._c() if m is not None else _NULL for m in W13])
    t2 = (_Tensor * E)(*[m._c() if m is not None else _NULL for m in W2])
    res = {
        "out": np.zeros((T, d), np.float64), "routed": np.zeros((T, d), np.float64),
        "shared": np.zeros((T, d), np.float64), "idx": np.zeros((T, k), np.int32),
        "gates": np.zeros((T, k), np.float64), "margin": np.zeros((T,), np.float64),
        "logits": np.zeros((T, E), np.float64),
    }
    c = cfg._c()
    st = lib.orc_forward(ctypes.byref(c), int(nthreads), x._c(), _ptr(W_r), _ptr(b), t13, t2,
                         Ws13._c() if Ws13 is not None else _NULL,
                         Ws2._c() if Ws2 is not None else _NULL,
                         W_down._c() if W_down is not None else _NULL,
                         W_up._c() if W_up is not None else _NULL,
                         _ptr(res["out"]), _ptr(res["idx"]), _ptr(res["gates"]),
                         _ptr(res["margin"]), _ptr(res["logits"]), _ptr(res["routed"]),
                         _ptr(res["shared"]))
    if st != 0:
        raise RuntimeError(f"orc_forward failed with status {st}")
    return res


def route(cfg: Config, x: Mat, W_r: np.ndarray, b: np.ndarray) -> dict:
    """The fp64 routing alone (logits, selection, gates, margin); reads no expert weight."""
    lib = _load()
    W_r = np.ascontiguousarray(W_r, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    T = x.data.shape[0]
    c = Config(**{**cfg.__dict__, "T": T})._c()
    res = {"idx": np.zeros((T, cfg.k), np.int32), "gates": np.zeros((T, cfg.k), np.float64),
           "margin": np.zeros((T,), np.float64), "logits": np.zeros((T, cfg.E), np.float64)}
    st = lib.orc_route(ctypes.byref(c), x._c(), _ptr(W_r), _ptr(b), _ptr(res["idx"]),
                       _ptr(res["gates"]), _ptr(res["margin"]), _ptr(res["logits"]))
    if st != 0:
        raise RuntimeError(f"orc_route failed with status {st}")
    return res


def route_from_logits(cfg: Config, z: np.ndarray, b: np.ndarray, with_keys: bool = False):
    """Selection and gates from given fp32 logits [T, E]; the key is fp32(fp32(sigmoid(z)) + b).
    Returns (idx [T,k] int32, gates [T,k] f64, margin [T] f64), and with ``with_keys`` also the
    selected experts' fp32 keys [T,k] in slot order."""
    lib = _load()
    z = np.ascontiguousarray(z, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    T = z.shape[0]
    c = Config(**{**cfg.__dict__, "T": T})._c()
    idx = np.zeros((T, cfg.k), np.int32)
    gates = np.zeros((T, cfg.k), np.float64)
    margin = np.zeros((T,), np.float64)
    keys = np.zeros((T, cfg.k), np.float32)
    st = lib.orc_route_from_logits(ctypes.byref(c), _ptr(z), _ptr(b), _ptr(idx), _ptr(gates),
                                   _ptr(margin), _ptr(keys))
    if st != 0:
        raise RuntimeError(f"orc_route_from_logits failed with status {st}")
    return (idx, gates, margin, keys) if with_keys else (idx, gates, margin)


def param_count(cfg: Config) -> int:
    c = cfg._c()
    return int(_load().orc_param_count(ctypes.byref(c)))


def param_breakdown(cfg: Config) -> dict:
    """Parameter count by component, from the shapes the forward indexes."""
    c = cfg._c()
    out = np.zeros((6,), np.int64)
    _load().orc_param_breakdown(ctypes.byref(c), _ptr(out))
    keys = ("router", "bias", "routed", "shared", "down", "up")
    return {kk: int(v) for kk, v in zip(keys, out)}


def e4m3_decode(code: int) -> float:
    return float(_load().orc_e4m3_decode(int(code)))


def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(v)))


def quantize_group_e4m3(v: np.ndarray, qb: int = 128):
    """Per-group e4m3 quantisation of a fp32 vector; returns (codes uint8, scales fp32)."""
    v = np.ascontiguousarray(v, dtype=np.float32).reshape(-1)
    q = np.zeros(v.shape, np.uint8)
    s = np.zeros(((v.size + qb - 1) // qb,), np.float32)
    _load().orc_quantize_group_e4m3(_ptr(v), v.size, qb, _ptr(q), _ptr(s))
    return q, s


def swiglu_row(x: np.ndarray, W13: Mat, W2: Mat, I: int, qb: int = 128,
               quant_act: bool = False) -> np.ndarray:
    """One dense SwiGLU MLP row: h = SiLU(x W1) * (x W3), y = h W2 (weights [out, in])."""
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(-1)
    dout = W2.data.shape[0]
    y = np.zeros((dout,), np.float64)
    st = _load().orc_swiglu_row(_ptr(x), x.size, int(I), int(dout), W13._c(), W2._c(), int(qb),
                                int(bool(quant_act)), _ptr(y))
    if st != 0:
        raise RuntimeError(f"orc_swiglu_row failed with status {st}")
    return y


def dequant_row(W: Mat, r: int, cols: int, qb: int = 128) -> np.ndarray:
    """Row r of W widened to fp64 as the oracle's GEMMs see it."""
    out = np.zeros((cols,), np.float64)
    st = _load().orc_dequant_row(W._c(), int(cols), int(qb), int(r), _ptr(out))
    if st != 0:
        raise RuntimeError(f"orc_dequant_row failed with status {st}")
    return out


def dense_mlp(x: Mat, W13: Mat, W2: Mat, nthreads: int = 1) -> np.ndarray:
    """The dense block MLP, y = (SiLU(x W1) * (x W3)) W2 per token, fp64 [T][d] (weights
    [out, in]; W13 holds the W1 rows, then the W3 rows)."""
    T, d = x.data.shape
    I = W2.data.shape[1]
    out = np.zeros((T, d), np.float64)
    st = _load().orc_dense_mlp(int(T), int(d), int(I), int(nthreads), x._c(), W13._c(), W2._c(),
                               _ptr(out))
    if st != 0:
        raise RuntimeError(f"orc_dense_mlp failed with status {st}")
    return out


def rmsnorm_unit(v: np.ndarray, eps: float) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64).reshape(-1)
    y = np.zeros_like(v)
    _load().orc_rmsnorm_unit(_ptr(v), v.size, float(eps), _ptr(y))
    return y
