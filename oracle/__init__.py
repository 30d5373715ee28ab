"""ORACLE — test infrastructure only (see the header of ``oracle/oracle.cpp``).

Python access to the plain FP32 (double-accumulating) C++ reference of the
SigLIP So400m/14 image encoder. Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may import this package. It never touches
the CUDA library: callers pass parameters and pixels drawn by ``synth``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_FP = ctypes.POINTER(ctypes.c_float)
_FPP = ctypes.POINTER(_FP)

_PER_LAYER = ("ln1_g", "ln1_b", "qkv_w", "qkv_b", "out_w", "out_b", "ln2_g", "ln2_b", "fc1_w", "fc1_b", "fc2_w",
              "fc2_b")
_GLOBAL_HEAD = ("patch_w", "patch_b", "pos")
_GLOBAL_TAIL = ("enc_ln_g", "enc_ln_b", "probe", "map_q_w", "map_q_b", "map_kv_w", "map_kv_b", "map_out_w",
                "map_out_b", "map_ln_g", "map_ln_b", "map_fc1_w", "map_fc1_b", "map_fc2_w", "map_fc2_b")


class Model(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int) for n in ("tokens", "patch_dim", "width", "heads", "head_dim", "mlp", "layers")]
                + [(n, _FP) for n in _GLOBAL_HEAD] + [(n, _FPP) for n in _PER_LAYER]
                + [(n, _FP) for n in _GLOBAL_TAIL])


def build(force: bool = False) -> str:
    """Compile liboracle.so with g++ (portable flags; no -march=native)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_SRC) > os.path.getmtime(_LIB):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O3", "-std=c++17", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_threads.restype = ctypes.c_int
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_e4m3.argtypes = [ctypes.c_float]
        L.oracle_e4m3.restype = ctypes.c_float
        L.oracle_gelu.argtypes = [_FP, _FP, ctypes.c_long]
        L.oracle_softmax_rows.argtypes = [_FP, _FP, ctypes.c_long, ctypes.c_long]
        L.oracle_linear.argtypes = [_FP, _FP, _FP, _FP, _FP, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                    ctypes.c_int, ctypes.c_int]
        L.oracle_layernorm.argtypes = [_FP, _FP, _FP, _FP, ctypes.c_long, ctypes.c_long, ctypes.c_float]
        L.oracle_attention.argtypes = [_FP, _FP, _FP, _FP, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                       ctypes.c_long, ctypes.c_float]
        L.oracle_patch_embed.argtypes = [_FP, _FP, _FP, _FP, _FP, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                         ctypes.c_long, ctypes.c_int]
        L.oracle_pack_patches.argtypes = [_FP, _FP, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long]
        L.oracle_attention_qk8.argtypes = [_FP, _FP, _FP, _FP, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                           ctypes.c_long, ctypes.c_float]
        L.oracle_map_pool.argtypes = [ctypes.POINTER(Model), _FP, _FP, ctypes.c_long, ctypes.c_int]
        L.oracle_encode.argtypes = [ctypes.POINTER(Model), _FP, _FP, ctypes.c_long, ctypes.c_int, ctypes.c_int, _FP]
        for f in ("oracle_gelu", "oracle_softmax_rows", "oracle_linear", "oracle_layernorm", "oracle_attention",
                  "oracle_patch_embed", "oracle_pack_patches", "oracle_attention_qk8", "oracle_map_pool", "oracle_encode",
                  "oracle_set_threads"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _p(a):
    return None if a is None else a.ctypes.data_as(_FP)


def threads() -> int:
    return lib().oracle_threads()


def e4m3(x: float) -> float:
    return lib().oracle_e4m3(float(x))


def gelu(x) -> np.ndarray:
    x = _f32(x)
    y = np.empty_like(x)
    lib().oracle_gelu(_p(x), _p(y), x.size)
    return y


def softmax_rows(x) -> np.ndarray:
    x = _f32(x)
    y = np.empty_like(x)
    lib().oracle_softmax_rows(_p(x), _p(y), x.shape[0], x.shape[1])
    return y


def linear(A, W, bias=None, residual=None, act: int = 0, fp8: bool = False) -> np.ndarray:
    """act(A @ W + bias) + residual, with W logical [K, N]."""
    A, W = _f32(A), _f32(W)
    M, K = A.shape
    N = W.shape[1]
    bias = None if bias is None else _f32(bias)
    residual = None if residual is None else _f32(residual)
    C = np.empty((M, N), dtype=np.float32)
    lib().oracle_linear(_p(A), _p(W), _p(bias), _p(residual), _p(C), M, N, K, act, int(fp8))
    return C


def layernorm(x, g, b, eps: float = 1e-6) -> np.ndarray:
    x = _f32(x)
    y = np.empty_like(x)
    lib().oracle_layernorm(_p(x), _p(_f32(g)), _p(_f32(b)), _p(y), x.shape[0], x.shape[1], eps)
    return y


def attention(q, k, v, heads: int, head_dim: int, scale: float | None = None, qk_fp8: bool = False) -> np.ndarray:
    """q, k, v: [B, T, heads*head_dim] token-major; returns o in the same layout.
    qk_fp8: Q and K rounded to E4M3 values (scale 2^-4) before the scores."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, T, _ = q.shape
    o = np.empty_like(q)
    s = 1.0 / np.sqrt(head_dim) if scale is None else scale
    f = lib().oracle_attention_qk8 if qk_fp8 else lib().oracle_attention
    f(_p(q), _p(k), _p(v), _p(o), B, heads, T, head_dim, s)
    return o


def pack_patches(img, patch: int = 14) -> np.ndarray:
    """[B, side, side, C] images -> [B, (side/patch)^2, patch*patch*C] patch rows."""
    img = _f32(img)
    B, S, S2, C = img.shape
    assert S == S2 and S % patch == 0
    G = S // patch
    pix = np.empty((B, G * G, patch * patch * C), dtype=np.float32)
    lib().oracle_pack_patches(_p(img), _p(pix), B, S, C, patch)
    return pix


def patch_embed(pix, Wp, bp, pos, fp8: bool = False) -> np.ndarray:
    pix = _f32(pix)
    B, T, P = pix.shape
    D = Wp.shape[1]
    X = np.empty((B, T, D), dtype=np.float32)
    lib().oracle_patch_embed(_p(pix), _p(_f32(Wp)), _p(_f32(bp)), _p(_f32(pos)), _p(X), B, T, P, D, int(fp8))
    return X


class OracleModel:
    """Float32 copies of a ``synth.model`` parameter dict plus the ctypes view the C side reads."""

    def __init__(self, params: dict, tokens: int, patch_dim: int, width: int, heads: int, mlp: int):
        self.arrays = {}
        keep = []
        m = Model()
        m.tokens, m.patch_dim, m.width, m.heads, m.mlp = tokens, patch_dim, width, heads, mlp
        m.head_dim = width // heads
        for n in _GLOBAL_HEAD + _GLOBAL_TAIL:
            a = _f32(params[n])
            self.arrays[n] = a
            setattr(m, n, _p(a))
        layers = len(params["qkv_w"])
        m.layers = layers
        for n in _PER_LAYER:
            arrs = [_f32(x) for x in params[n]]
            self.arrays[n] = arrs
            ptrs = (_FP * layers)(*[_p(a) for a in arrs])
            keep.append(ptrs)
            setattr(m, n, ctypes.cast(ptrs, _FPP))
        self._keep = keep
        self.struct = m
        self.layers = layers
        self.tokens, self.width = tokens, width

    @classmethod
    def from_synth(cls, seed: int, dims) -> "OracleModel":
        import synth
        return cls(synth.model(seed, dims), dims.tokens, dims.patch_dim, dims.width, dims.heads, dims.mlp)

    def encode(self, pix, layers: int | None = None, fp8: bool = False, want_xf: bool = False,
               fp8_attention: bool = False):
        """fp8: dense-GEMM operands rounded to E4M3; fp8_attention: Q and K rounded to E4M3
        before the attention scores."""
        pix = _f32(pix)
        B = pix.shape[0]
        L = self.layers if layers is None else layers
        out = np.empty((B, self.width), dtype=np.float32)
        xf = np.empty((B, self.tokens, self.width), dtype=np.float32) if want_xf else None
        mode = (1 if fp8 else 0) | (2 if fp8_attention else 0)
        lib().oracle_encode(ctypes.byref(self.struct), _p(pix), _p(out), B, L, mode, _p(xf))
        return (out, xf) if want_xf else out

    def map_pool(self, xf, fp8: bool = False) -> np.ndarray:
        xf = _f32(xf)
        B = xf.shape[0]
        out = np.empty((B, self.width), dtype=np.float32)
        lib().oracle_map_pool(ctypes.byref(self.struct), _p(xf), _p(out), B, int(fp8))
        return out
