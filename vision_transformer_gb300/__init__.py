"""Python binding of the GB300 SigLIP So400m/14 encoder library (``include/sv.h``).

Argument marshalling only: each function has the name of the C entry point it
calls, takes torch tensors (or raw device pointers) and the current torch CUDA
stream, and raises :class:`SvError` when the library returns an error. Every
step of the forward pass runs in the library's CUDA kernels; there is no
fallback path: importing works without a GPU, but the calls need one.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsv.so")
_lib = None

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_NOT_INITIALIZED, SV_ERR_CUDA, SV_ERR_OOM, SV_ERR_TIMEOUT = range(7)
SV_GEMM_F16, SV_GEMM_E4M3 = 0, 1
SV_DT_F16, SV_DT_E4M3 = 0, 1
SV_ACT_NONE, SV_ACT_GELU_TANH = 0, 1
KIND_GEMM, KIND_ATTN, KIND_LN, KIND_MAP_ATTN, KIND_OTHER = range(5)
KIND_NAMES = ("gemm_tc", "attention", "layernorm", "map_attention", "other")
STATUS_NAMES = ("SV_OK", "SV_ERR_INVALID_ARG", "SV_ERR_UNSUPPORTED", "SV_ERR_NOT_INITIALIZED", "SV_ERR_CUDA",
                "SV_ERR_OOM", "SV_ERR_TIMEOUT")

# (name, restype, argtypes) of every exported function, in header order.
_VP, _I, _U64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
_IP, _DP, _LLP = ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)
SIGNATURES = [
    ("sv_init_weights", _I, [_U64]),
    ("sv_init_weights_dims", _I, [_U64, _I, _I, _I, _I, _I, _I]),
    ("sv_model_dims", _I, [_IP, _IP, _IP, _IP, _IP, _IP]),
    ("sv_weights_count", _SZ, []),
    ("sv_export_weights", _I, [_VP, _SZ]),
    ("sv_weights_count_e4m3", _SZ, []),
    ("sv_export_weights_e4m3", _I, [_VP, _SZ]),
    ("sv_encode", _I, [_VP, _VP, _I, _I, _I, _VP]),
    ("sv_encode_ex", _I, [_VP, _VP, _I, _I, _I, _I, _VP]),
    ("sv_gemm_bias_act", _I, [_VP, _VP, _VP, _VP, _I, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _F, _VP]),
    ("sv_layernorm", _I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _F, _I, _VP]),
    ("sv_ln_gemm", _I, [_VP, _VP, _VP, _F, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    ("sv_pack_patches", _I, [_VP, _VP, _I, _I, _I, _I, _VP]),
    ("sv_attention", _I, [_VP, _VP, _I, _I, _I, _I, _F, _I, _VP]),
    ("sv_attention_ex", _I, [_VP, _VP, _I, _I, _I, _I, _F, _I, _I, _VP]),
    ("sv_attention_heads", _I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _I, _I, _VP]),
    ("sv_map_pool", _I, [_VP, _VP, _I, _I, _VP]),
    ("sv_map_pool_static", _I, [_VP, _VP, _I, _I, _VP]),
    ("sv_quantize_e4m3", _I, [_VP, _VP, _SZ, _VP]),
    ("sv_make_pixels", _I, [_U64, _I, _VP, _VP]),
    ("sv_sync", _I, [_VP]),
    ("sv_last_error", ctypes.c_char_p, []),
    ("sv_launch_count", ctypes.c_longlong, []),
    ("sv_profile_enable", _I, [_I]),
    ("sv_profile_read", _I, [_I, _DP, _DP, _DP, _LLP]),
    ("sv_debug_fill_workspace", _I, [_I, _I, _I]),
    ("sv_debug_wait_timeout", _I, [ctypes.c_uint, _VP]),
    ("sv_debug_gemm_plan", _I, [_I, _I, _I, _I, _I, _I, _IP, ctypes.POINTER(ctypes.c_size_t)]),
    ("sv_debug_attention_kernel", _I, [_I]),
    ("sv_debug_attention_plan", _I, [_I, _I, _I, _I, _IP, _IP]),
    ("sv_debug_encode_stage", _I, [_VP, _I, _I, _I, _I, _I, _VP, _SZ, _VP]),
    ("sv_shutdown", None, []),
]


class SvError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{fn}: {name}: {msg}")
        self.status = status


def load(path: str | None = None):
    """Loads libsv.so (building it first if it is absent). Raises if it cannot."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        from . import build as _b
        _b.build()
    L = ctypes.CDLL(p)
    for name, res, args in SIGNATURES:
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(fn: str, status: int):
    if status != SV_OK:
        raise SvError(status, fn, (_lib.sv_last_error() or b"").decode(errors="replace"))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _hptr(x):
    """Host buffer address: an int, or an object with a numpy-style ctypes.data."""
    if isinstance(x, int):
        return x
    return x.ctypes.data


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def sv_init_weights(seed: int = 0):
    _check("sv_init_weights", load().sv_init_weights(seed))


def sv_init_weights_dims(seed: int, tokens: int, patch_dim: int, width: int, heads: int, mlp: int, layers: int):
    _check("sv_init_weights_dims", load().sv_init_weights_dims(seed, tokens, patch_dim, width, heads, mlp, layers))


def sv_model_dims() -> dict:
    vals = [ctypes.c_int() for _ in range(6)]
    _check("sv_model_dims", load().sv_model_dims(*[ctypes.byref(v) for v in vals]))
    return dict(zip(("tokens", "patch_dim", "width", "heads", "mlp", "layers"), (v.value for v in vals)))


SV_ENCODE_UNFUSED_QKV = 1
SV_ENCODE_FP8_ATTENTION = 2
SV_ENCODE_EAGER = 4
SV_ATTENTION_QK_E4M3 = 1
(SV_STAGE_PATCH, SV_STAGE_QKV, SV_STAGE_ATTENTION, SV_STAGE_OUT_PROJ, SV_STAGE_MLP_UP, SV_STAGE_MLP_DOWN,
 SV_STAGE_FINAL_LN) = range(7)


def sv_encode_ex(pixels, out, batch: int, layers: int, gemm_dtype: int = SV_GEMM_F16, flags: int = 0, stream=None):
    _check("sv_encode_ex", load().sv_encode_ex(_ptr(pixels), _ptr(out), batch, layers, gemm_dtype, flags,
                                               _stream(stream)))


def sv_encode(pixels, out, batch: int, layers: int, gemm_dtype: int = SV_GEMM_F16, stream=None):
    _check("sv_encode", load().sv_encode(_ptr(pixels), _ptr(out), batch, layers, gemm_dtype, _stream(stream)))


def sv_gemm_bias_act(A, W, bias, pos, pos_rows: int, residual, C, M: int, N: int, K: int, act: int = 0,
                     in_dtype: int = 0, out_dtype: int = 0, scale_a: float = 1.0, scale_w: float = 1.0, stream=None):
    _check("sv_gemm_bias_act", load().sv_gemm_bias_act(_ptr(A), _ptr(W), _ptr(bias), _ptr(pos), pos_rows,
                                                       _ptr(residual), _ptr(C), M, N, K, act, in_dtype, out_dtype,
                                                       scale_a, scale_w, _stream(stream)))


def sv_pack_patches(images, pixels, batch: int, image_side: int = 378, channels: int = 3, patch: int = 14,
                    stream=None):
    _check("sv_pack_patches", load().sv_pack_patches(_ptr(images), _ptr(pixels), batch, image_side, channels, patch,
                                                     _stream(stream)))


def sv_ln_gemm(x, gamma, beta, W, bias, C, M: int, N: int, K: int, act: int = 0, eps: float = 1e-6, stream=None):
    _check("sv_ln_gemm", load().sv_ln_gemm(_ptr(x), _ptr(gamma), _ptr(beta), eps, _ptr(W), _ptr(bias), _ptr(C), M, N,
                                           K, act, _stream(stream)))


def sv_layernorm(x, residual, gamma, beta, y, rows: int, width: int, eps: float = 1e-6, out_dtype: int = 0,
                 stream=None):
    _check("sv_layernorm", load().sv_layernorm(_ptr(x), _ptr(residual), _ptr(gamma), _ptr(beta), _ptr(y), rows,
                                               width, eps, out_dtype, _stream(stream)))


def sv_attention(qkv, o, batch: int, heads: int, tokens: int, head_dim: int = 72, scale: float = 0.0,
                 out_dtype: int = 0, stream=None):
    """scale <= 0 lets the library use 1/sqrt(head_dim)."""
    _check("sv_attention", load().sv_attention(_ptr(qkv), _ptr(o), batch, heads, tokens, head_dim, scale, out_dtype,
                                               _stream(stream)))


def sv_attention_ex(qkv, o, batch: int, heads: int, tokens: int, head_dim: int = 72, scale: float = 0.0,
                    out_dtype: int = 0, flags: int = 0, stream=None):
    _check("sv_attention_ex", load().sv_attention_ex(_ptr(qkv), _ptr(o), batch, heads, tokens, head_dim, scale,
                                                     out_dtype, flags, _stream(stream)))


def sv_attention_heads(q, k, v, o, batch: int, heads: int, tokens: int, head_dim: int = 72, head_stride: int = 80,
                       scale: float = 0.0, out_dtype: int = 0, flags: int = 0, stream=None):
    _check("sv_attention_heads", load().sv_attention_heads(_ptr(q), _ptr(k), _ptr(v), _ptr(o), batch, heads, tokens,
                                                           head_dim, head_stride, scale, out_dtype, flags,
                                                           _stream(stream)))


def sv_weights_count() -> int:
    return int(load().sv_weights_count())


def sv_export_weights(host_dst, n_floats: int):
    """host_dst: a writable float32 buffer (e.g. a numpy array's ctypes data pointer) of n_floats values."""
    _check("sv_export_weights", load().sv_export_weights(_hptr(host_dst), n_floats))


def sv_weights_count_e4m3() -> int:
    return int(load().sv_weights_count_e4m3())


def sv_export_weights_e4m3(host_dst, n_bytes: int):
    _check("sv_export_weights_e4m3", load().sv_export_weights_e4m3(_hptr(host_dst), n_bytes))


def sv_map_pool(x, out, batch: int, gemm_dtype: int = SV_GEMM_F16, stream=None):
    _check("sv_map_pool", load().sv_map_pool(_ptr(x), _ptr(out), batch, gemm_dtype, _stream(stream)))


def sv_map_pool_static(x, out, batch: int, gemm_dtype: int = SV_GEMM_F16, stream=None):
    _check("sv_map_pool_static", load().sv_map_pool_static(_ptr(x), _ptr(out), batch, gemm_dtype, _stream(stream)))


def sv_quantize_e4m3(x, y, n: int, stream=None):
    _check("sv_quantize_e4m3", load().sv_quantize_e4m3(_ptr(x), _ptr(y), n, _stream(stream)))


def sv_make_pixels(seed: int, batch: int, dst, stream=None):
    _check("sv_make_pixels", load().sv_make_pixels(seed, batch, _ptr(dst), _stream(stream)))


def sv_sync(stream=None):
    _check("sv_sync", load().sv_sync(_stream(stream)))


def sv_last_error() -> str:
    return (load().sv_last_error() or b"").decode(errors="replace")


def sv_launch_count() -> int:
    return int(load().sv_launch_count())


def sv_profile_enable(on: bool = True):
    _check("sv_profile_enable", load().sv_profile_enable(1 if on else 0))


def sv_profile_read(kind: int) -> dict:
    ms, fl, by, n = ctypes.c_double(), ctypes.c_double(), ctypes.c_double(), ctypes.c_longlong()
    _check("sv_profile_read", load().sv_profile_read(kind, ctypes.byref(ms), ctypes.byref(fl), ctypes.byref(by),
                                                     ctypes.byref(n)))
    return {"ms": ms.value, "flops": fl.value, "bytes": by.value, "launches": n.value}


def sv_debug_fill_workspace(batch: int, gemm_dtype: int, byte_value: int):
    _check("sv_debug_fill_workspace", load().sv_debug_fill_workspace(batch, gemm_dtype, byte_value))


def sv_debug_gemm_plan(M: int, N: int, K: int, gemm_dtype: int = 0, sms: int = 152, max_splits: int = 8) -> dict:
    out = (ctypes.c_int * 8)()
    ws = ctypes.c_size_t(0)
    _check("sv_debug_gemm_plan", load().sv_debug_gemm_plan(M, N, K, gemm_dtype, sms, max_splits, out,
                                                           ctypes.byref(ws)))
    keys = ("bn", "pairs", "atoms", "tail_n", "tail_last", "k_splits", "kb_split", "n_main")
    return dict(zip(keys, list(out)), ws_bytes=ws.value)


def sv_debug_attention_kernel(choice: int) -> None:
    _check("sv_debug_attention_kernel", load().sv_debug_attention_kernel(choice))


def sv_debug_attention_plan(batch: int, tokens: int, heads: int, sms: int = 152) -> dict:
    kernel, grid = ctypes.c_int(0), ctypes.c_int(0)
    _check("sv_debug_attention_plan", load().sv_debug_attention_plan(batch, tokens, heads, sms, ctypes.byref(kernel),
                                                                     ctypes.byref(grid)))
    return {"kernel": kernel.value, "grid": grid.value}


def sv_debug_wait_timeout(limit_us: int, stream=None):
    _check("sv_debug_wait_timeout", load().sv_debug_wait_timeout(limit_us, _stream(stream)))


def sv_debug_encode_stage(pixels, batch: int, layers: int, gemm_dtype: int, flags: int, stage: int, dst,
                          dst_bytes: int, stream=None):
    _check("sv_debug_encode_stage", load().sv_debug_encode_stage(_ptr(pixels), batch, layers, gemm_dtype, flags, stage,
                                                                 _ptr(dst), dst_bytes, _stream(stream)))


def sv_shutdown():
    if _lib is not None:
        _lib.sv_shutdown()
