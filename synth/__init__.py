"""Seeded synthetic parameters and pixels (the recipe is in ``synth/synth.h``).

This is the only module shared by the CUDA library and the CPU oracle. It
draws inputs and holds none of the encoder's arithmetic. Values come back as
``numpy.float16`` arrays (the bits the C generator produced).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cpp")
_HDR = os.path.join(_HERE, "synth.h")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("tokens", "patch_dim", "width", "heads", "mlp", "layers")]


class TensorInfo(ctypes.Structure):
    _fields_ = [
        ("name", ctypes.c_char * 32),
        ("layer", ctypes.c_int),
        ("rows", ctypes.c_int),
        ("cols", ctypes.c_int),
        ("kind", ctypes.c_int),
        ("mean", ctypes.c_double),
        ("std", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile libsynth.so with g++ (portable flags: it runs on x86-64 and aarch64)."""
    stale = not os.path.exists(_LIB) or any(os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.POINTER
        L.synth_so400m.restype = Dims
        L.synth_so400m.argtypes = [ctypes.c_int]
        L.synth_tensor_count.argtypes = [P(Dims)]
        L.synth_tensor_info.argtypes = [P(Dims), ctypes.c_int, P(TensorInfo)]
        L.synth_fill_tensor_f16.argtypes = [ctypes.c_uint64, P(Dims), ctypes.c_int, ctypes.c_void_p]
        L.synth_fill_tensor_f16_t.argtypes = [ctypes.c_uint64, P(Dims), ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
        L.synth_pixels_f16.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        L.synth_pixels_f16.restype = None
        for fn in (L.synth_normal_f16, L.synth_uniform_f16):
            fn.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double, ctypes.c_double, ctypes.c_void_p,
                           ctypes.c_size_t]
            fn.restype = None
        L.synth_draw_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        L.synth_draw_u64.restype = ctypes.c_uint64
        L.synth_draw_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        L.synth_draw_normal.restype = ctypes.c_double
        L.synth_f16_from_double.argtypes = [ctypes.c_double]
        L.synth_f16_from_double.restype = ctypes.c_uint16
        _lib = L
    return _lib


def so400m(layers: int = 27) -> Dims:
    return lib().synth_so400m(layers)


def dims(tokens=729, patch_dim=588, width=1152, heads=16, mlp=4304, layers=27) -> Dims:
    return Dims(tokens, patch_dim, width, heads, mlp, layers)


def vit_small(layers: int = 1) -> Dims:
    """The pages' reduced graph: 28x28 image (4 tokens), width 144, 2 heads of 72, MLP 288."""
    return Dims(4, 588, 144, 2, 288, layers)


def four_token(layers: int = 1) -> Dims:
    """Four tokens at the full 1152/4304 widths and 16 heads (the pages' diagnostic shape)."""
    return Dims(4, 588, 1152, 16, 4304, layers)


def tensor_infos(d: Dims) -> list[TensorInfo]:
    L = lib()
    out = []
    for i in range(L.synth_tensor_count(ctypes.byref(d))):
        t = TensorInfo()
        if L.synth_tensor_info(ctypes.byref(d), i, ctypes.byref(t)) != 0:
            raise RuntimeError(f"synth_tensor_info({i}) failed")
        out.append(t)
    return out


def tensor(seed: int, d: Dims, tid: int) -> np.ndarray:
    """Tensor ``tid`` as float16, logical shape [rows, cols] ([K, N] for weights)."""
    t = tensor_infos(d)[tid]
    out = np.empty((t.rows, t.cols), dtype=np.float16)
    if lib().synth_fill_tensor_f16(seed, ctypes.byref(d), tid, out.ctypes.data) != 0:
        raise RuntimeError("synth_fill_tensor_f16 failed")
    return out


def model(seed: int, d: Dims) -> dict:
    """All parameters as {name: float16 array}; per-layer ones as lists indexed by layer."""
    out: dict = {}
    for tid, t in enumerate(tensor_infos(d)):
        name = t.name.decode()
        arr = tensor(seed, d, tid)
        if t.rows == 1 and name != "probe":
            arr = arr.reshape(-1)
        if t.layer >= 0:
            out.setdefault(name, []).append(arr)
        else:
            out[name] = arr
    return out


def pixels(seed: int, batch: int, tokens: int = 729, patch_dim: int = 588) -> np.ndarray:
    out = np.empty((batch, tokens, patch_dim), dtype=np.float16)
    lib().synth_pixels_f16(seed, batch, tokens, patch_dim, out.ctypes.data)
    return out


def normal(seed: int, tag: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float16)
    lib().synth_normal_f16(seed, tag, mean, std, out.ctypes.data, out.size)
    return out


def uniform(seed: int, tag: int, shape, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float16)
    lib().synth_uniform_f16(seed, tag, lo, hi, out.ctypes.data, out.size)
    return out
