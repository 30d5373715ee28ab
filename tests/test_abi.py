"""The C-ABI library: it loads without a GPU, exports every function include/sv.h
declares, the Python binding covers exactly those, and argument errors are
reported before any device work."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sv.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from vision_transformer_gb300 import build
    build.build()
    import vision_transformer_gb300 as vt
    return vt.load()


def test_header_declares_the_entry_points():
    names = _declared()
    for required in ("sv_init_weights", "sv_encode", "sv_gemm_bias_act", "sv_layernorm", "sv_attention",
                     "sv_map_pool", "sv_sync", "sv_last_error", "sv_shutdown"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from vision_transformer_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (sv_[a-z0-9_]+)$", out, flags=re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        assert hasattr(lib, n)


def test_binding_covers_exactly_the_header():
    import vision_transformer_gb300 as vt
    assert sorted(n for n, _, _ in vt.SIGNATURES) == _declared()
    for n, _, _ in vt.SIGNATURES:
        assert callable(getattr(vt, n))


def test_binding_constants_match_the_header():
    """Every enumerator include/sv.h defines has the same value in the binding."""
    import vision_transformer_gb300 as vt
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    values = dict((n, int(v)) for n, v in re.findall(r"\b(SV_[A-Z0-9_]+)\s*=\s*(\d+)", text))
    assert len(values) >= 17
    for name, value in values.items():
        assert getattr(vt, name) == value, name


def test_errors_before_device_work(lib):
    """Bad arguments are rejected on the host, so these calls need no GPU."""
    import vision_transformer_gb300 as vt
    buf = (ctypes.c_uint8 * 4096)()
    p16 = (ctypes.addressof(buf) + 15) // 16 * 16
    # N not a multiple of 16
    assert lib.sv_gemm_bias_act(p16, p16, None, None, 1, None, p16, 16, 15, 16, 0, 0, 0, 1.0, 1.0, None) == \
        vt.SV_ERR_INVALID_ARG
    # misaligned operand
    assert lib.sv_gemm_bias_act(p16 + 2, p16, None, None, 1, None, p16, 16, 16, 16, 0, 0, 0, 1.0, 1.0, None) == \
        vt.SV_ERR_INVALID_ARG
    # bad activation / dtype codes
    assert lib.sv_gemm_bias_act(p16, p16, None, None, 1, None, p16, 16, 16, 16, 7, 0, 0, 1.0, 1.0, None) == \
        vt.SV_ERR_INVALID_ARG
    assert lib.sv_gemm_bias_act(p16, p16, None, None, 1, None, p16, 16, 16, 16, 0, 3, 0, 1.0, 1.0, None) == \
        vt.SV_ERR_INVALID_ARG
    # image packing: side not a multiple of the patch
    assert lib.sv_pack_patches(p16, p16, 1, 30, 3, 14, None) == vt.SV_ERR_INVALID_ARG
    # LayerNorm folded into a GEMM: K beyond the LayerNorm's 4096, or N not a multiple of 16
    assert lib.sv_ln_gemm(p16, p16, p16, 1e-6, p16, None, p16, 16, 16, 8192, 0, None) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_ln_gemm(p16, p16, p16, 1e-6, p16, None, p16, 16, 24, 16, 0, None) == vt.SV_ERR_INVALID_ARG
    # LayerNorm width must be a multiple of 8 (even, unpadded rows: LayerNorm paragraph)
    assert lib.sv_layernorm(p16, None, p16, p16, p16, 4, 12, 1e-6, 0, None) == vt.SV_ERR_INVALID_ARG
    # ... and its residual operand 16-byte aligned
    assert lib.sv_layernorm(p16, p16 + 2, p16, p16, p16, 4, 16, 1e-6, 0, None) == vt.SV_ERR_INVALID_ARG
    # head width other than 72 is not implemented
    assert lib.sv_attention(p16, p16, 1, 2, 4, 64, 0.125, 0, None) == vt.SV_ERR_UNSUPPORTED
    assert lib.sv_attention(p16, p16, 0, 2, 4, 72, 0.125, 0, None) == vt.SV_ERR_INVALID_ARG
    # per-head operands: the row stride must cover the head and keep 16-byte rows
    assert lib.sv_attention_heads(p16, p16, p16, p16, 1, 2, 4, 72, 64, 0.0, 0, 0, None) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_attention_heads(p16, p16, p16, p16, 1, 2, 4, 72, 76, 0.0, 0, 0, None) == vt.SV_ERR_INVALID_ARG
    assert lib.sv_attention_heads(p16, p16, p16, p16, 1, 2, 4, 64, 80, 0.0, 0, 0, None) == vt.SV_ERR_UNSUPPORTED
    # unknown attention option bits
    assert lib.sv_attention_ex(p16, p16, 1, 2, 4, 72, 0.125, 0, 2, None) == vt.SV_ERR_INVALID_ARG
    # quantiser length
    assert lib.sv_quantize_e4m3(p16, p16, 15, None) == vt.SV_ERR_INVALID_ARG
    # wait-probe limits
    assert lib.sv_debug_wait_timeout(0, None) == vt.SV_ERR_INVALID_ARG
    # shapes the encoder does not implement
    assert lib.sv_init_weights_dims(0, 4, 588, 128, 2, 288, 1) == vt.SV_ERR_UNSUPPORTED
    assert lib.sv_init_weights_dims(0, 0, 588, 144, 2, 288, 1) == vt.SV_ERR_INVALID_ARG
    # nothing initialised yet
    assert lib.sv_encode(p16, p16, 1, 1, 0, None) == vt.SV_ERR_NOT_INITIALIZED
    assert lib.sv_map_pool(p16, p16, 1, 0, None) == vt.SV_ERR_NOT_INITIALIZED
    assert lib.sv_weights_count() == 0 and lib.sv_weights_count_e4m3() == 0
    assert lib.sv_export_weights(p16, 16) == vt.SV_ERR_NOT_INITIALIZED
    assert lib.sv_export_weights_e4m3(p16, 16) == vt.SV_ERR_NOT_INITIALIZED
    assert lib.sv_debug_encode_stage(p16, 1, 1, 0, 0, 0, p16, 16, None) == vt.SV_ERR_NOT_INITIALIZED
    assert b"sv_init_weights" in lib.sv_last_error()
