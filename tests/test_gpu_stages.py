"""Per-stage parity of the encoder as sv_encode runs it, single So400m/14 layer at
batch 8 (the per-op checks of the single-layer batch-8 configuration: patch GEMM,
LayerNorm + QKV, attention, output projection, LayerNorm + MLP, final LayerNorm,
MAP).

sv_debug_encode_stage stops the forward pass after a stage and returns that
stage's output tensor (the encoder's own workspace, in the launch sequence and
layouts sv_encode uses: the head-blocked QKV epilogue, the LayerNorms folded
into the QKV / MLP-up GEMMs with statistics from the X-writing epilogues). Each
stage is compared element by element with the oracle applied to the GPU's own
input of that stage (the previous stage's output), so every comparison has the
per-op tolerance of its kind:
  - GEMM results: 2^-10 |ref| + 2^-10 rms(ref) (one F16 rounding of an F32 sum);
  - a LayerNorm folded into the next GEMM: twice that scale term (gamma W is
    rounded to F16 where the unfolded order rounds LN(x));
  - attention: 2^-10 |ref| + 2^-10 max|v| (P is rounded to F16 before P V);
  - LayerNorm: 2^-10 |ref| + 2^-10;
  - MAP: 4 x the GEMM terms (five chained GEMMs and an attention);
  - E4M3 outputs: one E4M3 step (2^-3 relative) plus the F16 terms.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, decode_e4m3, host

pytestmark = pytest.mark.gpu

RT = 2.0 ** -10
B, T, D, H, F = 8, 729, 1152, 16, 4304


def _scale(ref):
    return float(np.sqrt(np.mean(np.asarray(ref, dtype=np.float64) ** 2))) + 1e-12


@pytest.fixture(scope="module")
def setup(sv):
    sv.sv_init_weights_dims(0, T, 588, D, H, F, 1)
    d = synth.so400m(1)
    params = synth.model(0, d)
    model = oracle.OracleModel(params, d.tokens, d.patch_dim, d.width, d.heads, d.mlp)
    pix = synth.pixels(3, B)
    return params, model, pix, torch.from_numpy(pix).cuda()


def _stage(sv, pix_dev, stage, cols, gemm_dtype=0, e4m3_out=False):
    dt = torch.uint8 if e4m3_out else torch.float16
    dst = torch.full((B * T, cols), 0xFF if e4m3_out else float("nan"), dtype=dt, device="cuda")
    sv.sv_debug_encode_stage(pix_dev, B, 1, gemm_dtype, 0, stage, dst, dst.numel() * dst.element_size())
    sv.sv_sync()
    if e4m3_out:
        return decode_e4m3(dst).reshape(B * T, cols)
    return host(dst)


def _f16(a):
    return np.asarray(a, dtype=np.float64).astype(np.float16)


def test_stages_f16_batch8(sv, setup):
    p, model, pix, pix_dev = setup
    # patch embedding (+ bias + positions) from the pixels
    x0 = _stage(sv, pix_dev, sv.SV_STAGE_PATCH, D)
    ref = oracle.patch_embed(pix, p["patch_w"], p["patch_b"], p["pos"]).reshape(B * T, D)
    assert_close(x0, ref, RT, RT * _scale(ref), "patch embedding")
    # LN1 folded into the fused QKV projection, from the GPU's X
    qkv = _stage(sv, pix_dev, sv.SV_STAGE_QKV, 3 * D)
    ref = oracle.linear(oracle.layernorm(_f16(x0), p["ln1_g"][0], p["ln1_b"][0]), p["qkv_w"][0], p["qkv_b"][0])
    assert_close(qkv, ref, RT, 2 * RT * _scale(ref), "LN1 + QKV")
    # attention over the GPU's Q, K, V
    o = _stage(sv, pix_dev, sv.SV_STAGE_ATTENTION, D)
    q3 = _f16(qkv).reshape(B, T, 3 * D)
    ref = oracle.attention(q3[..., :D], q3[..., D:2 * D], q3[..., 2 * D:], H, 72).reshape(B * T, D)
    vmax = float(np.abs(q3[..., 2 * D:].astype(np.float64)).max())
    assert_close(o, ref, RT, RT * vmax, "attention")
    # output projection + residual
    x1 = _stage(sv, pix_dev, sv.SV_STAGE_OUT_PROJ, D)
    ref = oracle.linear(_f16(o), p["out_w"][0], p["out_b"][0], residual=_f16(x0))
    assert_close(x1, ref, RT, RT * _scale(ref), "output projection + residual")
    # LN2 folded into MLP up + GELU
    hh = _stage(sv, pix_dev, sv.SV_STAGE_MLP_UP, F)
    ref = oracle.linear(oracle.layernorm(_f16(x1), p["ln2_g"][0], p["ln2_b"][0]), p["fc1_w"][0], p["fc1_b"][0],
                        act=1)
    assert_close(hh, ref, RT, 2 * RT * _scale(ref), "LN2 + MLP up + GELU")
    # MLP down + residual: X after the layer
    x2 = _stage(sv, pix_dev, sv.SV_STAGE_MLP_DOWN, D)
    ref = oracle.linear(_f16(hh), p["fc2_w"][0], p["fc2_b"][0], residual=_f16(x1))
    assert_close(x2, ref, RT, RT * _scale(ref), "MLP down + residual")
    # final LayerNorm
    y = _stage(sv, pix_dev, sv.SV_STAGE_FINAL_LN, D)
    ref = oracle.layernorm(_f16(x2), p["enc_ln_g"], p["enc_ln_b"])
    assert_close(y, ref, RT, RT, "final LayerNorm")
    # MAP pooling of the GPU's final-LN output (the whole forward pass's output)
    out = torch.empty(B, 1, D, dtype=torch.float16, device="cuda")
    sv.sv_encode_ex(pix_dev, out, B, 1, 0, sv.SV_ENCODE_EAGER)
    sv.sv_sync()
    got = host(out).reshape(B, D)
    ref = model.map_pool(_f16(y).reshape(B, T, D))
    assert np.abs(got - ref).max() <= 2e-2
    assert_close(got, ref, 4 * RT, 4 * RT * _scale(ref), "MAP")
    # the staged run changed nothing: the chained oracle agrees with the output at the one-layer bounds
    full = model.encode(pix, 1)
    cos = (got * full).sum(1) / np.linalg.norm(got, axis=1) / np.linalg.norm(full, axis=1)
    assert np.abs(got - full).max() <= 2e-2 and cos.min() >= 0.9999


def test_stages_e4m3_batch8(sv, setup):
    """E4M3 GEMM operands: the stages whose inputs both sides round identically
    (the pixels and weights to E4M3 at scale 2^-4; the attention output and the final
    LayerNorm quantised from F32 results) against the oracle's operand-rounding mode."""
    p, model, pix, pix_dev = setup
    x0 = _stage(sv, pix_dev, sv.SV_STAGE_PATCH, D, gemm_dtype=1)
    ref = oracle.patch_embed(pix, p["patch_w"], p["patch_b"], p["pos"], fp8=True).reshape(B * T, D)
    assert_close(x0, ref, RT, RT * _scale(ref), "patch embedding (E4M3 operands)")
    qkv = _stage(sv, pix_dev, sv.SV_STAGE_QKV, 3 * D, gemm_dtype=1)
    o = _stage(sv, pix_dev, sv.SV_STAGE_ATTENTION, D, gemm_dtype=1, e4m3_out=True)
    q3 = _f16(qkv).reshape(B, T, 3 * D)
    ref = oracle.attention(q3[..., :D], q3[..., D:2 * D], q3[..., 2 * D:], H, 72).reshape(B * T, D)
    vmax = float(np.abs(q3[..., 2 * D:].astype(np.float64)).max())
    assert_close(o, ref, 2.0 ** -3 + RT, RT * vmax, "attention (E4M3 output)")
    x2 = _stage(sv, pix_dev, sv.SV_STAGE_MLP_DOWN, D, gemm_dtype=1)
    y = _stage(sv, pix_dev, sv.SV_STAGE_FINAL_LN, D, gemm_dtype=1, e4m3_out=True)
    ref = oracle.layernorm(_f16(x2), p["enc_ln_g"], p["enc_ln_b"])
    assert_close(y, ref, 2.0 ** -3 + RT, 2.0 ** -10, "final LayerNorm (E4M3 output)")
