"""Split-K GEMMs (small M, long K) against the oracle, through the C ABI.

At small M a long-K GEMM's output tiles fill few SMs; the library then splits K
into ranges run by separate CTAs (pairs), writes their F32 partial sums to a
workspace and adds them in a fixed order in a reduction kernel that also runs
the epilogue (bias, positions, tanh-GELU, residual, F16 / E4M3 output, row
statistics for the next LayerNorm). A split GEMM is two library launches, which
sv_launch_count shows. Tolerances as in test_gpu_ops.py: one F16 rounding of an
F32 sum (2^-10 |ref| + 2^-10 rms(ref)); E4M3 outputs one E4M3 step.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_close, decode_e4m3, dev_f16, host

pytestmark = pytest.mark.gpu

RT = 2.0 ** -10
T, D, H, F = 729, 1152, 16, 4304


def _scale(ref):
    return float(np.sqrt(np.mean(np.asarray(ref, dtype=np.float64) ** 2))) + 1e-12


def _inputs(seed, M, N, K):
    A = synth.normal(seed, 1, (M, K))
    W = synth.normal(seed, 2, (K, N), std=1.0 / np.sqrt(K))
    b = synth.normal(seed, 3, (N,), std=0.01)
    return A, W, b


def _launches(sv, fn):
    sv.sv_launch_count()  # reads and resets the count
    fn()
    sv.sv_sync()
    return sv.sv_launch_count()


@pytest.mark.parametrize("M,N,K", [
    (729, 1152, 4304),   # the MLP-down projection of one image
    (300, 1040, 2560),   # ragged M, a 16-column last tile
    (1, 1152, 4304),     # the MAP head's second MLP projection, one image
    (1458, 1152, 4304),  # two images
])
def test_splitk_bias_residual(sv, M, N, K):
    A, W, b = _inputs(70 + M % 11, M, N, K)
    R = synth.normal(71, 4, (M, N))
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    n = _launches(sv, lambda: sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), None, 1, dev_f16(R), C, M,
                                                  N, K))
    assert n == 2, "the GEMM should split K (partial sums + reduction)"
    ref = oracle.linear(A, W, b, residual=R)
    assert_close(host(C), ref, RT, RT * _scale(ref), f"split-K {M}x{N}x{K} + residual")


def test_splitk_gelu_and_positions(sv):
    M, N, K = 300, 1040, 2560
    A, W, b = _inputs(72, M, N, K)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    assert _launches(sv, lambda: sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), None, 1, None, C, M, N, K,
                                                     act=1)) == 2
    ref = oracle.linear(A, W, b, act=1)
    assert_close(host(C), ref, RT, RT * _scale(ref), "split-K + GELU")
    # positional rows by m % 97
    pos = synth.normal(72, 5, (97, N), std=0.1)
    assert _launches(sv, lambda: sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), dev_f16(pos), 97, None, C,
                                                     M, N, K)) == 2
    ref = oracle.linear(A, W, b) + pos.astype(np.float32)[np.arange(M) % 97]
    assert_close(host(C), ref, RT, RT * _scale(ref), "split-K + positions")


def test_splitk_e4m3_operands_and_output(sv):
    """E4M3 operands at scale 2^-4 (the oracle's operand-rounding mode) and an E4M3
    GELU output at 100 rows (E4M3 GEMMs split only at small M: their main loop is
    short against the reduction)."""
    M, N, K = 100, 1152, 4304
    A, W, b = _inputs(73, M, N, K)
    A8 = torch.empty(M * K, dtype=torch.uint8, device="cuda")
    W8 = torch.empty(N * K, dtype=torch.uint8, device="cuda")
    sv.sv_quantize_e4m3(dev_f16(A), A8, M * K)
    sv.sv_quantize_e4m3(dev_f16(W.T), W8, N * K)
    C = torch.empty(M * N, dtype=torch.uint8, device="cuda")
    assert _launches(sv, lambda: sv.sv_gemm_bias_act(A8, W8, dev_f16(b), None, 1, None, C, M, N, K, act=1,
                                                     in_dtype=1, out_dtype=1, scale_a=1 / 16, scale_w=1 / 16)) == 2
    got = decode_e4m3(C).reshape(M, N)  # code values times 2^-4
    ref = oracle.linear(A, W, b, act=1, fp8=True)
    assert_close(got, ref, 2.0 ** -3 + RT, RT * _scale(ref), "split-K E4M3")


def test_splitk_repeats_bit_identical(sv):
    """The reduction adds the splits in a fixed order: repeated calls agree bit for bit."""
    M, N, K = 729, 1152, 4304
    A, W, b = _inputs(74, M, N, K)
    args = (dev_f16(A), dev_f16(W.T), dev_f16(b))
    outs = []
    for _ in range(4):
        C = torch.empty(M, N, dtype=torch.float16, device="cuda")
        sv.sv_gemm_bias_act(*args, None, 1, None, C, M, N, K)
        sv.sv_sync()
        outs.append(C.clone())
    assert all(torch.equal(outs[0], o) for o in outs[1:])


@pytest.fixture(scope="module")
def two_layers(sv):
    sv.sv_init_weights_dims(0, T, 588, D, H, F, 2)
    d = synth.so400m(2)
    params = synth.model(0, d)
    pix = synth.pixels(5, 1)
    return params, torch.from_numpy(pix).cuda()


def _stage(sv, pix_dev, layers, stage, cols):
    dst = torch.full((T, cols), float("nan"), dtype=torch.float16, device="cuda")
    sv.sv_debug_encode_stage(pix_dev, 1, layers, 0, 0, stage, dst, dst.numel() * 2)
    sv.sv_sync()
    return host(dst)


def test_encoder_batch1_split_mlp_down_and_statistics(sv, two_layers):
    """One image, F16: the MLP-down projection splits K. Its reduction's output
    (X after layer 1) and its row statistics (consumed by layer 2's LayerNorm,
    folded into the QKV projection) against the oracle on the GPU's own inputs;
    and layer 1's LN1 + QKV and LN2 + MLP up, whose statistics come from the patch
    embedding's and the output projection's epilogues at this size."""
    p, pix_dev = two_layers
    f16 = lambda a: np.asarray(a, dtype=np.float64).astype(np.float16)
    x0 = _stage(sv, pix_dev, 1, sv.SV_STAGE_PATCH, D)
    qkv1 = _stage(sv, pix_dev, 1, sv.SV_STAGE_QKV, 3 * D)
    ref = oracle.linear(oracle.layernorm(f16(x0), p["ln1_g"][0], p["ln1_b"][0]), p["qkv_w"][0], p["qkv_b"][0])
    assert_close(qkv1, ref, RT, 2 * RT * _scale(ref), "layer 1 LN1 (statistics from the patch GEMM) + QKV")
    hh = _stage(sv, pix_dev, 1, sv.SV_STAGE_MLP_UP, F)
    x1_in = _stage(sv, pix_dev, 1, sv.SV_STAGE_OUT_PROJ, D)
    ref = oracle.linear(oracle.layernorm(f16(x1_in), p["ln2_g"][0], p["ln2_b"][0]), p["fc1_w"][0], p["fc1_b"][0],
                        act=1)
    assert_close(hh, ref, RT, 2 * RT * _scale(ref), "layer 1 LN2 (statistics from the output projection) + MLP up")
    x1 = _stage(sv, pix_dev, 1, sv.SV_STAGE_MLP_DOWN, D)
    ref = oracle.linear(f16(hh), p["fc2_w"][0], p["fc2_b"][0], residual=f16(x1_in))
    assert_close(x1, ref, RT, RT * _scale(ref), "layer 1 MLP down (split K) + residual")
    qkv2 = _stage(sv, pix_dev, 2, sv.SV_STAGE_QKV, 3 * D)
    ref = oracle.linear(oracle.layernorm(f16(x1), p["ln1_g"][1], p["ln1_b"][1]), p["qkv_w"][1], p["qkv_b"][1])
    assert_close(qkv2, ref, RT, 2 * RT * _scale(ref), "layer 2 LN1 (statistics from the split reduction) + QKV")


def test_tail_split_gemm(sv):
    """The MLP-down shape at 32 images (23,328 x 1152 x 4304): 460 pair tiles on 76
    CTA pairs leave 4 for a seventh round, whose K is split over the idle pairs (two
    launches). Rows of whole tiles (the first 64) and of the split last tiles (the last
    64, whose columns 256.. are split) against the oracle on those rows."""
    M, N, K = 23328, 1152, 4304
    A, W, b = _inputs(76, M, N, K)
    R = synth.normal(76, 4, (M, N))
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    assert _launches(sv, lambda: sv.sv_gemm_bias_act(dev_f16(A), dev_f16(W.T), dev_f16(b), None, 1, dev_f16(R), C, M,
                                                     N, K)) == 2
    got = host(C)
    for rows in (slice(0, 64), slice(M - 64, M)):
        ref = oracle.linear(A[rows], W, b, residual=R[rows])
        assert_close(got[rows], ref, RT, RT * _scale(ref), f"tail split rows {rows}")


def test_encoder_batch32_tail_split_statistics(sv, two_layers):
    """32 images, F16: the MLP-down projection splits its last round's tiles; layer 2's
    folded LayerNorm reads row statistics from both the whole tiles' epilogues and the
    reduction. Layer 2's LN1 + QKV against the oracle on the GPU's X after layer 1, on
    rows of both kinds."""
    p, _ = two_layers
    B = 32
    pix = torch.from_numpy(synth.pixels(6, B)).cuda()
    f16 = lambda a: np.asarray(a, dtype=np.float64).astype(np.float16)

    def stage(layers, st, cols):
        dst = torch.full((B * T, cols), float("nan"), dtype=torch.float16, device="cuda")
        sv.sv_debug_encode_stage(pix, B, layers, 0, 0, st, dst, dst.numel() * 2)
        sv.sv_sync()
        return host(dst)

    x1 = stage(1, sv.SV_STAGE_MLP_DOWN, D)
    qkv2 = stage(2, sv.SV_STAGE_QKV, 3 * D)
    for rows in (slice(0, 64), slice(B * T - 64, B * T)):
        ref = oracle.linear(oracle.layernorm(f16(x1[rows]), p["ln1_g"][1], p["ln1_b"][1]), p["qkv_w"][1],
                            p["qkv_b"][1])
        assert_close(qkv2[rows], ref, RT, 2 * RT * _scale(ref), f"layer 2 LN1 + QKV rows {rows}")
